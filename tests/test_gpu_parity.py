"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tree attention as defined on the DeFT notes page ("Tree attention
definition") with scaled dot-product attention (FastTree review page,
"核心公式"); bars: max |err| <= 1e-2, mean |err| <= 1e-3 on the fp32 output,
|err| <= 1e-3 on lse."""
import numpy as np
import pytest
import torch

import workloads as W
from parity_utils import (compare, make_inputs, oracle_on_tokens, run_gpu,
                          sample_tokens)

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------- the five workloads
@pytest.mark.parametrize("name", ["tiny", "long", "wide", "three"])
def test_workload_parity_every_token(name):
    spec = W.CONFIGS[name]()
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, stats = run_gpu(spec, q, k, v)
    toks = list(range(spec.n_queries))
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, toks)
    compare(out, lse, ref, ref_lse, toks)


def _stratified_tokens(spec, per_kind=4, n_random=24, seed=7, **options):
    """Tokens chosen so that every kind of unit the plan holds, masked rows
    and every partial count are reached; returns (tokens, what was covered)."""
    import tree_structured_decode_gb300 as ta
    from schedule_check import check_schedule

    with ta.Plan.from_spec(spec, host_only=1, **options) as p:
        facts = check_schedule(spec, p.schedule(), collect=True)
    rng = np.random.default_rng(seed)
    picks, covered = set(), {}
    kinds = sorted(set().union(*facts["kinds"]))
    for kind in kinds:
        have = [t for t in range(spec.n_queries) if kind in facts["kinds"][t]]
        chosen = rng.choice(have, size=min(per_kind, len(have)), replace=False).tolist()
        picks.update(chosen)
        covered[kind] = chosen
    masked = np.nonzero(facts["masked"])[0]
    if len(masked):
        chosen = rng.choice(masked, size=min(per_kind, len(masked)), replace=False).tolist()
        picks.update(chosen)
        covered["masked"] = chosen
    for c in sorted(set(facts["pcount"].tolist())):
        have = np.nonzero(facts["pcount"] == c)[0]
        chosen = rng.choice(have, size=min(per_kind, len(have)), replace=False).tolist()
        picks.update(chosen)
        covered[f"partials={c}"] = chosen
    picks.update(sample_tokens(spec, n_random, seed=seed))
    return sorted(int(t) for t in picks), covered


def test_workload_parity_irregular_stratified():
    # the irregular tree: too many tokens for the oracle to check all of them,
    # so the sample reaches every kind of unit the plan holds (full 128-row
    # tiles, the 64-row leaf tiles held by kv-head pairs), rows masked inside a
    # tile (the causal tail of the 4 speculative tokens, node ends) and every
    # partial count
    spec = W.config_irregular()
    toks, covered = _stratified_tokens(spec)
    for kind in ("mma_full", "pairs", "masked", "partials=1", "partials=2", "partials=3"):
        assert kind in covered, (kind, sorted(covered))
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, stats = run_gpu(spec, q, k, v)
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, toks)
    compare(out, lse, ref, ref_lse, toks)


@pytest.mark.parametrize("options", [{}, {"split_tokens": 128}, {"num_sms": 4}])
def test_stratified_tokens_reach_every_packing_kind(options):
    # short and long thin leaves with 1-3 speculative tokens under a long root:
    # packed units (one or two phases), kv-head packed units and full tiles
    rng = np.random.default_rng(3)
    nleaf = 40
    lens = [900] + [int(x) for x in rng.integers(1, 129, size=nleaf - 8)] + \
        [int(x) for x in rng.integers(140, 500, size=8)]
    ntok = [int(rng.integers(1, 4)) for _ in range(nleaf)]
    qnode = [v for v in range(1, nleaf + 1) for _ in range(ntok[v - 1])]
    qend = [max(0, lens[v] - j) for v in range(1, nleaf + 1) for j in range(ntok[v - 1])]
    spec = W._finish("kinds", [-1] + [0] * nleaf, lens, qnode, qend, 32, 8, 128, seed=4)
    toks, covered = _stratified_tokens(spec, **options)
    assert "packed" in covered or "packed_phases" in covered
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, _ = run_gpu(spec, q, k, v, **options)
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, toks)
    compare(out, lse, ref, ref_lse, toks)


# ----------------------------------------------------------------- value range
@pytest.mark.parametrize("options", [{"split_tokens": 64}, {"split_tokens": 64, "merge_mode": 1},
                                     {"split_tokens": 64, "force_path": 1}])
def test_values_beyond_fp16_range(options):
    # V scaled by 2^17 (exact in bf16): |V| up to ~6.5e5, past fp16's 65504,
    # on a split plan where every token merges several partials.  Scaling V
    # by c scales the result by c, so out / c must match the oracle on V.
    spec = W.two_level(700, 5, 90, 8, 2, 128, seed=13)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    c = 2.0 ** 17
    vs = (v.float() * c).to(torch.bfloat16)
    assert torch.equal(vs.float()[torch.isfinite(v)], v.float()[torch.isfinite(v)] * c)
    out, lse, stats = run_gpu(spec, q, k, vs, **options)
    assert stats["n_merge_tokens"] == spec.n_queries
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out / c, lse, ref, ref_lse)


# ----------------------------------------------------------------- random trees
@pytest.mark.parametrize("seed", range(16))
def test_random_tree_parity(seed):
    rng = np.random.default_rng(seed)
    hkv = int(rng.choice([1, 2, 4]))
    spec = W.random_tree(seed, n_nodes=int(rng.integers(1, 40)),
                         max_len=int(rng.choice([20, 100, 700])),
                         hq=hkv * int(rng.choice([1, 4, 16])), hkv=hkv,
                         d=int(rng.choice([64, 128])), zero_len_prob=0.1,
                         max_queries_per_node=int(rng.integers(1, 5)))
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    opts = {}
    if seed % 3 == 1:
        opts["split_tokens"] = 128
    if seed % 4 == 2:
        opts["mma_min_rows"] = 4  # groups under 4 rows per kv head on CUDA cores
    out, lse, _ = run_gpu(spec, q, k, v, **opts)
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("seed", range(4))
def test_forced_paths_and_random_edges(path, seed):
    spec = W.random_tree(40 + seed, n_nodes=25, max_len=300, hq=8, hkv=2, d=128,
                         max_queries_per_node=3)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    rng = np.random.default_rng(seed)
    edges = rng.integers(0, 2, size=spec.n_nodes).astype(np.int8)
    out, lse, _ = run_gpu(spec, q, k, v, force_path=path, force_edges=edges,
                          split_tokens=int(rng.choice([0, 128, 256])))
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)


# ----------------------------------------------------------------- edge cases
def test_empty_paths_give_zero_and_neg_inf():
    spec = W._finish("empty", [-1, 0, 0], [0, 0, 5], [1, 2, 2], [0, 0, 3], 4, 2, 64, seed=1)
    q, k, v = make_inputs(spec)
    out, lse, _ = run_gpu(spec, q, k, v)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert (o[:2] == 0).all() and np.isneginf(l[:2]).all()
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, [2])
    compare(out, lse, ref, ref_lse, [2])


def test_no_queries_is_a_no_op():
    spec = W._finish("noq", [-1, 0], [20, 20], [], [], 4, 4, 64, seed=2)
    q, k, v = make_inputs(spec)
    import tree_structured_decode_gb300 as ta
    with ta.Plan.from_spec(spec) as p:
        out, lse = p.run(q, k, v)
        torch.cuda.synchronize()
        assert out.numel() == 0


def test_single_node_many_tokens_ragged():
    # one node, 16 * 37 + 5 tokens: many KV tiles and a ragged last page
    spec = W._finish("one", [-1], [597], [0] * 9, list(range(589, 598)), 8, 2, 128, seed=3)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    for opts in ({}, {"split_tokens": 128}, {"force_path": 1}):
        out, lse, _ = run_gpu(spec, q, k, v, **opts)
        ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(9)))
        compare(out, lse, ref, ref_lse)


def test_repeated_runs_reuse_the_plan():
    spec = W.config_tiny()
    q, k, v = make_inputs(spec)
    import tree_structured_decode_gb300 as ta
    with ta.Plan.from_spec(spec) as p:
        a, la = p.run(q, k, v)
        b, lb = p.run(q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(a, b) and torch.equal(la, lb)


def test_large_scores_do_not_overflow():
    spec = W.two_level(300, 3, 40, 4, 2, 128, seed=5)
    q, k, v = make_inputs(spec)
    q = (q.float() * 8).to(torch.bfloat16)  # scores of order +-100
    out, lse, _ = run_gpu(spec, q, k, v)
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)


# ----------------------------------------------------------------- merge modes
@pytest.mark.parametrize("merge_mode", [0, 1])
def test_fused_and_separate_merge(merge_mode):
    # many partials per row: a long split root and a chain of joined nodes
    spec = W.random_tree(91, n_nodes=20, max_len=500, hq=16, hkv=4, d=128,
                         max_queries_per_node=3)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, stats = run_gpu(spec, q, k, v, split_tokens=64, merge_mode=merge_mode)
    assert stats["n_merge_tokens"] > 0
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)


def test_merge_rows_past_one_grid_stride():
    # more merged (token, q head) rows than the merge grid covers in one
    # stride, with Hq = 24 not dividing the stride: each warp's later rows
    # come from the add-and-carry walk over (token, head)
    spec = W.two_level(2000, 1800, 16, 24, 4, 128, seed=77)
    q, k, v = make_inputs(spec)
    out, lse, stats = run_gpu(spec, q, k, v)
    assert stats["n_merge_tokens"] * spec.n_q_heads > 2 * 8 * 152 * 16
    toks = sample_tokens(spec, 48, seed=3)
    toks = sorted(set(toks) | set(range(spec.n_queries - 24, spec.n_queries)))
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, toks)
    compare(out, lse, ref, ref_lse, toks)


def test_fused_merge_counters_reset_between_runs():
    import tree_structured_decode_gb300 as ta
    spec = W.config_long()
    q, k, v = make_inputs(spec)
    with ta.Plan.from_spec(spec) as p:
        outs = [p.run(q, k, v) for _ in range(3)]
        torch.cuda.synchronize()
        assert p.device_status() == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    toks = [0, 5, 9]
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, toks)
    compare(outs[-1][0], outs[-1][1], ref, ref_lse, toks)


# ----------------------------------------------------------------- packed thin groups
@pytest.mark.parametrize("hq,hkv,path", [(4, 4, 2), (8, 4, 2), (16, 4, 2), (32, 4, 2), (8, 8, 1)])
def test_packed_thin_groups(hq, hkv, path):
    # many short leaves (<= 8 pages) under one root: leaves pack four to a
    # unit; force_path picks CUDA-core packs (<= 2 rows) or tensor-core packs
    spec = W.two_level(300, 23, 0, hq, hkv, 128, seed=hq + path)
    rng = np.random.default_rng(hq)
    lens = [300] + [int(x) for x in rng.integers(1, 129, size=23)]
    spec = W._finish("packs", spec.parent, lens,
                     [v for v in range(1, 24) for _ in range(1 + v % 2)],
                     [lens[v] - j for v in range(1, 24) for j in range(1 + v % 2)],
                     hq, hkv, 128, seed=5)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    for opts in ({"force_path": path}, {"force_path": path, "no_pack": 1}):
        out, lse, _ = run_gpu(spec, q, k, v, **opts)
        ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
        compare(out, lse, ref, ref_lse)


# ----------------------------------------------------------------- 64-row tiles in pairs
@pytest.mark.parametrize("hq,hkv,ntok,d", [(64, 4, 4, 128), (32, 8, 12, 128), (16, 2, 7, 128),
                                           (32, 4, 5, 128), (32, 4, 6, 64)])
@pytest.mark.parametrize("options", [{}, {"split_tokens": 96}, {"no_pack": 1},
                                     {"split_tokens": 96, "merge_mode": 1}])
def test_mid_size_tiles_held_by_kv_head_pairs(hq, hkv, ntok, d, options):
    # leaves whose query tile holds 33-64 rows (ntok tokens x GQA), with page
    # counts odd and even, under a root shared by all of them (whose larger
    # group takes 128-row tiles plus a remainder tile): pair units (two kv
    # heads per unit, two pages per slot per tile, a filler page for odd
    # counts), or plain tiles with no_pack; every token against the oracle
    rng = np.random.default_rng(hq + hkv + ntok)
    nleaf = 6
    lens = [333] + [int(x) for x in rng.integers(ntok, 260, size=nleaf)]
    qnode = [v for v in range(1, nleaf + 1) for _ in range(ntok)]
    qend = [lens[v] - ntok + 1 + j for v in range(1, nleaf + 1) for j in range(ntok)]
    spec = W._finish("pairs", [-1] + [0] * nleaf, lens, qnode, qend, hq, hkv, d, seed=5)
    toks, covered = _stratified_tokens(spec, **options)
    if not options.get("no_pack"):
        assert "pairs" in covered, sorted(covered)
    else:
        assert "pairs" not in covered
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, _ = run_gpu(spec, q, k, v, **options)
    toks = list(range(spec.n_queries))
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, toks)
    compare(out, lse, ref, ref_lse, toks)


# ----------------------------------------------------------------- kv-head packed units
@pytest.mark.parametrize("hq,hkv,ntok", [(16, 4, 1), (8, 4, 2), (32, 8, 6), (64, 8, 2)])
def test_kv_head_packed_units(hq, hkv, ntok):
    # leaves longer than 8 pages with a few (causal, speculative) query tokens
    # each, under a long root: groups of <= 32 rows per kv head run four kv
    # heads to a unit
    rng = np.random.default_rng(hq * 31 + ntok)
    nleaf = 6
    lens = [600] + [int(x) for x in rng.integers(140, 420, size=nleaf)]
    parent = [-1] + [0] * nleaf
    qnode = [v for v in range(1, nleaf + 1) for _ in range(ntok)]
    qend = [lens[v] - (ntok - 1 - j) for v in range(1, nleaf + 1) for j in range(ntok)]
    spec = W._finish("heads", parent, lens, qnode, qend, hq, hkv, 128, seed=11)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    units = {}
    for name, opts in (("auto", {}), ("split", {"split_tokens": 128}), ("unpacked", {"no_pack": 1})):
        out, lse, stats = run_gpu(spec, q, k, v, **opts)
        compare(out, lse, ref, ref_lse)
        units[name] = stats["n_units"]
    assert units["auto"] < units["unpacked"]  # the leaves were packed


# ----------------------------------------------------------------- extremes
def test_largest_gqa_ratio():
    # 128 q heads per kv head: one query token fills a 128-row tile, a few
    # tokens make several query tiles of one group
    spec = W._finish("gqa128", [-1, 0, 0], [300, 90, 33], [1, 1, 2, 2, 2], [90, 89, 33, 32, 31],
                     128, 1, 64, seed=21)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    for opts in ({}, {"split_tokens": 64}):
        out, lse, _ = run_gpu(spec, q, k, v, **opts)
        ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
        compare(out, lse, ref, ref_lse)


def test_tokens_with_more_partials_than_one_merge_round():
    # a 2000-token root split into 64-token chunks: every token folds 32 or
    # more partials (two phases of the wide merge)
    spec = W.two_level(2000, 3, 50, 8, 2, 128, seed=9)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, stats = run_gpu(spec, q, k, v, split_tokens=64)
    assert stats["n_partials"] >= 32 * spec.n_queries
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)


# ----------------------------------------------------------------- draft token trees
@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 4)])
def test_draft_token_tree_verification(hq, hkv):
    # six sequences below one prompt, each with a 3-level draft-token tree
    # (branching 3: 39 draft tokens); every draft token is a one-token node
    # that sees the prompt, its sequence and its draft ancestors
    spec = W.token_tree(700, 6, 130, 3, 3, hq, hkv, 128, seed=hq)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, _ = run_gpu(spec, q, k, v)
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)


# ----------------------------------------------------------------- grid size
def test_grid_larger_than_the_inline_unit_ranges():
    # more CTAs than the launch parameters carry unit ranges for (320): every
    # CTA reads its range from the table in global memory; the grid also
    # exceeds what is resident at once (two CTAs on each of the 152 SMs)
    spec = W.config_wide()
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, stats = run_gpu(spec, q, k, v, num_sms=200)
    assert stats["grid"] > 320
    toks = sample_tokens(spec, 24, seed=3)
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, toks)
    compare(out, lse, ref, ref_lse, toks)


@pytest.mark.parametrize("num_sms", [8, 37, 152])
def test_kv_head_packed_chunks_at_any_page(num_sms):
    # thin groups packed by kv head split into near-equal chunks whose
    # boundaries need not fall on a 4-page tile: the number of SMs the plan
    # assumes moves them (it sets the chunk length)
    rng = np.random.default_rng(num_sms)
    lens = [int(x) for x in rng.integers(150, 900, size=5)]
    parent = [-1, 0, 0, 1, 1]
    qnode = [2, 2, 3, 4, 4]
    qend = [lens[2], lens[2] - 1, lens[3], lens[4], lens[4] - 1]
    spec = W._finish("chunks", parent, lens, qnode, qend, 16, 8, 128, seed=num_sms)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    out, lse, stats = run_gpu(spec, q, k, v, num_sms=num_sms)
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)


@pytest.mark.parametrize("hq,hkv", [(32, 4), (16, 4), (64, 4)])
def test_two_phase_packed_units(hq, hkv):
    # short leaves under one root: those of at most 16 rows per kv head pack
    # eight to a unit in two phases (phase 0 in lanes 0-15 of each warp,
    # phase 1 in lanes 16-31; the tiles carry phase 0's pages, then phase
    # 1's), longer ones four to a unit; page counts differ inside a phase
    rng = np.random.default_rng(hq)
    nleaf = 27
    lens = [200] + [int(x) for x in rng.integers(1, 129, size=nleaf)]
    ntok = [1 + (v % 3 == 0) * int(rng.integers(1, 4)) for v in range(1, nleaf + 1)]
    qnode = [v for v in range(1, nleaf + 1) for _ in range(ntok[v - 1])]
    qend = [max(0, lens[v] - j) for v in range(1, nleaf + 1) for j in range(ntok[v - 1])]
    spec = W._finish("phases", [-1] + [0] * nleaf, lens, qnode, qend, hq, hkv, 128, seed=hq)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    units = {}
    # planned for one SM: two phases need three units per CTA, which a tree
    # this small has only for a grid of two CTAs
    for name, opts in (("phases", {"num_sms": 1}), ("one phase", {}), ("unpacked", {"no_pack": 1})):
        out, lse, stats = run_gpu(spec, q, k, v, **opts)
        compare(out, lse, ref, ref_lse)
        units[name] = stats["n_units"]
    assert units["phases"] < units["one phase"] < units["unpacked"]
