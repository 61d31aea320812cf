"""The native planner (C ABI, host only) against the reference planner.

Every decision must match exactly: the edge assignment (FastTree review page,
Algorithm 1 and its cost model), the groups of the virtual tree with their KV
chains, token lists and visible ends (DeFT notes page, "KV-Guided Tree
Split"), the path and query tiles of each group, the long-span chunks, the
partial count of every query token and the number of units."""
import numpy as np
import pytest

import workloads as W
from oracle import planner as P

ta = pytest.importorskip("tree_structured_decode_gb300")


def _native(spec, **opt):
    opt.setdefault("num_sms", 152)
    with ta.Plan.from_spec(spec, host_only=1, **opt) as p:
        return p.describe(), p.stats()


def _reference(spec, **opt):
    o = P.PlannerOptions(num_sms=opt.get("num_sms", 152))
    for k in ("gamma", "beta", "ts_c", "mma_min_rows", "split_tokens", "min_split_tokens",
              "split_waves", "force_path", "no_pack"):
        if k in opt:
            setattr(o, k, opt[k])
    if "ts_q_set" in opt:
        o.ts_q_set = tuple(opt["ts_q_set"])
    if "force_edges" in opt:
        o.edges = tuple(int(x) for x in opt["force_edges"])
    ref = P.build_plan(spec.parent, spec.node_kv_len, spec.node_page_offsets, spec.node_pages,
                       spec.page_size, spec.query_node, spec.query_kv_end, spec.n_q_heads,
                       spec.n_kv_heads, spec.head_dim, o)
    ref.pop("_blocks")
    return ref


def _same(spec, **opt):
    got, stats = _native(spec, **opt)
    ref = _reference(spec, **opt)
    assert got["edges"] == ref["edges"]
    assert got["chunk_blocks"] == ref["chunk_blocks"]
    assert len(got["groups"]) == len(ref["groups"])
    for a, b in zip(got["groups"], ref["groups"]):
        assert a == b
    assert got["partials"] == ref["partials"]
    assert got["units"] == ref["units"]
    assert stats["n_units"] == ref["units"]
    assert stats["n_groups"] == len(ref["groups"])
    return got, stats


@pytest.mark.parametrize("name", ["tiny", "long", "wide", "three", "irreg"])
def test_configs_match_reference(name):
    spec = W.CONFIGS[name]()
    got, stats = _same(spec)
    assert stats["unique_kv_tokens"] == int(spec.node_kv_len.sum())


@pytest.mark.parametrize("seed", range(300))
def test_random_trees_match_reference(seed):
    rng = np.random.default_rng(seed)
    hkv = int(rng.choice([1, 2, 4]))
    spec = W.random_tree(seed, n_nodes=int(rng.integers(1, 60)), max_len=int(rng.integers(1, 700)),
                         hq=hkv * int(rng.choice([1, 2, 4, 16])), hkv=hkv,
                         d=int(rng.choice([64, 128])), zero_len_prob=0.1,
                         max_queries_per_node=int(rng.integers(1, 5)))
    opt = {}
    if seed % 3 == 1:
        opt["gamma"] = int(rng.integers(0, 2000))
    if seed % 5 == 2:
        opt["split_tokens"] = int(rng.choice([-1, 16, 100, 300]))
    if seed % 7 == 3:
        opt["mma_min_rows"] = int(rng.integers(1, 200))
    if seed % 11 == 4:
        opt["ts_q_set"] = [8, 32]
        opt["beta"] = 3
    if seed % 13 == 5:
        opt["force_path"] = int(rng.integers(1, 3))
    _same(spec, **opt)


@pytest.mark.parametrize("seed", range(40))
def test_forced_edge_assignments_match_reference(seed):
    spec = W.random_tree(500 + seed, n_nodes=12, max_len=90, hq=4, hkv=2, d=64,
                         max_queries_per_node=3)
    rng = np.random.default_rng(seed)
    edges = rng.integers(0, 2, size=spec.n_nodes).astype(np.int8)
    edges[0] = 0
    _same(spec, force_edges=edges, split_tokens=int(rng.choice([0, 32, 64])))


@pytest.mark.parametrize("name", ["wide"])
def test_packing_can_be_disabled(name):
    spec = W.CONFIGS[name]()
    packed, _ = _same(spec)
    plain, _ = _same(spec, no_pack=1)
    assert packed["units"] < plain["units"]
    assert packed["groups"] == plain["groups"]


def test_planning_is_fast_on_the_irregular_tree():
    spec = W.config_irregular()
    _, stats = _native(spec)
    assert stats["plan_ms"] < 200.0


@pytest.mark.parametrize("hq,hkv,ntok", [(16, 4, 1), (8, 4, 2), (32, 8, 6), (64, 4, 3), (16, 2, 2),
                                         (64, 8, 1)])
def test_kv_head_packing_matches_reference(hq, hkv, ntok):
    # long thin leaves: groups of <= 32 rows per kv head pack four kv heads to
    # a unit with a quarter of the automatic chunk (hkv a multiple of 4);
    # others stay one unit per kv head
    rng = np.random.default_rng(hq * 31 + ntok)
    lens = [600] + [int(x) for x in rng.integers(140, 900, size=6)]
    qnode = [v for v in range(1, 7) for _ in range(ntok)]
    qend = [lens[v] - (ntok - 1 - j) for v in range(1, 7) for j in range(ntok)]
    spec = W._finish("heads", [-1] + [0] * 6, lens, qnode, qend, hq, hkv, 128, seed=11)
    for opt in ({}, {"split_tokens": 128}, {"no_pack": 1}, {"num_sms": 8}):
        _same(spec, **opt)


@pytest.mark.parametrize("depth,branching,hq,hkv", [(3, 3, 32, 8), (2, 4, 64, 4), (4, 2, 8, 8)])
def test_draft_token_trees_match_reference(depth, branching, hq, hkv):
    spec = W.token_tree(500, 4, 90, depth, branching, hq, hkv, 128, seed=depth)
    for opt in ({}, {"split_tokens": 128}, {"gamma": 2000}):
        _same(spec, **opt)


@pytest.mark.parametrize("num_sms", [1, 2, 5, 152])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (32, 4), (64, 4)])
def test_two_phase_packing_matches_reference(hq, hkv, num_sms):
    # short leaves with 1-3 query tokens: groups of at most 16 rows per kv
    # head pack eight to a unit in two phases while the plan keeps three
    # units per CTA (few SMs), else four to a unit like the longer ones
    rng = np.random.default_rng(hq * 7 + num_sms)
    nleaf = 40
    lens = [300] + [int(x) for x in rng.integers(1, 129, size=nleaf)]
    ntok = [int(rng.integers(1, 4)) for _ in range(nleaf)]
    qnode = [v for v in range(1, nleaf + 1) for _ in range(ntok[v - 1])]
    qend = [max(0, lens[v] - j) for v in range(1, nleaf + 1) for j in range(ntok[v - 1])]
    spec = W._finish("phases", [-1] + [0] * nleaf, lens, qnode, qend, hq, hkv, 128, seed=hq)
    _same(spec, num_sms=num_sms)
    _same(spec, num_sms=num_sms, no_pack=1)
