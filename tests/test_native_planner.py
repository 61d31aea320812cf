"""The native planner (C ABI, host only) against the reference planner and
against invariants of its schedule.

Decisions the pages define must match the reference planner exactly: the edge
assignment (FastTree review page, Algorithm 1 and its cost model), the groups
of the virtual tree with their KV chains, token lists, visible ends and rows
(DeFT notes page, "KV-Guided Tree Split"), each group's path, and, for a
given chunk length, the long-span chunks and every token's partial count.

How the native scheduler then turns groups into work units (query tiles,
packing of thin groups, the automatic chunk length, the CTA schedule) is a
performance choice the pages leave open.  It is checked by invariants on the
device tables the kernels read (``schedule_check``): every query token and q
head sees exactly its path's keys, each once, and each result lands exactly
once."""
import numpy as np
import pytest

import workloads as W
from oracle import planner as P
from schedule_check import check_schedule

ta = pytest.importorskip("tree_structured_decode_gb300")

PAGE_KEYS = ("node", "chain", "span", "tokens", "vis", "rows", "path")


def _native(spec, **opt):
    opt.setdefault("num_sms", 152)
    with ta.Plan.from_spec(spec, host_only=1, **opt) as p:
        return p.describe(), p.stats(), p.schedule()


PROXY = 1  # cost_model: the pages' padding-and-intermediate-result proxy


def _reference(spec, **opt):
    o = P.PlannerOptions()
    for k in ("gamma", "beta", "ts_c", "mma_min_rows", "force_path"):
        if k in opt:
            setattr(o, k, opt[k])
    if opt.get("split_tokens", 0) > 0:
        o.split_tokens = opt["split_tokens"]
    if "ts_q_set" in opt:
        o.ts_q_set = tuple(opt["ts_q_set"])
    if "force_edges" in opt:
        o.edges = tuple(int(x) for x in opt["force_edges"])
    return P.build_plan(spec.parent, spec.node_kv_len, spec.node_page_offsets, spec.node_pages,
                        spec.page_size, spec.query_node, spec.query_kv_end, spec.n_q_heads,
                        spec.n_kv_heads, spec.head_dim, o)


def _check_chunks(got):
    """Chunks partition each group's block list in order (any chunk length)."""
    for g in got["groups"]:
        ch = g["chunks"]
        assert ch[0][0] == 0
        for (a, b), (c, _) in zip(ch, ch[1:]):
            assert a < b == c
        assert ch[-1][1] >= ch[-1][0]
    parts = [0] * len(got["partials"])
    for g in got["groups"]:
        for t in g["tokens"]:
            parts[t] += len(g["chunks"])
    assert parts == got["partials"]


def _same(spec, **opt):
    # the pages' cost model: decisions compared with the reference planner
    opt.setdefault("cost_model", PROXY)
    got, stats, sched = _native(spec, **opt)
    ref = _reference(spec, **opt)
    assert got["edges"] == ref["edges"]
    assert len(got["groups"]) == len(ref["groups"])
    for a, b in zip(got["groups"], ref["groups"]):
        assert {k: a[k] for k in PAGE_KEYS} == {k: b[k] for k in PAGE_KEYS}
    # group blocks: the span in order, page by page (the chunks index them)
    _check_chunks(got)
    if opt.get("split_tokens", 0) != 0:  # a given chunk length (or none)
        for a, b in zip(got["groups"], ref["groups"]):
            assert a["chunks"] == b["chunks"]
        assert got["partials"] == ref["partials"]
    assert stats["n_groups"] == len(ref["groups"])
    assert stats["n_units"] == len(sched["units"]) // 8
    check_schedule(spec, sched, num_sms=opt["num_sms"] if "num_sms" in opt else 152)
    # the default (measured latency) model: another plan, the same invariants
    lat = {k: v for k, v in opt.items() if k != "cost_model"}
    _, _, sched_lat = _native(spec, **lat)
    check_schedule(spec, sched_lat, num_sms=lat.get("num_sms", 152))
    return got, stats, sched


@pytest.mark.parametrize("name", ["tiny", "long", "wide", "three", "irreg"])
def test_configs_match_reference(name):
    spec = W.CONFIGS[name]()
    got, stats, _ = _same(spec)
    assert stats["unique_kv_tokens"] == int(spec.node_kv_len.sum())


@pytest.mark.parametrize("name", ["long", "wide", "three"])
@pytest.mark.parametrize("split", [-1, 64, 400])
def test_configs_with_a_given_chunk_length(name, split):
    _same(W.CONFIGS[name](), split_tokens=split)


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
    if seed % 17 == 6:
        opt["num_sms"] = int(rng.choice([1, 3, 8]))
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
    packed, ps, _ = _same(spec)
    plain, qs, _ = _same(spec, no_pack=1)
    assert ps["n_units"] < qs["n_units"]
    assert packed["groups"] == plain["groups"]


def test_planning_is_fast_on_the_irregular_tree():
    spec = W.config_irregular()
    _, stats, _ = _native(spec)
    assert stats["plan_ms"] < 200.0


@pytest.mark.parametrize("hq,hkv,ntok", [(16, 4, 1), (8, 4, 2), (32, 8, 6), (64, 4, 3), (16, 2, 2),
                                         (64, 8, 1)])
def test_kv_head_packing_schedule(hq, hkv, ntok):
    # long thin leaves: groups of <= 32 rows per kv head pack four kv heads to
    # a unit (hkv a multiple of 4); others stay one unit per kv head
    rng = np.random.default_rng(hq * 31 + ntok)
    lens = [600] + [int(x) for x in rng.integers(140, 900, size=6)]
    qnode = [v for v in range(1, 7) for _ in range(ntok)]
    qend = [lens[v] - (ntok - 1 - j) for v in range(1, 7) for j in range(ntok)]
    spec = W._finish("heads", [-1] + [0] * 6, lens, qnode, qend, hq, hkv, 128, seed=11)
    for opt in ({}, {"split_tokens": 128}, {"no_pack": 1}, {"num_sms": 8}):
        _same(spec, **opt)


@pytest.mark.parametrize("hq,hkv,ntok,pairs", [
    (64, 4, 4, True),    # 64 rows (4 tokens x GQA 16): a pair slot
    (32, 4, 5, True),    # 40 rows
    (16, 2, 5, True),    # 40 rows, one kv-head pair
    (64, 4, 5, False),   # 80 rows: a 128-row tile
    (48, 3, 3, False),   # 48 rows but an odd kv-head count
    (32, 4, 4, False),   # 32 rows: packed four to a unit instead
    (128, 1, 1, False),  # GQA 128 does not divide a 64-row slot
])
def test_query_tiles_of_33_to_64_rows_form_kv_head_pairs(hq, hkv, ntok, pairs):
    # the tile choice near the leaves (FastTree review page, 高效树结构注意力
    # 内核设计): a leaf tile of 33-64 rows runs as one 64-row slot of a pair
    # unit exactly when the kv heads pair up and the GQA ratio divides 64;
    # the schedule stays valid either way
    from schedule_check import check_schedule

    rng = np.random.default_rng(hq + hkv + ntok)
    lens = [500] + [int(x) for x in rng.integers(ntok, 300, size=5)]
    qnode = [v for v in range(1, 6) for _ in range(ntok)]
    qend = [lens[v] - (ntok - 1 - j) for v in range(1, 6) for j in range(ntok)]
    spec = W._finish("tiles", [-1] + [0] * 5, lens, qnode, qend, hq, hkv, 128, seed=3)
    for opt in ({}, {"split_tokens": 128}, {"no_pack": 1}):
        _, _, sched = _native(spec, **opt)
        facts = check_schedule(spec, sched, collect=True)
        kinds = set().union(*facts["kinds"])
        assert ("pairs" in kinds) == (pairs and not opt.get("no_pack")), (opt, sorted(kinds))


@pytest.mark.parametrize("depth,branching,hq,hkv", [(3, 3, 32, 8), (2, 4, 64, 4), (4, 2, 8, 8)])
def test_draft_token_trees_match_reference(depth, branching, hq, hkv):
    spec = W.token_tree(500, 4, 90, depth, branching, hq, hkv, 128, seed=depth)
    for opt in ({}, {"split_tokens": 128}, {"gamma": 2000}):
        _same(spec, **opt)


@pytest.mark.parametrize("num_sms", [1, 2, 5, 152])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (32, 4), (64, 4)])
def test_two_phase_packing_schedule(hq, hkv, num_sms):
    # short leaves with 1-3 query tokens: groups of at most 16 rows per kv
    # head may pack eight to a unit in two phases, else four to a unit
    rng = np.random.default_rng(hq * 7 + num_sms)
    nleaf = 40
    lens = [300] + [int(x) for x in rng.integers(1, 129, size=nleaf)]
    ntok = [int(rng.integers(1, 4)) for _ in range(nleaf)]
    qnode = [v for v in range(1, nleaf + 1) for _ in range(ntok[v - 1])]
    qend = [max(0, lens[v] - j) for v in range(1, nleaf + 1) for j in range(ntok[v - 1])]
    spec = W._finish("phases", [-1] + [0] * nleaf, lens, qnode, qend, hq, hkv, 128, seed=hq)
    _same(spec, num_sms=num_sms)
    _same(spec, num_sms=num_sms, no_pack=1)


def test_schedule_check_catches_a_planted_fault():
    # the checker itself: a schedule with one block's valid count lowered, a
    # row record pointing at another token, or a unit dropped must fail
    spec = W.random_tree(7, n_nodes=15, max_len=120, hq=8, hkv=2, d=128, max_queries_per_node=3)
    _, _, sched = _native(spec)
    check_schedule(spec, sched)
    faults = []
    s1 = dict(sched)
    b = list(s1["blocks"])
    used = sorted({k for u in np.asarray(sched["units"]).reshape(-1, 8) for k in range(u[4], u[5])})
    i = next(2 * k + 1 for k in used if b[2 * k + 1] & 31 > 1)  # a block some unit reads
    b[i] -= 1
    s1["blocks"] = b
    faults.append(s1)
    s2 = dict(sched)
    rows = list(s2["rows"])
    read = sorted({int(u[0]) + (int(u[2]) + i) // sched["gqa"]
                   for u in np.asarray(sched["units"]).reshape(-1, 8) for i in range(min(int(u[3]), 128))})
    j = next(4 * k for k in read if rows[4 * k] >= 0 and rows[4 * k + 3] & 0xFFFFFF == 1)  # a record some unit reads
    rows[j + 1] -= 1  # visible end one short
    s2["rows"] = rows
    faults.append(s2)
    s3 = dict(sched)
    s3["units"] = list(sched["units"])[8:]
    s3["cta_off"] = [max(0, x - 1) for x in sched["cta_off"]]
    faults.append(s3)
    for f in faults:
        with pytest.raises(AssertionError):
            check_schedule(spec, f)


def _edge_of_child(lens, rows_root, rows_child, **opt):
    # root 0 with one child 1; GQA 1, one kv head; rows_root - rows_child
    # query tokens of the root itself, rows_child of the child
    qnode = [0] * (rows_root - rows_child) + [1] * rows_child
    qend = [lens[0]] * (rows_root - rows_child) + [lens[1]] * rows_child
    spec = W._finish("edge", [-1, 0], lens, qnode, qend, 1, 1, 128, seed=1)
    got, _, sched = _native(spec, **opt)
    check_schedule(spec, sched)
    return got["edges"][1]


def test_latency_model_decisions_worked_by_hand():
    # Latency model, in thousandths of one KV tile's time: a 128-row query
    # tile over len tokens costs ceil(len / 64) * 1000 + 8200 (its unit's
    # start-up and epilogue); a thin group (<= 32 rows, <= 128 tokens) a
    # quarter of ceil(len / 16) * 1000 + 8200 (four share a unit); an extra
    # partial 29 per row.
    # Root 2048 tokens with 250 rows, child 64 tokens with 100 of them:
    #   C0 = 2 * (32000 + 8200) + (1000 + 8200) + 29 * 100 = 92500
    #   C1 = 2 * (32000 + 8200) + (33000 + 8200)            = 121600  -> edge 0
    assert _edge_of_child([2048, 64], 250, 100) == 0
    # Root 64 tokens with 140 rows, child 64 tokens with 12 (a thin group):
    #   C0 = 2 * (1000 + 8200) + (4 * 1000 + 8200) / 4 + 29 * 12 = 21798
    #   C1 = 1 * (1000 + 8200) + (8 * 1000 + 8200) / 4            = 13250  -> edge 1
    assert _edge_of_child([64, 64], 140, 12) == 1
    # the pages' proxy on the same trees (d = 128, gamma = 64), by hand:
    #   first:  C0 = (6*2048 + 28*64 + 64*100) d = 20480 d < C1 = (106*2048 + 28*2112) d
    #   second: C0 = (116*64 + 4*64 + 64*12) d = 8448 d >= C1 = (4*128) d = 512 d
    assert _edge_of_child([2048, 64], 250, 100, cost_model=PROXY) == 0
    assert _edge_of_child([64, 64], 140, 12, cost_model=PROXY) == 1
