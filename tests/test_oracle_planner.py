"""Pins for the reference grouping planner (CPU only).

Greedy binary edge assignment and cost model: FastTree review page, sections
"二元边赋值", "算法1：贪心二元边赋值" and "开销模型"; KV-guided grouping:
DeFT notes page, "KV-Guided Tree Split".  The pins are the page's two worked
grouping cases (golden fixture), costs computed by hand from the printed
formulas, and a coverage invariant checked over every edge assignment of small
trees (whatever the assignment, each query's path is covered exactly once)."""
import itertools
import json
import os

import pytest

import oracle
from oracle import planner as P
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_pad_values_from_definition():
    # Pad(TS, N) = TS - ((N - 1) % TS + 1): the rows needed to fill the last tile.
    assert P.pad(16, 10) == 6
    assert P.pad(16, 16) == 0
    assert P.pad(16, 17) == 15
    assert P.pad(64, 10) == 54
    assert P.pad(64, 64) == 0
    assert P.pad(128, 1) == 127
    assert P.pad(64, 0) == 0  # reading: an empty group has no padding


def test_tile_choice():
    o = P.PlannerOptions()
    assert [P.ts_q(n, o.ts_q_set) for n in (0, 1, 16, 17, 64, 65, 128, 129, 1000)] == \
        [16, 16, 16, 64, 64, 128, 128, 128, 128]


@pytest.mark.parametrize("case", json.load(open(os.path.join(
    GOLDEN, "fasttree_grouping_cases.json")))["cases"], ids=lambda c: c["name"])
def test_worked_grouping_cases(case):
    spec = W._finish("case", [-1, 0, 0], case["node_len"],
                     [1] * case["queries_per_leaf"] + [2] * case["queries_per_leaf"],
                     [case["node_len"][1]] * case["queries_per_leaf"]
                     + [case["node_len"][2]] * case["queries_per_leaf"],
                     1, 1, 128, seed=0)
    o = P.PlannerOptions(ts_q_set=tuple(case["ts_q_set"]))
    plan = P.build_plan(spec.parent, spec.node_kv_len, spec.node_page_offsets,
                        spec.node_pages, 16, spec.query_node, spec.query_kv_end,
                        1, 1, 128, o)
    assert plan["edges"] == case["expect_edges"]
    got = [{"node": g["node"], "rows": g["rows"]} for g in plan["groups"]]
    assert got == case["expect_groups"]


def test_hand_computed_costs_long_tail_tree():
    # Root 4000 tokens shared by 10 single-row leaves of 400 (GQA 1, d = 128,
    # gamma = 64, TS_q in {16, 64, 128}, TS_c = 64).  First leaf, by hand:
    #   C0 = Pad(16,10)*4000 + 10*Pad(64,64) + Pad(16,1)*400 + 1*Pad(64,64) + 64*1
    #      = 6*4000 + 0 + 15*400 + 0 + 64 = 30064            (times d)
    #   C1 = Pad(16,9)*4000 + 9*0 + Pad(16,1)*4400 + 0 = 7*4000 + 15*4400 = 94000
    o = P.PlannerOptions()
    d = 128
    assert P.split_kv_cost(10, 1, 400, 4000, d, o) == 30064 * d
    assert P.split_q_cost(10, 1, 400, 4000, d, o) == 94000 * d
    spec = W.config_long()
    plan = P.build_plan(spec.parent, spec.node_kv_len, spec.node_page_offsets,
                        spec.node_pages, 16, spec.query_node, spec.query_kv_end,
                        32, 32, 128, o)
    assert plan["edges"] == [0] * 11
    assert [g["rows"] for g in plan["groups"]] == [10] + [1] * 10


def test_hand_computed_short_context_padding():
    # C_{P,c} charges context padding: 3 rows on a 10-token node pad 54 slots.
    o = P.PlannerOptions()
    assert P.cost_pc(3, 10, 1, o) == 3 * 54
    assert P.cost_pc(3, 100, 1, o) == 0
    # C_{P,q}: 17 rows take the 64 tile: 47 padded rows over len 5.
    assert P.cost_pq(17, 5, 2, o) == 47 * 5 * 2


def _span_tokens(group, node_kv_len):
    out = []
    for a in group["chain"]:
        out += [(a, i) for i in range(int(node_kv_len[a]))]
    return out


def _path_tokens(spec, t):
    u, e = int(spec.query_node[t]), int(spec.query_kv_end[t])
    path = oracle.node_path(spec.parent, u)
    out = []
    for a in path[:-1]:
        out += [(a, i) for i in range(int(spec.node_kv_len[a]))]
    return out + [(u, i) for i in range(e)]


def _check_coverage(spec, plan):
    toks_of = {}
    for gi, g in enumerate(plan["groups"]):
        span = _span_tokens(g, spec.node_kv_len)
        assert len(span) == g["span"]
        blocks = plan["_blocks"][gi]
        # chunks partition the block list in order
        assert g["chunks"][0][0] == 0 and g["chunks"][-1][1] == len(blocks)
        for (a, b), (c, _) in zip(g["chunks"], g["chunks"][1:]):
            assert b == c and a < b
        # blocks enumerate the span in order with the right pages
        pos = 0
        for page, bpos, nval in blocks:
            assert bpos == pos and 1 <= nval <= 16
            pos += nval
        assert pos == g["span"]
        for t, vis in zip(g["tokens"], g["vis"]):
            toks_of.setdefault(t, []).extend(span[:vis])
    for t in range(spec.n_queries):
        got = toks_of.get(t, [])
        assert sorted(got) == sorted(_path_tokens(spec, t)), t
        assert len(got) == len(set(got)), t  # exactly once
        n_groups = sum(1 for g in plan["groups"] if t in g["tokens"])
        n_parts = sum(len(g["chunks"]) for g in plan["groups"] if t in g["tokens"])
        assert plan["partials"][t] == n_parts and n_groups >= 1


@pytest.mark.parametrize("seed", range(8))
def test_coverage_over_all_edge_assignments(seed):
    spec = W.random_tree(100 + seed, n_nodes=2 + seed, max_len=40, hq=2, hkv=1,
                         d=64, zero_len_prob=0.1, max_queries_per_node=2)
    n_edges = spec.n_nodes - 1
    assert n_edges <= 10
    for bits in itertools.product((0, 1), repeat=n_edges):
        edges = (0,) + bits
        o = P.PlannerOptions(edges=edges, split_tokens=32 if seed % 2 else 0)
        plan = P.build_plan(spec.parent, spec.node_kv_len, spec.node_page_offsets,
                            spec.node_pages, 16, spec.query_node, spec.query_kv_end,
                            2, 1, 64, o)
        assert plan["edges"][1:] == list(bits)
        _check_coverage(spec, plan)


@pytest.mark.parametrize("name", ["tiny", "long", "wide", "three", "irreg"])
def test_coverage_of_greedy_plan_on_configs(name):
    spec = W.CONFIGS[name]()
    plan = P.build_plan(spec.parent, spec.node_kv_len, spec.node_page_offsets,
                        spec.node_pages, 16, spec.query_node, spec.query_kv_end,
                        spec.n_q_heads, spec.n_kv_heads, spec.head_dim)
    if name == "irreg":
        # full coverage check is quadratic; check partial counts and spans
        for g in plan["groups"]:
            assert g["span"] == sum(int(spec.node_kv_len[a]) for a in g["chain"])
        return
    _check_coverage(spec, plan)


def test_plan_cost_worked_by_hand():
    # Root 0 (100 tokens) with children 1 (30 tokens, 3 query rows) and 2 (70
    # tokens, 20 rows); GQA 1, d = 1, gamma = 64, TS_q in {16, 64, 128},
    # TS_c = 64.  A = [23, 3, 20].  Per virtual node: Pad(TS_q, rows) * len +
    # rows * Pad(TS_c, min(len, TS_c)), plus gamma * A[l] for every 0-edge:
    #  (0, 0): 41*100 + 13*30 + 3*34 + 44*70 + 64*3 + 64*20    = 9144
    #  (1, 0): 44*100 + 13*130 + 44*70 + 64*20                  = 10450
    #  (0, 1): 13*100 + 13*30 + 3*34 + 44*170 + 64*3            = 9464
    #  (1, 1): 0 + 13*130 + 44*170                              = 9170
    parent, lens = [-1, 0, 0], [100, 30, 70]
    qnode = [1] * 3 + [2] * 20
    o = P.PlannerOptions()
    A = P.subtree_rows(parent, qnode, 1)
    assert A == [23, 3, 20]
    want = {(0, 0): 9144, (1, 0): 10450, (0, 1): 9464, (1, 1): 9170}
    for (e1, e2), c in want.items():
        assert P.plan_cost(parent, lens, A, 1, [0, e1, e2], o) == c
        assert P.plan_cost(parent, lens, A, 128, [0, e1, e2], o) == 128 * c
    # Algorithm 1 on the same tree, by hand: child 1: C0 = 4100 + 390 + 102 +
    # 192 = 4784 < C1 = 4400 + 1690 = 6090; child 2: C0 = 4100 + 3080 + 1280 =
    # 8460 < C1 = 1300 + 7480 = 8780: both edges 0, the cheapest plan here.
    assert P.split_kv_cost(23, 3, 30, 100, 1, o) == 4784
    assert P.split_q_cost(23, 3, 30, 100, 1, o) == 6090
    assert P.split_kv_cost(23, 20, 70, 100, 1, o) == 8460
    assert P.split_q_cost(23, 20, 70, 100, 1, o) == 8780
    edge, _, rows, _ = P.greedy_edges(parent, lens, A, 1, o)
    assert edge == [0, 0, 0] and rows == [23, 3, 20]


def test_split_chunks_by_hand():
    # a span of at most one chunk stays whole; a longer one is cut into
    # ceil(n / chunk) chunks of equal, tile-rounded length, the last shorter
    assert P.split_chunks(7, 8, 4) == [[0, 7]]
    assert P.split_chunks(8, 8, 4) == [[0, 8]]
    assert P.split_chunks(9, 8, 4) == [[0, 8], [8, 9]]       # k = 2, ceil(9/2) = 5 -> 8
    assert P.split_chunks(250, 28, 4) == [[0, 28], [28, 56], [56, 84], [84, 112], [112, 140],
                                          [140, 168], [168, 196], [196, 224], [224, 250]]
    assert P.split_chunks(17, 4, 4) == [[0, 4], [4, 8], [8, 12], [12, 16], [16, 17]]
    assert P.split_chunks(0, 4, 4) == [[0, 0]]


@pytest.mark.parametrize("seed", range(6))
def test_greedy_against_brute_force_proxy(seed):
    spec = W.random_tree(200 + seed, n_nodes=4 + seed, max_len=300, hq=8, hkv=2,
                         d=64, max_queries_per_node=6)
    o = P.PlannerOptions(gamma=16)
    r = 4
    A = P.subtree_rows(spec.parent, spec.query_node, r)
    edge, _, _, _ = P.greedy_edges(spec.parent, spec.node_kv_len, A, 64, o)
    greedy = P.plan_cost(spec.parent, spec.node_kv_len, A, 64, edge, o)
    best = min(P.plan_cost(spec.parent, spec.node_kv_len, A, 64, (0,) + b, o)
               for b in itertools.product((0, 1), repeat=spec.n_nodes - 1))
    assert greedy >= best
    # all-zero (no KV duplicated) is one of the enumerated plans
    zero = P.plan_cost(spec.parent, spec.node_kv_len, A, 64, [0] * spec.n_nodes, o)
    assert best <= zero


def test_subtree_rows_counts_tokens_times_gqa():
    spec = W.config_three()
    A = P.subtree_rows(spec.parent, spec.query_node, 1)
    assert A[0] == 256 and all(A[c] == 16 for c in range(1, 17))
    assert all(A[x] == 1 for x in range(17, 273))
    spec = W.config_irregular()
    A = P.subtree_rows(spec.parent, spec.query_node, 16)
    assert A[0] == 16 * spec.n_queries
