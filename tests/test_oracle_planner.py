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
