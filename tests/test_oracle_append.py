"""Pins of the oracle's append step (each query token's own K/V written to
its own position of the paged cache before attention)."""
import numpy as np
import pytest

import workloads as W
from oracle import attention as A


def test_hand_placed_positions():
    # page size 4; node 0 (6 tokens) in pages [2, 0], node 1 (3 tokens) in
    # page [1].  Token 0 sees node 1 up to 3 -> its own position is node 1's
    # third token: page 1, slot 2.  Token 1 sees node 0 up to 6 -> position 5:
    # node 0's second page (page 0), slot 1.  Token 2 sees nothing of node 1.
    k = np.zeros((3, 1, 4, 2))
    v = np.zeros((3, 1, 4, 2))
    k_new = np.array([[[1.0, 2.0]], [[3.0, 4.0]], [[5.0, 6.0]]])
    v_new = -k_new
    ko, vo = A.append_kv([6, 3], [0, 2, 3], [2, 0, 1], [1, 0, 1], [3, 6, 0], k, v, k_new, v_new)
    want = np.zeros_like(k)
    want[1, 0, 2] = [1.0, 2.0]
    want[0, 0, 1] = [3.0, 4.0]
    assert np.array_equal(ko, want) and np.array_equal(vo, -want)
    assert not k.any()  # inputs untouched


@pytest.mark.parametrize("seed", range(6))
def test_written_positions_are_the_last_visible_tokens(seed):
    rng = np.random.default_rng(seed)
    spec = W.random_tree(seed, n_nodes=int(rng.integers(2, 30)), max_len=200, hq=4, hkv=2, d=64,
                         max_queries_per_node=3)
    k = rng.standard_normal((spec.num_pages, 2, 16, 64))
    v = rng.standard_normal((spec.num_pages, 2, 16, 64))
    k_new = rng.standard_normal((spec.n_queries, 2, 64)) + 100.0  # unlike any old value
    v_new = rng.standard_normal((spec.n_queries, 2, 64)) - 100.0
    ko, vo = A.append_kv(spec.node_kv_len, spec.node_page_offsets, spec.node_pages,
                         spec.query_node, spec.query_kv_end, k, v, k_new, v_new)
    changed = np.zeros(k.shape[:1] + k.shape[2:3], dtype=bool)  # [page, slot]
    for t in range(spec.n_queries):
        u, e = int(spec.query_node[t]), int(spec.query_kv_end[t])
        if e < 1:
            continue
        # read back through the gather of the attention oracle
        kk = A.gather_node_kv(ko, spec.node_page_offsets, spec.node_pages, u, e)
        vv = A.gather_node_kv(vo, spec.node_page_offsets, spec.node_pages, u, e)
        last = max(j for j in range(spec.n_queries)
                   if int(spec.query_node[j]) == u and int(spec.query_kv_end[j]) == e)
        assert np.array_equal(kk[-1], k_new[last]) and np.array_equal(vv[-1], v_new[last])
        p0 = int(spec.node_page_offsets[u])
        changed[int(spec.node_pages[p0 + (e - 1) // 16]), (e - 1) % 16] = True
    # every other slot keeps its value
    keep = ~changed
    assert np.array_equal(ko.transpose(0, 2, 1, 3)[keep], k.transpose(0, 2, 1, 3)[keep])
    assert np.array_equal(vo.transpose(0, 2, 1, 3)[keep], v.transpose(0, 2, 1, 3)[keep])


def test_append_restores_attention():
    # overwrite the query tokens' own positions with NaN, append the true
    # values back: attention equals the attention of the untouched cache
    spec = W.config_tiny()
    q, k, v = W.make_tensors(spec, seed=3)
    k, v = k.double().numpy(), v.double().numpy()
    ref, ref_lse = A.tree_attention_spec(spec, q.double().numpy(), k, v)
    k_own = np.stack([A.gather_node_kv(k, spec.node_page_offsets, spec.node_pages,
                                       int(spec.query_node[t]), int(spec.query_kv_end[t]))[-1]
                      for t in range(spec.n_queries)])
    v_own = np.stack([A.gather_node_kv(v, spec.node_page_offsets, spec.node_pages,
                                       int(spec.query_node[t]), int(spec.query_kv_end[t]))[-1]
                      for t in range(spec.n_queries)])
    nan = np.full_like(k_own, np.nan)
    args = (spec.node_kv_len, spec.node_page_offsets, spec.node_pages, spec.query_node,
            spec.query_kv_end)
    kb, vb = A.append_kv(*args, k, v, nan, nan)
    broken, _ = A.tree_attention_spec(spec, q.double().numpy(), kb, vb)
    assert np.isnan(broken).any()
    kf, vf = A.append_kv(*args, kb, vb, k_own, v_own)
    out, lse = A.tree_attention_spec(spec, q.double().numpy(), kf, vf)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
