"""Pins for the fp64 tree-attention oracle (CPU only).

Each test checks the oracle against something other than itself: a library
routine on the case that reduces to it, an independent dense tree-mask
formulation, scalar brute force, closed forms, and invariants the definition
implies (DeFT notes page, "Tree attention definition"; FastTree review page,
"核心公式")."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _np(x):
    return x.to(torch.float64).numpy()


def _run_spec(spec, q, k, v, tokens=None):
    return oracle.tree_attention_spec(spec, q, k, v, tokens=tokens)


# ---------------------------------------------------------------------------
# 1. Hand-computed example (values fixed by arithmetic, not by the oracle).
# ---------------------------------------------------------------------------
def test_hand_computed_two_token_example():
    # d = 2, scale = 1/sqrt(2): q = (1, 0); k0 = (0, 0) -> s0 = 0;
    # k1 = (sqrt(2) ln 3, 0) -> s1 = ln 3.  softmax = (1/4, 3/4).
    # v0 = (4, 0), v1 = (0, 4) -> out = (1, 3); lse = ln(1 + 3) = ln 4.
    parent = np.array([-1])
    lens = np.array([2])
    offs = np.array([0, 1])
    pages = np.array([0])
    kp = np.zeros((1, 1, 16, 2))
    vp = np.zeros((1, 1, 16, 2))
    kp[0, 0, 1] = [math.sqrt(2) * math.log(3), 0]
    vp[0, 0, 0] = [4, 0]
    vp[0, 0, 1] = [0, 4]
    q = np.array([[[1.0, 0.0]]])
    out, lse = oracle.tree_attention(parent, lens, offs, pages, [0], [2], q, kp, vp)
    assert np.allclose(out[0, 0], [1.0, 3.0], atol=1e-14)
    assert abs(lse[0, 0] - math.log(4)) < 1e-14
    # A causal end of 1 sees only k0: out = v0, lse = 0.
    out, lse = oracle.tree_attention(parent, lens, offs, pages, [0], [1], q, kp, vp)
    assert np.allclose(out[0, 0], [4.0, 0.0]) and abs(lse[0, 0]) < 1e-15


# ---------------------------------------------------------------------------
# 2. Single-node tree == ordinary attention (library routine, fp64 CPU).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n,hq,hkv,d", [(1, 2, 2, 64), (37, 4, 2, 64), (130, 8, 1, 128)])
def test_single_node_equals_sdpa(n, hq, hkv, d):
    spec = W._finish("single", [-1], [n], [0, 0], [n, max(1, n // 2)], hq, hkv, d,
                     seed=n)
    q, k, v = W.make_tensors(spec)
    out, lse = _run_spec(spec, q, k, v)
    # Library: torch SDPA in fp64 over the node's tokens in token order.
    kk = torch.cat([k[p] for p in spec.node_pages], dim=1)[:, :n].double()
    vv = torch.cat([v[p] for p in spec.node_pages], dim=1)[:, :n].double()
    r = hq // hkv
    kk = kk.repeat_interleave(r, dim=0)  # [hq, n, d]
    vv = vv.repeat_interleave(r, dim=0)
    for t, e in enumerate(spec.query_kv_end):
        qq = q[t].double()[:, None, :]  # [hq, 1, d]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, kk[:, :e], vv[:, :e])[:, 0]
        assert np.abs(out[t] - ref.numpy()).max() < 1e-12
        s = torch.einsum("hd,hjd->hj", qq[:, 0], kk[:, :e]) / math.sqrt(d)
        ref_lse = torch.logsumexp(s, dim=-1)
        assert np.abs(lse[t] - ref_lse.numpy()).max() < 1e-12


# ---------------------------------------------------------------------------
# 3. Independent formulation: flatten the tree, dense attention under a mask.
# ---------------------------------------------------------------------------
def _tree_mask_attention(spec, q, k, v):
    """All tree tokens in DFS order; token j is visible to query t iff its node
    is a strict ancestor of t's node, or is t's node with index < end."""
    n = spec.n_nodes
    ch = [[] for _ in range(n)]
    root = 0
    for x in range(n):
        if spec.parent[x] < 0:
            root = x
        else:
            ch[spec.parent[x]].append(x)
    order, stack = [], [root]
    while stack:
        x = stack.pop()
        order.append(x)
        stack.extend(reversed(ch[x]))
    tok_node, tok_idx = [], []
    ks, vs = [], []
    kd, vd = _np(k), _np(v)
    ps = spec.page_size
    for x in order:
        for i in range(int(spec.node_kv_len[x])):
            page = spec.node_pages[spec.node_page_offsets[x] + i // ps]
            ks.append(kd[page, :, i % ps])
            vs.append(vd[page, :, i % ps])
            tok_node.append(x)
            tok_idx.append(i)
    K = np.stack(ks) if ks else np.zeros((0, spec.n_kv_heads, spec.head_dim))
    V = np.stack(vs) if vs else np.zeros((0, spec.n_kv_heads, spec.head_dim))
    # ancestor sets by repeated parent lookups
    anc = [set() for _ in range(n)]
    for x in range(n):
        y = spec.parent[x]
        while y >= 0:
            anc[x].add(int(y))
            y = spec.parent[y]
    qd = _np(q)
    nq, hq, d = qd.shape
    r = hq // spec.n_kv_heads
    out = np.zeros((nq, hq, d))
    lse = np.full((nq, hq), -np.inf)
    for t in range(nq):
        u, e = int(spec.query_node[t]), int(spec.query_kv_end[t])
        mask = np.array([(tn in anc[u]) or (tn == u and ti < e)
                         for tn, ti in zip(tok_node, tok_idx)], dtype=bool)
        if not mask.any():
            continue
        for h in range(hq):
            s = (K[:, h // r, :] @ qd[t, h]) / math.sqrt(d)
            s = np.where(mask, s, -np.inf)
            m = s.max()
            w = np.exp(s - m)
            out[t, h] = (w @ V[:, h // r, :]) / w.sum()
            lse[t, h] = m + math.log(w.sum())
    return out, lse


@pytest.mark.parametrize("seed", range(6))
def test_tree_mask_formulation(seed):
    spec = W.random_tree(seed, n_nodes=3 + seed * 2, max_len=37, hq=4,
                         hkv=(1, 2, 4)[seed % 3], d=64, zero_len_prob=0.15,
                         max_queries_per_node=3)
    q, k, v = W.make_tensors(spec, tail_fill=float("nan"))
    out, lse = _run_spec(spec, q, k, v)
    ref, ref_lse = _tree_mask_attention(spec, q, k, v)
    assert np.array_equal(np.isfinite(lse), np.isfinite(ref_lse))
    fin = np.isfinite(ref_lse)
    assert np.abs(out - ref).max() < 1e-12
    assert np.abs(lse[fin] - ref_lse[fin]).max() < 1e-12


def test_tree_mask_on_config_tiny():
    spec = W.config_tiny()
    q, k, v = W.make_tensors(spec)
    out, lse = _run_spec(spec, q, k, v)
    ref, ref_lse = _tree_mask_attention(spec, q, k, v)
    assert np.abs(out - ref).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-12


# ---------------------------------------------------------------------------
# 4. Scalar brute force on tiny trees (pure Python loops, math.exp).
# ---------------------------------------------------------------------------
def test_scalar_brute_force_tiny():
    spec = W.random_tree(11, n_nodes=5, max_len=8, hq=2, hkv=1, d=8,
                         max_queries_per_node=2)
    q, k, v = W.make_tensors(spec)
    out, lse = _run_spec(spec, q, k, v)
    qd, kd, vd = _np(q), _np(k), _np(v)
    ps = spec.page_size
    for t in range(spec.n_queries):
        u, e = int(spec.query_node[t]), int(spec.query_kv_end[t])
        keys = []
        for x in range(spec.n_nodes):
            y, is_anc = u, False
            while y >= 0:
                y = int(spec.parent[y])
                if y == x:
                    is_anc = True
            n_vis = int(spec.node_kv_len[x]) if is_anc else (e if x == u else 0)
            for i in range(n_vis):
                keys.append((int(spec.node_pages[spec.node_page_offsets[x] + i // ps]),
                             i % ps))
        for h in range(spec.n_q_heads):
            g = h // spec.gqa
            if not keys:
                assert lse[t, h] == -np.inf and not out[t, h].any()
                continue
            ss = [sum(qd[t, h, c] * kd[p, g, s, c] for c in range(spec.head_dim))
                  / math.sqrt(spec.head_dim) for p, s in keys]
            mx = max(ss)
            ws = [math.exp(x - mx) for x in ss]
            tot = sum(ws)
            for c in range(spec.head_dim):
                o = sum(w * vd[p, g, s, c] for w, (p, s) in zip(ws, keys)) / tot
                assert abs(o - out[t, h, c]) < 1e-12
            assert abs(mx + math.log(tot) - lse[t, h]) < 1e-12


# ---------------------------------------------------------------------------
# 5. LSE merge of split partials is exact.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(5))
def test_merge_of_split_partials_is_exact(seed):
    rng = np.random.default_rng(seed)
    L, d, m = int(rng.integers(2, 300)), 64, 3
    qr = rng.standard_normal((m, d))
    k = rng.standard_normal((L, d)) * 2.0
    v = rng.standard_normal((L, d))
    full_o, full_l = oracle.attention_rows(qr, k, v, 0.125)
    cuts = sorted(set(rng.integers(0, L, size=int(rng.integers(1, 6))).tolist()))
    bounds = [0] + cuts + [L]
    os_, ls_ = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o, l = oracle.attention_rows(qr, k[a:b], v[a:b], 0.125)
        os_.append(o)
        ls_.append(l)
    mo, ml = oracle.merge_partials(os_, ls_)
    assert np.abs(mo - full_o).max() < 1e-12
    assert np.abs(ml - full_l).max() < 1e-12


def test_merge_all_empty_partials():
    o, l = oracle.merge_partials(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert (o == 0).all() and np.isneginf(l).all()


# ---------------------------------------------------------------------------
# 6. Closed forms.
# ---------------------------------------------------------------------------
def test_equal_keys_give_mean_of_values():
    spec = W.random_tree(5, n_nodes=6, max_len=20, hq=2, hkv=2, d=64)
    q, k, v = W.make_tensors(spec)
    k[:] = k[0, 0, 0]  # every key identical
    out, lse = _run_spec(spec, q, k, v)
    kd, vd, qd = _np(k), _np(v), _np(q)
    for t in range(spec.n_queries):
        _, vt = oracle.query_kv(spec.parent, spec.node_kv_len, spec.node_page_offsets,
                                spec.node_pages, kd, vd, int(spec.query_node[t]),
                                int(spec.query_kv_end[t]))
        n = vt.shape[0]
        for h in range(2):
            if n == 0:
                assert np.isneginf(lse[t, h])
                continue
            s = float(qd[t, h] @ kd[0, 0, 0]) / 8.0
            assert abs(lse[t, h] - (math.log(n) + s)) < 1e-12
            assert np.abs(out[t, h] - vt[:, h].mean(axis=0)).max() < 1e-12


def test_dominant_key_selects_its_value():
    spec = W.two_level(40, 2, 9, 1, 1, 64, seed=3)
    q, k, v = W.make_tensors(spec)
    # make token 17 of the root (page 1, slot 1) dominate for query 0
    page = spec.node_pages[spec.node_page_offsets[0] + 1]
    k[page, 0, 1] = (q[0, 0].float() * 40).to(torch.bfloat16)
    out, _ = _run_spec(spec, q, k, v, tokens=[0])
    assert np.abs(out[0, 0] - _np(v)[page, 0, 1]).max() < 1e-9


# ---------------------------------------------------------------------------
# 7. Invariants: GQA == MHA with repeated KV heads; page order irrelevant.
# ---------------------------------------------------------------------------
def test_gqa_equals_mha_with_repeated_kv():
    spec = W.random_tree(7, n_nodes=7, max_len=30, hq=8, hkv=2, d=64)
    q, k, v = W.make_tensors(spec)
    out, lse = _run_spec(spec, q, k, v)
    spec_mha = W._finish("mha", spec.parent, spec.node_kv_len, spec.query_node,
                         spec.query_kv_end, 8, 8, 64, seed=spec.seed, slack_pages=3)
    k2 = k.repeat_interleave(4, dim=1)
    v2 = v.repeat_interleave(4, dim=1)
    out2, lse2 = _run_spec(spec_mha, q, k2, v2)
    assert np.abs(out - out2).max() < 1e-12 and np.abs(lse - lse2).max() < 1e-12


def test_page_order_is_irrelevant():
    spec = W.random_tree(8, n_nodes=9, max_len=50, hq=4, hkv=2, d=64)
    q, k, v = W.make_tensors(spec)
    out, lse = _run_spec(spec, q, k, v)
    perm = np.random.default_rng(0).permutation(spec.num_pages)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    k2, v2 = k[torch.from_numpy(inv)], v[torch.from_numpy(inv)]
    spec.node_pages = perm[spec.node_pages].astype(np.int32)
    out2, lse2 = _run_spec(spec, q, k2, v2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_token_tree_verification_equals_masked_flat_attention():
    # Tree verification with a draft-token tree: the oracle on the tree of
    # one-token nodes equals dense attention over the flattened sequence
    # [prompt, context, drafts] with the usual verification mask (a draft
    # sees the prompt, its context and its draft ancestors), written here
    # directly from that mask.
    spec = W.token_tree(40, 2, 9, 3, 2, 4, 2, 16, seed=5)
    q, k, v = W.make_tensors(spec, seed=5)
    q, kp, vp = _np(q), _np(k), _np(v)
    out, lse = oracle.tree_attention_spec(spec, q, kp, vp)
    # flatten node by node (node ids are in DFS-compatible creation order)
    order = list(range(spec.n_nodes))
    tok_node, tok_k, tok_v = [], [], []
    for u in order:
        n = int(spec.node_kv_len[u])
        tok_node += [u] * n
        tok_k.append(oracle.gather_node_kv(kp, spec.node_page_offsets, spec.node_pages, u, n))
        tok_v.append(oracle.gather_node_kv(vp, spec.node_page_offsets, spec.node_pages, u, n))
    K, V = np.concatenate(tok_k), np.concatenate(tok_v)
    anc = {u: set(oracle.node_path(spec.parent, u)) for u in order}
    r = spec.n_q_heads // spec.n_kv_heads
    s = 1.0 / np.sqrt(spec.head_dim)
    for t in range(spec.n_queries):
        u = int(spec.query_node[t])
        mask = np.array([tn in anc[u] for tn in tok_node])
        for h in range(spec.n_q_heads):
            sc = s * (K[mask, h // r, :] @ q[t, h])
            w = np.exp(sc - sc.max())
            np.testing.assert_allclose(out[t, h], (w / w.sum()) @ V[mask, h // r, :], atol=1e-12)
            np.testing.assert_allclose(lse[t, h], sc.max() + np.log(w.sum()), atol=1e-12)
