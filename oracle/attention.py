"""Tree attention, written out as its definition in float64.

Oracle: test infrastructure only (see the package docstring).

Definition followed (DeFT notes page, "Tree attention definition"): for a
token n in node u, Tree-Attention(n) = Attention(P_root->n), where the path
P_root->n is every token of u's ancestors (root first) followed by the tokens
of u from its first up to n.  Attention is scaled dot-product attention,
softmax(Q K^T / sqrt(d)) V with d the head dimension (FastTree review page,
"核心公式").  The DeFT notes call the result a "sum" of the sequence
attentions along the path; the only reading under which it is the attention
of the concatenated path is the log-sum-exp weighted combination, which is
what ``merge_partials`` computes and what the tests pin as exact.

Inputs are the bf16 tensors of the GPU path, up-cast exactly to float64.
KV is paged: node v's tokens live, in order, in pages
node_pages[node_page_offsets[v]:node_page_offsets[v+1]], laid out
[page][kv_head][slot][d] (the block-table convention of the TGI FlashDecoding
pull request, "block_tables", with head-major pages).

GQA (TGI pull request, ``kv_head_mapping``): q head h reads kv head
h // (Hq / Hkv).
"""
from __future__ import annotations

import math

import numpy as np


def _as_f64(x) -> np.ndarray:
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def node_path(parent, u: int) -> list[int]:
    """Ancestors of u, root first, followed by u itself."""
    path = []
    v = int(u)
    seen = 0
    while v >= 0:
        path.append(v)
        v = int(parent[v])
        seen += 1
        if seen > len(parent):
            raise ValueError("parent array has a cycle")
    path.reverse()
    return path


def gather_node_kv(pages: np.ndarray, node_page_offsets, node_pages, node: int,
                   n_tokens: int) -> np.ndarray:
    """First ``n_tokens`` tokens of ``node`` from a page pool -> [n, Hkv, d]."""
    ps = pages.shape[2]
    out = []
    p0 = int(node_page_offsets[node])
    for i in range((n_tokens + ps - 1) // ps):
        page = int(node_pages[p0 + i])
        take = min(ps, n_tokens - i * ps)
        out.append(pages[page, :, :take, :].transpose(1, 0, 2))
    if not out:
        return np.zeros((0, pages.shape[1], pages.shape[3]), dtype=pages.dtype)
    return np.concatenate(out, axis=0)


def query_kv(parent, node_kv_len, node_page_offsets, node_pages, k_pages,
             v_pages, u: int, e: int):
    """K and V of a query token's path: ancestors in full, then u[0:e]."""
    path = node_path(parent, u)
    ks, vs = [], []
    for a in path[:-1]:
        n = int(node_kv_len[a])
        ks.append(gather_node_kv(k_pages, node_page_offsets, node_pages, a, n))
        vs.append(gather_node_kv(v_pages, node_page_offsets, node_pages, a, n))
    ks.append(gather_node_kv(k_pages, node_page_offsets, node_pages, u, e))
    vs.append(gather_node_kv(v_pages, node_page_offsets, node_pages, u, e))
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)


def attention_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray,
                   scale: float):
    """Exact softmax attention of rows q [m, d] over k, v [L, d] (float64).

    Returns (out [m, d], lse [m]) with lse = log sum_j exp(scale * q.k_j)
    (natural log).  An empty key set gives out = 0 and lse = -inf.
    """
    m = q_rows.shape[0]
    if k.shape[0] == 0:
        return np.zeros((m, v.shape[1])), np.full(m, -np.inf)
    s = scale * (q_rows @ k.T)
    mx = s.max(axis=1, keepdims=True)
    w = np.exp(s - mx)
    den = w.sum(axis=1, keepdims=True)
    out = (w @ v) / den
    lse = (mx + np.log(den))[:, 0]
    return out, lse


def tree_attention(parent, node_kv_len, node_page_offsets, node_pages,
                   query_node, query_kv_end, q, k_pages, v_pages,
                   scale: float | None = None, tokens=None):
    """Tree attention of every (or the listed) query token, all heads.

    q [nq, Hq, d]; k_pages, v_pages [num_pages, Hkv, page, d].
    Returns out [len(tokens), Hq, d] and lse [len(tokens), Hq], float64.
    """
    q = _as_f64(q)
    kp = _as_f64(k_pages)
    vp = _as_f64(v_pages)
    nq, hq, d = q.shape
    hkv = kp.shape[1]
    r = hq // hkv
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    toks = range(nq) if tokens is None else [int(t) for t in tokens]
    outs, lses = [], []
    for t in toks:
        u = int(query_node[t])
        e = int(query_kv_end[t])
        kt, vt = query_kv(parent, node_kv_len, node_page_offsets, node_pages,
                          kp, vp, u, e)
        o = np.zeros((hq, d))
        l = np.zeros(hq)
        for h in range(hq):
            g = h // r
            oh, lh = attention_rows(q[t, h][None, :], kt[:, g, :], vt[:, g, :],
                                    scale)
            o[h] = oh[0]
            l[h] = lh[0]
        outs.append(o)
        lses.append(l)
    if not outs:
        return np.zeros((0, hq, d)), np.zeros((0, hq))
    return np.stack(outs), np.stack(lses)


def tree_attention_spec(spec, q, k_pages, v_pages, scale=None, tokens=None):
    """``tree_attention`` with the arrays taken from a workload description."""
    return tree_attention(spec.parent, spec.node_kv_len, spec.node_page_offsets,
                          spec.node_pages, spec.query_node, spec.query_kv_end,
                          q, k_pages, v_pages, scale=scale, tokens=tokens)


def merge_partials(outs, lses):
    """Combine partial attentions over disjoint key sets into one.

    Tree-topology-aware global reduction (DeFT notes page, "Tree-Topology-Aware
    Global Reduction Strategy"): each partial i is (O_i, lse_i) over its own
    keys; the attention over the union is
        m = max_i lse_i,  w_i = exp(lse_i - m),
        O = sum_i w_i O_i / sum_i w_i,  lse = m + log sum_i w_i.
    Partials with lse = -inf (no keys) carry weight 0; if all are -inf the
    result is O = 0, lse = -inf.
    outs: [k, ..., d]; lses: [k, ...].
    """
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    m = lses.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - m_safe), 0.0)
    den = w.sum(axis=0)
    den_safe = np.where(den > 0, den, 1.0)
    o = (w[..., None] * outs).sum(axis=0) / den_safe[..., None]
    o = np.where(finite[..., None], o, 0.0)
    lse = np.where(finite, m_safe + np.log(den_safe), -np.inf)
    return o, lse


def append_kv(node_kv_len, node_page_offsets, node_pages, query_node, query_kv_end,
              k_pages, v_pages, k_new, v_new):
    """The step before attention in a decode step: every query token's own K
    and V go to its own position of the paged cache.

    Decode appends each new token's K/V to its node before attending, so a
    node's length already counts its query tokens, and a query token's own
    token is the last it sees: position e - 1 of its node, e being its
    visible end (DeFT notes page, "Tree attention definition"; the TGI
    FlashDecoding pull request gives each query token its own KV slot).  A
    token with e = 0 owns no position.  Returns new page pools (copies):
    k_pages[page, :, slot, :] = k_new[t] with page and slot of that position,
    likewise for V; everything else is unchanged.  Arrays are numpy (any
    dtype); tokens are applied in order."""
    k_out, v_out = np.array(k_pages, copy=True), np.array(v_pages, copy=True)
    ps = k_out.shape[2]
    for t, u in enumerate(query_node):
        u = int(u)
        e = int(node_kv_len[u]) if query_kv_end is None else int(query_kv_end[t])
        if e < 1:
            continue
        pos = e - 1
        page = int(node_pages[int(node_page_offsets[u]) + pos // ps])
        k_out[page, :, pos % ps, :] = k_new[t]
        v_out[page, :, pos % ps, :] = v_new[t]
    return k_out, v_out
