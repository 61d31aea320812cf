"""Seeded synthetic inputs for tree-structured decode attention.

This module builds decoding trees, their paged block tables and the Q/K/V
tensors that both the CUDA path and the oracle consume.  It holds none of the
method's arithmetic: no attention, no cost model, no grouping.  Everything here
is a pure function of a seed.

Structure (topology, lengths, page permutation) is drawn from SplitMix64, a
counter-based generator implemented below from its published definition
(Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014), so a tree is the same on every machine and numpy version.
Values (Q, K, V ~ N(0, 1), rounded to bf16) come from a seeded torch
generator.

Workloads (decoding trees as defined on the DeFT notes page, "Decoding tree
definition": the root is the prompt, every other node a generated span, and a
leaf's last token is the next decode input; tree shapes parameterised as on the
FastTree review page, section "内核基准测试", by nodes per level N, context per
node C and GQA ratio):

=======  ==========================================================  =========
name     tree                                                        heads, d
=======  ==========================================================  =========
tiny     root 256 + 4 leaves x 32, 1 query per leaf                  4/4, 64
long     root 4000 + 10 leaves x 400, 1 query per leaf               32/32, 128
wide     root 2048 + 256 leaves x 64, 1 query per leaf               32/8, 128
three    root 1024, 16 x 512, 16 x 16 leaves x 128, 1 q per leaf      32/32, 128
irreg    depth 4-5, branching U{1..8}, lengths log-uniform 16..2048, 64/4, 128
         ~1024 leaves, 4 speculative query tokens per leaf (causal)
=======  ==========================================================  =========
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE_SIZE = 16
MASK64 = (1 << 64) - 1


class SplitMix64:
    """SplitMix64 (Steele et al. 2014): state += golden gamma, then mix."""

    def __init__(self, seed: int):
        self.state = seed & MASK64

    def next_u64(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)

    def uniform(self) -> float:
        """Uniform double in [0, 1) from the top 53 bits."""
        return (self.next_u64() >> 11) * (1.0 / (1 << 53))

    def randint(self, lo: int, hi: int) -> int:
        """Uniform integer in [lo, hi] (inclusive)."""
        return lo + int(self.uniform() * (hi - lo + 1))

    def permutation(self, n: int) -> np.ndarray:
        """Fisher-Yates shuffle of range(n)."""
        p = np.arange(n, dtype=np.int64)
        for i in range(n - 1, 0, -1):
            j = self.randint(0, i)
            p[i], p[j] = p[j], p[i]
        return p


@dataclass
class TreeSpec:
    """A decoding tree with its decode queries and paged KV layout.

    parent[v]        parent node id, -1 for the root (node ids need not be
                     topologically ordered, but generators emit BFS order).
    node_kv_len[v]   tokens of KV held by node v (a leaf's length includes the
                     KV of its own decode query tokens).
    query_node[t]    node of query token t.
    query_kv_end[t]  how many tokens of query_node[t] that token sees (causal
                     prefix of its own node); ancestors are seen in full.
    node_page_offsets[v]..[v+1]  slice of node_pages holding v's pages, in
                     token order; node v owns ceil(len/16) pages.
    """

    name: str
    parent: np.ndarray
    node_kv_len: np.ndarray
    query_node: np.ndarray
    query_kv_end: np.ndarray
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int = PAGE_SIZE
    node_page_offsets: np.ndarray | None = None
    node_pages: np.ndarray | None = None
    num_pages: int = 0
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def n_nodes(self) -> int:
        return int(self.parent.shape[0])

    @property
    def n_queries(self) -> int:
        return int(self.query_node.shape[0])

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads


def _finish(name, parent, lens, qnode, qend, hq, hkv, d, seed, slack_pages=0,
            meta=None) -> TreeSpec:
    spec = TreeSpec(
        name=name,
        parent=np.asarray(parent, dtype=np.int32),
        node_kv_len=np.asarray(lens, dtype=np.int32),
        query_node=np.asarray(qnode, dtype=np.int32),
        query_kv_end=np.asarray(qend, dtype=np.int32),
        n_q_heads=hq, n_kv_heads=hkv, head_dim=d, seed=seed,
        meta=dict(meta or {}),
    )
    assign_pages(spec, seed, slack_pages=slack_pages)
    return spec


def assign_pages(spec: TreeSpec, seed: int, slack_pages: int = 0) -> None:
    """Give every node ceil(len/page) pages drawn from a shuffled pool.

    Page ids are a SplitMix64 permutation of the pool, so consecutive tokens of
    a node sit in scattered pages.  ``slack_pages`` extra pool pages belong to
    no node.
    """
    ps = spec.page_size
    counts = [(int(n) + ps - 1) // ps for n in spec.node_kv_len]
    offs = np.zeros(len(counts) + 1, dtype=np.int32)
    offs[1:] = np.cumsum(counts)
    total = int(offs[-1])
    num_pages = total + slack_pages
    perm = SplitMix64(seed ^ 0x5A5A_0F0F_1234).permutation(num_pages)
    spec.node_page_offsets = offs
    spec.node_pages = perm[:total].astype(np.int32)
    spec.num_pages = num_pages


def _leaf_queries(parent, lens, tokens_per_leaf=1):
    """Queries at every leaf: the last ``k`` tokens of the leaf, causal."""
    n = len(parent)
    has_child = np.zeros(n, dtype=bool)
    for v in range(n):
        if parent[v] >= 0:
            has_child[parent[v]] = True
    qn, qe = [], []
    for v in range(n):
        if not has_child[v]:
            for j in range(tokens_per_leaf):
                qn.append(v)
                qe.append(int(lens[v]) - tokens_per_leaf + j + 1)
    return qn, qe


def two_level(root_len, n_leaves, leaf_len, hq, hkv, d, seed=0, name="two_level",
              tokens_per_leaf=1):
    parent = [-1] + [0] * n_leaves
    lens = [root_len] + [leaf_len] * n_leaves
    qn, qe = _leaf_queries(parent, lens, tokens_per_leaf)
    return _finish(name, parent, lens, qn, qe, hq, hkv, d, seed)


def token_tree(prompt_len, n_ctx, ctx_len, depth, branching, hq, hkv, d, seed=0,
               name="token_tree"):
    """Speculative token trees for tree verification: a shared prompt, n_ctx
    sequences of ctx_len generated tokens below it, and under each a tree of
    draft tokens (depth levels, `branching` children per token).  Every draft
    token is its own one-token node and one query token that sees its node
    in full, so it attends to the prompt, its sequence and its draft-tree
    ancestors: an arbitrary intra-leaf token tree expressed as tree
    topology."""
    parent, lens = [-1], [prompt_len]
    qn, qe = [], []
    for _ in range(n_ctx):
        parent.append(0)
        lens.append(ctx_len)
        level = [len(parent) - 1]
        for _ in range(depth):
            nxt = []
            for par in level:
                for _ in range(branching):
                    parent.append(par)
                    lens.append(1)
                    qn.append(len(parent) - 1)
                    qe.append(1)
                    nxt.append(len(parent) - 1)
            level = nxt
    return _finish(name, parent, lens, qn, qe, hq, hkv, d, seed)


def config_tiny(seed=1):
    """Root 256 KV tokens, 4 leaves of 32; 4 q heads = 4 kv heads, d = 64."""
    return two_level(256, 4, 32, 4, 4, 64, seed, name="tiny")


def config_long(seed=2):
    """Llama-2-7B attention shape: root 4000, 10 leaves of 400, 32/32, d 128."""
    return two_level(4000, 10, 400, 32, 32, 128, seed, name="long")


def config_wide(seed=3):
    """Wide sharing with GQA 4: root 2048, 256 leaves of 64, 32/8 heads."""
    return two_level(2048, 256, 64, 32, 8, 128, seed, name="wide")


def config_three(seed=4):
    """Root 1024, 16 children of 512, each with 16 leaves of 128; 32/32."""
    parent = [-1] + [0] * 16
    lens = [1024] + [512] * 16
    for c in range(1, 17):
        parent += [c] * 16
        lens += [128] * 16
    qn, qe = _leaf_queries(parent, lens, 1)
    return _finish("three", parent, lens, qn, qe, 32, 32, 128, seed)


def irregular_topology(seed: int, max_depth=5, always_branch_below=4,
                       branch_max=8, len_lo=16, len_hi=2048):
    """BFS-expanded random tree.

    Nodes at depth < ``always_branch_below`` get U{1..branch_max} children;
    nodes at that depth get children with probability 1/2; nodes at
    ``max_depth`` are leaves.  Lengths are round(exp(U(ln lo, ln hi))).
    """
    rng = SplitMix64(seed)
    parent, depth, lens = [-1], [0], []
    lo, hi = math.log(len_lo), math.log(len_hi)
    head = 0
    while head < len(parent):
        v = head
        head += 1
        dv = depth[v]
        if dv < always_branch_below:
            nb = rng.randint(1, branch_max)
        elif dv < max_depth:
            nb = rng.randint(1, branch_max) if rng.uniform() < 0.5 else 0
        else:
            nb = 0
        for _ in range(nb):
            parent.append(v)
            depth.append(dv + 1)
    for _ in parent:
        lens.append(int(round(math.exp(lo + (hi - lo) * rng.uniform()))))
    return parent, lens


def config_irregular(seed=1000, leaf_lo=960, leaf_hi=1088, spec_tokens=4):
    """Irregular random tree, GQA 16 (64/4), 4 speculative tokens per leaf.

    Accepts the first sub-seed ``seed + k`` whose leaf count lies in
    [leaf_lo, leaf_hi].  Leaves shorter than ``spec_tokens`` are lengthened to
    hold the query tokens' own KV.
    """
    for k in range(10_000):
        parent, lens = irregular_topology(seed + k)
        n = len(parent)
        has_child = [False] * n
        for v in range(1, n):
            has_child[parent[v]] = True
        n_leaves = sum(1 for v in range(n) if not has_child[v])
        if leaf_lo <= n_leaves <= leaf_hi:
            for v in range(n):
                if not has_child[v] and lens[v] < spec_tokens:
                    lens[v] = spec_tokens
            qn, qe = _leaf_queries(parent, lens, spec_tokens)
            return _finish("irreg", parent, lens, qn, qe, 64, 4, 128, seed + k,
                           meta={"sub_seed": seed + k, "n_leaves": n_leaves})
    raise RuntimeError("no accepted sub-seed")


CONFIGS = {
    "tiny": config_tiny,
    "long": config_long,
    "wide": config_wide,
    "three": config_three,
    "irreg": config_irregular,
}


def random_tree(seed: int, n_nodes: int, max_len: int = 40, hq: int = 4,
                hkv: int = 2, d: int = 64, max_queries_per_node: int = 2,
                zero_len_prob: float = 0.0, internal_query_prob: float = 0.3,
                slack_pages: int = 3, name: str = "random") -> TreeSpec:
    """Small random tree for parity and invariant tests.

    Parents are drawn among earlier nodes, lengths from U{1..max_len} (or 0
    with ``zero_len_prob``); every leaf and some internal nodes carry 1..k
    query tokens, each seeing a random causal prefix of its own node.
    """
    rng = SplitMix64(seed)
    parent = [-1]
    for v in range(1, n_nodes):
        parent.append(rng.randint(0, v - 1))
    lens = []
    for _ in range(n_nodes):
        if zero_len_prob > 0 and rng.uniform() < zero_len_prob:
            lens.append(0)
        else:
            lens.append(rng.randint(1, max_len))
    has_child = [False] * n_nodes
    for v in range(1, n_nodes):
        has_child[parent[v]] = True
    qn, qe = [], []
    for v in range(n_nodes):
        if (not has_child[v]) or rng.uniform() < internal_query_prob:
            k = rng.randint(1, max_queries_per_node)
            for _ in range(k):
                qn.append(v)
                qe.append(rng.randint(0, lens[v]) if lens[v] > 0 else 0)
    return _finish(name, parent, lens, qn, qe, hq, hkv, d, seed,
                   slack_pages=slack_pages)


def make_tensors(spec: TreeSpec, seed: int | None = None, device="cpu",
                 tail_fill: float | None = None):
    """Q [nq, Hq, d], K/V pages [num_pages, Hkv, 16, d], all bf16 ~ N(0, 1).

    ``tail_fill`` overwrites every slot that holds no token (the tail of a
    node's last page and unowned pages), e.g. with NaN, so a test can show that
    those slots never reach a result.
    """
    import torch

    seed = spec.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 7919 + 17)
    hq, hkv, d, ps = spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.page_size
    q = torch.randn((spec.n_queries, hq, d), generator=gen, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    shape = (spec.num_pages, hkv, ps, d)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    k = k.to(torch.bfloat16)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    v = v.to(torch.bfloat16)
    if tail_fill is not None:
        valid = valid_slot_mask(spec)
        inval = torch.from_numpy(~valid).to(device)[:, None, :, None]
        k.masked_fill_(inval, tail_fill)
        v.masked_fill_(inval, tail_fill)
    return q, k, v


def valid_slot_mask(spec: TreeSpec) -> np.ndarray:
    """Boolean [num_pages, page] mask of slots that hold a node's token."""
    ps = spec.page_size
    m = np.zeros((spec.num_pages, ps), dtype=bool)
    for v in range(spec.n_nodes):
        n = int(spec.node_kv_len[v])
        pages = spec.node_pages[spec.node_page_offsets[v]:spec.node_page_offsets[v + 1]]
        for i, p in enumerate(pages):
            m[p, :min(ps, n - i * ps)] = True
    return m


def summary(spec: TreeSpec) -> dict:
    """Sizes of a workload (no method arithmetic: counts only)."""
    return {
        "name": spec.name,
        "nodes": spec.n_nodes,
        "queries": spec.n_queries,
        "kv_tokens": int(spec.node_kv_len.sum()),
        "pages": int(spec.num_pages),
        "heads": [spec.n_q_heads, spec.n_kv_heads],
        "d": spec.head_dim,
    }
