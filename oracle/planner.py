"""Reference grouping planner (greedy binary edge assignment): ORACLE.

Test infrastructure only.  Written from the FastTree review page, section
"二元边赋值" (binary edge assignment), "算法1：贪心二元边赋值" (Algorithm 1)
and "开销模型" (cost model), and the DeFT notes page, "KV-Guided Tree Split".
It exists to check the native planner decision by decision; it is plain
Python over ints, with the pages' names.

The problem (FastTree page, "问题形式化"): choose f: E -> {0, 1}.  An edge
v -> l with f = 1 joins l to v in the virtual tree VT(T, f): l's group
carries v's (cumulative) KV and takes l's queries away from v's group
("SplitQ").  f = 0 keeps them apart: l's queries read v's KV inside v's group
and their own KV in l's group, and the two partial results are merged
("SplitKV").  Groups(VT) maps each virtual node with queries left to one
context-query group (KV-guided split, DeFT page: a node's KV grouped with
every query that shares it).

Readings taken where the page is silent or garbled (each is listed with its
reason in the design notes of the repository):
  * "for l in leaves(v)" is read as the children of v, visited in ascending
    node id; BFS is FIFO from the root.
  * nQ counts query *rows*: query tokens x GQA ratio (rows fill the MMA M).
  * SplitKVCost / SplitQCost are the sums of the printed padding components
    over the groups each choice produces, plus the printed intermediate-result
    term gamma * nQ_l * d for SplitKV; beta (default 0) optionally charges the
    duplicated KV of v under SplitQ.
  * Pad(TS, 0) = 0 (an empty group does not exist); TS_q(n) = the smallest
    tile of the tile set >= n, else the largest; TS_c = 64.
  * The ">=" tie of the algorithm assigns 1.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass
class PlannerOptions:
    gamma: int = 64                      # intermediate-result weight
    beta: int = 0                        # optional SplitQ duplicate-KV weight
    ts_q_set: tuple = (16, 64, 128)      # query tile sizes (multi-stage tiling)
    ts_c: int = 64                       # context tile size
    mma_min_rows: int = 1                # rows per kv head to use tensor cores
    force_path: int = 0                  # 0 by rows, 1 CUDA cores, 2 tensor cores
    kv_tile_tokens: int = 64             # chunk granularity (tokens)
    split_tokens: int = 0                # chunk length (tokens); <= 0: no split
    edges: tuple | None = field(default=None)  # force an assignment (tests)


def children_lists(parent):
    n = len(parent)
    ch = [[] for _ in range(n)]
    root = -1
    for v in range(n):
        p = int(parent[v])
        if p < 0:
            root = v
        else:
            ch[p].append(v)
    return root, ch  # children in ascending id by construction


def subtree_rows(parent, query_node, r):
    """A[v]: query rows (tokens x r) whose path contains v (Algorithm 1, step 1)."""
    n = len(parent)
    A = [0] * n
    for u in query_node:
        v = int(u)
        while v >= 0:
            A[v] += r
            v = int(parent[v])
    return A


def pad(ts, n):
    """Pad(TS, N) = TS - ((N - 1) % TS + 1), with Pad(TS, 0) = 0."""
    if n == 0:
        return 0
    return ts - ((n - 1) % ts + 1)


def ts_q(n, ts_set):
    for t in sorted(ts_set):
        if t >= n:
            return t
    return max(ts_set)


def cost_pq(nq, length, d, o):
    """C_{P,q}(nQ, len) = Pad(TS_q, nQ) * len * d."""
    return pad(ts_q(nq, o.ts_q_set), nq) * length * d


def cost_pc(nq, length, d, o):
    """C_{P,c}(nQ, len) = nQ * Pad(TS_c, min(len, TS_c)) * d."""
    return nq * pad(o.ts_c, min(length, o.ts_c)) * d


def split_kv_cost(nq_curr, nq_l, len_l, len_v, d, o):
    """C_0: keep l separate; l's rows also stay in v's group (two partials)."""
    return (cost_pq(nq_curr, len_v, d, o) + cost_pc(nq_curr, len_v, d, o)
            + cost_pq(nq_l, len_l, d, o) + cost_pc(nq_l, len_l, d, o)
            + o.gamma * nq_l * d)


def split_q_cost(nq_curr, nq_l, len_l, len_v, d, o):
    """C_1: join l to v; l's group carries v's KV, v's group loses l's rows."""
    rest = nq_curr - nq_l
    c = (cost_pq(rest, len_v, d, o) + cost_pc(rest, len_v, d, o)
         + cost_pq(nq_l, len_l + len_v, d, o) + cost_pc(nq_l, len_l + len_v, d, o))
    if rest > 0:
        c += o.beta * len_v * d
    return c


def greedy_edges(parent, node_kv_len, A, d, o: PlannerOptions):
    """Algorithm 1: BFS over nodes, decide every edge v -> l greedily.

    Returns (edge, L, rows): edge[l] in {0, 1} (root: 0), L the cumulative
    context lengths after the pass, rows[v] = nQ_curr left at v.
    """
    root, ch = children_lists(parent)
    n = len(parent)
    L = [int(x) for x in node_kv_len]
    edge = [0] * n
    rows = [0] * n
    queue = [root]
    head = 0
    while head < len(queue):
        v = queue[head]
        head += 1
        nq_curr = A[v]
        len_v = L[v]
        for l in ch[v]:
            nq_l, len_l = A[l], L[l]
            if o.edges is not None:
                take = int(o.edges[l]) == 1
            else:
                c0 = split_kv_cost(nq_curr, nq_l, len_l, len_v, d, o)
                c1 = split_q_cost(nq_curr, nq_l, len_l, len_v, d, o)
                take = c0 >= c1
            if take:
                edge[l] = 1
                nq_curr -= nq_l
                L[l] = len_l + len_v
            else:
                edge[l] = 0
            queue.append(l)
        rows[v] = nq_curr
    return edge, L, rows, queue


def plan_groups(parent, node_kv_len, query_node, query_kv_end, edge, bfs_order):
    """Groups(VT(T, f)): one group per virtual node that keeps query tokens.

    A group of node v carries the KV chain of v and its ancestors joined by
    1-edges (root first) and the query tokens of v's subtree that no 1-edge
    child took.  For each token, ``vis`` is how many span positions it sees:
    the whole span, or for a token of v itself the span up to its own causal
    end.
    """
    n = len(parent)
    # token -> the groups it belongs to: nodes x on its path with x == u or
    # edge(next on path) == 0.
    members = [[] for _ in range(n)]
    for t, u in enumerate(query_node):
        u = int(u)
        x = u
        child = -1
        while x >= 0:
            if x == u or edge[child] == 0:
                members[x].append(t)
            child = x
            x = int(parent[x])
    groups = []
    for v in bfs_order:
        toks = sorted(members[v])
        if not toks:
            continue
        chain = [v]
        x = v
        while edge[x] == 1 and parent[x] >= 0:
            x = int(parent[x])
            chain.append(x)
        chain.reverse()
        span = sum(int(node_kv_len[a]) for a in chain)
        lv = int(node_kv_len[v])
        vis = [span - lv + int(query_kv_end[t]) if int(query_node[t]) == v else span
               for t in toks]
        groups.append({"node": v, "chain": chain, "span": span, "tokens": toks,
                       "vis": vis})
    return groups


def group_blocks(group, node_kv_len, node_page_offsets, node_pages, page_size):
    """The group's KV span as blocks: (page, span position, valid slots)."""
    blocks = []
    pos = 0
    for a in group["chain"]:
        n = int(node_kv_len[a])
        p0 = int(node_page_offsets[a])
        for i in range((n + page_size - 1) // page_size):
            blocks.append((int(node_pages[p0 + i]), pos + i * page_size,
                           min(page_size, n - i * page_size)))
        pos += n
    return blocks


def _ceil(a, b):
    return -(-a // b)


def split_chunks(n_blocks, chunk_blocks, tile_blocks):
    """The long-context split of one group span (FastTree review page,
    "GPU高效的长上下文分割": a span longer than the threshold is cut into
    chunks that run as separate work, and their partial results are merged).
    Reading taken: a span of at most ``chunk_blocks`` blocks stays whole; a
    longer one is cut into k = ceil(n / chunk) equal chunks, each rounded up
    to a whole KV tile, the last one shorter.  Returns [[lo, hi), ...] in
    blocks of the span."""
    if n_blocks <= chunk_blocks:
        return [[0, n_blocks]]
    k = _ceil(n_blocks, chunk_blocks)
    cb = _ceil(_ceil(n_blocks, k), tile_blocks) * tile_blocks
    return [[s, min(n_blocks, s + cb)] for s in range(0, n_blocks, cb)]


def build_plan(parent, node_kv_len, node_page_offsets, node_pages, page_size,
               query_node, query_kv_end, n_q_heads, n_kv_heads, d,
               o: PlannerOptions | None = None):
    """The plan's decisions that the pages define, in canonical form: the
    edge assignment (Algorithm 1), the groups of the virtual tree with their
    KV chains, tokens and visible ends, rows and path, the chunks of each
    group span for the given chunk length, and each token's partial count
    (one per chunk of every group it belongs to)."""
    o = o or PlannerOptions()
    r = n_q_heads // n_kv_heads
    A = subtree_rows(parent, query_node, r)
    edge, L, rows, bfs = greedy_edges(parent, node_kv_len, A, d, o)
    groups = plan_groups(parent, node_kv_len, query_node, query_kv_end, edge, bfs)
    tile_blocks = o.kv_tile_tokens // page_size
    chunk = None
    if o.split_tokens > 0:
        chunk = _ceil(_ceil(o.split_tokens, page_size), tile_blocks) * tile_blocks
    for g in groups:
        g["blocks"] = group_blocks(g, node_kv_len, node_page_offsets, node_pages,
                                   page_size)
        g["rows"] = len(g["tokens"]) * r
        assert g["rows"] == rows[g["node"]]
        assert g["span"] == L[g["node"]]
        # path (spec: tensor cores once a group's stacked query rows
        # make an MMA tile worth issuing; the threshold is an option)
        if o.force_path == 1:
            g["path"] = "simt"
        elif o.force_path == 2:
            g["path"] = "mma"
        else:
            g["path"] = "mma" if g["rows"] >= o.mma_min_rows else "simt"
        nb = len(g["blocks"])
        g["chunks"] = split_chunks(nb, chunk, tile_blocks) if chunk else [[0, nb]]
    nq = len(query_node)
    count = [0] * nq
    for g in groups:
        for t in g["tokens"]:
            count[t] += len(g["chunks"])
    return {
        "edges": edge,
        "groups": [{k: g[k] for k in ("node", "chain", "span", "tokens", "vis",
                                      "rows", "path", "chunks")}
                   for g in groups],
        "partials": count,
        "_blocks": [g["blocks"] for g in groups],
    }


def plan_cost(parent, node_kv_len, A, d, edge, o: PlannerOptions):
    """Proxy cost of a whole assignment: the same components, summed over the
    groups the assignment makes (padding of every group plus gamma per row
    that gets an extra partial).  Used to compare the greedy result with the
    best assignment found by brute force on small trees."""
    root, ch = children_lists(parent)
    n = len(parent)
    L = [int(x) for x in node_kv_len]
    rows = list(A)
    order = [root]
    head = 0
    while head < len(order):
        v = order[head]
        head += 1
        for l in ch[v]:
            if edge[l] == 1:
                rows[v] -= A[l]
                L[l] += L[v]
            order.append(l)
    total = 0
    for v in range(n):
        total += cost_pq(rows[v], L[v], d, o) + cost_pc(rows[v], L[v], d, o)
        if v != root and edge[v] == 0:
            total += o.gamma * A[v] * d
    return total
