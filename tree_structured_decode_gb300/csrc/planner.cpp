// Host planner: validation, greedy edge assignment, groups, long-span split,
// partial-result slots, work units and the persistent schedule.
#include "planner.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <queue>
#include <utility>

namespace ta {
namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Pad(TS, N) = TS - ((N - 1) % TS + 1): rows (or slots) that fill the last
// tile; an empty group has none.
inline int64_t pad(int64_t ts, int64_t n) {
  return n == 0 ? 0 : ts - ((n - 1) % ts + 1);
}

struct CostModel {
  const Options& o;
  int64_t d;
  int64_t hkv;
  int r;
  int64_t ts_q(int64_t n) const {
    int64_t best = -1, mx = 0;
    for (int32_t t : o.ts_q) {
      mx = std::max<int64_t>(mx, t);
      if (t >= n && (best < 0 || t < best)) best = t;
    }
    return best < 0 ? mx : best;
  }
  // C_{P,q}(nQ, len) = Pad(TS_q, nQ) * len * d
  int64_t pq(int64_t nq, int64_t len) const { return pad(ts_q(nq), nq) * len * d; }
  // C_{P,c}(nQ, len) = nQ * Pad(TS_c, min(len, TS_c)) * d
  int64_t pc(int64_t nq, int64_t len) const {
    return nq * pad(o.ts_c, std::min<int64_t>(len, o.ts_c)) * d;
  }
  // Latency of one kv head's share of a group of n rows over len tokens
  // (latency model): tensor-core query tiles of 128 rows, each streaming
  // the span in 64-token tiles as one unit; thin groups (at most one warp's
  // 32 rows) share a unit four ways, one page of each per tile.
  int64_t lat_group(int64_t n, int64_t len) const {
    if (n <= 0) return 0;
    if (!o.no_pack && n <= kPackMmaRows && kPackMmaRows % r == 0 &&
        (len <= (int64_t)kPackMaxBlocks * kPageSize || hkv % kPackSlots == 0))
      return (ceil_div(len, kPageSize) * kLatTile + kLatUnit) / kPackSlots;
    return ceil_div(n, kMmaTileRows) * (ceil_div(len, kKvTileTokens) * kLatTile + kLatUnit);
  }
  // C_0: l keeps its own group; its rows also stay in v's (two partials).
  int64_t split_kv(int64_t nq_curr, int64_t nq_l, int64_t len_l, int64_t len_v) const {
    if (o.cost_model == 0)
      return lat_group(nq_curr, len_v) + lat_group(nq_l, len_l) + kLatMergeRow * nq_l;
    return pq(nq_curr, len_v) + pc(nq_curr, len_v) + pq(nq_l, len_l) +
           pc(nq_l, len_l) + o.gamma * nq_l * d;
  }
  // C_1: l joins v; l's group carries v's KV and takes l's rows.
  int64_t split_q(int64_t nq_curr, int64_t nq_l, int64_t len_l, int64_t len_v) const {
    int64_t rest = nq_curr - nq_l;
    if (o.cost_model == 0) return lat_group(rest, len_v) + lat_group(nq_l, len_l + len_v);
    int64_t c = pq(rest, len_v) + pc(rest, len_v) + pq(nq_l, len_l + len_v) +
                pc(nq_l, len_l + len_v);
    if (rest > 0) c += o.beta * len_v * d;
    return c;
  }
};

tree_attn_status fail(std::string* err, tree_attn_status s, const char* fmt,
                      long long a = 0, long long b = 0, long long c = 0) {
  char buf[256];
  std::snprintf(buf, sizeof buf, fmt, a, b, c);
  if (err) *err = buf;
  return s;
}

}  // namespace

tree_attn_status build_host_plan(
    const int32_t* parent, int32_t n, const int32_t* node_kv_len,
    const int32_t* node_page_offsets, const int32_t* node_pages,
    int32_t page_size, int32_t num_pages, const int32_t* query_node,
    const int32_t* query_kv_end, int32_t nq, int32_t hq, int32_t hkv, int32_t d,
    float scale, const Options& opt, HostPlan* P, std::string* err) {
  // ---------------------------------------------------------------- checks
  if (!P) return fail(err, TA_ERR_INVALID_ARG, "plan_out is NULL");
  if (n < 1) return fail(err, TA_ERR_INVALID_ARG, "n_nodes = %lld < 1", n);
  if (nq < 0) return fail(err, TA_ERR_INVALID_ARG, "n_query_tokens = %lld < 0", nq);
  if (!parent || !node_kv_len || !node_page_offsets || (!node_pages && num_pages > 0) ||
      (nq > 0 && !query_node))
    return fail(err, TA_ERR_INVALID_ARG, "required array is NULL");
  if (d != 64 && d != 128)
    return fail(err, TA_ERR_UNSUPPORTED, "head_dim %lld not in {64, 128}", d);
  if (page_size != kPageSize)
    return fail(err, TA_ERR_UNSUPPORTED, "page_size %lld != 16", page_size);
  if (hq < 1 || hkv < 1 || hq % hkv != 0 || hq / hkv > 128)
    return fail(err, TA_ERR_UNSUPPORTED, "heads %lld/%lld: need Hkv | Hq, Hq/Hkv <= 128",
                hq, hkv);
  if (num_pages < 0) return fail(err, TA_ERR_INVALID_ARG, "num_pages < 0");
  if (opt.ts_q.empty() || opt.ts_c < 1)
    return fail(err, TA_ERR_INVALID_ARG, "empty tile set");
  for (int32_t t : opt.ts_q)
    if (t < 1) return fail(err, TA_ERR_INVALID_ARG, "tile size %lld < 1", t);
  if (!opt.force_edges.empty() && (int64_t)opt.force_edges.size() != n)
    return fail(err, TA_ERR_INVALID_ARG, "force_edges size");

  int root = -1;
  for (int v = 0; v < n; ++v) {
    int p = parent[v];
    if (p == -1) {
      if (root >= 0) return fail(err, TA_ERR_NOT_A_TREE, "two roots: %lld and %lld", root, v);
      root = v;
    } else if (p < 0 || p >= n || p == v) {
      return fail(err, TA_ERR_NOT_A_TREE, "parent[%lld] = %lld out of range", v, p);
    }
    if (node_kv_len[v] < 0)
      return fail(err, TA_ERR_INVALID_ARG, "node_kv_len[%lld] = %lld < 0", v, node_kv_len[v]);
  }
  if (root < 0) return fail(err, TA_ERR_NOT_A_TREE, "no root (parent == -1)");

  // children in ascending id (counting sort by parent)
  std::vector<int32_t> ch_off(n + 1, 0), ch(std::max(n - 1, 0));
  for (int v = 0; v < n; ++v)
    if (v != root) ch_off[parent[v] + 1]++;
  for (int v = 0; v < n; ++v) ch_off[v + 1] += ch_off[v];
  {
    std::vector<int32_t> cur(ch_off.begin(), ch_off.end() - 1);
    for (int v = 0; v < n; ++v)
      if (v != root) ch[cur[parent[v]]++] = v;
  }
  // BFS order; a node never reached lies on a cycle
  std::vector<int32_t> bfs;
  bfs.reserve(n);
  bfs.push_back(root);
  for (size_t h = 0; h < bfs.size(); ++h) {
    int v = bfs[h];
    for (int i = ch_off[v]; i < ch_off[v + 1]; ++i) bfs.push_back(ch[i]);
  }
  if ((int)bfs.size() != n)
    return fail(err, TA_ERR_NOT_A_TREE, "%lld of %lld nodes unreachable from the root (cycle)",
                n - (long long)bfs.size(), n);

  // block table
  if (node_page_offsets[0] != 0)
    return fail(err, TA_ERR_PAGE_RANGE, "node_page_offsets[0] = %lld != 0", node_page_offsets[0]);
  int64_t unique_tokens = 0;
  for (int v = 0; v < n; ++v) {
    int64_t need = ceil_div(node_kv_len[v], page_size);
    int64_t have = (int64_t)node_page_offsets[v + 1] - node_page_offsets[v];
    if (have != need)
      return fail(err, TA_ERR_PAGE_RANGE, "node %lld has %lld pages, needs %lld", v, have, need);
    for (int i = node_page_offsets[v]; i < node_page_offsets[v + 1]; ++i)
      if (node_pages[i] < 0 || node_pages[i] >= num_pages)
        return fail(err, TA_ERR_PAGE_RANGE, "page id %lld of node %lld not in [0, %lld)",
                    node_pages[i], v, num_pages);
    unique_tokens += node_kv_len[v];
  }
  for (int t = 0; t < nq; ++t) {
    int u = query_node[t];
    if (u < 0 || u >= n)
      return fail(err, TA_ERR_INVALID_ARG, "query_node[%lld] = %lld out of range", t, u);
    if (query_kv_end) {
      int e = query_kv_end[t];
      if (e < 0 || e > node_kv_len[u])
        return fail(err, TA_ERR_INVALID_ARG, "query_kv_end[%lld] = %lld not in [0, len]", t, e);
    }
  }

  HostPlan& p = *P;
  p = HostPlan();
  // Each query token's own KV position: the last position it sees in its
  // node (decode appends the token's K/V before attention).
  p.append_dst.assign(nq, -1);
  for (int t = 0; t < nq; ++t) {
    const int u = query_node[t];
    const int e = query_kv_end ? query_kv_end[t] : node_kv_len[u];
    if (e >= 1)
      p.append_dst[t] = node_pages[node_page_offsets[u] + (e - 1) / kPageSize] * kPageSize +
                        (e - 1) % kPageSize;
  }
  p.n_nodes = n;
  p.nq = nq;
  p.hq = hq;
  p.hkv = hkv;
  p.d = d;
  p.gqa = hq / hkv;
  p.page_size = page_size;
  p.num_pages = num_pages;
  p.scale = scale > 0.f ? scale : 1.0f / std::sqrt((float)d);
  p.opt = opt;
  p.unique_kv_tokens = unique_tokens;
  const int r = p.gqa;

  // ------------------------------------------ A[v]: query rows per subtree
  std::vector<int64_t> A(n, 0);
  for (int t = 0; t < nq; ++t) A[query_node[t]] += r;
  for (int i = n - 1; i >= 1; --i) A[parent[bfs[i]]] += A[bfs[i]];

  // ------------------------------------------ Algorithm 1 (greedy, BFS)
  CostModel cm{p.opt, d, hkv, r};
  p.L.assign(n, 0);
  for (int v = 0; v < n; ++v) p.L[v] = node_kv_len[v];
  p.edge.assign(n, 0);
  std::vector<int64_t> rows(n, 0);
  for (int v : bfs) {
    int64_t nq_curr = A[v];
    const int64_t len_v = p.L[v];
    for (int i = ch_off[v]; i < ch_off[v + 1]; ++i) {
      int l = ch[i];
      int64_t nq_l = A[l], len_l = p.L[l];
      bool take;
      if (!opt.force_edges.empty()) {
        take = opt.force_edges[l] == 1;
      } else {
        take = cm.split_kv(nq_curr, nq_l, len_l, len_v) >=
               cm.split_q(nq_curr, nq_l, len_l, len_v);
      }
      if (take) {
        p.edge[l] = 1;
        nq_curr -= nq_l;
        p.L[l] = len_l + len_v;
      }
    }
    rows[v] = nq_curr;
  }

  // ------------------------------------------ groups of the virtual tree
  // token t belongs to the group of x on its path iff x == node(t) or the
  // edge from x to the next node on the path is 0.
  std::vector<int32_t> mem_cnt(n + 1, 0);
  for (int t = 0; t < nq; ++t) {
    int x = query_node[t], c = -1;
    while (x >= 0) {
      if (c < 0 || p.edge[c] == 0) mem_cnt[x + 1]++;
      c = x;
      x = parent[x];
    }
  }
  for (int v = 0; v < n; ++v) mem_cnt[v + 1] += mem_cnt[v];
  std::vector<int32_t> mem(mem_cnt[n]);
  {
    std::vector<int32_t> cur(mem_cnt.begin(), mem_cnt.end() - 1);
    for (int t = 0; t < nq; ++t) {  // ascending t: lists come out sorted
      int x = query_node[t], c = -1;
      while (x >= 0) {
        if (c < 0 || p.edge[c] == 0) mem[cur[x]++] = t;
        c = x;
        x = parent[x];
      }
    }
  }
  const bool force_simt = opt.force_path == 1, force_mma = opt.force_path == 2;
  std::vector<int32_t> chain_tmp;
  for (int v : bfs) {
    int ntok = mem_cnt[v + 1] - mem_cnt[v];
    if (ntok == 0) continue;
    GroupInfo g{};
    g.node = v;
    chain_tmp.clear();
    int x = v;
    chain_tmp.push_back(x);
    while (p.edge[x] == 1 && parent[x] >= 0) {
      x = parent[x];
      chain_tmp.push_back(x);
    }
    std::reverse(chain_tmp.begin(), chain_tmp.end());
    g.chain_off = (int32_t)p.chain_nodes.size();
    g.chain_len = (int32_t)chain_tmp.size();
    p.chain_nodes.insert(p.chain_nodes.end(), chain_tmp.begin(), chain_tmp.end());
    int64_t span = 0;
    g.blk_off = (int32_t)p.blk_page.size();
    for (int a : chain_tmp) {
      int64_t la = node_kv_len[a];
      int pg0 = node_page_offsets[a];
      for (int64_t i = 0; i * page_size < la; ++i) {
        int64_t pos = span + i * page_size;
        int64_t valid = std::min<int64_t>(page_size, la - i * page_size);
        if (pos >= (1ll << 26))
          return fail(err, TA_ERR_UNSUPPORTED, "group span exceeds 2^26 tokens");
        p.blk_page.push_back(node_pages[pg0 + i]);
        p.blk_meta.push_back((int32_t)(pos * 32 + valid));
      }
      span += la;
    }
    g.nblk = (int32_t)p.blk_page.size() - g.blk_off;
    g.span = span;
    if (span != p.L[v])
      return fail(err, TA_ERR_INVALID_ARG, "internal: span %lld != L %lld", span, p.L[v]);
    g.tok_off = (int32_t)p.gtok.size();
    g.ntok = ntok;
    const int64_t lv = node_kv_len[v];
    for (int i = mem_cnt[v]; i < mem_cnt[v + 1]; ++i) {
      int t = mem[i];
      int64_t vis = span;
      if (query_node[t] == v) vis = span - lv + (query_kv_end ? query_kv_end[t] : lv);
      p.gtok.push_back(t);
      p.gvis.push_back((int32_t)vis);
      p.gpbase.push_back(-1);
      p.visible_pairs += vis;
    }
    g.rows = ntok * r;
    if ((int64_t)g.rows != rows[v])
      return fail(err, TA_ERR_INVALID_ARG, "internal: rows %lld != %lld", g.rows, rows[v]);
    g.path = force_simt ? kPathSimt
             : force_mma ? kPathMma
             : (g.rows >= opt.mma_min_rows ? kPathMma : kPathSimt);
    g.qtiles = (int32_t)ceil_div(g.rows, g.path == kPathMma ? kMmaTileRows : kSimtTileRows);
    p.group_kv_tokens += span;
    p.groups.push_back(g);
  }

  // ------------------------------------------ long-span split (chunks)
  int64_t chunk;
  int64_t work = 0;  // page-heads streamed, summed over query tiles
  for (auto& g : p.groups) work += (int64_t)g.nblk * hkv * g.qtiles;
  if (opt.split_tokens < 0) {
    int64_t mx = 1;
    for (auto& g : p.groups) mx = std::max<int64_t>(mx, g.nblk);
    chunk = ceil_div(mx, kBlocksPerTile) * kBlocksPerTile;
  } else if (opt.split_tokens > 0) {
    chunk = ceil_div(ceil_div(opt.split_tokens, page_size), kBlocksPerTile) * kBlocksPerTile;
  } else {
    int64_t target = ceil_div(work, (int64_t)std::max(1, opt.split_waves) * std::max(1, opt.num_sms));
    chunk = std::max(ceil_div(opt.min_split_tokens, page_size),
                     ceil_div(target, kBlocksPerTile) * kBlocksPerTile);
  }
  chunk = std::max<int64_t>(chunk, kBlocksPerTile);
  p.chunk_blocks = chunk;
  // Thin tensor-core groups longer than a packable group run packed by kv
  // head (see the units below): a unit covers four kv heads and one page of
  // each per tile, so its chunks need no tile alignment.  The automatic
  // split sizes them for one unit per CTA (the page-heads of the whole plan
  // over the CTAs, a quarter of that in pages), in near-equal chunks of at
  // least half the minimum split: one long unit per CTA beats two short
  // ones (each pays start-up and epilogue), and equal units leave no CTA
  // with the tail.
  auto head_thin = [&](const GroupInfo& g) {
    return !opt.no_pack && g.path == kPathMma && g.qtiles == 1 && g.rows <= kPackMmaRows &&
           kPackMmaRows % r == 0 && hkv % kPackSlots == 0 && g.nblk > kPackMaxBlocks;
  };
  const int64_t thin_chunk =
      std::max(ceil_div(ceil_div(opt.min_split_tokens, page_size), 2),
               ceil_div(work, (int64_t)kPackSlots * std::max(1, opt.num_sms) * kCtasPerSm));
  for (auto& g : p.groups) {
    g.chunk_off = (int32_t)p.chunk_lo.size();
    int64_t nb = g.nblk;
    int64_t cg = chunk;
    if (opt.split_tokens == 0 && head_thin(g)) {
      const int64_t k = ceil_div(nb, thin_chunk);
      for (int64_t i = 0, s = 0; i < k; ++i) {
        const int64_t len = nb / k + (i < nb % k ? 1 : 0);
        p.chunk_lo.push_back((int32_t)s);
        p.chunk_hi.push_back((int32_t)(s + len));
        s += len;
      }
    } else if (nb <= cg) {
      p.chunk_lo.push_back(0);
      p.chunk_hi.push_back((int32_t)nb);
    } else {
      int64_t k = ceil_div(nb, cg);
      int64_t cb = ceil_div(ceil_div(nb, k), kBlocksPerTile) * kBlocksPerTile;
      for (int64_t s = 0; s < nb; s += cb) {
        p.chunk_lo.push_back((int32_t)s);
        p.chunk_hi.push_back((int32_t)std::min(nb, s + cb));
      }
    }
    g.nchunks = (int32_t)p.chunk_lo.size() - g.chunk_off;
  }

  // ------------------------------------------ partial-result slots
  p.pcount.assign(nq, 0);
  for (auto& g : p.groups)
    for (int i = 0; i < g.ntok; ++i) p.pcount[p.gtok[g.tok_off + i]] += g.nchunks;
  p.poff.assign(nq, -1);
  int64_t np = 0;
  for (int t = 0; t < nq; ++t)
    if (p.pcount[t] >= 2) {
      p.poff[t] = (int32_t)np;
      np += p.pcount[t];
      p.merge_tok.push_back(t);
    }
  p.n_partials = np;
  {
    std::vector<int32_t> cursor(nq, 0);
    for (auto& g : p.groups)
      for (int i = 0; i < g.ntok; ++i) {
        int t = p.gtok[g.tok_off + i];
        if (p.pcount[t] >= 2) {
          p.gpbase[g.tok_off + i] = p.poff[t] + cursor[t];
          cursor[t] += g.nchunks;
        }
      }
  }

  // ------------------------------------------ units and LPT schedule
  p.gslot.assign(p.gtok.size(), -1);
  auto packable = [&](const GroupInfo& g) {
    if (opt.no_pack || g.nchunks != 1 || g.qtiles != 1 || g.nblk < 1 || g.nblk > kPackMaxBlocks)
      return -1;
    if (g.path == kPathMma && g.rows <= kPackMmaRows && kPackMmaRows % r == 0) return (int)kPathMma;
    // CUDA-core groups are not packed: measured slower (fewer, longer units
    // balance worse than the per-unit overhead they save)
    return -1;
  };
  // tensor-core groups of at most half a slot pack two phases to a unit
  auto half_slot = [&](const GroupInfo& g) {
    return g.rows <= kPackMmaRows / 2 && (kPackMmaRows / 2) % r == 0;
  };
  std::vector<int32_t> pack_mma, pack_mma2, pack_simt;  // group indices, in group order
  for (size_t gi = 0; gi < p.groups.size(); ++gi) {
    const int k = packable(p.groups[gi]);
    if (k == kPathMma) (half_slot(p.groups[gi]) ? pack_mma2 : pack_mma).push_back((int32_t)gi);
    if (k == kPathSimt) pack_simt.push_back((int32_t)gi);
  }
  // A tensor-core query tile of 33-64 rows runs as one slot of a pair unit
  // (kUnitPairs): two kv heads of the group share the unit's 128 rows.
  auto tile_rows = [&](const GroupInfo& g, int qt) {
    return std::min(kMmaTileRows, g.rows - qt * kMmaTileRows);
  };
  auto pair_tile = [&](const GroupInfo& g, int qt) {
    const int n = tile_rows(g, qt);
    return !opt.no_pack && g.path == kPathMma && hkv % 2 == 0 && kPairRows % r == 0 &&
           n > kPackMmaRows && n <= kPairRows;
  };
  // Longer thin tensor-core groups are packed by kv head: four kv heads of
  // the group share a unit, slot k holding kv head kvh + k, and KV tile j
  // holds page j of the chunk once per slot.
  for (auto& g : p.groups) {
    if (packable(g) >= 0 || head_thin(g)) continue;
    const int tile = g.path == kPathMma ? kMmaTileRows : kSimtTileRows;
    for (int kvh = 0; kvh < hkv; ++kvh)
      for (int c = 0; c < g.nchunks; ++c)
        for (int qt = 0; qt < g.qtiles; ++qt) {
          if (pair_tile(g, qt)) continue;  // emitted as a pair unit below
          UnitDesc u;
          u.tok_off = g.tok_off;
          u.kvh = kvh;
          u.row0 = qt * tile;
          u.nrows = std::min(tile, g.rows - qt * tile);
          u.blk0 = g.blk_off + p.chunk_lo[g.chunk_off + c];
          u.blk1 = g.blk_off + p.chunk_hi[g.chunk_off + c];
          u.chunk = c;
          u.path = g.path;
          p.units.push_back(u);
        }
  }
  // Packed units: row records laid out slot by slot (slot_rows rows per
  // slot; filler records have tok -1), and an interleaved block list
  // (tile j = page j of each slot's group, zero-valid filler pages past a
  // group's end or for an empty slot).  In two phases, a slot's rows are
  // phase 0's group then phase 1's (half a slot each) and the tiles carry
  // phase 0's pages, then phase 1's, each page record marked with its
  // phase.  Records and blocks do not depend on the kv head, so all kv
  // heads share them.
  auto emit_packs = [&](const std::vector<int32_t>& list, int path, int phases) {
    const int slot_rows = path == kPathMma ? kPackMmaRows : kPackSimtRows;
    const int phase_rows = slot_rows / phases;
    const size_t per_unit = (size_t)kPackSlots * phases;
    for (size_t s0 = 0; s0 < list.size(); s0 += per_unit) {
      const size_t ns = std::min<size_t>(per_unit, list.size() - s0);
      auto grp = [&](int rho, int k) -> const GroupInfo* {
        const size_t i = (size_t)rho * kPackSlots + k;
        return i < ns ? &p.groups[list[s0 + i]] : nullptr;
      };
      const int32_t tok_off = (int32_t)p.gtok.size();
      for (int k = 0; k < kPackSlots; ++k)
        for (int rho = 0; rho < phases; ++rho) {
          const GroupInfo* g = grp(rho, k);
          for (int e = 0; e < phase_rows / r; ++e) {
            if (g && e < g->ntok) {
              p.gtok.push_back(p.gtok[g->tok_off + e]);
              p.gvis.push_back(p.gvis[g->tok_off + e]);
              p.gpbase.push_back(p.gpbase[g->tok_off + e]);
            } else {
              p.gtok.push_back(-1);
              p.gvis.push_back(0);
              p.gpbase.push_back(-1);
            }
            p.gslot.push_back(k);
          }
        }
      const int32_t blk0 = (int32_t)p.blk_page.size();
      const int32_t filler_page = p.blk_page[p.groups[list[s0]].blk_off];
      for (int rho = 0; rho < phases; ++rho) {
        const int32_t mark = phases > 1 ? (int32_t)rho << kPhaseShift : 0;
        int tiles = 0;
        for (int k = 0; k < kPackSlots; ++k)
          if (const GroupInfo* g = grp(rho, k)) tiles = std::max(tiles, g->nblk);
        for (int t = 0; t < tiles; ++t)
          for (int k = 0; k < kPackSlots; ++k) {
            const GroupInfo* g = grp(rho, k);
            if (g && t < g->nblk) {
              p.blk_page.push_back(p.blk_page[g->blk_off + t]);
              p.blk_meta.push_back(p.blk_meta[g->blk_off + t] | mark);
            } else {
              p.blk_page.push_back(filler_page);
              p.blk_meta.push_back(mark);
            }
          }
      }
      const int32_t blk1 = (int32_t)p.blk_page.size();
      for (int kvh = 0; kvh < hkv; ++kvh) {
        UnitDesc u;
        u.tok_off = tok_off;
        u.kvh = kvh;
        u.row0 = 0;
        u.nrows = kPackSlots * slot_rows;
        u.blk0 = blk0;
        u.blk1 = blk1;
        u.chunk = 0;
        u.path = path | (phases > 1 ? kUnitPhases : 0);
        p.units.push_back(u);
      }
    }
  };
  // Two phases halve the units of the short groups; they pay only while the
  // plan keeps enough units to balance the CTAs (at least three per CTA),
  // else the half-slot groups pack one phase, four to a unit, as the others.
  {
    const int64_t others = (int64_t)p.units.size() +
                           hkv * (ceil_div((int64_t)pack_mma.size(), kPackSlots) +
                                  ceil_div((int64_t)pack_simt.size(), kPackSlots));
    const int64_t with_phases = others + hkv * ceil_div((int64_t)pack_mma2.size(), 2 * kPackSlots);
    if (with_phases < (int64_t)kPhasesMinUnitsPerCta * std::max(1, opt.num_sms) * kCtasPerSm) {
      pack_mma.insert(pack_mma.end(), pack_mma2.begin(), pack_mma2.end());
      std::sort(pack_mma.begin(), pack_mma.end());
      pack_mma2.clear();
    }
  }
  emit_packs(pack_mma2, kPathMma, 2);
  emit_packs(pack_mma, kPathMma, 1);
  emit_packs(pack_simt, kPathSimt, 1);
  for (size_t gi = 0; gi < p.groups.size(); ++gi) {
    const GroupInfo& g = p.groups[gi];
    if (!head_thin(g)) continue;
    // row records slot by slot: the group's tokens once per slot
    const int32_t tok_off = (int32_t)p.gtok.size();
    for (int k = 0; k < kPackSlots; ++k)
      for (int e = 0; e < kPackMmaRows / r; ++e) {
        if (e < g.ntok) {
          p.gtok.push_back(p.gtok[g.tok_off + e]);
          p.gvis.push_back(p.gvis[g.tok_off + e]);
          p.gpbase.push_back(p.gpbase[g.tok_off + e]);
        } else {
          p.gtok.push_back(-1);
          p.gvis.push_back(0);
          p.gpbase.push_back(-1);
        }
        p.gslot.push_back(k);
      }
    for (int c = 0; c < g.nchunks; ++c) {
      const int32_t blk0 = (int32_t)p.blk_page.size();
      for (int32_t b = p.chunk_lo[g.chunk_off + c]; b < p.chunk_hi[g.chunk_off + c]; ++b)
        for (int k = 0; k < kPackSlots; ++k) {
          p.blk_page.push_back(p.blk_page[g.blk_off + b]);
          p.blk_meta.push_back(p.blk_meta[g.blk_off + b]);
        }
      const int32_t blk1 = (int32_t)p.blk_page.size();
      for (int kvh = 0; kvh < hkv; kvh += kPackSlots) {
        UnitDesc u;
        u.tok_off = tok_off;
        u.kvh = kvh;
        u.row0 = 0;
        u.nrows = kPackSlots * kPackMmaRows;
        u.blk0 = blk0;
        u.blk1 = blk1;
        u.chunk = c;
        u.path = kPathMma | kUnitHeads;
        p.units.push_back(u);
      }
    }
  }
  // Pair units: row records slot by slot (the tile's rows for kv head kvh,
  // then the same rows for kvh + 1; filler records past the tile's rows),
  // shared by every chunk and head pair; per chunk a block list whose tile j
  // holds pages 2j, 2j + 1 for the first head and again for the second (a
  // zero-valid filler page when the chunk has an odd page count).
  for (auto& g : p.groups) {
    if (packable(g) >= 0 || head_thin(g)) continue;
    for (int qt = 0; qt < g.qtiles; ++qt) {
      if (!pair_tile(g, qt)) continue;
      const int32_t tok_off = (int32_t)p.gtok.size();
      const int t0 = qt * kMmaTileRows / r, nt = tile_rows(g, qt) / r;
      for (int k = 0; k < 2; ++k)
        for (int e = 0; e < kPairRows / r; ++e) {
          if (e < nt) {
            p.gtok.push_back(p.gtok[g.tok_off + t0 + e]);
            p.gvis.push_back(p.gvis[g.tok_off + t0 + e]);
            p.gpbase.push_back(p.gpbase[g.tok_off + t0 + e]);
          } else {
            p.gtok.push_back(-1);
            p.gvis.push_back(0);
            p.gpbase.push_back(-1);
          }
          p.gslot.push_back(k);
        }
      for (int c = 0; c < g.nchunks; ++c) {
        const int32_t lo = p.chunk_lo[g.chunk_off + c], hi = p.chunk_hi[g.chunk_off + c];
        const int32_t blk0 = (int32_t)p.blk_page.size();
        for (int32_t b = lo; b < hi; b += 2)
          for (int k = 0; k < 2; ++k) {
            p.blk_page.push_back(p.blk_page[g.blk_off + b]);
            p.blk_meta.push_back(p.blk_meta[g.blk_off + b]);
            const bool second = b + 1 < hi;
            p.blk_page.push_back(p.blk_page[g.blk_off + (second ? b + 1 : b)]);
            p.blk_meta.push_back(second ? p.blk_meta[g.blk_off + b + 1] : 0);
          }
        const int32_t blk1 = (int32_t)p.blk_page.size();
        for (int kvh = 0; kvh < hkv; kvh += 2) {
          UnitDesc u;
          u.tok_off = tok_off;
          u.kvh = kvh;
          u.row0 = 0;
          u.nrows = 2 * kPairRows;
          u.blk0 = blk0;
          u.blk1 = blk1;
          u.chunk = c;
          u.path = kPathMma | kUnitPairs;
          p.units.push_back(u);
        }
      }
    }
  }
  // Units whose K/V no other unit reads (counted per page and kv head; a
  // pair unit's zero-valid filler pages do not count)
  {
    auto head_of = [&](const UnitDesc& u, int32_t b) {
      const int bb = (b - u.blk0) % kBlocksPerTile;
      return u.kvh + ((u.path & kUnitHeads) ? bb : (u.path & kUnitPairs) ? bb / 2 : 0);
    };
    std::vector<uint8_t> reads((size_t)num_pages * hkv, 0);
    for (const UnitDesc& u : p.units)
      for (int32_t b = u.blk0; b < u.blk1; ++b)
        if (p.blk_meta[b] & 31) {
          uint8_t& c = reads[(size_t)p.blk_page[b] * hkv + head_of(u, b)];
          c = c < 2 ? c + 1 : 2;
        }
    int64_t tiles = 0, once_tiles = 0;
    for (UnitDesc& u : p.units) {
      bool once = true;
      for (int32_t b = u.blk0; b < u.blk1 && once; ++b)
        once = !(p.blk_meta[b] & 31) || reads[(size_t)p.blk_page[b] * hkv + head_of(u, b)] == 1;
      if (once && u.blk1 > u.blk0) u.path |= kUnitReadOnce;
      const int64_t t = ceil_div(u.blk1 - u.blk0, kBlocksPerTile);
      tiles += t;
      once_tiles += (u.path & kUnitReadOnce) ? t : 0;
    }
    p.kv_evict = tiles > 0 && 4 * once_tiles >= 3 * tiles;
  }
  const int64_t nu = (int64_t)p.units.size();
  p.grid = (int32_t)std::min<int64_t>(nu, (int64_t)std::max(1, opt.num_sms) * kCtasPerSm);
  {
    std::vector<int32_t> order(nu);
    for (int64_t i = 0; i < nu; ++i) order[i] = (int32_t)i;
    // blocks streamed plus a fixed start-up and epilogue cost per unit (the
    // latency model: its measured per-tile and per-unit times)
    auto cost = [&](int32_t i) {
      const int64_t nb = p.units[i].blk1 - p.units[i].blk0;
      if (opt.cost_model == 0)
        return (p.units[i].path & kPathMma) ? ceil_div(nb, kBlocksPerTile) * kLatTile + kLatUnit
                                            : (nb + 3) * kLatTile / kBlocksPerTile;
      return nb + ((p.units[i].path & kPathMma) ? 6 : 3);
    };
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return cost(a) > cost(b); });
    using Item = std::pair<int64_t, int32_t>;  // (load, cta), min-heap
    std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
    for (int32_t c = 0; c < p.grid; ++c) heap.push({0, c});
    std::vector<std::vector<int32_t>> lists(p.grid);
    for (int32_t i : order) {
      Item it = heap.top();
      heap.pop();
      lists[it.second].push_back(i);
      heap.push({it.first + cost(i), it.second});
    }
    // store the units CTA-major: CTA c runs units [cta_off[c], cta_off[c+1])
    p.cta_off.assign(p.grid + 1, 0);
    std::vector<UnitDesc> sched;
    sched.reserve(nu);
    for (int32_t c = 0; c < p.grid; ++c) {
      p.cta_off[c + 1] = p.cta_off[c] + (int32_t)lists[c].size();
      for (int32_t i : lists[c]) sched.push_back(p.units[i]);
    }
    p.units.swap(sched);
  }
  return TA_OK;
}

namespace {
void put_list(std::string& s, const int32_t* a, int64_t n) {
  s += '[';
  char b[24];
  for (int64_t i = 0; i < n; ++i) {
    std::snprintf(b, sizeof b, i ? ",%d" : "%d", a[i]);
    s += b;
  }
  s += ']';
}
}  // namespace

std::string describe_json(const HostPlan& p) {
  std::string s;
  s.reserve(1024 + p.gtok.size() * 16);
  char b[64];
  s += "{\"chunk_blocks\":";
  s += std::to_string(p.chunk_blocks);
  s += ",\"edges\":[";
  for (int v = 0; v < p.n_nodes; ++v) {
    std::snprintf(b, sizeof b, v ? ",%d" : "%d", (int)p.edge[v]);
    s += b;
  }
  s += "],\"groups\":[";
  for (size_t gi = 0; gi < p.groups.size(); ++gi) {
    const GroupInfo& g = p.groups[gi];
    if (gi) s += ',';
    s += "{\"chain\":";
    put_list(s, p.chain_nodes.data() + g.chain_off, g.chain_len);
    s += ",\"chunks\":[";
    for (int c = 0; c < g.nchunks; ++c) {
      std::snprintf(b, sizeof b, c ? ",[%d,%d]" : "[%d,%d]", p.chunk_lo[g.chunk_off + c],
                    p.chunk_hi[g.chunk_off + c]);
      s += b;
    }
    std::snprintf(b, sizeof b, "],\"node\":%d,\"path\":\"%s\",\"qtiles\":%d,\"rows\":%d,", g.node,
                  g.path == kPathMma ? "mma" : "simt", g.qtiles, g.rows);
    s += b;
    s += "\"span\":" + std::to_string(g.span) + ",\"tokens\":";
    put_list(s, p.gtok.data() + g.tok_off, g.ntok);
    s += ",\"vis\":";
    put_list(s, p.gvis.data() + g.tok_off, g.ntok);
    s += '}';
  }
  s += "],\"partials\":";
  put_list(s, p.pcount.data(), p.nq);
  s += ",\"units\":" + std::to_string(p.units.size()) + "}";
  return s;
}

}  // namespace ta
