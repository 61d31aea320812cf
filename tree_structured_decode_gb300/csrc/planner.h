// Host planner for tree-structured decode attention.
//
// Turns a decoding tree, its block table and its decode queries into the
// context-query groups, work units and schedule that the kernels execute.
// Grouping follows the KV-guided split of the DeFT notes page ("KV-Guided
// Tree Split": each node's KV grouped with every query that shares it); the
// edge assignment is Algorithm 1 and the cost model of the FastTree review
// page ("算法1：贪心二元边赋值", "开销模型"); long spans are split as in
// "GPU高效的长上下文分割" of the same page.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/tree_attn.h"

namespace ta {

constexpr int kPageSize = 16;
constexpr int kKvTileTokens = 64;                  // one KV tile = 4 pages
constexpr int kBlocksPerTile = kKvTileTokens / kPageSize;
constexpr int kMmaTileRows = 128;                  // tcgen05 M
constexpr int kSimtTileRows = 8;                   // CUDA-core rows per unit
constexpr int kCtasPerSm = 2;                      // co-resident persistent CTAs per SM
// Thin-group packing: up to kPackSlots short groups of one kv head share a
// unit; tile j carries page j of every packed group (one page per slot) and
// each group's rows see only their slot.
constexpr int kPackSlots = 4;
constexpr int kPackMaxBlocks = 8;   // groups of at most 8 pages (128 tokens)
constexpr int kPackMmaRows = 32;    // rows per slot on tensor cores (one warp)
constexpr int kPackSimtRows = 2;    // rows per slot on CUDA cores
static_assert(kPackSlots == kBlocksPerTile, "one page per slot per tile");
constexpr int kPathSimt = 0;
constexpr int kPathMma = 1;
constexpr int kUnitHeads = 2;  // with kPathMma: slot k of the unit is kv head kvh + k
// with kPathMma: a packed unit in two phases; each slot (warp) holds two
// groups of at most 16 rows, phase 0's in lanes 0-15 and phase 1's in lanes
// 16-31, and the unit's tiles carry phase 0's pages, then phase 1's
constexpr int kUnitPhases = 4;
// with kPathMma: a query tile of 33-64 rows held once per kv head of a pair
// (FastTree review page, 高效树结构注意力内核设计: smaller tiles near the
// leaves): rows [64k, 64k + 64) are the tile for kv head kvh + k, and KV
// tile j holds pages 2j and 2j + 1 of the chunk for each of the two heads
constexpr int kUnitPairs = 16;
constexpr int kPairRows = 64;
// every page (and kv head) the unit reads is read by no other unit: its K/V
// copies ask L2 to evict those lines first
constexpr int kUnitReadOnce = 32;
constexpr int kPhasesMinUnitsPerCta = 3;         // two phases only with this many units per CTA
constexpr int kPhaseShift = 30;                  // phase of a packed tile's page record
constexpr int32_t kPosMask = (1 << kPhaseShift) - 1;

struct Options {
  int64_t gamma = 64;
  int64_t beta = 0;
  std::vector<int32_t> ts_q{16, 64, 128};
  int32_t ts_c = 64;
  int32_t mma_min_rows = 1;
  int32_t split_tokens = 0;
  int32_t min_split_tokens = 256;
  int32_t split_waves = 2;
  int32_t num_sms = 152;
  int32_t force_path = 0;
  int32_t host_only = 0;
  int32_t wait_timeout_us = 2000000;
  std::vector<int8_t> force_edges;  // empty = greedy
  int32_t debug_stuck_wait = 0;
  int32_t merge_mode = 0;  // 0 separate merge kernel, 1 fused into the partial kernel
  int32_t no_pack = 0;     // 1: never pack thin groups
  int32_t cost_model = 0;  // 0: the measured latency model, 1: the pages' padding proxy
};

// Measured latency model (the plan objective Latency(Groups(VT(T, f))) of
// the FastTree review page, "问题形式化", with costs measured on GB300).
// Times in thousandths of the period of one 64-token KV tile on a CTA, fitted
// to per-CTA timelines of the partial-attention kernel: a work unit costs
// kLatTile per KV tile plus kLatUnit of start-up and epilogue (the same for
// 64- and 128-row tiles), and a query row's extra partial result costs
// kLatMergeRow (written by the kernel, folded by the merge pass).
constexpr int64_t kLatTile = 1000;
constexpr int64_t kLatUnit = 8200;
constexpr int64_t kLatMergeRow = 29;

// One work unit as the kernels read it (32 bytes, device POD).
struct UnitDesc {
  int32_t tok_off;  // first entry of the group's token list
  int32_t kvh;      // kv head
  int32_t row0;     // first row (token-major, head-minor) of this query tile
  int32_t nrows;    // rows in this tile
  int32_t blk0;     // first block (absolute index into the block list)
  int32_t blk1;     // one past the last block
  int32_t chunk;    // chunk index inside the group (selects the partial slot)
  int32_t path;     // kPathSimt, kPathMma, or kPathMma | kUnitHeads
};

struct GroupInfo {
  int32_t node;
  int32_t chain_off, chain_len;  // into HostPlan::chain_nodes (root first)
  int64_t span;                  // KV tokens of the chain
  int32_t tok_off, ntok;         // into gtok / gvis / gpbase
  int32_t rows;                  // ntok * gqa
  int32_t path;
  int32_t qtiles;
  int32_t blk_off, nblk;         // into blk_page / blk_meta
  int32_t chunk_off, nchunks;    // into chunk_lo / chunk_hi (relative blocks)
};

struct HostPlan {
  // problem
  int32_t n_nodes = 0, nq = 0, hq = 0, hkv = 0, d = 0, gqa = 0;
  int32_t page_size = kPageSize, num_pages = 0;
  float scale = 0.f;
  Options opt;
  // decisions
  std::vector<int8_t> edge;
  std::vector<int64_t> L;
  std::vector<GroupInfo> groups;
  std::vector<int32_t> chain_nodes;
  std::vector<int32_t> gtok, gvis, gpbase;
  std::vector<int32_t> gslot;                // -1, or the page slot of a packed row (tok -1: filler row)
  std::vector<int32_t> blk_page, blk_meta;   // meta = span_pos * 32 + valid
  std::vector<int32_t> chunk_lo, chunk_hi;
  int64_t chunk_blocks = 0;
  std::vector<int32_t> pcount, poff;          // per query token
  std::vector<int32_t> append_dst;            // per query token: page * 16 + slot of its own
                                              // position (visible end - 1), or -1
  int64_t n_partials = 0;
  std::vector<int32_t> merge_tok;             // tokens with >= 2 partials
  std::vector<UnitDesc> units;                // in schedule order (CTA-major)
  std::vector<int32_t> cta_off;               // CTA c runs units [cta_off[c], cta_off[c+1])
  int32_t grid = 0;
  // the plan's K/V mostly streams once: at least 3/4 of its KV tiles are in
  // units flagged kUnitReadOnce, and the kernel's copies carry L2 policies
  // (evict-first for those units, evict-last for the others).  Measured: a
  // plan that re-reads much of its K/V runs slower with the policies, one
  // that streams it once faster.
  bool kv_evict = false;
  // sizes
  int64_t unique_kv_tokens = 0, group_kv_tokens = 0, visible_pairs = 0;
};

// Validate and plan.  On failure returns the status and fills *err.
tree_attn_status build_host_plan(
    const int32_t* parent, int32_t n_nodes, const int32_t* node_kv_len,
    const int32_t* node_page_offsets, const int32_t* node_pages,
    int32_t page_size, int32_t num_pages, const int32_t* query_node,
    const int32_t* query_kv_end, int32_t nq, int32_t hq, int32_t hkv,
    int32_t d, float scale, const Options& opt, HostPlan* plan,
    std::string* err);

// Canonical JSON of the decisions (see tree_attn_plan_describe).
std::string describe_json(const HostPlan& plan);

}  // namespace ta
