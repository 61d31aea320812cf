/*
 * tree_attn.h -- C ABI of the tree-structured decode attention library
 * (libtreeattn.so, sm_103a).
 *
 * What it computes.  A decoding tree holds a KV cache: the root is the
 * prompt, every other node a span of generated tokens, and each decode query
 * token sits in some node u (DeFT notes page, "Decoding tree definition").
 * Query token t sees every token of u's ancestors, root first, then the
 * first e_t tokens of u itself (DeFT notes page, "Tree attention
 * definition").  For every q head h the output is scaled dot-product attention
 * softmax(s * Q K^T) V over those keys (FastTree review page, "核心公式"),
 * with s = 1/sqrt(d) unless given, and kv head h / (Hq/Hkv) (grouped-query
 * attention, the kv_head_mapping of the TGI FlashDecoding pull request).
 * The log-sum-exp lse = ln sum_j exp(s q.k_j) is returned beside it.
 *
 * How.  tree_attn_plan() runs on the host: it groups each node's KV with every
 * query that shares it (DeFT notes page, "KV-Guided Tree Split"), assigns
 * every edge 0/1 with the greedy heuristic and cost model of the FastTree
 * review page ("算法1：贪心二元边赋值", "开销模型"), splits long spans to fill
 * the GPU (FastTree review page, "GPU高效的长上下文分割"), and uploads the
 * plan.  tree_attn_run() launches a persistent grouped partial-attention
 * kernel (tensor cores for stacked query rows, CUDA cores for thin groups)
 * and a log-sum-exp merge of partial results (DeFT notes page,
 * "Tree-Topology-Aware Global Reduction Strategy").
 *
 * Conventions.
 *   - All index arrays are int32, host memory, read during the call only (the
 *     plan keeps its own copies).  Variable-length lists use CSR offsets: an
 *     array of n+1 prefix sums starting at 0 (the cu_seqlen convention of the
 *     TGI FlashDecoding pull request).
 *   - Device tensors are caller-owned, contiguous, 16-byte aligned:
 *       q        bf16 [n_query_tokens][n_q_heads][head_dim]
 *       k_pages  bf16 [num_pages][n_kv_heads][page_size][head_dim]
 *       v_pages  bf16 [num_pages][n_kv_heads][page_size][head_dim]
 *       out      fp32 [n_query_tokens][n_q_heads][head_dim]
 *       lse      fp32 [n_query_tokens][n_q_heads] (natural log), may be NULL
 *     Slots of a page past the end of its node are never read into a result
 *     (they may hold anything, NaN included).
 *   - A query whose path holds no visible key gets out = 0, lse = -inf.
 *   - Any finite bf16 values are valid input: partial results are kept in
 *     fp16 divided by a per-row power of two when they would leave fp16's
 *     range, with the divisor stored beside their log-sum-exp.
 *   - Every call returns a status; nothing is thrown across the ABI.  On
 *     failure tree_attn_last_error() describes the cause (thread-local).
 *   - Supported: head_dim in {64, 128}, page_size == 16, n_q_heads a multiple
 *     of n_kv_heads, n_q_heads / n_kv_heads <= 128.
 */
#ifndef TREE_ATTN_H_
#define TREE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tree_attn_plan_s* tree_attn_plan_t; /* opaque, library-owned */

typedef enum {
  TA_OK = 0,
  TA_ERR_INVALID_ARG = 1,    /* null pointer, bad size or count            */
  TA_ERR_NOT_A_TREE = 2,     /* parent[] is not one rooted tree             */
  TA_ERR_PAGE_RANGE = 3,     /* page id or page count out of range          */
  TA_ERR_UNSUPPORTED = 4,    /* head_dim / page_size / head ratio not built */
  TA_ERR_ALIGNMENT = 5,      /* device pointer not 16-byte aligned          */
  TA_ERR_CUDA = 6,           /* a CUDA runtime call failed                  */
  TA_ERR_OOM = 7,            /* device or host allocation failed            */
  TA_ERR_DEVICE = 8,         /* a kernel reported an error (see below)      */
  TA_ERR_HOST_ONLY_PLAN = 9, /* run() on a plan made with host_only = 1     */
  TA_ERR_BUFFER_TOO_SMALL = 10
} tree_attn_status;

/* Planner and launch options.  A zero field means "default" (in brackets);
 * a NULL options pointer means all defaults. */
typedef struct {
  int64_t gamma;            /* [64] weight of an intermediate result per row
                               (the cost model's SplitKVCost_R = gamma*nQ*d;
                               gamma, beta, ts_q_set and ts_c act with
                               cost_model = 1)                               */
  int64_t beta;             /* [0] optional weight of KV duplicated by a join */
  int32_t ts_q_set[4];      /* [16,64,128] query tile sizes of the cost model;
                               zero entries end the list                     */
  int32_t ts_c;             /* [64] context tile size of the cost model      */
  int32_t mma_min_rows;     /* [1] rows per kv head from which a group runs
                               on tensor cores; fewer run on CUDA cores
                               (thin groups are packed four to a tile)      */
  int32_t split_tokens;     /* [0 = automatic] chunk length for splitting
                               long spans; < 0 disables splitting            */
  int32_t min_split_tokens; /* [256] smallest automatic chunk (half of it
                               for thin groups packed by kv head)           */
  int32_t split_waves;      /* [2] automatic split aims at waves x SMs units
                               (thin groups packed by kv head: one unit per
                               CTA, two CTAs per SM)                         */
  int32_t num_sms;          /* [0 = the current device's, else 152]          */
  int32_t force_path;       /* [0 = by rows] 1 = CUDA cores, 2 = tensor cores */
  int32_t host_only;        /* [0] 1: plan on the host only (describe/stats),
                               no device state; run() then fails             */
  int32_t wait_timeout_us;  /* [2000000] limit of every in-kernel wait; a
                               wait that runs out makes the kernel record
                               TA_DEVERR_TIMEOUT and return                   */
  const int8_t* force_edges;/* [NULL = greedy] per node 0/1 (root ignored):
                               use this edge assignment instead             */
  int32_t debug_stuck_wait; /* [0] testing aid: 1 makes every CTA first wait
                               on a barrier that nothing signals, so the
                               kernel must take its timeout path (records
                               TA_DEVERR_TIMEOUT, results undefined)        */
  int32_t merge_mode;       /* [0] 0: a separate merge kernel folds partial
                               results after the partial-attention kernel;
                               1: the unit that writes a row's last partial
                               folds them (no second launch; measured slower
                               on GB300: per-row release fences sit on the
                               compute warps' path)                          */
  int32_t no_pack;          /* [0] 1: never pack thin groups (up to four
                               short groups of one kv head sharing a unit,
                               one page of each per KV tile)                 */
  int32_t cost_model;       /* [0] the cost the planner minimises.  0: a
                               latency model with per-tile, per-unit and
                               per-partial times measured on GB300 (the
                               FastTree review page's objective, "问题形式化",
                               is the plan's latency), used for the edge
                               decisions and the CTA schedule; 1: the pages'
                               padding-and-intermediate-result proxy
                               ("开销模型": gamma, beta, ts_q_set, ts_c).  The
                               chunk length follows split_waves either way */
} tree_attn_options;

/* Sizes of a plan, for logging and roofline accounting. */
typedef struct {
  int32_t n_nodes, n_query_tokens, n_q_heads, n_kv_heads, head_dim;
  int32_t n_groups;           /* context-query groups                        */
  int32_t n_groups_mma;       /* of which on tensor cores                    */
  int32_t n_units;            /* (group, kv head, query tile, chunk) units   */
  int32_t grid;               /* persistent CTAs launched by run()           */
  int32_t n_merge_tokens;     /* query tokens with more than one partial     */
  int64_t n_partials;         /* partial (O, lse) slots per q head           */
  int64_t chunk_tokens;       /* chunk length chosen by the split            */
  int64_t group_kv_tokens;    /* sum of group spans (KV read once per unit)  */
  int64_t unique_kv_tokens;   /* tokens in the tree                          */
  int64_t visible_pairs;      /* sum over query tokens of visible keys       */
  int64_t workspace_bytes;    /* partial results, device                     */
  int64_t metadata_bytes;     /* plan tables, device                         */
  double plan_ms;             /* host time spent in tree_attn_plan()         */
} tree_attn_plan_stats;

/* Device-side error codes read by tree_attn_device_status(). */
enum { TA_DEVERR_NONE = 0, TA_DEVERR_TIMEOUT = 1, TA_DEVERR_BOUNDS = 2 };

/* Fill *o with the defaults spelled out above. */
void tree_attn_options_init(tree_attn_options* o);

/* Build a plan for one tree and one set of decode queries.
 *
 * parent[n_nodes]           parent id, -1 for exactly one root; must form a
 *                           tree (no cycle, every node reaches the root).
 * node_kv_len[n_nodes]      KV tokens per node (>= 0); a node holding the KV
 *                           of its own decode tokens counts them.
 * node_page_offsets[n_nodes+1], node_pages[...]
 *                           CSR block table: node v's tokens sit in order in
 *                           pages node_pages[off[v]..off[v+1]), and
 *                           off[v+1]-off[v] == ceil(len_v / page_size); every
 *                           page id in [0, num_pages).
 * query_node[n_query_tokens]   node of each decode query token.
 * query_kv_end[n_query_tokens] tokens of its own node the query sees, in
 *                           [0, len]; NULL = the whole node.
 * softmax_scale             <= 0 selects 1/sqrt(head_dim).
 * opts                      NULL = defaults.
 * *plan_out                 receives the plan; release it with
 *                           tree_attn_plan_destroy().  Unless host_only, the
 *                           plan owns device memory on the current device
 *                           (tables and the partial-result workspace),
 *                           allocated and filled here (synchronously).
 * Errors: TA_ERR_INVALID_ARG, TA_ERR_NOT_A_TREE, TA_ERR_PAGE_RANGE,
 * TA_ERR_UNSUPPORTED, TA_ERR_CUDA, TA_ERR_OOM; *plan_out is then NULL. */
tree_attn_status tree_attn_plan(
    const int32_t* parent, int32_t n_nodes, const int32_t* node_kv_len,
    const int32_t* node_page_offsets, const int32_t* node_pages,
    int32_t page_size, int32_t num_pages, const int32_t* query_node,
    const int32_t* query_kv_end, int32_t n_query_tokens, int32_t n_q_heads,
    int32_t n_kv_heads, int32_t head_dim, float softmax_scale,
    const tree_attn_options* opts, tree_attn_plan_t* plan_out);

/* Run the attention of a plan on `stream` (a cudaStream_t; NULL = the legacy
 * default stream).  Asynchronous: no allocation and no host synchronisation.
 * Device pointers as in the conventions above; q, k_pages, v_pages are read,
 * out (and lse if non-NULL) written in full.  One plan may be run any number
 * of times (e.g. once per layer) but by one stream at a time: its workspace
 * is shared by all runs.  The runs of a decode step (one per layer) may be
 * captured into one CUDA graph and replayed.  The first kernel of a run is
 * a programmatic dependent of the stream's previous kernel: its CTAs may be
 * scheduled and set themselves up while that kernel finishes, but they read
 * q, the pages and the plan's workspace, and write out and lse, only once
 * that kernel has completed and its writes are visible (the usual stream
 * order, for the data).  A run's last kernel may in turn let the stream's
 * next kernel be scheduled before it ends; a next kernel launched with
 * programmatic stream serialization must therefore wait for its
 * prerequisite grid (griddepcontrol.wait, cudaGridDependencySynchronize)
 * before it reads out or lse, as such launches require anyway; any other
 * launch sees the usual order.  The current device must be
 * the one the plan was made on.  Errors: TA_ERR_INVALID_ARG (also: another
 * device is current),
 * TA_ERR_ALIGNMENT, TA_ERR_HOST_ONLY_PLAN, TA_ERR_CUDA (launch failure). */
tree_attn_status tree_attn_run(tree_attn_plan_t plan, const void* q,
                               const void* k_pages, const void* v_pages,
                               float* out, float* lse, void* stream);

/* The step before the attention of a decode step: write the key and value
 * of every query token into its own position of the paged cache.  A decode
 * step appends the new tokens' K/V to their leaves before attending, so a
 * node's length counts its query tokens (DeFT notes page, "Tree attention
 * definition": the query's own token is the last one it sees); the TGI
 * FlashDecoding pull request gives every query token its own KV slot.
 * Token t of node u with visible end e (query_kv_end[t], or len_u) owns
 * position e - 1 of u: page node_pages[off[u] + (e - 1) / 16], slot
 * (e - 1) % 16; tokens with e = 0 own none and are skipped.
 *   k_new, v_new      device bf16 [n_query_tokens][n_kv_heads][head_dim]: the
 *                     tokens' keys and values (16-byte aligned), read.
 *   k_pages, v_pages  the page pools of tree_attn_run(); only the tokens'
 *                     positions are written, every kv head.
 * Asynchronous on `stream`, no allocation.  Two tokens at one position leave
 * either's values.  Errors: TA_ERR_INVALID_ARG, TA_ERR_ALIGNMENT,
 * TA_ERR_HOST_ONLY_PLAN (the destinations live in the device plan),
 * TA_ERR_CUDA. */
tree_attn_status tree_attn_append_kv(tree_attn_plan_t plan, const void* k_new,
                                     const void* v_new, void* k_pages, void* v_pages,
                                     void* stream);

/* Size of the scratch array compiled into the library for
 * tree_attn_run_static(): 32 MiB, held on every GPU where that entry point's
 * code is loaded, until the process exits. */
#define TREE_ATTN_STATIC_SCRATCH_BYTES (32u << 20)

/* Run without allocating device memory.  The method's pages have no
 * counterpart for this: it serves callers that may not call cudaMalloc, such
 * as a plug-in whose host engine owns all device memory, or a serving loop
 * whose memory budget was fixed at start-up.  Same arguments, results and
 * asynchrony as tree_attn_run(), and `plan` may be a host_only plan (which
 * holds no device memory), so planning and running allocate nothing on the
 * GPU.  The plan's tables and its partial results go into one static
 * scratch array of TREE_ATTN_STATIC_SCRATCH_BYTES on the current device
 * (whichever device the plan was made on); each call copies the plan's
 * table image (one host-to-device copy, stream-ordered) and clears what
 * must start at zero.
 *   - The image sits in ordinary (pageable) host memory, so the runtime
 *     stages that copy through its own buffer: the call returns once the
 *     copy is staged, and is not fully asynchronous to the host.
 *   - The first call on a device (and again after its context is made
 *     anew) looks up the scratch address on that device.
 *   - Its copy from pageable host memory is not for stream capture: run
 *     this entry point outside a capture (tree_attn_run() captures).
 *   - Every call shares the one array: calls that overlap on the GPU (other
 *     streams, other threads) race and corrupt each other's results.
 *     Serialise them, e.g. on one stream.
 *   - A plan whose tables and partials exceed the scratch is rejected with
 *     TA_ERR_UNSUPPORTED (tree_attn_last_error() gives the size it needs);
 *     nothing is launched.
 *   - In-kernel wait errors of this path are not reported through
 *     tree_attn_device_status().
 * Errors: as tree_attn_run(), plus TA_ERR_UNSUPPORTED (too large) and
 * TA_ERR_CUDA (scratch lookup or copy failed). */
tree_attn_status tree_attn_run_static(tree_attn_plan_t plan, const void* q,
                                      const void* k_pages, const void* v_pages,
                                      float* out, float* lse, void* stream);

/* Wait for `stream`, then read and clear the plan's device error word.
 * *code receives a TA_DEVERR_* value; returns TA_ERR_DEVICE if it is not
 * TA_DEVERR_NONE, TA_ERR_CUDA if the stream reported an error. */
tree_attn_status tree_attn_device_status(tree_attn_plan_t plan, void* stream,
                                         int32_t* code);

/* Kernel timing.  With enable = 1, every later tree_attn_run() of this plan
 * records CUDA events on its stream before and after each of its kernels
 * (the partial-attention pass and the merge pass); enable = 0 stops it.
 * Needs a device plan; events are created here.  Errors: TA_ERR_INVALID_ARG,
 * TA_ERR_HOST_ONLY_PLAN, TA_ERR_CUDA. */
tree_attn_status tree_attn_profile_enable(tree_attn_plan_t plan, int32_t enable);

/* Device durations of the last profiled run, in milliseconds: waits for its
 * last event.  *merge_ms is 0 when the run needed no merge pass.  Either
 * pointer may be NULL.  Errors: TA_ERR_INVALID_ARG (profiling not enabled or
 * nothing run yet), TA_ERR_CUDA. */
tree_attn_status tree_attn_profile_read(tree_attn_plan_t plan, float* partial_ms,
                                        float* merge_ms);

/* Canonical JSON of the plan's decisions: edge assignment, groups (node,
 * KV chain, span, tokens, visible ends, rows, path, query tiles, chunks),
 * partial counts per query token and the unit count.  Writes at most cap
 * bytes including the terminating NUL; *needed (if non-NULL) receives the
 * full size.  Returns TA_ERR_BUFFER_TOO_SMALL if cap is too small. */
tree_attn_status tree_attn_plan_describe(tree_attn_plan_t plan, char* buf,
                                         size_t cap, size_t* needed);

/* Canonical JSON of the tables the kernels of a run read, exactly as they
 * are copied to the device: the work units in schedule order (8 ints each:
 * first row record, kv head, first row, rows, first block, end block,
 * chunk, path flags: 1 tensor cores, 2 slots are kv heads, 4 two phases,
 * 16 a pair unit, 32 K/V no other unit reads), each CTA's unit range
 * (cta_off), the blocks (page,
 * span position * 32 + valid slots, bit 30 the phase of a two-phase unit),
 * the row records (token, visible end, first partial slot, partial count |
 * (slot + 1) << 24), the merge items (token, first slot, count, 0) and each
 * token's first partial slot; kv_evict = 1 when the plan's K/V mostly
 * streams once and its copies carry L2 policies.  For tests and tools that
 * check a schedule;
 * same buffer rules as tree_attn_plan_describe(). */
tree_attn_status tree_attn_plan_describe_schedule(tree_attn_plan_t plan, char* buf,
                                                  size_t cap, size_t* needed);

/* Copy the plan's sizes into *stats. */
tree_attn_status tree_attn_plan_get_stats(tree_attn_plan_t plan,
                                          tree_attn_plan_stats* stats);

/* Release a plan and its device memory (NULL is ignored).  The caller must
 * make sure no run() of the plan is still executing on the GPU. */
void tree_attn_plan_destroy(tree_attn_plan_t plan);

/* Static string naming a status. */
const char* tree_attn_status_string(tree_attn_status s);

/* Thread-local description of the last failure in this thread ("" if none). */
const char* tree_attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TREE_ATTN_H_ */
