// C ABI of libtreeattn: plan construction, device upload, launches, status.
#include <cuda_runtime.h>

#include <algorithm>

#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>

#include "../../include/tree_attn.h"
#include "kernels.h"
#include "plan_state.h"
#include "planner.h"

namespace {

thread_local std::string g_last_error;

tree_attn_status set_err(tree_attn_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

tree_attn_status cuda_err(cudaError_t e, const char* what) {
  return set_err(TA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

ta::Options to_options(const tree_attn_options* o) {
  ta::Options r;
  if (!o) return r;
  if (o->gamma) r.gamma = o->gamma;
  if (o->beta) r.beta = o->beta;
  if (o->ts_q_set[0]) {
    r.ts_q.clear();
    for (int i = 0; i < 4 && o->ts_q_set[i]; ++i) r.ts_q.push_back(o->ts_q_set[i]);
  }
  if (o->ts_c) r.ts_c = o->ts_c;
  if (o->mma_min_rows) r.mma_min_rows = o->mma_min_rows;
  r.split_tokens = o->split_tokens;
  if (o->min_split_tokens) r.min_split_tokens = o->min_split_tokens;
  if (o->split_waves) r.split_waves = o->split_waves;
  r.num_sms = o->num_sms;  // 0 resolved by the caller
  r.force_path = o->force_path;
  r.host_only = o->host_only;
  if (o->wait_timeout_us) r.wait_timeout_us = o->wait_timeout_us;
  r.debug_stuck_wait = o->debug_stuck_wait;
  r.merge_mode = o->merge_mode;
  r.no_pack = o->no_pack;
  return r;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Lay out every table of the plan in one device buffer and upload it.
tree_attn_status upload(tree_attn_plan_s* P) {
  const ta::HostPlan& h = P->hp;
  std::vector<ta::GroupTok> gt(h.gtok.size());
  for (size_t i = 0; i < gt.size(); ++i)
    gt[i] = {h.gtok[i], h.gvis[i], h.gpbase[i],
             ta::pack_pc_slot(h.gtok[i] >= 0 ? h.pcount[h.gtok[i]] : 0, h.gslot[i])};
  std::vector<int2> blocks(h.blk_page.size());
  for (size_t i = 0; i < blocks.size(); ++i) blocks[i] = make_int2(h.blk_page[i], h.blk_meta[i]);
  std::vector<ta::MergeItem> merge(h.merge_tok.size());
  for (size_t i = 0; i < merge.size(); ++i) {
    int t = h.merge_tok[i];
    merge[i] = {t, h.poff[t], h.pcount[t], 0};
  }
  struct Sec {
    const void* src;
    size_t bytes;
    size_t off;
  };
  Sec secs[8] = {
      {h.units.data(), h.units.size() * sizeof(ta::UnitDesc), 0},
      {blocks.data(), blocks.size() * sizeof(int2), 0},
      {gt.data(), gt.size() * sizeof(ta::GroupTok), 0},
      {h.cta_off.data(), h.cta_off.size() * sizeof(int32_t), 0},
      {merge.data(), merge.size() * sizeof(ta::MergeItem), 0},
      {nullptr, 16 * sizeof(int32_t), 0},  // error word(s)
      {h.poff.data(), h.poff.size() * sizeof(int32_t), 0},
      {h.append_dst.data(), h.append_dst.size() * sizeof(int32_t), 0},
  };
  size_t off = 0;
  for (auto& s : secs) {
    s.off = off;
    off = align_up(off + std::max<size_t>(s.bytes, 16), 256);
  }
  std::vector<uint8_t> host(off, 0);
  for (auto& s : secs)
    if (s.src && s.bytes) std::memcpy(host.data() + s.off, s.src, s.bytes);
  cudaError_t e = cudaMalloc(&P->dmeta, off);
  if (e != cudaSuccess) {
    P->dmeta = nullptr;
    return set_err(TA_ERR_OOM, std::string("cudaMalloc(plan tables): ") + cudaGetErrorString(e));
  }
  P->meta_bytes = off;
  e = cudaMemcpy(P->dmeta, host.data(), off, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_err(e, "cudaMemcpy(plan tables)");
  uint8_t* b = static_cast<uint8_t*>(P->dmeta);
  P->d_units = reinterpret_cast<const ta::UnitDesc*>(b + secs[0].off);
  P->d_blocks = reinterpret_cast<const int2*>(b + secs[1].off);
  P->d_gtoks = reinterpret_cast<const ta::GroupTok*>(b + secs[2].off);
  P->d_cta_off = reinterpret_cast<const int32_t*>(b + secs[3].off);
  P->d_merge = reinterpret_cast<const ta::MergeItem*>(b + secs[4].off);
  P->d_err = reinterpret_cast<int32_t*>(b + secs[5].off);
  P->d_tok_poff = reinterpret_cast<const int32_t*>(b + secs[6].off);
  P->d_append = reinterpret_cast<const int32_t*>(b + secs[7].off);

  const size_t np = (size_t)h.n_partials * h.hq;
  const size_t o_bytes = align_up(np * h.d * sizeof(uint16_t), 256);  // fp16 partial O
  const size_t l_bytes = align_up(np * sizeof(float), 256);
  const size_t c_bytes = h.n_partials ? align_up((size_t)h.nq * h.hq * sizeof(int32_t), 256) : 0;
  P->work_bytes = o_bytes + l_bytes + c_bytes;
  if (P->work_bytes) {
    e = cudaMalloc(&P->dwork, P->work_bytes);
    if (e != cudaSuccess) {
      P->dwork = nullptr;
      return set_err(TA_ERR_OOM, std::string("cudaMalloc(workspace): ") + cudaGetErrorString(e));
    }
    P->d_part_o = static_cast<uint16_t*>(P->dwork);
    P->d_part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(P->dwork) + o_bytes);
    if (c_bytes) {
      P->d_merge_cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(P->dwork) + o_bytes + l_bytes);
      P->merge_cnt_bytes = c_bytes;
      e = cudaMemset(P->d_merge_cnt, 0, c_bytes);
      if (e != cudaSuccess) return cuda_err(e, "cudaMemset(merge counters)");
    }
  }
  return TA_OK;
}

void release(tree_attn_plan_s* P) {
  if (!P) return;
  for (auto& e : P->ev)
    if (e) cudaEventDestroy(e);
  if (P->dmeta || P->dwork) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (P->device >= 0 && cur != P->device) cudaSetDevice(P->device);
    if (P->dmeta) cudaFree(P->dmeta);
    if (P->dwork) cudaFree(P->dwork);
    if (P->device >= 0 && cur >= 0 && cur != P->device) cudaSetDevice(cur);
  }
  delete P;
}

}  // namespace

namespace ta {
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace ta

extern "C" {

void tree_attn_options_init(tree_attn_options* o) {
  if (!o) return;
  std::memset(o, 0, sizeof *o);
  ta::Options d;
  o->gamma = d.gamma;
  o->beta = d.beta;
  for (size_t i = 0; i < d.ts_q.size() && i < 4; ++i) o->ts_q_set[i] = d.ts_q[i];
  o->ts_c = d.ts_c;
  o->mma_min_rows = d.mma_min_rows;
  o->split_tokens = d.split_tokens;
  o->min_split_tokens = d.min_split_tokens;
  o->split_waves = d.split_waves;
  o->num_sms = 0;
  o->wait_timeout_us = d.wait_timeout_us;
}

tree_attn_status tree_attn_plan(const int32_t* parent, int32_t n_nodes, const int32_t* node_kv_len,
                                const int32_t* node_page_offsets, const int32_t* node_pages,
                                int32_t page_size, int32_t num_pages, const int32_t* query_node,
                                const int32_t* query_kv_end, int32_t n_query_tokens,
                                int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                float softmax_scale, const tree_attn_options* opts,
                                tree_attn_plan_t* plan_out) {
  g_last_error.clear();
  if (!plan_out) return set_err(TA_ERR_INVALID_ARG, "plan_out is NULL");
  *plan_out = nullptr;
  const auto t0 = std::chrono::steady_clock::now();
  ta::Options opt = to_options(opts);
  if (opts && opts->force_edges) opt.force_edges.assign(opts->force_edges, opts->force_edges + n_nodes);
  const bool host_only = opt.host_only != 0;
  int device = -1;
  if (!host_only) {
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
  }
  if (opt.num_sms <= 0) {
    int sms = 0;
    if (device >= 0 &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) == cudaSuccess &&
        sms > 0)
      opt.num_sms = sms;
    else
      opt.num_sms = 152;
  }
  tree_attn_plan_s* P = new (std::nothrow) tree_attn_plan_s();
  if (!P) return set_err(TA_ERR_OOM, "host allocation of the plan failed");
  std::string err;
  tree_attn_status st;
  try {
    st = ta::build_host_plan(parent, n_nodes, node_kv_len, node_page_offsets, node_pages,
                             page_size, num_pages, query_node, query_kv_end, n_query_tokens,
                             n_q_heads, n_kv_heads, head_dim, softmax_scale, opt, &P->hp, &err);
  } catch (const std::bad_alloc&) {
    st = TA_ERR_OOM;
    err = "host allocation failed while planning";
  }
  if (st != TA_OK) {
    delete P;
    return set_err(st, err);
  }
  P->host_only = host_only;
  P->device = device;
  if (!host_only) {
    st = upload(P);
    if (st != TA_OK) {
      std::string m = g_last_error;
      release(P);
      return set_err(st, m);
    }
  }
  P->plan_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  *plan_out = P;
  return TA_OK;
}

tree_attn_status tree_attn_append_kv(tree_attn_plan_t P, const void* k_new, const void* v_new,
                                     void* k_pages, void* v_pages, void* stream) {
  g_last_error.clear();
  if (!P) return set_err(TA_ERR_INVALID_ARG, "plan is NULL");
  if (P->host_only) return set_err(TA_ERR_HOST_ONLY_PLAN, "plan was made with host_only = 1");
  const ta::HostPlan& h = P->hp;
  if (h.nq == 0) return TA_OK;
  if (!k_new || !v_new || !k_pages || !v_pages)
    return set_err(TA_ERR_INVALID_ARG, "k_new, v_new, k_pages and v_pages must be non-NULL");
  auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (mis(k_new) || mis(v_new) || mis(k_pages) || mis(v_pages))
    return set_err(TA_ERR_ALIGNMENT, "k_new, v_new, k_pages and v_pages must be 16-byte aligned");
  cudaError_t e = ta::launch_append_kv(static_cast<const uint16_t*>(k_new),
                                       static_cast<const uint16_t*>(v_new), P->d_append, h.nq,
                                       h.hkv, h.d, static_cast<uint16_t*>(k_pages),
                                       static_cast<uint16_t*>(v_pages),
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_err(e, "append launch");
  return TA_OK;
}

tree_attn_status tree_attn_run(tree_attn_plan_t P, const void* q, const void* k_pages,
                               const void* v_pages, float* out, float* lse, void* stream) {
  g_last_error.clear();
  if (!P) return set_err(TA_ERR_INVALID_ARG, "plan is NULL");
  if (P->host_only) return set_err(TA_ERR_HOST_ONLY_PLAN, "plan was made with host_only = 1");
  const ta::HostPlan& h = P->hp;
  if (h.nq == 0) return TA_OK;
  if (!q || !out || (h.num_pages > 0 && (!k_pages || !v_pages)))
    return set_err(TA_ERR_INVALID_ARG, "q, k_pages, v_pages and out must be non-NULL");
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k_pages, 16) || mis(v_pages, 16) || mis(out, 16) || mis(lse, 4))
    return set_err(TA_ERR_ALIGNMENT, "q/k_pages/v_pages/out must be 16-byte aligned, lse 4-byte");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ta::AttnParams ap{};
  ap.units = P->d_units;
  ap.blocks = P->d_blocks;
  ap.gtoks = P->d_gtoks;
  ap.cta_off = P->d_cta_off;
  ap.q = static_cast<const uint16_t*>(q);
  ap.k = static_cast<const uint16_t*>(k_pages);
  ap.v = static_cast<const uint16_t*>(v_pages);
  ap.out = out;
  ap.lse = lse;
  ap.part_o = P->d_part_o;
  ap.part_lse = P->d_part_lse;
  ap.err = P->d_err;
  ap.hq = h.hq;
  ap.hkv = h.hkv;
  ap.gqa = h.gqa;
  ap.n_units = (int32_t)h.units.size();
  ap.scale_log2 = h.scale * 1.4426950408889634f;
  ap.wait_timeout_ns = (long long)h.opt.wait_timeout_us * 1000ll;
  ap.debug_stuck_wait = h.opt.debug_stuck_wait;
  ap.merge_cnt = P->d_merge_cnt;
  ap.tok_poff = P->d_tok_poff;
  ap.merge_fused = h.opt.merge_mode == 1 ? 1 : 0;
  ap.cta_inline = h.grid <= ta::kInlineCtas ? 1 : 0;
  if (ap.cta_inline)
    for (int c = 0; c <= h.grid; ++c) ap.cta_off_inline[c] = h.cta_off[c];
  cudaError_t e;
  if (P->profiling) {
    e = cudaEventRecord(P->ev[0], s);
    if (e != cudaSuccess) return cuda_err(e, "cudaEventRecord");
  }
  e = ta::launch_tree_attention(ap, h.d, h.grid, h.num_pages, s);
  if (e != cudaSuccess) return cuda_err(e, "partial attention launch");
  if (P->profiling) {
    e = cudaEventRecord(P->ev[1], s);
    if (e != cudaSuccess) return cuda_err(e, "cudaEventRecord");
  }
  if (!h.merge_tok.empty() && !ap.merge_fused) {
    ta::MergeParams mp{};
    mp.items = P->d_merge;
    mp.n_items = (int32_t)h.merge_tok.size();
    mp.hq = h.hq;
    mp.max_count = h.pcount.empty() ? 0 : *std::max_element(h.pcount.begin(), h.pcount.end());
    mp.part_o = P->d_part_o;
    mp.part_lse = P->d_part_lse;
    mp.out = out;
    mp.lse = lse;
    e = ta::launch_lse_merge(mp, h.d, s);
    if (e != cudaSuccess) return cuda_err(e, "merge launch");
    if (P->profiling) {
      e = cudaEventRecord(P->ev[2], s);
      if (e != cudaSuccess) return cuda_err(e, "cudaEventRecord");
    }
  }
  if (P->profiling) {
    P->profiled_run = true;
    P->profiled_merge = !h.merge_tok.empty() && !ap.merge_fused;
  }
  return TA_OK;
}

tree_attn_status tree_attn_profile_enable(tree_attn_plan_t P, int32_t enable) {
  g_last_error.clear();
  if (!P) return set_err(TA_ERR_INVALID_ARG, "plan is NULL");
  if (P->host_only) return set_err(TA_ERR_HOST_ONLY_PLAN, "plan was made with host_only = 1");
  if (enable) {
    for (auto& ev : P->ev)
      if (!ev) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) {
          ev = nullptr;
          return cuda_err(e, "cudaEventCreate");
        }
      }
  }
  P->profiling = enable != 0;
  P->profiled_run = false;
  return TA_OK;
}

tree_attn_status tree_attn_profile_read(tree_attn_plan_t P, float* partial_ms, float* merge_ms) {
  g_last_error.clear();
  if (!P) return set_err(TA_ERR_INVALID_ARG, "plan is NULL");
  if (!P->profiled_run) return set_err(TA_ERR_INVALID_ARG, "no profiled run to read");
  cudaEvent_t last = P->profiled_merge ? P->ev[2] : P->ev[1];
  cudaError_t e = cudaEventSynchronize(last);
  if (e != cudaSuccess) return cuda_err(e, "cudaEventSynchronize");
  float a = 0.f, b = 0.f;
  e = cudaEventElapsedTime(&a, P->ev[0], P->ev[1]);
  if (e != cudaSuccess) return cuda_err(e, "cudaEventElapsedTime");
  if (P->profiled_merge) {
    e = cudaEventElapsedTime(&b, P->ev[1], P->ev[2]);
    if (e != cudaSuccess) return cuda_err(e, "cudaEventElapsedTime");
  }
  if (partial_ms) *partial_ms = a;
  if (merge_ms) *merge_ms = b;
  return TA_OK;
}

tree_attn_status tree_attn_device_status(tree_attn_plan_t P, void* stream, int32_t* code) {
  g_last_error.clear();
  if (!P || !code) return set_err(TA_ERR_INVALID_ARG, "plan or code is NULL");
  *code = TA_DEVERR_NONE;
  if (P->host_only) return set_err(TA_ERR_HOST_ONLY_PLAN, "plan was made with host_only = 1");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_err(e, "stream synchronize");
  int32_t w[2] = {0, 0};
  e = cudaMemcpy(w, P->d_err, sizeof w, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_err(e, "read device status");
  e = cudaMemset(P->d_err, 0, sizeof w);
  if (e != cudaSuccess) return cuda_err(e, "clear device status");
  *code = w[0];
  if (w[0] != TA_DEVERR_NONE && P->d_merge_cnt) {
    // an aborted run can leave merge counters part-way: start them afresh
    e = cudaMemset(P->d_merge_cnt, 0, P->merge_cnt_bytes);
    if (e != cudaSuccess) return cuda_err(e, "clear merge counters");
  }
  if (w[0] != TA_DEVERR_NONE)
    return set_err(TA_ERR_DEVICE, "kernel reported device error " + std::to_string(w[0]) +
                                      " (detail " + std::to_string(w[1]) + ")");
  return TA_OK;
}

tree_attn_status tree_attn_plan_describe(tree_attn_plan_t P, char* buf, size_t cap, size_t* needed) {
  g_last_error.clear();
  if (!P) return set_err(TA_ERR_INVALID_ARG, "plan is NULL");
  std::string s = ta::describe_json(P->hp);
  if (needed) *needed = s.size() + 1;
  if (!buf || cap < s.size() + 1) return set_err(TA_ERR_BUFFER_TOO_SMALL, "describe buffer too small");
  std::memcpy(buf, s.c_str(), s.size() + 1);
  return TA_OK;
}

tree_attn_status tree_attn_plan_get_stats(tree_attn_plan_t P, tree_attn_plan_stats* st) {
  g_last_error.clear();
  if (!P || !st) return set_err(TA_ERR_INVALID_ARG, "plan or stats is NULL");
  const ta::HostPlan& h = P->hp;
  std::memset(st, 0, sizeof *st);
  st->n_nodes = h.n_nodes;
  st->n_query_tokens = h.nq;
  st->n_q_heads = h.hq;
  st->n_kv_heads = h.hkv;
  st->head_dim = h.d;
  st->n_groups = (int32_t)h.groups.size();
  for (auto& g : h.groups) st->n_groups_mma += g.path == ta::kPathMma;
  st->n_units = (int32_t)h.units.size();
  st->grid = h.grid;
  st->n_merge_tokens = (int32_t)h.merge_tok.size();
  st->n_partials = h.n_partials;
  st->chunk_tokens = h.chunk_blocks * h.page_size;
  st->group_kv_tokens = h.group_kv_tokens;
  st->unique_kv_tokens = h.unique_kv_tokens;
  st->visible_pairs = h.visible_pairs;
  st->workspace_bytes = (int64_t)P->work_bytes;
  st->metadata_bytes = (int64_t)P->meta_bytes;
  st->plan_ms = P->plan_ms;
  return TA_OK;
}

void tree_attn_plan_destroy(tree_attn_plan_t P) { release(P); }

const char* tree_attn_status_string(tree_attn_status s) {
  switch (s) {
    case TA_OK: return "TA_OK";
    case TA_ERR_INVALID_ARG: return "TA_ERR_INVALID_ARG";
    case TA_ERR_NOT_A_TREE: return "TA_ERR_NOT_A_TREE";
    case TA_ERR_PAGE_RANGE: return "TA_ERR_PAGE_RANGE";
    case TA_ERR_UNSUPPORTED: return "TA_ERR_UNSUPPORTED";
    case TA_ERR_ALIGNMENT: return "TA_ERR_ALIGNMENT";
    case TA_ERR_CUDA: return "TA_ERR_CUDA";
    case TA_ERR_OOM: return "TA_ERR_OOM";
    case TA_ERR_DEVICE: return "TA_ERR_DEVICE";
    case TA_ERR_HOST_ONLY_PLAN: return "TA_ERR_HOST_ONLY_PLAN";
    case TA_ERR_BUFFER_TOO_SMALL: return "TA_ERR_BUFFER_TOO_SMALL";
  }
  return "TA_ERR_UNKNOWN";
}

const char* tree_attn_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
