// C ABI of libtreeattn: plan construction, device upload, launches, status.
#include <cuda_runtime.h>

#include <algorithm>

#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstdio>
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
  r.cost_model = o->cost_model;
  return r;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Partial-result workspace sizes: O (fp16), {lse, scale} and the fused
// merge's arrival counters.
struct WorkSizes {
  size_t o_bytes, ml_bytes, cnt_bytes;
  size_t total() const { return o_bytes + ml_bytes + cnt_bytes; }
};
WorkSizes work_sizes(const ta::HostPlan& h) {
  const size_t np = (size_t)h.n_partials * h.hq;
  WorkSizes w;
  w.o_bytes = align_up(np * h.d * sizeof(uint16_t), 256);
  w.ml_bytes = align_up(np * sizeof(float2), 256);
  w.cnt_bytes = h.n_partials ? align_up((size_t)h.nq * h.hq * sizeof(int32_t), 256) : 0;
  return w;
}

// Upload the plan's table image and allocate its partial-result workspace.
tree_attn_status upload(tree_attn_plan_s* P) {
  const ta::TableImage& img = P->img;
  const size_t off = img.bytes.size();
  cudaError_t e = cudaMalloc(&P->dmeta, off);
  if (e != cudaSuccess) {
    P->dmeta = nullptr;
    return set_err(TA_ERR_OOM, std::string("cudaMalloc(plan tables): ") + cudaGetErrorString(e));
  }
  P->meta_bytes = off;
  e = cudaMemcpy(P->dmeta, img.bytes.data(), off, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_err(e, "cudaMemcpy(plan tables)");
  uint8_t* b = static_cast<uint8_t*>(P->dmeta);
  P->d_units = reinterpret_cast<const ta::UnitDesc*>(b + img.off_units);
  P->d_blocks = reinterpret_cast<const int2*>(b + img.off_blocks);
  P->d_gtoks = reinterpret_cast<const ta::GroupTok*>(b + img.off_gtoks);
  P->d_cta_off = reinterpret_cast<const int32_t*>(b + img.off_cta);
  P->d_merge = reinterpret_cast<const ta::MergeItem*>(b + img.off_merge);
  P->d_err = reinterpret_cast<int32_t*>(b + img.off_err);
  P->d_tok_poff = reinterpret_cast<const int32_t*>(b + img.off_poff);
  P->d_append = reinterpret_cast<const int32_t*>(b + img.off_append);

  const WorkSizes w = work_sizes(P->hp);
  P->work_bytes = w.total();
  if (P->work_bytes) {
    e = cudaMalloc(&P->dwork, P->work_bytes);
    if (e != cudaSuccess) {
      P->dwork = nullptr;
      return set_err(TA_ERR_OOM, std::string("cudaMalloc(workspace): ") + cudaGetErrorString(e));
    }
    uint8_t* wb = static_cast<uint8_t*>(P->dwork);
    P->d_part_o = reinterpret_cast<uint16_t*>(wb);
    P->d_part_ml = reinterpret_cast<float2*>(wb + w.o_bytes);
    if (w.cnt_bytes) {
      P->d_merge_cnt = reinterpret_cast<int32_t*>(wb + w.o_bytes + w.ml_bytes);
      P->merge_cnt_bytes = w.cnt_bytes;
      e = cudaMemset(P->d_merge_cnt, 0, w.cnt_bytes);
      if (e != cudaSuccess) return cuda_err(e, "cudaMemset(merge counters)");
    }
  }
  return TA_OK;
}

// The plan's device memory and tables belong to the device that was current
// when it was made; launching it from another device would read them there.
tree_attn_status check_device(const tree_attn_plan_s* P) {
  int cur = -1;
  const cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
  if (cur != P->device)
    return set_err(TA_ERR_INVALID_ARG, "the current device (" + std::to_string(cur) +
                                           ") is not the plan's device (" +
                                           std::to_string(P->device) + ")");
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

TableImage build_table_image(const HostPlan& h) {
  TableImage img;
  std::vector<GroupTok> gt(h.gtok.size());
  for (size_t i = 0; i < gt.size(); ++i)
    gt[i] = {h.gtok[i], h.gvis[i], h.gpbase[i],
             pack_pc_slot(h.gtok[i] >= 0 ? h.pcount[h.gtok[i]] : 0, h.gslot[i])};
  std::vector<int2> blocks(h.blk_page.size());
  for (size_t i = 0; i < blocks.size(); ++i) blocks[i] = make_int2(h.blk_page[i], h.blk_meta[i]);
  std::vector<MergeItem> merge(h.merge_tok.size());
  for (size_t i = 0; i < merge.size(); ++i) {
    const int t = h.merge_tok[i];
    merge[i] = {t, h.poff[t], h.pcount[t], 0};
  }
  struct Sec {
    const void* src;
    size_t bytes;
    size_t* off;
  } secs[8] = {
      {h.units.data(), h.units.size() * sizeof(UnitDesc), &img.off_units},
      {blocks.data(), blocks.size() * sizeof(int2), &img.off_blocks},
      {gt.data(), gt.size() * sizeof(GroupTok), &img.off_gtoks},
      {h.cta_off.data(), h.cta_off.size() * sizeof(int32_t), &img.off_cta},
      {merge.data(), merge.size() * sizeof(MergeItem), &img.off_merge},
      {nullptr, 16 * sizeof(int32_t), &img.off_err},  // error word(s), zero
      {h.poff.data(), h.poff.size() * sizeof(int32_t), &img.off_poff},
      {h.append_dst.data(), h.append_dst.size() * sizeof(int32_t), &img.off_append},
  };
  size_t off = 0;
  for (auto& sec : secs) {
    *sec.off = off;
    off = align_up(off + std::max<size_t>(sec.bytes, 16), 256);
  }
  img.bytes.assign(off, 0);
  for (auto& sec : secs)
    if (sec.src && sec.bytes) std::memcpy(img.bytes.data() + *sec.off, sec.src, sec.bytes);
  img.n_units = h.units.size();
  img.n_blocks = blocks.size();
  img.n_gtoks = gt.size();
  img.n_cta = h.cta_off.size();
  img.n_merge = merge.size();
  img.n_tok = (size_t)h.nq;
  img.max_count = h.pcount.empty() ? 0 : *std::max_element(h.pcount.begin(), h.pcount.end());
  return img;
}
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
  try {
    P->img = ta::build_table_image(P->hp);
  } catch (const std::bad_alloc&) {
    delete P;
    return set_err(TA_ERR_OOM, "host allocation failed while building the plan tables");
  }
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
  {
    const tree_attn_status ds = check_device(P);
    if (ds != TA_OK) return ds;
  }
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
  {
    const tree_attn_status ds = check_device(P);
    if (ds != TA_OK) return ds;
  }
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
  ap.part_ml = P->d_part_ml;
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
  e = ta::launch_tree_attention(ap, h.d, h.grid, h.num_pages, h.kv_evict, s);
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
    mp.max_count = P->img.max_count;
    mp.part_o = P->d_part_o;
    mp.part_ml = P->d_part_ml;
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

tree_attn_status tree_attn_plan_describe_schedule(tree_attn_plan_t P, char* buf, size_t cap,
                                                  size_t* needed) {
  g_last_error.clear();
  if (!P) return set_err(TA_ERR_INVALID_ARG, "plan is NULL");
  const ta::TableImage& img = P->img;
  const ta::HostPlan& h = P->hp;
  std::string s;
  s.reserve(64 + img.bytes.size() * 3);
  auto ints = [&](const char* key, size_t off, size_t n_ints) {
    s += ",\"";
    s += key;
    s += "\":[";
    char b[16];
    for (size_t i = 0; i < n_ints; ++i) {
      int32_t v;
      std::memcpy(&v, img.bytes.data() + off + 4 * i, 4);
      std::snprintf(b, sizeof b, i ? ",%d" : "%d", v);
      s += b;
    }
    s += ']';
  };
  s += "{\"hq\":" + std::to_string(h.hq) + ",\"hkv\":" + std::to_string(h.hkv) +
       ",\"gqa\":" + std::to_string(h.gqa) + ",\"d\":" + std::to_string(h.d) +
       ",\"grid\":" + std::to_string(h.grid) + ",\"n_partials\":" + std::to_string(h.n_partials) +
       ",\"num_pages\":" + std::to_string(h.num_pages) + ",\"n_tokens\":" + std::to_string(h.nq) +
       ",\"kv_evict\":" + std::to_string(h.kv_evict ? 1 : 0);
  ints("units", img.off_units, img.n_units * sizeof(ta::UnitDesc) / 4);
  ints("cta_off", img.off_cta, img.n_cta);
  ints("blocks", img.off_blocks, img.n_blocks * 2);
  ints("rows", img.off_gtoks, img.n_gtoks * sizeof(ta::GroupTok) / 4);
  ints("merge", img.off_merge, img.n_merge * sizeof(ta::MergeItem) / 4);
  ints("poff", img.off_poff, img.n_tok);
  s += '}';
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
