// tree_attn_run_static(): the attention of a plan without any device
// allocation, for callers that may not call cudaMalloc.
//
// Some callers cannot allocate device memory: a plug-in inside a host engine
// that owns every byte of the GPU, or a serving loop that reserved its whole
// memory budget at start-up.  For them this entry point uses one fixed
// scratch array compiled into the library (TREE_ATTN_STATIC_SCRATCH_BYTES),
// and works even with a plan made with host_only = 1, which holds no device
// memory.  Every call copies the plan's table image (built once, when the
// plan was made) into the scratch with one copy, clears the fused merge's
// arrival counters, and runs the same partial-attention and merge kernels as
// tree_attn_run() with their tables and partial results in the scratch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "../../include/tree_attn.h"
#include "kernels.h"
#include "plan_state.h"

namespace ta {
namespace {

constexpr size_t kScratchBytes = TREE_ATTN_STATIC_SCRATCH_BYTES;

// The scratch itself.  Host code must not use this name as a device address
// (on the host it names a stand-in); scratch_base() resolves the address.
static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

// The scratch address is looked up once per device and context: a context
// made anew (after cudaDeviceReset, say) loads the module again, and the
// address is looked up again.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  CUcontext ctx;
  void* addr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on `dev` (the current device).
cudaError_t scratch_base(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get = ctx_get_current();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  CUcontext ctx = nullptr;
  if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  ScratchAddr& a = g_scratch_addr[dev];
  if (!a.addr || !ctx || a.ctx != ctx) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return e;
    if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    a.addr = ptr;
    a.ctx = ctx;
  }
  *out = a.addr;
  return cudaSuccess;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

tree_attn_status fail(tree_attn_status s, const std::string& msg) {
  set_last_error(msg);
  return s;
}

}  // namespace
}  // namespace ta

extern "C" tree_attn_status tree_attn_run_static(tree_attn_plan_t P, const void* q,
                                                 const void* k_pages, const void* v_pages,
                                                 float* out, float* lse, void* stream) {
  using namespace ta;
  set_last_error("");
  if (!P) return fail(TA_ERR_INVALID_ARG, "plan is NULL");
  const HostPlan& h = P->hp;
  const TableImage& img = P->img;
  if (h.nq == 0) return TA_OK;
  if (!q || !out || (h.num_pages > 0 && (!k_pages || !v_pages)))
    return fail(TA_ERR_INVALID_ARG, "q, k_pages, v_pages and out must be non-NULL");
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k_pages, 16) || mis(v_pages, 16) || mis(out, 16) || mis(lse, 4))
    return fail(TA_ERR_ALIGNMENT, "q/k_pages/v_pages/out must be 16-byte aligned, lse 4-byte");

  // ---- scratch layout: the table image, then the partial results (every
  // section 256-byte aligned)
  const size_t np = (size_t)h.n_partials * (size_t)h.hq;
  const size_t o_po = up256(img.bytes.size());
  const size_t o_pml = o_po + up256(np * (size_t)h.d * sizeof(uint16_t));  // fp16 partial O
  const size_t o_cnt = o_pml + up256(np * sizeof(float2));
  const size_t ncnt = h.n_partials ? (size_t)h.nq * (size_t)h.hq : 0;
  const size_t need = o_cnt + up256(ncnt * sizeof(int32_t));
  if (need > kScratchBytes)
    return fail(TA_ERR_UNSUPPORTED,
                "this plan needs " + std::to_string(need) + " bytes of scratch; the static scratch "
                "holds " + std::to_string(kScratchBytes) + " (TREE_ATTN_STATIC_SCRATCH_BYTES); use "
                "tree_attn_run() with a device plan instead");

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  void* basev = nullptr;
  e = scratch_base(dev, &basev);
  if (e != cudaSuccess)
    return fail(TA_ERR_CUDA, std::string("cudaGetSymbolAddress(static scratch): ") +
                                 cudaGetErrorString(e));
  uint8_t* base = static_cast<uint8_t*>(basev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // ---- tables: one copy of the image (its error words are zero), then the
  // fused merge's counters start at zero
  e = cudaMemcpyAsync(base, img.bytes.data(), img.bytes.size(), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("cudaMemcpyAsync: ") + cudaGetErrorString(e));
  if (ncnt) {
    e = cudaMemsetAsync(base + o_cnt, 0, ncnt * sizeof(int32_t), s);
    if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  }

  // ---- the same kernels as tree_attn_run(), tables and partials in the scratch
  AttnParams ap{};
  ap.units = reinterpret_cast<const UnitDesc*>(base + img.off_units);
  ap.blocks = reinterpret_cast<const int2*>(base + img.off_blocks);
  ap.gtoks = reinterpret_cast<const GroupTok*>(base + img.off_gtoks);
  ap.cta_off = reinterpret_cast<const int32_t*>(base + img.off_cta);
  ap.q = static_cast<const uint16_t*>(q);
  ap.k = static_cast<const uint16_t*>(k_pages);
  ap.v = static_cast<const uint16_t*>(v_pages);
  ap.out = out;
  ap.lse = lse;
  ap.part_o = reinterpret_cast<uint16_t*>(base + o_po);
  ap.part_ml = reinterpret_cast<float2*>(base + o_pml);
  ap.err = reinterpret_cast<int32_t*>(base + img.off_err);
  ap.hq = h.hq;
  ap.hkv = h.hkv;
  ap.gqa = h.gqa;
  ap.n_units = (int32_t)img.n_units;
  ap.scale_log2 = h.scale * 1.4426950408889634f;
  ap.wait_timeout_ns = (long long)h.opt.wait_timeout_us * 1000ll;
  ap.debug_stuck_wait = h.opt.debug_stuck_wait;
  ap.merge_cnt = reinterpret_cast<int32_t*>(base + o_cnt);
  ap.tok_poff = reinterpret_cast<const int32_t*>(base + img.off_poff);
  ap.merge_fused = h.opt.merge_mode == 1 ? 1 : 0;
  ap.cta_inline = h.grid <= ta::kInlineCtas ? 1 : 0;
  if (ap.cta_inline)
    for (int c = 0; c <= h.grid; ++c) ap.cta_off_inline[c] = h.cta_off[c];
  e = launch_tree_attention(ap, h.d, h.grid, h.num_pages, h.kv_evict, s);
  if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("partial attention launch: ") + cudaGetErrorString(e));
  if (img.n_merge && !ap.merge_fused) {
    MergeParams mp{};
    mp.items = reinterpret_cast<const MergeItem*>(base + img.off_merge);
    mp.n_items = (int32_t)img.n_merge;
    mp.hq = h.hq;
    mp.max_count = img.max_count;
    mp.part_o = ap.part_o;
    mp.part_ml = ap.part_ml;
    mp.out = out;
    mp.lse = lse;
    e = launch_lse_merge(mp, h.d, s);
    if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("merge launch: ") + cudaGetErrorString(e));
  }
  return TA_OK;
}
