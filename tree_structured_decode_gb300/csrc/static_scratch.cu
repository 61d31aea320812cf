// tree_attn_run_static(): the attention of a plan without any device
// allocation, for callers that may not call cudaMalloc.
//
// Some callers cannot allocate device memory: a plug-in inside a host engine
// that owns every byte of the GPU, or a serving loop that reserved its whole
// memory budget at start-up.  For them this entry point uses one fixed
// scratch array compiled into the library (TREE_ATTN_STATIC_SCRATCH_BYTES),
// and works even with a plan made with host_only = 1, which holds no device
// memory.  Every call copies the plan's tables into the scratch, packs them
// with a small kernel (which also clears the error word), and runs the same
// partial-attention and merge kernels as tree_attn_run() with their tables
// and partial results in the scratch.
#include <cuda_runtime.h>

#include <algorithm>
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

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on `dev` (the current device), looked up once
// per device.
cudaError_t scratch_base(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

// Interleave the plan's flat tables into the records the kernels read, and
// clear the error words.
__global__ void pack_tables(const int32_t* blk_page, const int32_t* blk_meta, int nblk,
                            int2* blocks, const int32_t* gtok, const int32_t* gvis,
                            const int32_t* gpbase, const int32_t* gslot, int ntok, GroupTok* gtoks,
                            const int32_t* merge_tok, const int32_t* poff, const int32_t* pcount,
                            int nmerge, MergeItem* merge, int32_t* err, int32_t* cnt, int ncnt) {
  const int n = max(max(nblk, ntok), max(nmerge, ncnt));
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (i < nblk) blocks[i] = make_int2(blk_page[i], blk_meta[i]);
    if (i < ntok)
      gtoks[i] = GroupTok{gtok[i], gvis[i], gpbase[i],
                          pack_pc_slot(gtok[i] >= 0 ? pcount[gtok[i]] : 0, gslot[i])};
    if (i < ncnt) cnt[i] = 0;  // fused-merge arrival counters start at zero
    if (i < nmerge) {
      const int t = merge_tok[i];
      merge[i] = MergeItem{t, poff[t], pcount[t], 0};
    }
  }
  if (blockIdx.x == 0 && threadIdx.x < 16) err[threadIdx.x] = 0;
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
  if (h.nq == 0) return TA_OK;
  if (!q || !out || (h.num_pages > 0 && (!k_pages || !v_pages)))
    return fail(TA_ERR_INVALID_ARG, "q, k_pages, v_pages and out must be non-NULL");
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k_pages, 16) || mis(v_pages, 16) || mis(out, 16) || mis(lse, 4))
    return fail(TA_ERR_ALIGNMENT, "q/k_pages/v_pages/out must be 16-byte aligned, lse 4-byte");

  // ---- scratch layout (every section 256-byte aligned)
  const size_t nu = h.units.size(), nblk = h.blk_page.size(), ntok = h.gtok.size();
  const size_t nmerge = h.merge_tok.size(), nq = (size_t)h.nq;
  const size_t np = (size_t)h.n_partials * (size_t)h.hq;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up256(bytes ? bytes : 16);
    return o;
  };
  const size_t o_units = take(nu * sizeof(UnitDesc));
  const size_t o_cta = take(h.cta_off.size() * sizeof(int32_t));
  const size_t o_bpage = take(nblk * 4), o_bmeta = take(nblk * 4), o_blocks = take(nblk * 8);
  const size_t o_gtok = take(ntok * 4), o_gvis = take(ntok * 4), o_gpb = take(ntok * 4);
  const size_t o_gslot = take(ntok * 4);
  const size_t o_gtoks = take(ntok * sizeof(GroupTok));
  const size_t o_mtok = take(nmerge * 4), o_poff = take(nq * 4), o_pcnt = take(nq * 4);
  const size_t o_merge = take(nmerge * sizeof(MergeItem));
  const size_t o_err = take(16 * sizeof(int32_t));
  const size_t o_po = take(np * (size_t)h.d * sizeof(uint16_t));  // fp16 partial O
  const size_t o_pl = take(np * sizeof(float));
  const size_t ncnt = h.n_partials ? nq * (size_t)h.hq : 0;
  const size_t o_cnt = take(ncnt * sizeof(int32_t));
  if (off > kScratchBytes)
    return fail(TA_ERR_UNSUPPORTED,
                "this plan needs " + std::to_string(off) + " bytes of scratch; the static scratch "
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

  // ---- tables: host -> scratch, then pack
  struct Copy {
    size_t dst;
    const void* src;
    size_t bytes;
  } copies[] = {
      {o_units, h.units.data(), nu * sizeof(UnitDesc)},
      {o_cta, h.cta_off.data(), h.cta_off.size() * sizeof(int32_t)},
      {o_bpage, h.blk_page.data(), nblk * 4},
      {o_bmeta, h.blk_meta.data(), nblk * 4},
      {o_gtok, h.gtok.data(), ntok * 4},
      {o_gvis, h.gvis.data(), ntok * 4},
      {o_gpb, h.gpbase.data(), ntok * 4},
      {o_gslot, h.gslot.data(), ntok * 4},
      {o_mtok, h.merge_tok.data(), nmerge * 4},
      {o_poff, h.poff.data(), nq * 4},
      {o_pcnt, h.pcount.data(), nq * 4},
  };
  for (const Copy& c : copies) {
    if (!c.bytes) continue;
    e = cudaMemcpyAsync(base + c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("cudaMemcpyAsync: ") + cudaGetErrorString(e));
  }
  const size_t nmax = std::max(std::max(nblk, ntok), std::max(nmerge, ncnt));
  const int pack_blocks = (int)std::min<size_t>(std::max<size_t>((nmax + 255) / 256, 1), 1024);
  pack_tables<<<pack_blocks, 256, 0, s>>>(
      reinterpret_cast<const int32_t*>(base + o_bpage), reinterpret_cast<const int32_t*>(base + o_bmeta),
      (int)nblk, reinterpret_cast<int2*>(base + o_blocks),
      reinterpret_cast<const int32_t*>(base + o_gtok), reinterpret_cast<const int32_t*>(base + o_gvis),
      reinterpret_cast<const int32_t*>(base + o_gpb), reinterpret_cast<const int32_t*>(base + o_gslot),
      (int)ntok,
      reinterpret_cast<GroupTok*>(base + o_gtoks), reinterpret_cast<const int32_t*>(base + o_mtok),
      reinterpret_cast<const int32_t*>(base + o_poff), reinterpret_cast<const int32_t*>(base + o_pcnt),
      (int)nmerge, reinterpret_cast<MergeItem*>(base + o_merge),
      reinterpret_cast<int32_t*>(base + o_err), reinterpret_cast<int32_t*>(base + o_cnt), (int)ncnt);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("table pack launch: ") + cudaGetErrorString(e));

  // ---- the same kernels as tree_attn_run(), tables and partials in the scratch
  AttnParams ap{};
  ap.units = reinterpret_cast<const UnitDesc*>(base + o_units);
  ap.blocks = reinterpret_cast<const int2*>(base + o_blocks);
  ap.gtoks = reinterpret_cast<const GroupTok*>(base + o_gtoks);
  ap.cta_off = reinterpret_cast<const int32_t*>(base + o_cta);
  ap.q = static_cast<const uint16_t*>(q);
  ap.k = static_cast<const uint16_t*>(k_pages);
  ap.v = static_cast<const uint16_t*>(v_pages);
  ap.out = out;
  ap.lse = lse;
  ap.part_o = reinterpret_cast<uint16_t*>(base + o_po);
  ap.part_lse = reinterpret_cast<float*>(base + o_pl);
  ap.err = reinterpret_cast<int32_t*>(base + o_err);
  ap.hq = h.hq;
  ap.hkv = h.hkv;
  ap.gqa = h.gqa;
  ap.n_units = (int32_t)nu;
  ap.scale_log2 = h.scale * 1.4426950408889634f;
  ap.wait_timeout_ns = (long long)h.opt.wait_timeout_us * 1000ll;
  ap.debug_stuck_wait = h.opt.debug_stuck_wait;
  ap.merge_cnt = reinterpret_cast<int32_t*>(base + o_cnt);
  ap.tok_poff = reinterpret_cast<const int32_t*>(base + o_poff);
  ap.merge_fused = h.opt.merge_mode == 1 ? 1 : 0;
  ap.cta_inline = h.grid <= ta::kInlineCtas ? 1 : 0;
  if (ap.cta_inline)
    for (int c = 0; c <= h.grid; ++c) ap.cta_off_inline[c] = h.cta_off[c];
  e = launch_tree_attention(ap, h.d, h.grid, h.num_pages, s);
  if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("partial attention launch: ") + cudaGetErrorString(e));
  if (nmerge && !ap.merge_fused) {
    MergeParams mp{};
    mp.items = reinterpret_cast<const MergeItem*>(base + o_merge);
    mp.n_items = (int32_t)nmerge;
    mp.hq = h.hq;
    mp.max_count = h.pcount.empty() ? 0 : *std::max_element(h.pcount.begin(), h.pcount.end());
    mp.part_o = ap.part_o;
    mp.part_lse = ap.part_lse;
    mp.out = out;
    mp.lse = lse;
    e = launch_lse_merge(mp, h.d, s);
    if (e != cudaSuccess) return fail(TA_ERR_CUDA, std::string("merge launch: ") + cudaGetErrorString(e));
  }
  return TA_OK;
}
