// The plan object behind tree_attn_plan_t, shared by the translation units
// that implement the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <string>
#include <vector>

#include "kernels.h"
#include "planner.h"

namespace ta {
// The tables the kernels read, laid out as one host image (every section
// 256-byte aligned): tree_attn_plan() copies it to the device once,
// tree_attn_run_static() copies it into its scratch on every call, and
// tree_attn_plan_describe_schedule() prints it.  Offsets are in bytes.
struct TableImage {
  std::vector<uint8_t> bytes;
  size_t off_units = 0, off_blocks = 0, off_gtoks = 0, off_cta = 0, off_merge = 0;
  size_t off_err = 0, off_poff = 0, off_append = 0;
  size_t n_units = 0, n_blocks = 0, n_gtoks = 0, n_cta = 0, n_merge = 0, n_tok = 0;
  int32_t max_count = 0;  // most partials of any query token
};
TableImage build_table_image(const HostPlan& h);
}  // namespace ta

struct tree_attn_plan_s {
  ta::HostPlan hp;
  ta::TableImage img;
  bool host_only = true;
  int device = -1;
  void* dmeta = nullptr;
  size_t meta_bytes = 0;
  void* dwork = nullptr;
  size_t work_bytes = 0;
  const ta::UnitDesc* d_units = nullptr;
  const int2* d_blocks = nullptr;
  const ta::GroupTok* d_gtoks = nullptr;
  const int32_t* d_cta_off = nullptr;
  const ta::MergeItem* d_merge = nullptr;
  int32_t* d_err = nullptr;
  uint16_t* d_part_o = nullptr;  // fp16
  float2* d_part_ml = nullptr;  // {lse (base 2), scale of the stored O}
  int32_t* d_merge_cnt = nullptr;
  size_t merge_cnt_bytes = 0;
  const int32_t* d_tok_poff = nullptr;
  const int32_t* d_append = nullptr;  // per query token: page * 16 + slot of its own KV, or -1
  double plan_ms = 0.0;
  bool profiling = false;
  bool profiled_run = false;
  bool profiled_merge = false;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
};

namespace ta {
// Record the thread-local message returned by tree_attn_last_error().
void set_last_error(const std::string& msg);
}  // namespace ta
