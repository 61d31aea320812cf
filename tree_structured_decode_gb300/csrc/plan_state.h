// The plan object behind tree_attn_plan_t, shared by the translation units
// that implement the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <string>

#include "kernels.h"
#include "planner.h"

struct tree_attn_plan_s {
  ta::HostPlan hp;
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
  float* d_part_lse = nullptr;
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
