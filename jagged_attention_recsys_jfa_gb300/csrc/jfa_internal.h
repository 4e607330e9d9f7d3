// Host-side interfaces between the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "jfa_common.cuh"

namespace jfa {

struct Problem {
  int B, H, d;
  int64_t total_q, total_kv;
  const int64_t* q_off;
  const int64_t* kv_off;
  float scale;
  int causal;
  const float* bias_table;  // nullptr = no bias
  int num_buckets, center;
};

struct PlanMaps {
  CUtensorMap tmpl[kNumMapSlots];  // whole-tensor templates; the planner patches per-sequence copies
  const void* base[kNumMapSlots];  // tensor base pointers (row 0)
  uint32_t row_bytes[kNumMapSlots];
  int used[kNumMapSlots];
};

// Launch the planner: validates offsets, writes per-sequence tensor maps and the
// longest-first work lists for the forward (backward = false) or the two backward passes.
cudaError_t launch_plan(const Problem& p, const PlanMaps& maps, void* ws, const WsLayout& L, bool backward,
                        cudaStream_t stream);

cudaError_t launch_forward(const Problem& p, void* ws, const WsLayout& L, void* out, float* lse,
                           int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const Problem& p, const void* dout, const void* out, void* ws,
                                  const WsLayout& L, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const Problem& p, const float* lse, void* ws, const WsLayout& L, void* dk,
                            void* dv, int num_sms, cudaStream_t stream);
cudaError_t launch_bwd_dq(const Problem& p, const float* lse, void* ws, const WsLayout& L, void* dq,
                          int num_sms, cudaStream_t stream);

}  // namespace jfa
