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
  float* bias_grad;         // [H][num_buckets] fp32 gradient of the bias table (backward), or nullptr
  const void* jbias;        // general jagged bias: bf16 [H][jb_plane], or nullptr
  const int64_t* jb_off;    // its block offsets [B+1]
  int64_t jb_plane;
  void* jb_grad;            // its gradient (backward), bf16 [H][jb_plane], or nullptr
  TraceBuf trace[JFA_NUM_KERNEL_KINDS];  // per kernel kind (JFA_KERNEL_*): developer tracing, buf == nullptr when off
  int nsp_max_tiles;        // backward: query tiles up to which a sequence takes the non-sequence-parallel pass
};

struct PlanMaps {
  CUtensorMap tmpl[kNumMapSlots];  // whole-tensor templates; the planner patches per-sequence copies
  const void* base[kNumMapSlots];  // tensor base pointers (row 0)
  uint32_t row_bytes[kNumMapSlots];
  int used[kNumMapSlots];
};

// Record which CUDA call failed (what jfa_last_error then returns, for the calling thread)
// and return JFA_ERR_CUDA.
jfa_status cuda_fail(cudaError_t e, const char* where);

// setmaxnreg.inc waits until the registers it asks for are free, so a kernel that
// rebalances registers must be launched with the full allocation the split assumes.
// Checked once per kernel before its first launch: a build that lowered the kernel's
// register count is refused (cudaErrorInvalidConfiguration) instead of launched.
template <typename K>
cudaError_t check_launch_registers(K kern, uint32_t launch_regs = kLaunchRegs) {
  static int verdict = -1;  // -1 unknown, 0 ok, 1 refused
  if (verdict < 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    verdict = fa.numRegs >= int(launch_regs) ? 0 : 1;
  }
  return verdict == 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Launch with programmatic stream serialization: the kernel's CTAs may be scheduled while the
// previous kernel on the stream finishes (they take SMs as its CTAs exit), and every kernel
// of this library executes griddepcontrol.wait before its first access to memory that
// earlier work wrote, so the results are those of plain stream order.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Launch the planner: validates offsets, writes per-sequence tensor maps and the
// longest-first work lists for the forward (backward = false) or the two backward passes.
cudaError_t launch_plan(const Problem& p, const PlanMaps& maps, void* ws, const WsLayout& L, bool backward,
                        int num_sms, cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(void* ws, uint64_t timeout_ns, cudaStream_t stream);

cudaError_t launch_forward(const Problem& p, void* ws, const WsLayout& L, void* out, float* lse,
                           int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const Problem& p, const void* dout, const void* out, const float* lse,
                                  void* ws, const WsLayout& L, int num_sms, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const Problem& p, const float* lse, void* ws, const WsLayout& L, void* dk,
                            void* dv, int num_sms, cudaStream_t stream);
cudaError_t launch_bwd_dq(const Problem& p, const float* lse, void* ws, const WsLayout& L, void* dq,
                          int num_sms, cudaStream_t stream);
// Sequences of 2 .. kNspMaxTiles query tiles: one CTA per sequence and head, every tile
// pair once, dQ summed over key tiles in the workspace.
cudaError_t launch_bwd_nsp(const Problem& p, const float* lse, void* ws, const WsLayout& L, void* dq, void* dk,
                           void* dv, int num_sms, cudaStream_t stream);
// Sequences whose queries fit one tile: dQ, dK and dV in one pass over K and V.
cudaError_t launch_bwd_fused(const Problem& p, const float* lse, void* ws, const WsLayout& L, void* dq, void* dk,
                             void* dv, int num_sms, cudaStream_t stream);

}  // namespace jfa
