// jfa_forward_noalloc: the forward for callers that cannot allocate device memory.
//
// Some hosts hand a kernel library nothing but its input and output buffers: plugin
// interfaces of inference runtimes and services that run on a fixed, pre-planned
// memory arena.  They cannot call cudaMalloc on their hot path (it can synchronise
// the whole device and breaks the arena's budget), so they cannot provide the
// workspace jfa_forward needs.  This entry point runs the same forward with its
// scratch (work list, per-sequence tensor maps, status word) in a file-scope device
// array instead.
#include <cuda_runtime.h>

#include <mutex>

#include "jfa_internal.h"

namespace {

// Fixed scratch for the no-allocation forward.  Every GPU that loads this library holds
// it until the process exits.  Its size bounds the problems this entry point accepts
// (jfa_workspace_size(..., 0) <= 8 MiB, e.g. B = 4096 sequences, H = 8, 1M query rows).
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
jfa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return JFA_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return JFA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return JFA_OK;
}

}  // namespace

extern "C" jfa_status jfa_forward_noalloc(const void* q, const void* k, const void* v, const int64_t* q_offsets,
                                          const int64_t* kv_offsets, int B, int H, int d, int64_t total_q,
                                          int64_t total_kv, const jfa_bias* bias, float scale, int causal,
                                          void* out, float* lse, jfa_stream_t stream) {
  const size_t need = jfa_workspace_size(B, H, d, total_q, total_kv, 0);
  if (need == 0) return (d == 64 || d == 128) ? JFA_ERR_INVALID_ARG : JFA_ERR_UNSUPPORTED;
  if (need > kNoAllocScratchBytes) return JFA_ERR_WORKSPACE;
  void* ws = nullptr;
  const jfa_status st = scratch_address(&ws);
  if (st != JFA_OK) return st;
  // The planner rewrites everything the forward reads from the scratch (status word,
  // item count, work list, tensor maps, scaled bias) at the start of each call, so
  // the previous call's contents need no clearing.
  return jfa_forward(q, k, v, q_offsets, kv_offsets, B, H, d, total_q, total_kv, bias, scale, causal, out, lse,
                     ws, kNoAllocScratchBytes, stream);
}
