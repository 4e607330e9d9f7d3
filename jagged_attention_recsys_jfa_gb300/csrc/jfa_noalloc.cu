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
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return jfa::cuda_fail(e, "jfa_forward_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return jfa::cuda_fail(cudaErrorInvalidDevice, "jfa_forward_noalloc: device index");
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t es = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (es != cudaSuccess) return jfa::cuda_fail(es, "jfa_forward_noalloc: cudaGetSymbolAddress");
    if (p == nullptr) return jfa::cuda_fail(cudaErrorInvalidSymbol, "jfa_forward_noalloc: scratch address");
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
  // The planner rewrites everything the forward kernels read from the scratch (item
  // counts, claim counters, work list, tensor maps, scaled bias) at the start of each
  // call, so the previous call's contents need no clearing.  The status word is the
  // exception: the planner only sets it when an error is found (compare-and-swap from 0)
  // and nothing here reads or clears it, so in this shared array the first device-side
  // error stays latched for the life of the process.  No kernel reads the word (aborts
  // travel through per-CTA shared memory), so a latched error changes no result; callers
  // of this entry point simply get no device-side error report.
  return jfa_forward(q, k, v, q_offsets, kv_offsets, B, H, d, total_q, total_kv, bias, scale, causal, out, lse,
                     ws, kNoAllocScratchBytes, stream);
}
