// The library's C ABI (declared in include/jfa.h): host-side argument checks,
// workspace layout, tensor-map templates and the launch sequence.  No device
// memory is allocated here; every kernel is enqueued on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "jfa_internal.h"

namespace jfa {
namespace {
thread_local int g_last_launches = 0;
// query tiles up to which a sequence's backward takes the non-sequence-parallel pass
std::atomic<int> g_nsp_max_tiles{kNspDefaultMaxTiles};
bool nsp_enabled() { return g_nsp_max_tiles.load(std::memory_order_relaxed) >= 2; }
thread_local char g_last_error[256] = "";
}  // namespace

// Record which CUDA call failed (readable through jfa_last_error) and map it to JFA_ERR_CUDA.
jfa_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return JFA_ERR_CUDA;
}

namespace {
#define JFA_CHECK_LAUNCH(call, where)            \
  do {                                           \
    cudaError_t e_ = (call);                     \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

// ---- optional per-kernel event timing (benchmarks)
struct TimingRec {
  int kind;
  cudaEvent_t start, stop;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<TimingRec> g_timing;

// ---- optional developer tracing (one kernel kind at a time)
std::mutex g_trace_mu;
TraceBuf g_trace = {nullptr, 0};
int g_trace_kind = -1;

struct KernelTimer {
  int kind;
  cudaStream_t stream;
  cudaEvent_t start = nullptr, stop = nullptr;
  bool on;
  KernelTimer(int k, cudaStream_t s) : kind(k), stream(s) {
    {
      std::lock_guard<std::mutex> g(g_timing_mu);
      on = g_timing_on;
    }
    if (on && cudaEventCreate(&start) == cudaSuccess && cudaEventCreate(&stop) == cudaSuccess) {
      cudaEventRecord(start, stream);
    } else {
      on = false;
    }
  }
  ~KernelTimer() {
    if (!on) return;
    cudaEventRecord(stop, stream);
    std::lock_guard<std::mutex> g(g_timing_mu);
    g_timing.push_back(TimingRec{kind, start, stop});
  }
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// SM count of the current device.  Also binds the device's primary context to the
// calling thread (cudaSetDevice initialises it), which the driver-level tensor-map
// encoder needs on threads that have made no CUDA call yet (e.g. autograd workers).
int sm_count() {
  int dev = 0, n = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cuda_fail(e, "device query");
    return 0;
  }
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whole-tensor template for a bf16 [rows, H*d] row-major tensor: boxes of 64 columns
// (128 bytes, the 128-byte swizzle span) by 128 rows; out-of-bounds elements read as 0.
jfa_status encode_template(CUtensorMap* m, const void* base, int64_t rows, int H, int d) {
  auto fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled entry point not available");
    return JFA_ERR_CUDA;
  }
  const cuuint64_t dims[2] = {cuuint64_t(H) * cuuint64_t(d), cuuint64_t(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {cuuint64_t(H) * cuuint64_t(d) * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled: CUresult %d", int(r));
    return JFA_ERR_CUDA;
  }
  return JFA_OK;
}

jfa_status check_common(int B, int H, int d, int64_t total_q, int64_t total_kv, const jfa_bias* bias,
                        float scale, const int64_t* q_off, const int64_t* kv_off) {
  if (B < 1 || H < 1 || H > 4096 || total_q < 0 || total_kv < 0) return JFA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return JFA_ERR_INVALID_ARG;
  if (!q_off || !kv_off) return JFA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return JFA_ERR_UNSUPPORTED;
  if ((total_q + 1) * int64_t(H) * d > (int64_t(1) << 40)) return JFA_ERR_INVALID_ARG;
  if (bias && bias->kind == 2) {
    if (bias->grad) return JFA_ERR_UNSUPPORTED;
    if (!bias->values || !bias->block_offsets || bias->plane < 0 || !aligned16(bias->values) ||
        (reinterpret_cast<uintptr_t>(bias->block_offsets) & 7u) != 0 ||
        (bias->values_grad && !aligned16(bias->values_grad)))
      return JFA_ERR_INVALID_ARG;
  } else if (bias && bias->kind != 0) {
    if (bias->kind != 1) return JFA_ERR_UNSUPPORTED;
    if (!bias->table || bias->num_buckets < 1 || bias->num_buckets > kMaxBuckets) return JFA_ERR_INVALID_ARG;
    if (!aligned16(bias->table)) return JFA_ERR_INVALID_ARG;
    if (bias->grad && (reinterpret_cast<uintptr_t>(bias->grad) & 3u) != 0) return JFA_ERR_INVALID_ARG;
  }
  return JFA_OK;
}

Problem make_problem(int B, int H, int d, int64_t total_q, int64_t total_kv, const int64_t* q_off,
                     const int64_t* kv_off, const jfa_bias* bias, float scale, int causal) {
  Problem p;
  p.B = B;
  p.H = H;
  p.d = d;
  p.total_q = total_q;
  p.total_kv = total_kv;
  p.q_off = q_off;
  p.kv_off = kv_off;
  p.scale = scale;
  p.causal = causal ? 1 : 0;
  const bool has_bias = bias && bias->kind == 1;
  p.bias_table = has_bias ? bias->table : nullptr;
  p.num_buckets = has_bias ? bias->num_buckets : 0;
  p.center = has_bias ? bias->center : 0;
  p.bias_grad = has_bias ? bias->grad : nullptr;
  const bool has_jbias = bias && bias->kind == 2;
  p.jbias = has_jbias ? bias->values : nullptr;
  p.jb_off = has_jbias ? bias->block_offsets : nullptr;
  p.jb_plane = has_jbias ? bias->plane : 0;
  p.jb_grad = has_jbias ? bias->values_grad : nullptr;
  std::lock_guard<std::mutex> g(g_trace_mu);
  for (int k = 0; k < JFA_NUM_KERNEL_KINDS; ++k) p.trace[k] = (k == g_trace_kind) ? g_trace : TraceBuf{nullptr, 0};
  p.nsp_max_tiles = g_nsp_max_tiles.load(std::memory_order_relaxed);
  return p;
}

jfa_status check_workspace(void* ws, size_t bytes, const WsLayout& L) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || bytes < L.total) return JFA_ERR_WORKSPACE;
  return JFA_OK;
}

}  // namespace
}  // namespace jfa

using namespace jfa;

extern "C" {

size_t jfa_workspace_size(int B, int H, int d, int64_t total_q, int64_t total_kv, int is_backward) {
  if (B < 1 || H < 1 || (d != 64 && d != 128) || total_q < 0 || total_kv < 0) return 0;
  return make_layout(B, H, d, total_q, total_kv, is_backward != 0, nsp_enabled()).total;
}

jfa_status jfa_forward(const void* q, const void* k, const void* v, const int64_t* q_offsets,
                       const int64_t* kv_offsets, int B, int H, int d, int64_t total_q, int64_t total_kv,
                       const jfa_bias* bias, float scale, int causal, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, jfa_stream_t stream) {
  g_last_launches = 0;
  jfa_status st = check_common(B, H, d, total_q, total_kv, bias, scale, q_offsets, kv_offsets);
  if (st != JFA_OK) return st;
  if (total_q > 0 && (!q || !out || !lse || !aligned16(q) || !aligned16(out) || !aligned16(lse)))
    return JFA_ERR_INVALID_ARG;
  if (total_kv > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return JFA_ERR_INVALID_ARG;
  const WsLayout L = make_layout(B, H, d, total_q, total_kv, false);
  if ((st = check_workspace(workspace, workspace_bytes, L)) != JFA_OK) return st;
  const Problem pr = make_problem(B, H, d, total_q, total_kv, q_offsets, kv_offsets, bias, scale, causal);
  const int nsm = sm_count();
  if (nsm <= 0) return JFA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  PlanMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const void* kbase = total_kv > 0 ? k : q;  // k/v maps are never read when there are no keys
  const void* vbase = total_kv > 0 ? v : q;
  const void* qbase = total_q > 0 ? q : kbase;
  if (!qbase) return JFA_ERR_INVALID_ARG;
  if ((st = encode_template(&maps.tmpl[kMapQ], qbase, total_q, H, d)) != JFA_OK) return st;
  if ((st = encode_template(&maps.tmpl[kMapK], kbase, total_kv, H, d)) != JFA_OK) return st;
  if ((st = encode_template(&maps.tmpl[kMapV], vbase, total_kv, H, d)) != JFA_OK) return st;
  maps.base[kMapQ] = qbase;
  maps.base[kMapK] = kbase;
  maps.base[kMapV] = vbase;
  for (int i = 0; i < 3; ++i) {
    maps.row_bytes[i] = uint32_t(H) * uint32_t(d) * 2;
    maps.used[i] = 1;
  }
  {
    KernelTimer t(JFA_KERNEL_PLAN, s);
    JFA_CHECK_LAUNCH(launch_plan(pr, maps, workspace, L, false, nsm, s), "planner launch");
  }
  {
    KernelTimer t(JFA_KERNEL_FORWARD, s);
    JFA_CHECK_LAUNCH(launch_forward(pr, workspace, L, out, lse, nsm, s), "forward launch");
  }
  g_last_launches = 2;
  return JFA_OK;
}

jfa_status jfa_backward(const void* dout, const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const int64_t* q_offsets, const int64_t* kv_offsets, int B, int H,
                        int d, int64_t total_q, int64_t total_kv, const jfa_bias* bias, float scale,
                        int causal, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        jfa_stream_t stream) {
  g_last_launches = 0;
  jfa_status st = check_common(B, H, d, total_q, total_kv, bias, scale, q_offsets, kv_offsets);
  if (st != JFA_OK) return st;
  if (total_q > 0 && (!dout || !q || !out || !lse || !dq || !aligned16(dout) || !aligned16(q) ||
                      !aligned16(out) || !aligned16(lse) || !aligned16(dq)))
    return JFA_ERR_INVALID_ARG;
  if (total_kv > 0 && (!k || !v || !dk || !dv || !aligned16(k) || !aligned16(v) || !aligned16(dk) ||
                       !aligned16(dv)))
    return JFA_ERR_INVALID_ARG;
  // the non-sequence-parallel setting is read once (in pr) for the layout, the lists and the launches
  const Problem pr = make_problem(B, H, d, total_q, total_kv, q_offsets, kv_offsets, bias, scale, causal);
  const bool nsp = pr.nsp_max_tiles >= 2;
  const WsLayout L = make_layout(B, H, d, total_q, total_kv, true, nsp);
  if ((st = check_workspace(workspace, workspace_bytes, L)) != JFA_OK) return st;
  const int nsm = sm_count();
  if (nsm <= 0) return JFA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  PlanMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const void* kbase = total_kv > 0 ? k : (total_q > 0 ? q : nullptr);
  const void* vbase = total_kv > 0 ? v : kbase;
  const void* qbase = total_q > 0 ? q : kbase;
  const void* dobase = total_q > 0 ? dout : kbase;
  if (!qbase) return JFA_ERR_INVALID_ARG;
  if ((st = encode_template(&maps.tmpl[kMapQ], qbase, total_q, H, d)) != JFA_OK) return st;
  if ((st = encode_template(&maps.tmpl[kMapK], kbase, total_kv, H, d)) != JFA_OK) return st;
  if ((st = encode_template(&maps.tmpl[kMapV], vbase, total_kv, H, d)) != JFA_OK) return st;
  if ((st = encode_template(&maps.tmpl[kMapDO], dobase, total_q, H, d)) != JFA_OK) return st;
  maps.base[kMapQ] = qbase;
  maps.base[kMapK] = kbase;
  maps.base[kMapV] = vbase;
  maps.base[kMapDO] = dobase;
  for (int i = 0; i < kNumMapSlots; ++i) {
    maps.row_bytes[i] = uint32_t(H) * uint32_t(d) * 2;
    maps.used[i] = 1;
  }
  if (pr.jb_grad)  // pairs no pass visits (hidden by the causal mask) and the row padding read as 0
    JFA_CHECK_LAUNCH(cudaMemsetAsync(pr.jb_grad, 0, size_t(H) * size_t(pr.jb_plane) * 2, s), "bias gradient clear");
  {
    KernelTimer t(JFA_KERNEL_PLAN, s);
    JFA_CHECK_LAUNCH(launch_plan(pr, maps, workspace, L, true, nsm, s), "planner launch");
  }
  {
    KernelTimer t(JFA_KERNEL_BWD_PREPROCESS, s);
    JFA_CHECK_LAUNCH(launch_bwd_preprocess(pr, dout, out, lse, workspace, L, nsm, s), "backward preprocess launch");
  }
  {
    KernelTimer t(JFA_KERNEL_BWD_DKDV, s);
    JFA_CHECK_LAUNCH(launch_bwd_dkdv(pr, lse, workspace, L, dk, dv, nsm, s), "dK/dV launch");
  }
  {
    KernelTimer t(JFA_KERNEL_BWD_DQ, s);
    JFA_CHECK_LAUNCH(launch_bwd_dq(pr, lse, workspace, L, dq, nsm, s), "dQ launch");
  }
  {
    KernelTimer t(JFA_KERNEL_BWD_FUSED, s);
    JFA_CHECK_LAUNCH(launch_bwd_fused(pr, lse, workspace, L, dq, dk, dv, nsm, s), "fused short-query launch");
  }
  if (nsp) {  // otherwise its list is empty: no sequence is routed to the pass
    KernelTimer t(JFA_KERNEL_BWD_NSP, s);
    JFA_CHECK_LAUNCH(launch_bwd_nsp(pr, lse, workspace, L, dq, dk, dv, nsm, s), "non-sequence-parallel launch");
  }
  g_last_launches = nsp ? 6 : 5;
  return JFA_OK;
}

jfa_status jfa_check_status(void* workspace, jfa_stream_t stream) {
  if (!workspace) return JFA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  JFA_CHECK_LAUNCH(cudaStreamSynchronize(s), "stream synchronize");
  int status = 0;
  JFA_CHECK_LAUNCH(cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost), "status read");
  if (status != 0) JFA_CHECK_LAUNCH(cudaMemset(workspace, 0, sizeof(int)), "status clear");
  return static_cast<jfa_status>(status);
}

const char* jfa_status_string(jfa_status s) {
  switch (s) {
    case JFA_OK: return "ok";
    case JFA_ERR_INVALID_ARG: return "invalid argument";
    case JFA_ERR_UNSUPPORTED: return "unsupported configuration (head_dim must be 64 or 128; bias kind 0 or 1)";
    case JFA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case JFA_ERR_CUDA: return "CUDA runtime or driver call failed";
    case JFA_ERR_BAD_OFFSETS: return "offsets must start at 0, be non-decreasing and end at the row count";
    case JFA_ERR_TIMEOUT: return "a bounded pipeline wait ran out on the device; outputs are unspecified";
  }
  return "unknown status";
}

int jfa_last_launch_count(void) { return g_last_launches; }

const char* jfa_last_error(void) { return g_last_error; }

int jfa_set_nsp_max_tiles(int max_tiles) {
  if (max_tiles < 0) return g_nsp_max_tiles.load();
  if (max_tiles > kNspMaxTiles) return -1;
  return g_nsp_max_tiles.exchange(max_tiles);
}

uint64_t jfa_wait_limit_ns(int64_t planned_tile_pairs, int ctas, int64_t max_item_tile_pairs) {
  return wait_limit_ns(planned_tile_pairs, ctas, max_item_tile_pairs);
}

jfa_status jfa_selftest_wait_timeout(void* workspace, uint64_t timeout_ns, jfa_stream_t stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return JFA_ERR_WORKSPACE;
  if (timeout_ns == 0 || timeout_ns > kWaitTimeoutNs) return JFA_ERR_INVALID_ARG;
  JFA_CHECK_LAUNCH(launch_wait_timeout_selftest(workspace, timeout_ns, reinterpret_cast<cudaStream_t>(stream)),
                   "self-test launch");
  return JFA_OK;
}

jfa_status jfa_trace_configure(void* device_buffer, size_t bytes, int kernel_kind) {
  std::lock_guard<std::mutex> g(g_trace_mu);
  if (!device_buffer || kernel_kind < 0 || kernel_kind >= JFA_NUM_KERNEL_KINDS) {
    g_trace = TraceBuf{nullptr, 0};
    g_trace_kind = -1;
    return JFA_OK;
  }
  const size_t cap = bytes / (sizeof(unsigned long long) * kTraceRoles);
  if (cap == 0 || (reinterpret_cast<uintptr_t>(device_buffer) & 7u) != 0) return JFA_ERR_INVALID_ARG;
  g_trace = TraceBuf{static_cast<unsigned long long*>(device_buffer), int(cap > (1u << 30) ? (1u << 30) : cap)};
  g_trace_kind = kernel_kind;
  return JFA_OK;
}

jfa_status jfa_timing_enable(int on) {
  std::lock_guard<std::mutex> g(g_timing_mu);
  g_timing_on = on != 0;
  return JFA_OK;
}

jfa_status jfa_timing_read(double* ms, int* launches, int n_kinds) {
  std::vector<TimingRec> recs;
  {
    std::lock_guard<std::mutex> g(g_timing_mu);
    recs.swap(g_timing);
  }
  jfa_status st = JFA_OK;
  for (const TimingRec& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      st = JFA_ERR_CUDA;
    else if (r.kind < n_kinds) {
      if (ms) ms[r.kind] += t;
      if (launches) launches[r.kind] += 1;
    }
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  return st;
}

}  // extern "C"
