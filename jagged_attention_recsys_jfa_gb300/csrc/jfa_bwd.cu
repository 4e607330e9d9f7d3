// Jagged Flash Attention backward for sm_103a.
//
// The gradients of sum(dO * O) (standard FlashAttention-2 backward, the lineage
// "Jagged Flash Attention (JFA)" builds on) computed in the split scheme of "Four
// generations" item 2 -- no atomics on dQ, dK or dV: every gradient tile has exactly one
// writer.  (The one exception is the optional relative-position table gradient, whose
// per-warp diagonal sums are added into the caller's table with fp32 reductions in L2;
// its last bits can therefore differ between calls, while dQ, dK and dV are
// bit-reproducible.)
//   preprocess   D_i = sum_c dO_ic O_ic                            (HBM-bound)
//   dK/dV pass   one CTA work item per (sequence, head, key tile); loops over the
//                query tiles that see it: S^T = K Q^T, P^T = exp(S^T - lse),
//                dV += P^T dO, dP^T = V dO^T, dS^T = P^T o (dP^T - D), dK += dS^T Q
//   dQ pass      one item per (sequence, head, query tile), the only writer of its
//                dQ tile: S = Q K^T, P, dP = dO V^T, dS = P o (dP - D), dQ += dS K
// Rows past a sequence end arrive as zeros (per-sequence tensor maps); padded query
// rows carry lse = D = 0, so they add nothing to dK/dV, and padded key rows add
// nothing to dQ.  The passes are persistent (grid = #SMs) over longest-first lists and
// warp specialised, 16 warps: warpgroup 0 holds the roles (warp 0 streams tiles with
// TMA, warp 1 issues the tcgen05 MMAs and owns TMEM, warp 2 loads the item's resident
// tiles, warp 3 claims work items and publishes them to the others); warpgroups 1 and 2
// split the 128 columns of each S/dP tile (64 each); warpgroup 3 is the epilogue, which
// drains the finished accumulators from TMEM and writes the gradient rows while the
// compute warpgroups start the next tile.  TMEM: S [0,128), dP [128,256), two d-column
// accumulators from 256.  P and dS are written back as bf16 (over the S / dP columns the
// warpgroup owns at d = 128, in the free columns from 384 at d = 64 in the dK/dV pass) and
// feed the accumulating MMAs straight from TMEM.
#include <cuda_bf16.h>

#include "jfa_internal.h"
#include "sm100_ptx.cuh"
#include "jfa_sched.cuh"

namespace jfa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kRegsLoad = 104, kRegsCompute = 200;
static_assert(reg_split_fits(kRegsLoad, kRegsCompute), "register split exceeds the launch allocation");
// dK/dV pass (512 threads): role warps, compute warpgroups, epilogue warpgroup
constexpr uint32_t kRegsLoadDkdv = 96, kRegsComputeDkdv = 168, kRegsEpiDkdv = 72;
static_assert(reg_split_fits_dkdv(kRegsLoadDkdv, kRegsComputeDkdv, kRegsEpiDkdv),
              "register split exceeds the launch allocation");
// the non-sequence-parallel pass: the epilogue warps also sum and finish the dQ rows
constexpr uint32_t kRegsLoadNsp = 104, kRegsComputeNsp = 160, kRegsEpiNsp = 88;
static_assert(reg_split_fits_dkdv(kRegsLoadNsp, kRegsComputeNsp, kRegsEpiNsp),
              "register split exceeds the launch allocation");
// the fused short-query pass: more issue state in warpgroup 0, lighter compute warps
constexpr uint32_t kRegsLoadFused = 112, kRegsComputeFused = 168, kRegsEpiFused = 64;
static_assert(reg_split_fits_dkdv(kRegsLoadFused, kRegsComputeFused, kRegsEpiFused),
              "register split exceeds the launch allocation");

struct BwdParams {
  const int64_t* q_off;
  const int64_t* kv_off;
  int B, H;
  int64_t total_q, total_kv;
  float scale, scale_log2;
  int causal;
  const float* bias2;  // [H][num_buckets] bias * log2(e), or nullptr
  float* bias_grad;    // [H][num_buckets] gradient of the bias table (cleared by the planner), or nullptr
  int num_buckets, center;
  const __nv_bfloat16* jbias;  // general jagged bias [H][jb_plane], or nullptr
  const int64_t* jb_off;       // its block offsets [B+1]
  int64_t jb_plane;
  __nv_bfloat16* jb_grad;      // its gradient (dK/dV and fused passes), or nullptr
  const CUtensorMap* maps;
  const WorkItem* items;
  const int* n_items;
  int* claim;  // the list's claim counter (zeroed by the planner)
  int* status;
  const uint64_t* wait_ns;  // the planner's item hand-off wait limit for this launch (ns)
  const float* lse2;    // [H][qpad_cap]  -lse * log2(e), padded per sequence to 128 rows
  const float* delta;   // [H][qpad_cap]  -D, same layout
  const int64_t* qpad;  // [B+1] sequence offsets in the padded vectors
  int64_t qpad_cap;
  __nv_bfloat16* g0;   // dK (dK/dV and fused passes) or dQ (dQ pass)
  __nv_bfloat16* g1;   // dV (dK/dV and fused passes)
  __nv_bfloat16* g2;   // dQ (fused and non-sequence-parallel passes)
  float* dqacc;        // non-sequence-parallel pass: fp32 dQ sums [total_q][H][D]
  TraceBuf trace;
};

__device__ __forceinline__ void raise_status(int* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

// ---------------------------------------------------------------- preprocess
// For every query row of the 128-row-padded per-query vectors (every sequence's rows,
// each sequence rounded up to whole tiles): -D_i = -sum_c dO_ic O_ic and -lse_i * log2(e)
// (-inf where lse = -inf, so exp2(s - lse) = 0 for a row that sees no key), for every
// head; zeros on padding rows.  Both are stored negated so the consumers add them with
// packed fp32x2 instructions.  Two kernels, chosen by the width of a token row (H*d):
// - preprocess_kernel (H*d >= 1024): one warp per padded row.  It finds the row's sequence
//   by binary search in the padded offsets, reads the token's whole dO and O rows (H*d
//   contiguous bf16 each, 16-byte chunks across the lanes, all loads and the row's lse
//   values in flight before any reduction), and reduces each head's products within its
//   group of d/8 lanes.  Consecutive warps take consecutive rows, so the reads stream.
// - preprocess_items_kernel (narrower rows): one block per item of the dQ and fused lists,
//   one warp per 16 rows of one head, which keeps enough loads in flight when a token row
//   is only a few hundred bytes.
struct PreParams {
  const int64_t* q_off;
  int B, H;
  int64_t total_q;
  const WorkItem* items;      // dQ list: units are query tiles
  const int* n_items;
  const WorkItem* items2;     // fused list: the sequence's one query tile
  const int* n_items2;
  const WorkItem* items3;     // non-sequence-parallel list: all of the sequence's query tiles
  const int* n_items3;
  const int64_t* qpad;        // [B+1] padded row offsets
  const int64_t* total_qpad;  // qpad[B], written by the planner
  int64_t qpad_cap;
  const __nv_bfloat16* dout;
  const __nv_bfloat16* out;
  const float* lse;
  float* lse2;
  float* delta;
};

template <int D>
__global__ void __launch_bounds__(256) preprocess_items_kernel(const PreParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n1 = *p.n_items, n2 = *p.n_items2, n3 = *p.n_items3;
  for (int idx = blockIdx.x; idx < n1 + n2 + n3; idx += gridDim.x) {
    const bool whole = idx >= n1;  // fused or non-sequence-parallel: every query tile of the sequence
    const WorkItem it = idx < n1 ? p.items[idx] : idx < n1 + n2 ? p.items2[idx - n1] : p.items3[idx - n1 - n2];
    const int64_t qo = p.q_off[it.b];
    const int Lq = int(p.q_off[it.b + 1] - qo);
    const int64_t pad0 = int64_t(it.h) * p.qpad_cap + p.qpad[it.b];
    const int t_lo = whole ? 0 : it.u0, t_hi = whole ? (Lq + kBM - 1) / kBM : it.u1;
    for (int t = t_lo; t < t_hi; ++t) {
      // 8 warps x 16 rows.  A row of one head is D/8 16-byte chunks: a warp covers
      // 32 / (D/8) rows per load, and all of its 16 rows' loads are in flight at once.
      constexpr int kLanesPerRow = D / 8, kRowsPerLoad = 32 / kLanesPerRow, kLoads = 16 / kRowsPerLoad;
      const int sub = lane / kLanesPerRow, chunk = lane % kLanesPerRow;
      float acc[kLoads];
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        const int i = t * kBM + warp * 16 + k * kRowsPerLoad + sub;
        acc[k] = 0.f;
        if (i < Lq) {
          const int64_t e0 = ((qo + i) * p.H + it.h) * int64_t(D);
          const uint4 a = __ldg(reinterpret_cast<const uint4*>(p.dout + e0) + chunk);
          const uint4 c = __ldg(reinterpret_cast<const uint4*>(p.out + e0) + chunk);
          acc[k] = fmaf(bf16lo(a.x), bf16lo(c.x), bf16hi(a.x) * bf16hi(c.x)) +
                   fmaf(bf16lo(a.y), bf16lo(c.y), bf16hi(a.y) * bf16hi(c.y)) +
                   fmaf(bf16lo(a.z), bf16lo(c.z), bf16hi(a.z) * bf16hi(c.z)) +
                   fmaf(bf16lo(a.w), bf16lo(c.w), bf16hi(a.w) * bf16hi(c.w));
        }
      }
#pragma unroll
      for (int o = kLanesPerRow / 2; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < kLoads; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
      }
      if (chunk == 0) {
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
          const int i = t * kBM + warp * 16 + k * kRowsPerLoad + sub;
          float nl2 = 0.f;
          if (i < Lq) {
            const float l = __ldg(p.lse + int64_t(it.h) * p.total_q + qo + i);
            nl2 = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
          }
          p.delta[pad0 + i] = i < Lq ? -acc[k] : 0.f;
          p.lse2[pad0 + i] = nl2;
        }
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256, 4) preprocess_kernel(const PreParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  constexpr int kLanesPerHead = D / 8;  // 16-byte chunks per head row
  constexpr int kLoads = 4;             // chunks per lane in flight (rows of up to 128 chunks per pass)
  const int lane = threadIdx.x & 31;
  const int64_t total = *p.total_qpad;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int nchunks = p.H * kLanesPerHead;
  for (int64_t pr = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; pr < total; pr += nwarps) {
    int lo = 0, hi = p.B;  // the last b with qpad[b] <= pr (qpad[0] = 0 <= pr < qpad[B])
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.qpad + mid) <= pr) lo = mid; else hi = mid;
    }
    const int64_t qo = __ldg(p.q_off + lo);
    const int64_t i = pr - __ldg(p.qpad + lo);
    if (i >= __ldg(p.q_off + lo + 1) - qo) {  // padding row
      for (int h = lane; h < p.H; h += 32) {
        p.delta[int64_t(h) * p.qpad_cap + pr] = 0.f;
        p.lse2[int64_t(h) * p.qpad_cap + pr] = 0.f;
      }
      continue;
    }
    const int64_t row = qo + i;
    const uint4* drow = reinterpret_cast<const uint4*>(p.dout + row * p.H * int64_t(D));
    const uint4* orow = reinterpret_cast<const uint4*>(p.out + row * p.H * int64_t(D));
    for (int c0 = 0; c0 < nchunks; c0 += 32 * kLoads) {
      // this pass covers heads [h0, h0 + 32 * kLoads / kLanesPerHead): lane t fetches head
      // h0 + t's lse with the row loads, handed to the storing lanes by shuffle
      const int h0 = c0 / kLanesPerHead;
      const float l_own = h0 + lane < p.H ? __ldg(p.lse + int64_t(h0 + lane) * p.total_q + row) : 0.f;
      uint4 a[kLoads], c[kLoads];
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        const int ch = c0 + 32 * k + lane;
        if (ch < nchunks) {
          a[k] = __ldg(drow + ch);
          c[k] = __ldg(orow + ch);
        }
      }
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        const int ch0 = c0 + 32 * k;  // warp-uniform
        if (ch0 >= nchunks) break;
        const int ch = ch0 + lane;
        float acc = 0.f;
        if (ch < nchunks)
          acc = fmaf(bf16lo(a[k].x), bf16lo(c[k].x), bf16hi(a[k].x) * bf16hi(c[k].x)) +
                fmaf(bf16lo(a[k].y), bf16lo(c[k].y), bf16hi(a[k].y) * bf16hi(c[k].y)) +
                fmaf(bf16lo(a[k].z), bf16lo(c[k].z), bf16hi(a[k].z) * bf16hi(c[k].z)) +
                fmaf(bf16lo(a[k].w), bf16lo(c[k].w), bf16hi(a[k].w) * bf16hi(c[k].w));
#pragma unroll
        for (int o = kLanesPerHead / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        const int h = ch / kLanesPerHead;
        const float l = __shfl_sync(0xffffffffu, l_own, (h - h0) & 31);
        if (ch < nchunks && lane % kLanesPerHead == 0) {
          p.delta[int64_t(h) * p.qpad_cap + pr] = -acc;
          p.lse2[int64_t(h) * p.qpad_cap + pr] = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
        }
      }
    }
  }
}

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kRingDkdv = D == 128 ? 4 : 8;  // single-tile ring entries
  static constexpr int kRingDq = D == 128 ? 5 : 8;
  static constexpr int kVecSlots = 4;                  // dK/dV: per-query-tile lse2 / D vectors
  // dK/dV pass: S^T, dP^T, dK, dV.   dQ pass: S, dP (two buffers), dQ.
  static constexpr uint32_t kColS = 0, kColP = 128, kColA0 = 256, kColA1 = 256 + D;
  static constexpr uint32_t kColP1 = 256, kColDQ = 384;
  // dK/dV pass: P^T and dS^T (bf16, keys x 128 queries, each compute warpgroup's 64 queries
  // in 32 columns) over S^T / dP^T at d = 128, two 64-column halves apart; at d = 64 in the
  // spare columns [384, 448) and [448, 512), so the next S^T / dP^T MMA does not write the
  // columns the previous dV / dK MMA is still reading
  static constexpr uint32_t kColPT = D == 64 ? 384 : kColS, kColDST = D == 64 ? 448 : kColP;
  static constexpr uint32_t kXHalf = D == 64 ? 32 : 64;
  // dQ pass at d = 64: the query tile's Q and dO rows copied into the free columns
  // [448, 480) and [480, 512) by the compute warpgroups feed the S and dP MMAs from TMEM, and
  // the shared-memory buffers are free for the next query tile once both copies are done
  static constexpr bool kDqQTmem = D == 64;
  static constexpr uint32_t kColDqQ = 448, kColDqDO = 480;
  static constexpr int kSmemDkdv = 2 * kTileBytes + kRingDkdv * kTileBytes + kVecSlots * 1024 + 1024;
  static constexpr int kSmemDq = 2 * kTileBytes + kRingDq * kTileBytes + 1024;
  // Fused short-query pass: Q and dO resident, K/V ring, dS^T staging (keys x 128 queries,
  // bf16), lse2 / D vectors.  TMEM: S^T [0,128), dP^T then dK [128,256), dV, dQ.
  static constexpr int kRingFused = D == 128 ? 3 : 8;
  static constexpr uint32_t kColFdV = 256, kColFdQ = 256 + D;
  static constexpr int kSmemFused = 2 * kTileBytes + kRingFused * kTileBytes + 32768 + 1024 + 1024;
  // Non-sequence-parallel pass: K, V resident, dO / Q ring, dS^T staging, lse2 / D vectors.
  // dQ_ij over dP^T at d = 128, in the columns d = 64 leaves free otherwise.
  static constexpr int kRingNsp = D == 128 ? 3 : 8;
  static constexpr uint32_t kColNspDq = D == 128 ? kColP : 384;
  static constexpr int kSmemNsp = 2 * kTileBytes + kRingNsp * kTileBytes + 32768 + kVecSlots * 1024 + 1024;
  static_assert(kSmemDkdv <= 232448 && kSmemDq <= 232448 && kSmemFused + 1024 <= 232448 && kSmemNsp + 1024 <= 232448,
                "shared memory per CTA");
};

// Load one row-tile (128 rows x D columns, D/64 boxes of 16 KB) through a tensor map.
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int col0, int row0) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) tma_load_2d(dst + c * 16384, m, bar, col0 + c * 64, row0);
}

// 64 columns from TMEM -> floats, both loads in flight before one wait.
__device__ __forceinline__ void ld_cols64(uint32_t taddr, float* x) {
  uint32_t r0[32], r1[32];
  tmem_ld32(taddr, r0);
  tmem_ld32(taddr + 32, r1);
  tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    x[c] = __uint_as_float(r0[c]);
    x[32 + c] = __uint_as_float(r1[c]);
  }
}

// Store 64 fp32 values as 32 packed bf16x2 TMEM columns.
__device__ __forceinline__ void st_bf16_64(uint32_t taddr, const float* v) {
  uint32_t pk[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) pk[t] = pack_bf16x2(v[2 * t], v[2 * t + 1]);
  tmem_st32(taddr, pk);
}

// ---------------------------------------------------------------- bias-table gradient
// Table entry (h, n) collects dS_ij over the pairs of bucket n = clamp(j - i + center, 0,
// nb - 1).  A warp holds dS^T for its 32 key rows j = j0 + lane against 64 query columns
// i = i0 + c: entry (lane, c) lies on relative position j - i = (j0 - i0 - 63) + b with
// b = lane - c + 63 in [0, 95).  The warp sums along these diagonals in registers: in
// round k (0..31) each lane takes columns k and k + 32 of lane (lane + k) mod 32 with one
// shuffle each.  Every value a lane receives this way lies on the same diagonal --
// b = lane + 63 for column k, lane + 31 for column k + 32 -- except those whose source
// wrapped around the warp (lane + k >= 32), which lie 32 lower.  So each lane ends with
// three sums, b = lane + 63, lane + 31 and lane - 1, and adds them to the table with one
// coalesced fp32 reduction each (rel0 = j0 - i0 - 63 + center is the unclamped bucket of
// b = 0).  No shared memory, two shuffles and two packed adds per round.
__device__ __forceinline__ void dbias_flush(float s_hi, float s_mid, float s_lo, float* grad_row, int nb, int rel0,
                                            int lane) {
  const int top = nb - 1;
  if (s_hi != 0.f) red_add_global(grad_row + min(max(rel0 + lane + 63, 0), top), s_hi);
  if (s_mid != 0.f) red_add_global(grad_row + min(max(rel0 + lane + 31, 0), top), s_mid);
  if (s_lo != 0.f) red_add_global(grad_row + min(max(rel0 + lane - 1, 0), top), s_lo);  // lane 0: always 0
}

__device__ __forceinline__ void dbias_warp_tile(const float* ds, float* grad_row, int nb, int rel0, int lane) {
  uint64_t straight = 0, wrapped = 0;  // packed (column k, column k + 32) sums
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const int src = (lane + k) & 31;
    const uint64_t v = f2_pack(__shfl_sync(0xffffffffu, ds[k], src), __shfl_sync(0xffffffffu, ds[k + 32], src));
    if (lane + k < 32)
      straight = f2_add(straight, v);
    else
      wrapped = f2_add(wrapped, v);
  }
  float s0, s1, w0, w1;
  f2_unpack(straight, s0, s1);
  f2_unpack(wrapped, w0, w1);
  dbias_flush(s0, w0 + s1, w1, grad_row, nb, rel0, lane);
}

// Write NC (32 or 64) accumulator columns of this thread's TMEM lane, times `mul`, as bf16
// to global (or zeros when `zero`), one thread per row.
template <int NC>
__device__ __forceinline__ void store_acc_row_own(uint32_t taddr, float mul, __nv_bfloat16* dst, bool valid,
                                                  bool zero) {
#pragma unroll
  for (int cc = 0; cc < NC / 32; ++cc) {
    uint32_t r[32];
    if (!zero) {
      tmem_ld32(taddr + cc * 32, r);
      tmem_ld_wait();
    }
    uint32_t pk[16];
#pragma unroll
    for (int t = 0; t < 16; ++t)
      pk[t] = zero ? 0u : pack_bf16x2(__uint_as_float(r[2 * t]) * mul, __uint_as_float(r[2 * t + 1]) * mul);
    if (valid) {
      st_global_v8(dst + cc * 32, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
      st_global_v8(dst + cc * 32 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
    }
  }
}
// All D accumulator columns of this thread's TMEM lane, times `mul`, as bf16 to its own row,
// 32 columns at a time; arrives on `empty` as soon as the last columns are in registers.
template <int D>
__device__ __forceinline__ void drain_row_own(uint32_t taddr, float mul, __nv_bfloat16* dst, bool valid,
                                              uint64_t* empty) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + c0, r);
    tmem_ld_wait();
    if (c0 + 32 == D) {
      tc_fence_before();
      mbar_arrive(empty);
    }
    uint32_t pk[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(__uint_as_float(r[2 * t]) * mul, __uint_as_float(r[2 * t + 1]) * mul);
    if (valid) {
      st_global_v8(dst + c0, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
      st_global_v8(dst + c0 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
    }
  }
}

// Write NC (32 or 64) accumulator columns of this thread's TMEM lane, times `mul`, as bf16
// to global (or zeros when `zero`).  All 32 lanes of the warp call it together: the rows'
// stores are shared across lanes so that each store instruction writes whole row segments.
template <int NC>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, float mul, __nv_bfloat16* dst, bool valid, bool zero) {
  uint4 c[NC / 8];  // the row's NC bf16 values as 16-byte chunks
#pragma unroll
  for (int cc = 0; cc < NC / 32; ++cc) {
    uint32_t r[32];
    if (!zero) {
      tmem_ld32(taddr + cc * 32, r);
      tmem_ld_wait();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w4[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int e = 8 * q + 2 * t;
        w4[t] = zero ? 0u : pack_bf16x2(__uint_as_float(r[e]) * mul, __uint_as_float(r[e + 1]) * mul);
      }
      c[4 * cc + q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
  }
  st_rows_coalesced<NC * 2>(c, valid ? static_cast<void*>(dst) : nullptr);
}

// Writes the D accumulator columns of this thread's TMEM lane, times `mul`, as bf16 to the
// row at `dst`, 32 columns at a time (coalesced across the warp), and arrives on `empty`
// once the last columns are in registers: the accumulator may be overwritten from then on.
// All 32 lanes of the warp call it together.
template <int D>
__device__ __forceinline__ void drain_acc_rows(uint32_t taddr, float mul, __nv_bfloat16* dst, bool valid,
                                               uint64_t* empty) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + c0, r);
    tmem_ld_wait();
    if (c0 + 32 == D) {
      tc_fence_before();
      mbar_arrive(empty);
    }
    uint4 c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      c[q] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * q]) * mul, __uint_as_float(r[8 * q + 1]) * mul),
                        pack_bf16x2(__uint_as_float(r[8 * q + 2]) * mul, __uint_as_float(r[8 * q + 3]) * mul),
                        pack_bf16x2(__uint_as_float(r[8 * q + 4]) * mul, __uint_as_float(r[8 * q + 5]) * mul),
                        pack_bf16x2(__uint_as_float(r[8 * q + 6]) * mul, __uint_as_float(r[8 * q + 7]) * mul));
    st_rows_coalesced<64>(c, valid ? static_cast<void*>(dst + c0) : nullptr);
  }
}

// ================================================================== dK / dV pass
// Ring of single tiles, filled in the order dO_i, Q_i for the query tiles i of each key
// tile: dO_i is released after dV(i) and Q_i after dK(i), i.e. in fill order.  Each Q_i
// brings its tile's lse2 and D vectors (vector slot = query tile count mod kVecSlots; a
// slot is refilled only after dK of its previous tile completed).
template <int D, bool kBias, bool kJBias = false>
__global__ void __launch_bounds__(kThreadsDkdv, 1) dkdv_kernel(const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int R = C::kRingDkdv;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kTileBytes;
  uint8_t* sRing = smem + 2 * C::kTileBytes;
  float* sVec = reinterpret_cast<float*>(sRing + R * C::kTileBytes);  // [kVecSlots][2][128]: lse2, D

  // dV and dK hand over to the epilogue separately: dV(last) completes one MMA group
  // before dK(last), and the next key tile's dV(0) only needs dV stored, not dK.
  __shared__ uint64_t kv_full, kv_empty, st_full, dpt_full, p_full, ds_full, mma_done;
  __shared__ uint64_t dv_full, dv_empty, dk_full, dk_empty;
  __shared__ uint64_t ring_full[R], ring_empty[R];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ MetaRing meta;
  __shared__ uint4 jb_scratch[kJBias ? 8 * 128 : 1];  // general bias: 2 KB transpose scratch per compute warp

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    mbar_init(&st_full, 1);
    mbar_init(&dpt_full, 1);
    mbar_init(&p_full, 256);
    mbar_init(&ds_full, 256);
    mbar_init(&dv_full, 1);
    mbar_init(&dv_empty, 128);
    mbar_init(&dk_full, 1);
    mbar_init(&dk_empty, 128);
    mbar_init(&mma_done, 1);
    for (int i = 0; i < R; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    meta_init(meta, p.wait_ns, 3 + (kThreadsDkdv / 32 - kFirstComputeWarp));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  grid_dependency_wait();  // the planner's lists and maps, the previous kernels' outputs
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int n_items = *p.n_items;
  volatile int* abort_flag = &abort_sh;
  const bool causal = p.causal != 0;
  auto seq_len = [&](int b, int* Lq, int* Lk) {
    *Lq = int(p.q_off[b + 1] - p.q_off[b]);
    *Lk = int(p.kv_off[b + 1] - p.kv_off[b]);
  };

  if (warp < kFirstComputeWarp) {
   setmaxnreg_dec<kRegsLoadDkdv>();
   if (warp == 2) {
    // ------------------------------------------------------------ K/V loader
    // Its own warp, so a key tile's K/V load starts as soon as the previous tile's last
    // dP^T MMA frees the buffers, whatever the ring producer is waiting on.
    if (lane == 0) {
      uint32_t item_n = 0, tn = 0;
      int acq_b = -1;  // sequence whose maps this thread has acquired
      bool ok = true;
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
        if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
        const ItemMeta& wi = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
        if (wi.b < 0) break;  // end of this CTA's items
        const int Lq = wi.Lq, Lk = wi.Lk;
        const int64_t k0 = wi.ko;
        acquire_seq_maps(p.maps, wi.b, kMapK, kMapV, acq_b, false);
        for (int kt = wi.u0; kt < wi.u1 && ok; ++kt) {
          int first, count;
          q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
          if (count == 0) continue;
          const TileMap mk = tile_map(p.maps, p.B, kMapK, wi.b, k0, kt, p.total_kv);
          const TileMap mv = tile_map(p.maps, p.B, kMapV, wi.b, k0, kt, p.total_kv);
          if (mk.tail) {
            tmap_acquire(mk.map);
            tmap_acquire(mv.map);
          }
          if (!mbar_wait(&kv_empty, (item_n & 1) ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
          trace_event(p.trace, kTraceLoader, tn, 1);
          mbar_arrive_expect_tx(&kv_full, 2 * C::kTileBytes);
          load_tile<D>(sK, mk.map, &kv_full, wi.h * D, mk.y);
          load_tile<D>(sV, mv.map, &kv_full, wi.h * D, mv.y);
          ++item_n;
          // pull the next key tile into L2 meanwhile: the next of this range, else the first
          // of this CTA's next item
          {
            int nb = -1, nh = 0, nt = 0;
            if (kt + 1 < wi.u1) {
              nb = wi.b, nh = wi.h, nt = kt + 1;
            } else if (const ItemMeta* wn = meta_peek_next(meta, item_k)) {
              nb = wn->b, nh = wn->h, nt = wn->u0;
            }
            if (nb >= 0) {
              const int64_t nko = p.kv_off[nb];
              acquire_seq_maps(p.maps, nb, kMapK, kMapV, acq_b, true);
              if (nt * kBN < int(p.kv_off[nb + 1] - nko)) {
                prefetch_tile<D / 64>(p.maps, p.B, kMapK, nb, nko, nt, p.total_kv, nh * D);
                prefetch_tile<D / 64>(p.maps, p.B, kMapV, nb, nko, nt, p.total_kv, nh * D);
              }
            }
          }
        }
        if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      if (item_n > 0) drain_wait(&kv_full, (item_n - 1) & 1);
    }
   } else if (warp == 0) {
    // ------------------------------------------------------------ dO / Q ring producer
    if (lane == 0) {
      uint32_t ring_n = 0, qtile_n = 0, tn = 0;
      int acq_b = -1;  // sequence whose maps this thread has acquired
      bool ok = true;
      auto fill = [&](const TileMap& m, int col, const float* l2src, const float* dsrc) {
        const uint32_t e = ring_n % R, ph = (ring_n / R) & 1;
        if (m.tail) tmap_acquire(m.map);
        if (!mbar_wait(&ring_empty[e], ph ^ 1, abort_flag, kWaitTimeoutNs)) return false;
        trace_event(p.trace, kTraceProducer, tn, 2);
        mbar_arrive_expect_tx(&ring_full[e], C::kTileBytes + (l2src ? 2 * kBM * 4 : 0));
        load_tile<D>(sRing + e * C::kTileBytes, m.map, &ring_full[e], col, m.y);
        if (l2src) {
          float* v = sVec + (qtile_n % C::kVecSlots) * 256;
          bulk_load(v, l2src, kBM * 4, &ring_full[e]);
          bulk_load(v + 128, dsrc, kBM * 4, &ring_full[e]);
        }
        ++ring_n;
        return true;
      };
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
        if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
        const ItemMeta& wi = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
        if (wi.b < 0) break;  // end of this CTA's items
        const int Lq = wi.Lq, Lk = wi.Lk;
        const int64_t q0 = wi.qo;
        acquire_seq_maps(p.maps, wi.b, kMapQ, kMapDO, acq_b, false);
        const int64_t vec0 = int64_t(wi.h) * p.qpad_cap + wi.qp;
        for (int kt = wi.u0; kt < wi.u1 && ok; ++kt) {
          int first, count;
          q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
          if (const ItemMeta* wnp = kt + 1 == wi.u1 ? meta_peek_next(meta, item_k) : nullptr) {
            // pull the first query tiles of this CTA's next item into L2 meanwhile
            const ItemMeta& wn = *wnp;
            int nLq, nLk, nfirst, ncount;
            seq_len(wn.b, &nLq, &nLk);
            q_tiles_for_kv_tile(wn.u0, nLq, nLk, causal, &nfirst, &ncount);
            const int64_t nqo = p.q_off[wn.b];
            acquire_seq_maps(p.maps, wn.b, kMapQ, kMapDO, acq_b, true);
            for (int t = nfirst; t < nfirst + min(ncount, 2); ++t) {
              prefetch_tile<D / 64>(p.maps, p.B, kMapDO, wn.b, nqo, t, p.total_q, wn.h * D);
              prefetch_tile<D / 64>(p.maps, p.B, kMapQ, wn.b, nqo, t, p.total_q, wn.h * D);
            }
          }
          for (int i = 0; i < count && ok; ++i) {
            const int qt = first + i;
            const TileMap mdo = tile_map(p.maps, p.B, kMapDO, wi.b, q0, qt, p.total_q);
            const TileMap mq = tile_map(p.maps, p.B, kMapQ, wi.b, q0, qt, p.total_q);
            if (!fill(mdo, wi.h * D, nullptr, nullptr)) { ok = false; break; }
            if (!fill(mq, wi.h * D, p.lse2 + vec0 + qt * kBM, p.delta + vec0 + qt * kBM)) {
              ok = false;
              break;
            }
            ++qtile_n;
          }
        }
        if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      const uint32_t f = ring_n > uint32_t(R) ? ring_n - R : 0;
      for (uint32_t n = f; n < ring_n; ++n) drain_wait(&ring_full[n % R], (n / R) & 1);
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, false, true);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aR = smem_u32(sRing);
      uint32_t ring_n = 0, item_n = 0, tile_n = 0, acc_n = 0, tn = 0;
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        if (!mbar_wait(bar, par, abort_flag, kWaitTimeoutNs)) return false;
        tc_fence_after();
        return true;
      };
      auto wait_ring = [&](uint32_t n) { return wait(&ring_full[n % R], (n / R) & 1); };
      auto ra = [&](uint32_t n) { return aR + (n % R) * C::kTileBytes; };
      // S^T (or dP^T) = A_tile(keys x D) * B_tile(queries x D)^T, both K-major
      auto mma_nt = [&](uint32_t dcol, uint32_t a, uint32_t b) {
        const uint64_t ad = sdesc_sw128(a, 16, 1024), bd = sdesc_sw128(b, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ss(tmem + dcol, ad + o, bd + o, kIdS, kk > 0);
        }
      };
      // acc(keys x D) += X^T (TMEM bf16, keys x 128 queries, two halves kXHalf columns apart) * B(queries x D, MN-major)
      auto mma_acc = [&](uint32_t dcol, uint32_t xcol, uint32_t b, bool acc) {
        const uint64_t bd = sdesc_sw128(b, 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          umma_ts(tmem + dcol, tmem + xcol + (kk >> 2) * C::kXHalf + (kk & 3) * 8, bd + uint32_t(kk * 2048 >> 4),
                  kIdAcc, (acc || kk > 0) ? 1u : 0u);
      };
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
       if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
       if (wi.b < 0) break;  // end of this CTA's items
       const int Lq = wi.Lq, Lk = wi.Lk;
       for (int kt = wi.u0; kt < wi.u1 && ok; ++kt) {
        int first, count;
        q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
        if (count == 0) continue;
        if (!wait(&kv_full, item_n & 1)) { ok = false; break; }
        ++item_n;
        trace_event(p.trace, kTraceMma, tn, 10);
        const uint32_t n0 = ring_n;  // dO_i at n0 + 2i, Q_i at n0 + 2i + 1
        if (!wait_ring(n0 + 1)) { ok = false; break; }
        mma_nt(C::kColS, aK, ra(n0 + 1));
        umma_commit(&st_full);
        if (!wait_ring(n0)) { ok = false; break; }
        mma_nt(C::kColP, aV, ra(n0));
        umma_commit(&dpt_full);
        // K and V are read only by S^T and dP^T: once the last dP^T is issued the loader
        // may bring in the next key tile while dV / dK of this one still run
        if (count == 1) umma_commit(&kv_empty);
        for (int i = 0; i < count && ok; ++i) {
          const uint32_t nd = n0 + 2 * i, nq = nd + 1;
          if (!wait(&p_full, tile_n & 1)) { ok = false; break; }
          trace_event(p.trace, kTraceMma, tn, 11);
          if (i == 0 && !wait(&dv_empty, (acc_n & 1) ^ 1)) { ok = false; break; }
          mma_acc(C::kColA1, C::kColPT, ra(nd), i > 0);  // dV += P^T dO
          umma_commit(&ring_empty[nd % R]);
          if (i + 1 == count) umma_commit(&dv_full);
          trace_event(p.trace, kTraceMma, tn, 12);
          if (i + 1 < count) {
            if (!wait_ring(nq + 2)) { ok = false; break; }
            mma_nt(C::kColS, aK, ra(nq + 2));
            umma_commit(&st_full);
            trace_event(p.trace, kTraceMma, tn, 13);
          }
          if (!wait(&ds_full, tile_n & 1)) { ok = false; break; }
          trace_event(p.trace, kTraceMma, tn, 14);
          ++tile_n;
          if (i == 0 && !wait(&dk_empty, (acc_n & 1) ^ 1)) { ok = false; break; }
          mma_acc(C::kColA0, C::kColDST, ra(nq), i > 0);  // dK += dS^T Q
          umma_commit(&ring_empty[nq % R]);
          trace_event(p.trace, kTraceMma, tn, 15);
          if (i + 1 < count) {
            if (!wait_ring(nd + 2)) { ok = false; break; }
            mma_nt(C::kColP, aV, ra(nd + 2));
            umma_commit(&dpt_full);
            if (i + 2 == count) umma_commit(&kv_empty);
            trace_event(p.trace, kTraceMma, tn, 16);
          }
        }
        if (!ok) break;
        ring_n = n0 + 2 * count;
        ++acc_n;
        umma_commit(&dk_full);
       }
       if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      umma_commit(&mma_done);
      drain_wait(&mma_done, 0);
    }
   } else if (warp == 3) {
    // ------------------------------------------------------------ scheduler
    if (lane == 0 && !meta_publish(meta, p.items, n_items, p.claim, p.q_off, p.kv_off, p.qpad, p.jb_off, abort_flag))
      raise_status(p.status, JFA_ERR_TIMEOUT);
   }
  } else if (warp < kFirstEpilogueWarp) {
    setmaxnreg_inc<kRegsComputeDkdv>();
    // ------------------------------------------------------------ compute warpgroups
    const int w = (warp - kFirstComputeWarp) >> 2;  // column half owned: queries [64w, 64w+64)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row within the tile
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kColS + 64 * w;
    const uint32_t tP = tmem + lane_addr + C::kColP + 64 * w;
    const uint32_t tPT = tmem + lane_addr + C::kColPT + C::kXHalf * w;    // P^T, bf16
    const uint32_t tDST = tmem + lane_addr + C::kColDST + C::kXHalf * w;  // dS^T, bf16
    const float sl2 = p.scale_log2;
    uint32_t ring_n = 0, tile_n = 0, qtile_n = 0, tn = 0;
    const bool leader = (warp & 3) == 0 && lane == 0;
    bool ok = true;
    uint32_t item_k = 0;
    for (; ok; ++item_k) {
     if (!meta_wait_warp(meta, item_k, abort_flag)) { ok = false; break; }
     const ItemMeta& it = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
     if (it.b < 0) break;  // end of this CTA's items
     const int Lq = it.Lq, Lk = it.Lk;
     for (int kt = it.u0; kt < it.u1 && ok; ++kt) {
      int first, count;
      q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
      const int j = kt * kBN + row;  // local key index
      if (count == 0) continue;  // rows of zeros: written by the epilogue warpgroup
      const int diag = Lk - Lq;  // key j visible to query i iff i >= j - diag
      const float* brow = kBias ? p.bias2 + size_t(it.h) * p.num_buckets : nullptr;
      for (int i = 0; i < count && ok; ++i) {
        const int qt = first + i;
        uint4 jbw[8];  // general bias for this tile (row order), loaded before the waits
        if (kJBias) {
          const int64_t pitch = (Lk + 7) / 8 * 8;  // rows of the sequence's block: bias[i][j] at i * pitch + j
          const int qi0 = qt * kBM + 64 * w, kj0 = kt * kBN + quarter * 32;
          jbias_load_cols_vec(jbw, p.jbias + size_t(it.h) * p.jb_plane + it.jb + int64_t(qi0) * pitch + kj0, pitch,
                              Lq - qi0, Lk - kj0, lane);
          if (kj0 < Lk) {  // the next query tile's rows of these keys into L2 meanwhile
            const int nq0 = qi0 + kBM;
            const __nv_bfloat16* nb = p.jbias + size_t(it.h) * p.jb_plane + it.jb + int64_t(nq0) * pitch + kj0;
            if (nq0 + lane < Lq) prefetch_l2(nb + int64_t(lane) * pitch);
            if (nq0 + 32 + lane < Lq) prefetch_l2(nb + int64_t(32 + lane) * pitch);
          }
        }
        // relative-position bias * log2(e) of this tile (bucket of column c: idx0 - c), loaded
        // before the waits so the loads overlap the MMAs
        float bw[kBias ? 64 : 1];
        if (kBias) {
          const int idx0 = j - (qt * kBM + 64 * w) + p.center;
          if (idx0 - 63 >= 0 && idx0 < p.num_buckets) {
#pragma unroll
            for (int c = 0; c < 64; ++c) bw[c] = __ldg(brow + idx0 - c);
          } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) bw[c] = __ldg(brow + min(max(idx0 - c, 0), p.num_buckets - 1));
          }
        }
        // Q_i's ring slot carries this tile's lse2 / D vectors: wait for it
        const uint32_t nq = ring_n + 1;
        if (!mbar_wait(&ring_full[nq % R], (nq / R) & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        ring_n += 2;
        const float* vec = sVec + (qtile_n % C::kVecSlots) * 256;
        ++qtile_n;
        const uint64_t* nlse2 = reinterpret_cast<const uint64_t*>(vec + 64 * w);  // -lse2 pairs
        const uint64_t* ndvec = reinterpret_cast<const uint64_t*>(vec + 128 + 64 * w);  // -D pairs
        if (!mbar_wait(&st_full, tile_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 20);
        float x[64];
        ld_cols64(tS, x);
        const int i0 = qt * kBM + 64 * w;  // local query index of column 0 of this half
        if (kJBias) {
          uint32_t jbk[32];
          jbias_col_transpose(jbk, jbw, jb_scratch + (warp - kFirstComputeWarp) * 128, j < Lk, lane);
          jbias_apply<64>(x, jbk, sl2, kLog2e);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)
            f2_unpack(f2_add(f2_pack(x[2 * c2], x[2 * c2 + 1]), nlse2[c2]), x[2 * c2], x[2 * c2 + 1]);
        } else if (kBias) {
          const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)  // packed: x*scale + bias - lse2, two columns per op
            f2_unpack(f2_add(f2_fma(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2, f2_pack(bw[2 * c2], bw[2 * c2 + 1])),
                             nlse2[c2]),
                      x[2 * c2], x[2 * c2 + 1]);
        } else {
          const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)
            f2_unpack(f2_fma(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2, nlse2[c2]), x[2 * c2], x[2 * c2 + 1]);
        }
        if (causal) {
          const int lim = j - diag - i0;  // columns c < lim are hidden
          if (lim > 0) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c < lim) x[c] = -INFINITY;
          }
        }
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = ex2_approx(x[c]);  // P^T
        st_bf16_64(tPT, x);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full);
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 21);
        if (!mbar_wait(&dpt_full, tile_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        ++tile_n;
        tc_fence_after();
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 22);
        float dp[64];
        ld_cols64(tP, dp);
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2)  // dS^T = P^T o (dP^T - D)
          f2_unpack(f2_mul(f2_pack(x[2 * c2], x[2 * c2 + 1]), f2_add(f2_pack(dp[2 * c2], dp[2 * c2 + 1]), ndvec[c2])),
                    dp[2 * c2], dp[2 * c2 + 1]);
        st_bf16_64(tDST, dp);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_full);
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 23);
        if (kJBias && p.jb_grad) {  // the general bias's gradient is dS itself
          const int64_t pitch = (Lk + 7) / 8 * 8;
          const int kj0 = kt * kBN + quarter * 32;
          uint32_t gk[32];
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2) gk[c2] = pack_bf16x2(dp[2 * c2], dp[2 * c2 + 1]);
          jbias_store_cols(gk, jb_scratch + (warp - kFirstComputeWarp) * 128,
                           p.jb_grad + size_t(it.h) * p.jb_plane + it.jb + int64_t(i0) * pitch + kj0, pitch, Lq - i0,
                           Lk - kj0, j < Lk, lane);
        }
        if (kBias && p.bias_grad) {
          // dS^T of a padded key row is not zero (k = 0 but lse2 of the query is not), and
          // padded query columns only give 0 while their P^T stays finite: count neither
          const int ncols = j < Lk ? Lq - i0 : 0;
          if (ncols < 64) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c >= ncols) dp[c] = 0.f;
          }
          dbias_warp_tile(dp, p.bias_grad + size_t(it.h) * p.num_buckets, p.num_buckets,
                          kt * kBN + quarter * 32 - i0 - 63 + p.center, lane);
        }
      }
      if (!ok) break;
     }
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, item_k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  } else {
    setmaxnreg_dec<kRegsEpiDkdv>();
    // ------------------------------------------------------------ epilogue warpgroup
    // Writes each key tile's dV and dK rows (this thread's TMEM lane = one key row, all D
    // columns, 32 at a time) while the compute warpgroups go on with the next key tile;
    // an accumulator is released as soon as its last columns are in registers.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    uint32_t acc_n = 0;
    bool ok = true;
    uint32_t item_k = 0;
    for (; ok; ++item_k) {
     if (!meta_wait_warp(meta, item_k, abort_flag)) { ok = false; break; }
     const ItemMeta& it = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
     if (it.b < 0) break;  // end of this CTA's items
     const int64_t ko = it.ko;
     const int Lq = it.Lq, Lk = it.Lk;
     for (int kt = it.u0; kt < it.u1 && ok; ++kt) {
      int first, count;
      q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
      const int j = kt * kBN + row;  // local key index
      const bool valid = j < Lk;
      __nv_bfloat16* dk_row = p.g0 + ((ko + j) * p.H + it.h) * int64_t(D);
      __nv_bfloat16* dv_row = p.g1 + ((ko + j) * p.H + it.h) * int64_t(D);
      if (count == 0) {  // no query sees these keys
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          store_acc_row<32>(0, 0.f, dk_row + c0, valid, true);
          store_acc_row<32>(0, 0.f, dv_row + c0, valid, true);
        }
        continue;
      }
      if (!mbar_wait(&dv_full, acc_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      tc_fence_after();
      drain_acc_rows<D>(tmem + lane_addr + C::kColA1, 1.f, dv_row, valid, &dv_empty);
      if (!mbar_wait(&dk_full, acc_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      ++acc_n;
      tc_fence_after();
      drain_acc_rows<D>(tmem + lane_addr + C::kColA0, p.scale, dk_row, valid, &dk_empty);
     }
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, item_k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================================== dQ pass
// Ring of single tiles, filled V_j, K_j per key tile: V_j is released after dP(j), K_j
// after dQ(j), i.e. in fill order.  S and dP of the next key tile are issued as soon as
// the warpgroups hold S in registers, so the dP/dS buffer alternates by tile parity.
template <int D, bool kBias, bool kJBias = false>
__global__ void __launch_bounds__(kThreadsDkdv, 1) dq_kernel(const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int R = C::kRingDq;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::kTileBytes;
  uint8_t* sRing = smem + 2 * C::kTileBytes;

  __shared__ uint64_t qdo_full, qdo_empty, qt_full, s_full, s_free, acc_full, acc_empty, mma_done;
  // dp_full / ds_full of global tile g live at index g & 1: dP(g+1) is issued before dQ(g)
  // waits for dS(g), so one warpgroup may finish tile g+1 while the other still works on
  // tile g (never further: S(g+2) waits for both warpgroups' s_free(g+1)); separate
  // barriers per tile parity keep their arrivals apart.
  __shared__ uint64_t dp_full[2], ds_full[2];
  __shared__ uint64_t ring_full[R], ring_empty[R];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ MetaRing meta;
  __shared__ float rb_scr[kBias && D == 64 ? 8 * 96 : 1];  // relative-position bias windows (d = 64)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&qdo_full, 1);
    mbar_init(&qdo_empty, C::kDqQTmem ? 256 : 1);  // both compute warpgroups, else the last dP MMA
    mbar_init(&qt_full, 256);
    mbar_init(&s_full, 1);
    mbar_init(&s_free, 256);
    mbar_init(&dp_full[0], 1);
    mbar_init(&dp_full[1], 1);
    mbar_init(&ds_full[0], 256);
    mbar_init(&ds_full[1], 256);
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, 128);
    mbar_init(&mma_done, 1);
    for (int i = 0; i < R; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    meta_init(meta, p.wait_ns, 3 + (kThreadsDkdv / 32 - kFirstComputeWarp));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  grid_dependency_wait();  // the planner's lists and maps, the previous kernels' outputs
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int n_items = *p.n_items;
  volatile int* abort_flag = &abort_sh;
  const bool causal = p.causal != 0;
  auto colP = [](uint32_t g) { return (g & 1) ? C::kColP1 : C::kColP; };
  auto seq_len = [&](int b, int* Lq, int* Lk) {
    *Lq = int(p.q_off[b + 1] - p.q_off[b]);
    *Lk = int(p.kv_off[b + 1] - p.kv_off[b]);
  };

  if (warp < kFirstComputeWarp) {
   setmaxnreg_dec<kRegsLoadDkdv>();
   if (warp == 2) {
    // ------------------------------------------------------------ Q / dO loader
    if (lane == 0) {
      uint32_t item_n = 0, tn = 0;
      int acq_b = -1;  // sequence whose maps this thread has acquired
      bool ok = true;
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
       if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
       if (wi.b < 0) break;  // end of this CTA's items
       const int Lq = wi.Lq, Lk = wi.Lk;
       const int64_t q0 = wi.qo;
       acquire_seq_maps(p.maps, wi.b, kMapQ, kMapDO, acq_b, false);
       for (int qt = wi.u0; qt < wi.u1 && ok; ++qt) {
        if (kv_tiles_for_q_tile(qt, Lq, Lk, causal) == 0) continue;
        const TileMap mq = tile_map(p.maps, p.B, kMapQ, wi.b, q0, qt, p.total_q);
        const TileMap mdo = tile_map(p.maps, p.B, kMapDO, wi.b, q0, qt, p.total_q);
        if (mq.tail) {
          tmap_acquire(mq.map);
          tmap_acquire(mdo.map);
        }
        if (!mbar_wait(&qdo_empty, (item_n & 1) ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        trace_event(p.trace, kTraceLoader, tn, 1);
        mbar_arrive_expect_tx(&qdo_full, 2 * C::kTileBytes);
        load_tile<D>(sQ, mq.map, &qdo_full, wi.h * D, mq.y);
        load_tile<D>(sDO, mdo.map, &qdo_full, wi.h * D, mdo.y);
        ++item_n;
        // pull the next query tile into L2 meanwhile: the next of this range, else the first
        // of this CTA's next item
        {
          int nb = -1, nh = 0, nt = 0;
          if (qt + 1 < wi.u1) {
            nb = wi.b, nh = wi.h, nt = qt + 1;
          } else if (const ItemMeta* wn = meta_peek_next(meta, item_k)) {
            nb = wn->b, nh = wn->h, nt = wn->u0;
          }
          if (nb >= 0) {
            const int64_t nqo = p.q_off[nb];
            acquire_seq_maps(p.maps, nb, kMapQ, kMapDO, acq_b, true);
            if (nt * kBM < int(p.q_off[nb + 1] - nqo)) {
              prefetch_tile<D / 64>(p.maps, p.B, kMapQ, nb, nqo, nt, p.total_q, nh * D);
              prefetch_tile<D / 64>(p.maps, p.B, kMapDO, nb, nqo, nt, p.total_q, nh * D);
            }
          }
        }
       }
       if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      if (item_n > 0) drain_wait(&qdo_full, (item_n - 1) & 1);
    }
   } else if (warp == 0) {
    // ------------------------------------------------------------ V / K ring producer
    if (lane == 0) {
      uint32_t ring_n = 0, tn = 0;
      int acq_b = -1;  // sequence whose maps this thread has acquired
      bool ok = true;
      auto fill = [&](const TileMap& m, int col) {
        const uint32_t e = ring_n % R, ph = (ring_n / R) & 1;
        if (m.tail) tmap_acquire(m.map);
        if (!mbar_wait(&ring_empty[e], ph ^ 1, abort_flag, kWaitTimeoutNs)) return false;
        trace_event(p.trace, kTraceProducer, tn, 2);
        mbar_arrive_expect_tx(&ring_full[e], C::kTileBytes);
        load_tile<D>(sRing + e * C::kTileBytes, m.map, &ring_full[e], col, m.y);
        ++ring_n;
        return true;
      };
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
       if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
       if (wi.b < 0) break;  // end of this CTA's items
       const int Lq = wi.Lq, Lk = wi.Lk;
       const int64_t k0 = wi.ko;
       acquire_seq_maps(p.maps, wi.b, kMapK, kMapV, acq_b, false);
       for (int qt = wi.u0; qt < wi.u1 && ok; ++qt) {
        const int nkv = kv_tiles_for_q_tile(qt, Lq, Lk, causal);
        if (const ItemMeta* wnp = qt + 1 == wi.u1 ? meta_peek_next(meta, item_k) : nullptr) {
          // pull the first key tiles of this CTA's next item into L2 meanwhile
          const ItemMeta& wn = *wnp;
          const int64_t nko = p.kv_off[wn.b];
          const int nLk = int(p.kv_off[wn.b + 1] - nko);
          acquire_seq_maps(p.maps, wn.b, kMapK, kMapV, acq_b, true);
          for (int t = 0; t < 2 && t * kBN < nLk; ++t) {
            prefetch_tile<D / 64>(p.maps, p.B, kMapV, wn.b, nko, t, p.total_kv, wn.h * D);
            prefetch_tile<D / 64>(p.maps, p.B, kMapK, wn.b, nko, t, p.total_kv, wn.h * D);
          }
        }
        for (int jt = 0; jt < nkv && ok; ++jt) {
          const TileMap mv = tile_map(p.maps, p.B, kMapV, wi.b, k0, jt, p.total_kv);
          const TileMap mk = tile_map(p.maps, p.B, kMapK, wi.b, k0, jt, p.total_kv);
          if (!fill(mv, wi.h * D) || !fill(mk, wi.h * D)) { ok = false; break; }
        }
       }
       if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      const uint32_t f = ring_n > uint32_t(R) ? ring_n - R : 0;
      for (uint32_t n = f; n < ring_n; ++n) drain_wait(&ring_full[n % R], (n / R) & 1);
    }
   } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, false, true);
      const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO), aR = smem_u32(sRing);
      uint32_t ring_n = 0, item_n = 0, tile_n = 0, acc_n = 0, tn = 0;
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        if (!mbar_wait(bar, par, abort_flag, kWaitTimeoutNs)) return false;
        tc_fence_after();
        return true;
      };
      auto wait_ring = [&](uint32_t n) { return wait(&ring_full[n % R], (n / R) & 1); };
      auto ra = [&](uint32_t n) { return aR + (n % R) * C::kTileBytes; };
      // S (dp = false: Q K^T) or dP (dp = true: dO V^T) of a query tile and the key tile at b
      auto mma_nt = [&](uint32_t dcol, bool dp, uint32_t b) {
        const uint64_t ad = sdesc_sw128(dp ? aDO : aQ, 16, 1024), bd = sdesc_sw128(b, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          if (C::kDqQTmem)
            umma_ts(tmem + dcol, tmem + (dp ? C::kColDqDO : C::kColDqQ) + kk * 8, bd + o, kIdS, kk > 0);
          else
            umma_ss(tmem + dcol, ad + o, bd + o, kIdS, kk > 0);
        }
      };
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
       if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
       if (wi.b < 0) break;  // end of this CTA's items
       const int Lq = wi.Lq, Lk = wi.Lk;
       for (int qt = wi.u0; qt < wi.u1 && ok; ++qt) {
        const int nkv = kv_tiles_for_q_tile(qt, Lq, Lk, causal);
        if (nkv == 0) continue;
        if (!wait(C::kDqQTmem ? &qt_full : &qdo_full, item_n & 1)) { ok = false; break; }
        ++item_n;
        trace_event(p.trace, kTraceMma, tn, 10);
        const uint32_t n0 = ring_n;  // V_j at n0 + 2j, K_j at n0 + 2j + 1
        if (!wait_ring(n0 + 1)) { ok = false; break; }
        mma_nt(C::kColS, false, ra(n0 + 1));
        umma_commit(&s_full);
        if (!wait_ring(n0)) { ok = false; break; }
        mma_nt(colP(tile_n), true, ra(n0));
        umma_commit(&dp_full[tile_n & 1]);
        umma_commit(&ring_empty[n0 % R]);
        // Q and dO are read only by S and dP: once the last dP is issued the loader may
        // bring in the next query tile while dQ of this one still runs (at d = 64 the compute
        // warpgroups free them after copying them into TMEM)
        if (nkv == 1 && !C::kDqQTmem) umma_commit(&qdo_empty);
        for (int jt = 0; jt < nkv && ok; ++jt) {
          const uint32_t g = tile_n;  // global tile index
          const uint32_t nv = n0 + 2 * jt, nk = nv + 1;
          if (jt + 1 < nkv) {
            // next S once the warpgroups hold this S in registers; next dP into the
            // other buffer (its dS was consumed by the dQ MMA issued before)
            if (!wait(&s_free, g & 1)) { ok = false; break; }
            trace_event(p.trace, kTraceMma, tn, 11);
            if (!wait_ring(nk + 2)) { ok = false; break; }
            mma_nt(C::kColS, false, ra(nk + 2));
            umma_commit(&s_full);
            trace_event(p.trace, kTraceMma, tn, 12);
            if (!wait_ring(nv + 2)) { ok = false; break; }
            mma_nt(colP(g + 1), true, ra(nv + 2));
            umma_commit(&dp_full[(g + 1) & 1]);
            umma_commit(&ring_empty[(nv + 2) % R]);
            if (jt + 2 == nkv && !C::kDqQTmem) umma_commit(&qdo_empty);
            trace_event(p.trace, kTraceMma, tn, 13);
          }
          if (!wait(&ds_full[g & 1], (g >> 1) & 1)) { ok = false; break; }
          trace_event(p.trace, kTraceMma, tn, 14);
          ++tile_n;
          if (jt == 0 && !wait(&acc_empty, (acc_n & 1) ^ 1)) { ok = false; break; }
          // dQ += dS (TMEM, queries x keys) * K (keys x D, MN-major)
          const uint64_t kd = sdesc_sw128(ra(nk), 16384, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            umma_ts(tmem + C::kColDQ, tmem + colP(g) + (kk >> 2) * 64 + (kk & 3) * 8, kd + uint32_t(kk * 2048 >> 4),
                    kIdAcc, (jt > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&ring_empty[nk % R]);
          trace_event(p.trace, kTraceMma, tn, 15);
        }
        if (!ok) break;
        // the last tile's s_free arrival has no consumer above: take it here
        if (!wait(&s_free, (tile_n - 1) & 1)) { ok = false; break; }
        ring_n = n0 + 2 * nkv;
        ++acc_n;
        umma_commit(&acc_full);
       }
       if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      umma_commit(&mma_done);
      drain_wait(&mma_done, 0);
    }
   } else if (warp == 3) {
    // ------------------------------------------------------------ scheduler
    if (lane == 0 && !meta_publish(meta, p.items, n_items, p.claim, p.q_off, p.kv_off, p.qpad, p.jb_off, abort_flag))
      raise_status(p.status, JFA_ERR_TIMEOUT);
   }
  } else if (warp < kFirstEpilogueWarp) {
    setmaxnreg_inc<kRegsComputeDkdv>();
    const int w = (warp - kFirstComputeWarp) >> 2;  // key columns [64w, 64w+64)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kColS + 64 * w;
    const float sl2 = p.scale_log2;
    uint32_t tile_n = 0, q_n = 0, tn = 0;
    const bool leader = (warp & 3) == 0 && lane == 0;
    bool ok = true;
    uint32_t item_k = 0;
    for (; ok; ++item_k) {
     if (!meta_wait_warp(meta, item_k, abort_flag)) { ok = false; break; }
     const ItemMeta& it = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
     if (it.b < 0) break;  // end of this CTA's items
     const int Lq = it.Lq, Lk = it.Lk;
     const int64_t vec0 = int64_t(it.h) * p.qpad_cap + it.qp;
     for (int qt = it.u0; qt < it.u1 && ok; ++qt) {
      const int nkv = kv_tiles_for_q_tile(qt, Lq, Lk, causal);
      const int i = qt * kBM + row;
      const bool valid = i < Lq;
      if (nkv == 0) continue;  // rows of zeros: written by the epilogue warpgroup
      if (C::kDqQTmem) {
        // this query tile's rows into TMEM: warpgroup 0 copies Q, warpgroup 1 dO (row `row`
        // of a 128-byte-swizzled tile: 16-byte chunk c at chunk position c ^ (row & 7))
        if (!mbar_wait(&qdo_full, q_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        ++q_n;
        const uint4* src = reinterpret_cast<const uint4*>((w ? sDO : sQ) + row * 128);
        uint32_t cw[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = src[c ^ (row & 7)];
          cw[4 * c] = v.x;
          cw[4 * c + 1] = v.y;
          cw[4 * c + 2] = v.z;
          cw[4 * c + 3] = v.w;
        }
        tmem_st32(tmem + lane_addr + (w ? C::kColDqDO : C::kColDqQ), cw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&qt_full);
        mbar_arrive(&qdo_empty);
      }
      // padded per-query vectors (stored negated): 0 past the sequence end, -inf for rows
      // that see no key
      const float nl2 = __ldg(p.lse2 + vec0 + i);
      const uint64_t k_nl2 = f2_pack(nl2, nl2);
      const float nd = __ldg(p.delta + vec0 + i);
      const uint64_t k_nd = f2_pack(nd, nd);
      const int diag = Lk - Lq;
      const float* brow = kBias ? p.bias2 + size_t(it.h) * p.num_buckets : nullptr;
      // relative-position bias at d = 64: this warp's window of the table for key tile jt (the
      // bucket of (lane, column c) is lo0 + jt * 128 + 31 + c - lane), fetched into registers a
      // tile ahead and staged in the warp's scratch when its tile comes up
      float* scr = kBias && D == 64 ? rb_scr + (warp - kFirstComputeWarp) * 96 : nullptr;
      const int lo0 = 64 * w - (i - lane) + p.center - 31;
      float rbv[3];  // dead unless kBias at d = 64
      if (kBias && D == 64) relbias_fetch<3>(rbv, brow, lo0, 64 + 31, p.num_buckets, lane);
      for (int jt = 0; jt < nkv && ok; ++jt) {
        uint32_t jbk[kJBias ? 32 : 1];  // general bias for this tile, loaded before the wait
        if (kJBias) {
          const int64_t pitch = (Lk + 7) / 8 * 8;  // rows of the sequence's block: bias[i][j] at i * pitch + j
          const int jj0 = jt * kBN + 64 * w;
          const __nv_bfloat16* brow_i = p.jbias + size_t(it.h) * p.jb_plane + it.jb + int64_t(i) * pitch;
          jbias_load_row<64>(jbk, valid ? brow_i + jj0 : nullptr, min(64, Lk - jj0));
          if (valid && jj0 + kBN < Lk) {  // the next key tile's row segment into L2 meanwhile
            prefetch_l2(brow_i + jj0 + kBN);
            prefetch_l2(brow_i + jj0 + kBN + 56);
          }
        }
        // relative-position bias * log2(e) of this tile (bucket of column c: idx0 + c), loaded
        // before the wait so the loads overlap the MMAs
        float bw[kBias ? 64 : 1];
        if (kBias && D == 64) {
          relbias_store<3>(scr, rbv, 64 + 31, lane);
#pragma unroll
          for (int c = 0; c < 64; ++c) bw[c] = scr[c + 31 - lane];
          if (jt + 1 < nkv) relbias_fetch<3>(rbv, brow, lo0 + (jt + 1) * kBN, 64 + 31, p.num_buckets, lane);
        } else if (kBias) {  // d = 128: no shared memory to spare, gathered from global memory
          const int idx0 = jt * kBN + 64 * w - i + p.center;
          if (idx0 >= 0 && idx0 + 63 < p.num_buckets) {
#pragma unroll
            for (int c = 0; c < 64; ++c) bw[c] = __ldg(brow + idx0 + c);
          } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) bw[c] = __ldg(brow + min(max(idx0 + c, 0), p.num_buckets - 1));
          }
        }
        if (!mbar_wait(&s_full, tile_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 20);
        float x[64];
        ld_cols64(tS, x);
        tc_fence_before();
        mbar_arrive(&s_free);
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 21);
        const int j0 = jt * kBN + 64 * w;  // local key index of column 0 of this half
        const int n_real = Lk - j0;        // columns >= n_real are past the sequence end
        if (kJBias) {
          jbias_apply<64>(x, jbk, sl2, kLog2e);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)
            f2_unpack(f2_add(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_nl2), x[2 * c2], x[2 * c2 + 1]);
        } else if (kBias) {
          const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)  // packed: x*scale + bias - lse2, two columns per op
            f2_unpack(f2_add(f2_fma(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2, f2_pack(bw[2 * c2], bw[2 * c2 + 1])),
                             k_nl2),
                      x[2 * c2], x[2 * c2 + 1]);
        } else {
          const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)
            f2_unpack(f2_fma(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2, k_nl2), x[2 * c2], x[2 * c2 + 1]);
        }
        if (causal) {
          const int lim = i + diag - j0;  // columns c > lim are hidden
          if (lim < 63) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c > lim) x[c] = -INFINITY;
          }
        }
        if (n_real < 64) {
          // padded keys (zero rows) would score exp2(-lse): keep them out of dS so it stays finite
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c >= n_real) x[c] = -INFINITY;
        }
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = ex2_approx(x[c]);  // P
        const uint32_t g = tile_n;
        const uint32_t tP = tmem + lane_addr + colP(g) + 64 * w;
        if (!mbar_wait(&dp_full[g & 1], (g >> 1) & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        ++tile_n;
        tc_fence_after();
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 22);
        float dp[64];
        ld_cols64(tP, dp);
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2)  // dS = P o (dP - D)
          f2_unpack(f2_mul(f2_pack(x[2 * c2], x[2 * c2 + 1]), f2_add(f2_pack(dp[2 * c2], dp[2 * c2 + 1]), k_nd)),
                    dp[2 * c2], dp[2 * c2 + 1]);
        st_bf16_64(tP, dp);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_full[g & 1]);
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 23);
      }
      if (!ok) break;
     }
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, item_k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  } else {
    setmaxnreg_dec<kRegsEpiDkdv>();
    // ------------------------------------------------------------ epilogue warpgroup
    // Writes each query tile's dQ rows (this thread's TMEM lane = one query row, all D
    // columns, 32 at a time) while warpgroups 1 and 2 start the next query tile; the
    // accumulator is released as soon as its last columns are in registers.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    uint32_t acc_n = 0;
    bool ok = true;
    uint32_t item_k = 0;
    for (; ok; ++item_k) {
     if (!meta_wait_warp(meta, item_k, abort_flag)) { ok = false; break; }
     const ItemMeta& it = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
     if (it.b < 0) break;  // end of this CTA's items
     const int Lq = it.Lq, Lk = it.Lk;
     for (int qt = it.u0; qt < it.u1 && ok; ++qt) {
      const int i = qt * kBM + row;
      const bool valid = i < Lq;
      __nv_bfloat16* dq_row = p.g0 + ((it.qo + i) * p.H + it.h) * int64_t(D);
      if (kv_tiles_for_q_tile(qt, Lq, Lk, causal) == 0) {  // the query tile sees no key
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) store_acc_row<32>(0, 0.f, dq_row + c0, valid, true);
        continue;
      }
      if (!mbar_wait(&acc_full, acc_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      ++acc_n;
      tc_fence_after();
      drain_acc_rows<D>(tmem + lane_addr + C::kColDQ, p.scale, dq_row, valid, &acc_empty);
     }
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, item_k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================================== fused short-query pass
// For sequences whose queries fit one 128-row tile ("Four generations" item 2 splits the
// backward to avoid atomics; with a single query tile one CTA per (sequence, head) can
// own dQ outright): Q, dO and the tile's lse2 / D vectors stay resident while the key
// tiles stream once.  Per visible key tile j:
//   S^T = K_j Q^T, dP^T = V_j dO^T                  (SS, fp32 in TMEM)
//   P^T, dS^T = P^T o (dP^T - D) by the warpgroups   (P^T -> TMEM, dS^T -> shared memory)
//   dV_j = P^T dO (TS), dK_j = dS^T Q (SS)          (one query tile: stored directly)
//   dQ += dS K_j (SS, dS^T read as an MN-major A)   (accumulated in TMEM, stored at the end)
// so K and V are read once instead of once per pass, still without atomics.  Key tiles
// the query tile cannot see (causal) get zero dK / dV rows and no MMAs.
template <int D, bool kBias, bool kJBias = false>
__global__ void __launch_bounds__(kThreadsDkdv, 1) fused_kernel(const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int R = C::kRingFused;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::kTileBytes;
  uint8_t* sRing = smem + 2 * C::kTileBytes;                 // K_j, V_j single tiles
  uint8_t* sDS = sRing + R * C::kTileBytes;                  // dS^T: [keys][queries], two 64-query atoms
  float* sVec = reinterpret_cast<float*>(sDS + 32768);       // lse2[128], D[128] of the query tile

  __shared__ uint64_t q_full, q_empty, st_full, dpt_full, p_full, ds_full, dv_full, dv_empty, dk_full, dk_empty;
  __shared__ uint64_t dsm_empty, dq_full, dq_empty, mma_done;
  __shared__ uint64_t ring_full[R], ring_empty[R];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ MetaRing meta;
  __shared__ uint4 jb_scratch[kJBias ? 8 * 128 : 1];  // general bias: 2 KB transpose scratch per compute warp

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 1);
    mbar_init(&st_full, 1);
    mbar_init(&dpt_full, 1);
    mbar_init(&p_full, 256);
    mbar_init(&ds_full, 256);
    mbar_init(&dv_full, 1);
    mbar_init(&dv_empty, 128);
    mbar_init(&dk_full, 1);
    mbar_init(&dk_empty, 128);
    mbar_init(&dsm_empty, 1);
    mbar_init(&dq_full, 1);
    mbar_init(&dq_empty, 128);
    mbar_init(&mma_done, 1);
    for (int i = 0; i < R; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    meta_init(meta, p.wait_ns, 3 + (kThreadsDkdv / 32 - kFirstComputeWarp));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  grid_dependency_wait();  // the planner's lists and maps, the previous kernels' outputs
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int n_items = *p.n_items;
  volatile int* abort_flag = &abort_sh;
  const bool causal = p.causal != 0;
  // key tile kt of a sequence is visible to its (single) query tile
  auto visible = [&](int kt, int Lq, int Lk) {
    int first, count;
    q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
    return count > 0;
  };
  auto any_visible = [&](int u0, int u1, int Lq, int Lk) {
    for (int kt = u0; kt < u1; ++kt)
      if (visible(kt, Lq, Lk)) return true;
    return false;
  };

  if (warp < kFirstComputeWarp) {
   setmaxnreg_dec<kRegsLoadFused>();
   if (warp == 2) {
    // ------------------------------------------------------------ Q / dO / vector loader
    if (lane == 0) {
      uint32_t item_n = 0, tn = 0;
      int acq_b = -1;
      bool ok = true;
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
        if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
        const ItemMeta& wi = meta.e[item_k % kMetaSlots];
        if (wi.b < 0) break;  // end of this CTA's items
        if (any_visible(wi.u0, wi.u1, wi.Lq, wi.Lk)) {
          acquire_seq_maps(p.maps, wi.b, kMapQ, kMapDO, acq_b, false);
          const TileMap mq = tile_map(p.maps, p.B, kMapQ, wi.b, wi.qo, 0, p.total_q);
          const TileMap mdo = tile_map(p.maps, p.B, kMapDO, wi.b, wi.qo, 0, p.total_q);
          if (mq.tail) {
            tmap_acquire(mq.map);
            tmap_acquire(mdo.map);
          }
          const float* l2src = p.lse2 + int64_t(wi.h) * p.qpad_cap + wi.qp;
          const float* dsrc = p.delta + int64_t(wi.h) * p.qpad_cap + wi.qp;
          if (!mbar_wait(&q_empty, (item_n & 1) ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
          trace_event(p.trace, kTraceLoader, tn, 1);
          mbar_arrive_expect_tx(&q_full, 2 * C::kTileBytes + 2 * kBM * 4);
          load_tile<D>(sQ, mq.map, &q_full, wi.h * D, mq.y);
          load_tile<D>(sDO, mdo.map, &q_full, wi.h * D, mdo.y);
          bulk_load(sVec, l2src, kBM * 4, &q_full);
          bulk_load(sVec + kBM, dsrc, kBM * 4, &q_full);
          ++item_n;
        }
        meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      if (item_n > 0) drain_wait(&q_full, (item_n - 1) & 1);
    }
   } else if (warp == 0) {
    // ------------------------------------------------------------ K / V ring producer
    if (lane == 0) {
      uint32_t ring_n = 0, tn = 0;
      int acq_b = -1;
      bool ok = true;
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
        if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
        const ItemMeta& wi = meta.e[item_k % kMetaSlots];
        if (wi.b < 0) break;  // end of this CTA's items
        for (int kt = wi.u0; kt < wi.u1 && ok; ++kt) {
          if (!visible(kt, wi.Lq, wi.Lk)) continue;
          acquire_seq_maps(p.maps, wi.b, kMapK, kMapV, acq_b, false);
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const TileMap m = tile_map(p.maps, p.B, kv ? kMapV : kMapK, wi.b, wi.ko, kt, p.total_kv);
            if (m.tail) tmap_acquire(m.map);
            const uint32_t e = ring_n % R, ph = (ring_n / R) & 1;
            if (!mbar_wait(&ring_empty[e], ph ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
            trace_event(p.trace, kTraceProducer, tn, 2);
            mbar_arrive_expect_tx(&ring_full[e], C::kTileBytes);
            load_tile<D>(sRing + e * C::kTileBytes, m.map, &ring_full[e], wi.h * D, m.y);
            ++ring_n;
          }
        }
        if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      const uint32_t f = ring_n > uint32_t(R) ? ring_n - R : 0;
      for (uint32_t n = f; n < ring_n; ++n) drain_wait(&ring_full[n % R], (n / R) & 1);
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdS64 = idesc_bf16_f32(128, 64, false, false);  // Lq <= 64: 64 query columns
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, false, true);  // A K-major, B MN-major
      constexpr uint32_t kIdDq = idesc_bf16_f32(128, D, true, true);    // A (dS) and B (K) MN-major
      const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO), aR = smem_u32(sRing), aDS = smem_u32(sDS);
      uint32_t ring_n = 0, item_n = 0, g = 0, tn = 0;
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        if (!mbar_wait(bar, par, abort_flag, kWaitTimeoutNs)) return false;
        tc_fence_after();
        return true;
      };
      auto ra = [&](uint32_t n) { return aR + (n % R) * C::kTileBytes; };
      // D(128 x nq) = A(128 x D) * B(nq x D)^T, both K-major (S^T, dP^T; nq = 128, or 64 query
      // columns when the sequence has at most 64 queries)
      auto mma_nt = [&](uint32_t dcol, uint32_t a, uint32_t b, uint32_t idesc) {
        const uint64_t ad = sdesc_sw128(a, 16, 1024), bd = sdesc_sw128(b, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ss(tmem + dcol, ad + o, bd + o, idesc, kk > 0);
        }
      };
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
       if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[item_k % kMetaSlots];
       if (wi.b < 0) break;  // end of this CTA's items
       const int Lq = wi.Lq, Lk = wi.Lk;
       // at most 64 queries: S^T and dP^T with 64 query columns, dV and dK over K = 64
       const bool half = Lq <= 64;
       const uint32_t idS = half ? kIdS64 : kIdS;
       const int kq = half ? 4 : kBM / 16;  // K-steps of dV and dK
       if (any_visible(wi.u0, wi.u1, Lq, Lk)) {
        if (!wait(&q_full, item_n & 1)) { ok = false; break; }
        if (!wait(&dq_empty, (item_n & 1) ^ 1)) { ok = false; break; }
        trace_event(p.trace, kTraceMma, tn, 10);
        bool first = true;
        for (int kt = wi.u0; kt < wi.u1 && ok; ++kt) {
          if (!visible(kt, Lq, Lk)) continue;
          const uint32_t nk = ring_n, nv = ring_n + 1;
          ring_n += 2;
          // S^T = K Q^T
          if (!wait(&ring_full[nk % R], (nk / R) & 1)) { ok = false; break; }
          mma_nt(C::kColS, ra(nk), aQ, idS);
          umma_commit(&st_full);
          trace_event(p.trace, kTraceMma, tn, 13);
          // dP^T = V dO^T, into the columns dK of the previous tile is read from
          if (!wait(&dk_empty, (g & 1) ^ 1) || !wait(&ring_full[nv % R], (nv / R) & 1)) { ok = false; break; }
          mma_nt(C::kColP, ra(nv), aDO, idS);
          umma_commit(&dpt_full);
          umma_commit(&ring_empty[nv % R]);  // V is read by dP^T only
          trace_event(p.trace, kTraceMma, tn, 14);
          // dV = P^T dO  (P^T from TMEM: each warpgroup's 64 queries in its own S half)
          if (!wait(&p_full, g & 1) || !wait(&dv_empty, (g & 1) ^ 1)) { ok = false; break; }
          {
            const uint64_t bd = sdesc_sw128(aDO, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < kBM / 16 && kk < kq; ++kk)
              umma_ts(tmem + C::kColFdV, tmem + C::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                      bd + uint32_t(kk * 2048 >> 4), kIdAcc, kk > 0 ? 1u : 0u);
          }
          umma_commit(&dv_full);
          trace_event(p.trace, kTraceMma, tn, 11);
          // dK = dS^T Q (dS^T staged in shared memory, K-major over queries), into the
          // dP^T columns; then dQ += dS K (the same staging read as an MN-major A; with at
          // most 64 queries its rows 64..127 read the second atom's stale values and are
          // never stored)
          if (!wait(&ds_full, g & 1)) { ok = false; break; }
          {
            const uint64_t ad = sdesc_sw128(aDS, 16, 1024), bd = sdesc_sw128(aQ, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < kBM / 16 && kk < kq; ++kk) {
              const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
              umma_ss(tmem + C::kColP, ad + o, bd + uint32_t(kk * 2048 >> 4), kIdAcc, kk > 0 ? 1u : 0u);
            }
          }
          umma_commit(&dk_full);
          {
            const uint64_t ad = sdesc_sw128(aDS, 16384, 1024), bd = sdesc_sw128(ra(nk), 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              umma_ss(tmem + C::kColFdQ, ad + uint32_t(kk * 2048 >> 4), bd + uint32_t(kk * 2048 >> 4), kIdDq,
                      (!first || kk > 0) ? 1u : 0u);
          }
          umma_commit(&dsm_empty);
          trace_event(p.trace, kTraceMma, tn, 12);
          umma_commit(&ring_empty[nk % R]);  // K is read by S^T and dQ
          first = false;
          ++g;
        }
        if (!ok) break;
        umma_commit(&dq_full);
        umma_commit(&q_empty);
        ++item_n;
       }
       meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      umma_commit(&mma_done);
      drain_wait(&mma_done, 0);
    }
   } else if (warp == 3) {
    // ------------------------------------------------------------ scheduler
    if (lane == 0 && !meta_publish(meta, p.items, n_items, p.claim, p.q_off, p.kv_off, p.qpad, p.jb_off, abort_flag))
      raise_status(p.status, JFA_ERR_TIMEOUT);
   }
  } else if (warp < kFirstEpilogueWarp) {
    setmaxnreg_inc<kRegsComputeFused>();
    // ------------------------------------------------------------ compute warpgroups
    const int w = (warp - kFirstComputeWarp) >> 2;  // queries [64w, 64w+64)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row of S^T / dP^T / dV / dK; query row of dQ
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kColS + 64 * w;
    const uint32_t tP = tmem + lane_addr + C::kColP + 64 * w;
    const float sl2 = p.scale_log2;
    const uint64_t* nlse2v = reinterpret_cast<const uint64_t*>(sVec + 64 * w);  // -lse2 pairs
    const uint64_t* ndvec = reinterpret_cast<const uint64_t*>(sVec + kBM + 64 * w);  // -D pairs
    uint32_t g = 0, item_n = 0, tn = 0;
    const bool leader = (warp & 3) == 0 && lane == 0;
    bool ok = true;
    uint32_t item_k = 0;
    for (; ok; ++item_k) {
     if (!meta_wait_warp(meta, item_k, abort_flag)) { ok = false; break; }
     const ItemMeta& it = meta.e[item_k % kMetaSlots];
     if (it.b < 0) break;  // end of this CTA's items
     const int Lq = it.Lq, Lk = it.Lk;
     const int diag = Lk - Lq;  // key j visible to query i iff i >= j - diag
     const float* brow = kBias ? p.bias2 + size_t(it.h) * p.num_buckets : nullptr;
     const bool live = any_visible(it.u0, it.u1, Lq, Lk);
     if (live && !__all_sync(0xffffffffu, mbar_wait(&q_full, item_n & 1, abort_flag, kWaitTimeoutNs))) {
       ok = false;
       break;
     }
     for (int kt = it.u0; kt < it.u1 && ok; ++kt) {
      const int j = kt * kBN + row;  // local key index
      const bool valid = j < Lk;
      if (!visible(kt, Lq, Lk)) continue;  // zero dK / dV rows: written by the epilogue warpgroup
      if (Lq <= 64 && w == 1) {
        // every query is in warpgroup 0's columns (the MMAs run 64 query columns wide):
        // only the hand-offs, so that each barrier phase still sees both warpgroups once
        if (!mbar_wait(&st_full, g & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        tc_fence_before();
        mbar_arrive(&p_full);
        if (!mbar_wait(&dpt_full, g & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        if (!mbar_wait(&dsm_empty, (g & 1) ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        tc_fence_before();
        mbar_arrive(&ds_full);
        ++g;
        continue;
      }
      uint4 jbw[8];  // general bias for this tile (row order), loaded before the wait
      if (kJBias) {
        const int64_t pitch = (Lk + 7) / 8 * 8;  // rows of the sequence's block: bias[i][j] at i * pitch + j
        const int kj0 = kt * kBN + quarter * 32;
        jbias_load_cols_vec(jbw, p.jbias + size_t(it.h) * p.jb_plane + it.jb + int64_t(64 * w) * pitch + kj0, pitch,
                            Lq - 64 * w, Lk - kj0, lane);
      }
      // relative-position bias * log2(e) (bucket of column c: j - 64 w + center - c), loaded
      // before the wait so the loads overlap the MMAs
      float bw[kBias ? 64 : 1];
      if (kBias) {
        const int idx0 = j - 64 * w + p.center;
#pragma unroll
        for (int c = 0; c < 64; ++c) bw[c] = __ldg(brow + min(max(idx0 - c, 0), p.num_buckets - 1));
      }
      // ---- P^T = exp2(S^T * scale * log2e (+ bias) - lse2), 0 on padding and hidden pairs
      if (!mbar_wait(&st_full, g & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      tc_fence_after();
      if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 20);
      float x[64];
      ld_cols64(tS, x);
      const int i0 = 64 * w;  // query of column 0 of this half
      if (kJBias) {
        uint32_t jbk[32];
        jbias_col_transpose(jbk, jbw, jb_scratch + (warp - kFirstComputeWarp) * 128, valid, lane);
        jbias_apply<64>(x, jbk, sl2, kLog2e);
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2)
          f2_unpack(f2_add(f2_pack(x[2 * c2], x[2 * c2 + 1]), nlse2v[c2]), x[2 * c2], x[2 * c2 + 1]);
      } else if (kBias) {
        const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2)  // packed: x*scale + bias - lse2, two columns per op
          f2_unpack(f2_add(f2_fma(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2, f2_pack(bw[2 * c2], bw[2 * c2 + 1])),
                           nlse2v[c2]),
                    x[2 * c2], x[2 * c2 + 1]);
      } else {
        const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2)
          f2_unpack(f2_fma(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2, nlse2v[c2]), x[2 * c2], x[2 * c2 + 1]);
      }
      {
        // hidden: padded keys (whole row), padded queries, and i < j - diag when causal
        const int lim_q = Lq - i0;                       // columns c >= lim_q are padding
        const int lim_c = causal ? j - diag - i0 : -1;   // columns c < lim_c are hidden
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (!valid || c >= lim_q || c < lim_c) x[c] = -INFINITY;
      }
#pragma unroll
      for (int c = 0; c < 64; ++c) x[c] = ex2_approx(x[c]);
      st_bf16_64(tS, x);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full);
      if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 21);
      // ---- dS^T = P^T o (dP^T - D) -> shared memory (keys x queries, 128-byte swizzle)
      if (!mbar_wait(&dpt_full, g & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      tc_fence_after();
      if (!mbar_wait(&dsm_empty, (g & 1) ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      // bias gradient: diagonal sums of this warp's dS^T (as in dbias_warp_tile, one column
      // half at a time); hidden and padded pairs have P^T = 0, so dS^T = 0 there
      float db_straight[2] = {0.f, 0.f}, db_wrapped[2] = {0.f, 0.f};
      uint32_t gk[32];  // general bias: this key's dS^T as packed bf16 pairs of query rows
      {
        uint8_t* drow = sDS + w * 16384 + row * 128;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {  // 32 columns at a time
          uint32_t r[32];
          tmem_ld32(tP + 32 * hf, r);
          tmem_ld_wait();
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            float d8[8];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const int c = 32 * hf + 8 * ch + 2 * e2;
              const uint64_t dpp = f2_pack(__uint_as_float(r[8 * ch + 2 * e2]), __uint_as_float(r[8 * ch + 2 * e2 + 1]));
              f2_unpack(f2_mul(f2_pack(x[c], x[c + 1]), f2_add(dpp, ndvec[c >> 1])), d8[2 * e2], d8[2 * e2 + 1]);
            }
            if (kBias && p.bias_grad) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int kk = 8 * ch + e;  // round: column 32 * hf + kk of lane (lane + kk) mod 32
                const float v = __shfl_sync(0xffffffffu, d8[e], (lane + kk) & 31);
                if (lane + kk < 32)
                  db_straight[hf] += v;
                else
                  db_wrapped[hf] += v;
              }
            }
            uint4 v;
            v.x = pack_bf16x2(d8[0], d8[1]);
            v.y = pack_bf16x2(d8[2], d8[3]);
            v.z = pack_bf16x2(d8[4], d8[5]);
            v.w = pack_bf16x2(d8[6], d8[7]);
            const int chunk = 4 * hf + ch;
            *reinterpret_cast<uint4*>(drow + ((chunk ^ (row & 7)) << 4)) = v;
            if (kJBias) {  // query rows 8 chunk .. + 7 of this key, for the general bias's gradient
              gk[4 * chunk + 0] = v.x;
              gk[4 * chunk + 1] = v.y;
              gk[4 * chunk + 2] = v.z;
              gk[4 * chunk + 3] = v.w;
            }
          }
        }
      }
      fence_proxy_async_smem();  // the MMAs read the staging through the async proxy
      tc_fence_before();
      mbar_arrive(&ds_full);
      if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 22);
      if (kJBias && p.jb_grad) {  // the general bias's gradient is dS itself
        const int64_t pitch = (Lk + 7) / 8 * 8;
        const int kj0 = kt * kBN + quarter * 32;
        jbias_store_cols(gk, jb_scratch + (warp - kFirstComputeWarp) * 128,
                         p.jb_grad + size_t(it.h) * p.jb_plane + it.jb + int64_t(64 * w) * pitch + kj0, pitch,
                         Lq - 64 * w, Lk - kj0, valid, lane);
      }
      if (kBias && p.bias_grad)
        dbias_flush(db_straight[0], db_wrapped[0] + db_straight[1], db_wrapped[1],
                    p.bias_grad + size_t(it.h) * p.num_buckets, p.num_buckets,
                    kt * kBN + quarter * 32 - i0 - 63 + p.center, lane);
      ++g;
     }
     if (!ok) break;
     if (live) ++item_n;  // the item's dQ rows: written by the epilogue warpgroup
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, item_k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  } else {
    setmaxnreg_dec<kRegsEpiFused>();
    // ------------------------------------------------------------ epilogue warpgroup
    // Each key tile's dV_j and dK_j rows (this thread = one key row, all D columns; zeros
    // for tiles the query tile cannot see) and, at the item's end, its dQ rows (this thread =
    // one query row), each accumulator released once its last columns are in registers.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    uint32_t g = 0, item_n = 0;
    bool ok = true;
    uint32_t item_k = 0;
    for (; ok; ++item_k) {
     if (!meta_wait_warp(meta, item_k, abort_flag)) { ok = false; break; }
     const ItemMeta& it = meta.e[item_k % kMetaSlots];
     if (it.b < 0) break;  // end of this CTA's items
     const int Lq = it.Lq, Lk = it.Lk;
     const bool live = any_visible(it.u0, it.u1, Lq, Lk);
     for (int kt = it.u0; kt < it.u1 && ok; ++kt) {
      const int j = kt * kBN + row;  // local key index
      const bool valid = j < Lk;
      __nv_bfloat16* dk_row = p.g0 + ((it.ko + j) * p.H + it.h) * int64_t(D);
      __nv_bfloat16* dv_row = p.g1 + ((it.ko + j) * p.H + it.h) * int64_t(D);
      if (!visible(kt, Lq, Lk)) {
        store_acc_row_own<D>(0, 0.f, dk_row, valid, true);
        store_acc_row_own<D>(0, 0.f, dv_row, valid, true);
        continue;
      }
      if (!mbar_wait(&dv_full, g & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      tc_fence_after();
      drain_row_own<D>(tmem + lane_addr + C::kColFdV, 1.f, dv_row, valid, &dv_empty);
      if (!mbar_wait(&dk_full, g & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      tc_fence_after();
      drain_row_own<D>(tmem + lane_addr + C::kColP, p.scale, dk_row, valid, &dk_empty);
      ++g;
     }
     if (!ok) break;
     const bool qvalid = row < Lq;
     __nv_bfloat16* dq_row = p.g2 + ((it.qo + row) * p.H + it.h) * int64_t(D);
     if (live) {
       if (!mbar_wait(&dq_full, item_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
       ++item_n;
       tc_fence_after();
       drain_row_own<D>(tmem + lane_addr + C::kColFdQ, p.scale, dq_row, qvalid, &dq_empty);
     } else {
       store_acc_row_own<D>(0, 0.f, dq_row, qvalid, true);
     }
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, item_k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================================== non-sequence-parallel pass
// One CTA owns a (sequence, head) whose queries span 2 .. kNspMaxTiles tiles (the reading of
// "Jagged Flash Attention (JFA)", "Four generations" item 2, in which the backward is not
// parallel over a sequence's query tiles).  For each key tile j (K_j, V_j resident) and each
// query tile i that sees it (Q_i, dO_i and the tile's lse2 / D vectors through a ring),
// S^T, P^T, dP^T and dS^T are formed once and feed all three products
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i   (accumulated over i in TMEM, as in the dK/dV pass)
//   dQ_ij = dS K_j                        (dS from a shared-memory staging of dS^T)
// so a tile pair costs the five algorithmic GEMMs instead of the split passes' seven.  dQ_i
// is summed over the key tiles in an fp32 buffer of the workspace by the epilogue thread
// that owns the row -- a store at the first key tile, fp32 additions in key-tile order after
// it, the bf16 dq row written at the last key tile that sees the query tile -- so every row
// has one writer and one summation order: no atomics race and the result is deterministic.
// TMEM: S^T [0,128), dP^T [128,256), dK [256,256+D), dV [256+D,256+2D); dQ_ij goes over dP^T
// at d = 128 (after dK(i) has read dS^T there; the next dP^T waits for the dQ_ij drain) and
// into [384,448) at d = 64.
template <int D, bool kBias, bool kJBias = false>
__global__ void __launch_bounds__(kThreadsDkdv, 1) nsp_kernel(const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int R = C::kRingNsp;
  constexpr bool kDqOverDp = C::kColNspDq == C::kColP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kTileBytes;
  uint8_t* sRing = smem + 2 * C::kTileBytes;
  uint8_t* sDS = sRing + R * C::kTileBytes;             // dS^T: [keys][queries], two 64-query atoms
  float* sVec = reinterpret_cast<float*>(sDS + 32768);   // [kVecSlots][2][128]: lse2, D

  __shared__ uint64_t kv_full, kv_empty, st_full, dpt_full, p_full, ds_full, mma_done;
  __shared__ uint64_t dv_full, dv_empty, dk_full, dk_empty, dq_full, dq_empty, dsm_empty;
  __shared__ uint64_t ring_full[R], ring_empty[R];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ MetaRing meta;
  __shared__ uint4 jb_scratch[kJBias ? 8 * 128 : 1];  // general bias: 2 KB transpose scratch per compute warp

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    mbar_init(&st_full, 1);
    mbar_init(&dpt_full, 1);
    mbar_init(&p_full, 256);
    mbar_init(&ds_full, 256);
    mbar_init(&dv_full, 1);
    mbar_init(&dv_empty, 128);
    mbar_init(&dk_full, 1);
    mbar_init(&dk_empty, 128);
    mbar_init(&dq_full, 1);
    mbar_init(&dq_empty, 128);
    mbar_init(&dsm_empty, 1);
    mbar_init(&mma_done, 1);
    for (int i = 0; i < R; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    meta_init(meta, p.wait_ns, 3 + (kThreadsDkdv / 32 - kFirstComputeWarp));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  grid_dependency_wait();  // the planner's lists and maps, the previous kernels' outputs
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int n_items = *p.n_items;
  volatile int* abort_flag = &abort_sh;
  const bool causal = p.causal != 0;

  if (warp < kFirstComputeWarp) {
   setmaxnreg_dec<kRegsLoadNsp>();
   if (warp == 2) {
    // ------------------------------------------------------------ K/V loader
    if (lane == 0) {
      uint32_t item_n = 0;
      int acq_b = -1;  // sequence whose maps this thread has acquired
      bool ok = true;
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
        if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
        const ItemMeta& wi = meta.e[item_k % kMetaSlots];  // read in place, freed after the item
        if (wi.b < 0) break;  // end of this CTA's items
        const int Lq = wi.Lq, Lk = wi.Lk;
        acquire_seq_maps(p.maps, wi.b, kMapK, kMapV, acq_b, false);
        for (int kt = wi.u0; kt < wi.u1 && ok; ++kt) {
          int first, count;
          q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
          if (count == 0) continue;
          const TileMap mk = tile_map(p.maps, p.B, kMapK, wi.b, wi.ko, kt, p.total_kv);
          const TileMap mv = tile_map(p.maps, p.B, kMapV, wi.b, wi.ko, kt, p.total_kv);
          if (mk.tail) {
            tmap_acquire(mk.map);
            tmap_acquire(mv.map);
          }
          if (!mbar_wait(&kv_empty, (item_n & 1) ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
          mbar_arrive_expect_tx(&kv_full, 2 * C::kTileBytes);
          load_tile<D>(sK, mk.map, &kv_full, wi.h * D, mk.y);
          load_tile<D>(sV, mv.map, &kv_full, wi.h * D, mv.y);
          ++item_n;
          // the next key tile of this item, else the first of this CTA's next item, into L2
          int nb = -1, nh = 0, nt = 0;
          if (kt + 1 < wi.u1) {
            nb = wi.b, nh = wi.h, nt = kt + 1;
          } else if (const ItemMeta* wn = meta_peek_next(meta, item_k)) {
            nb = wn->b, nh = wn->h, nt = wn->u0;
          }
          if (nb >= 0) {
            const int64_t nko = p.kv_off[nb];
            acquire_seq_maps(p.maps, nb, kMapK, kMapV, acq_b, true);
            if (nt * kBN < int(p.kv_off[nb + 1] - nko)) {
              prefetch_tile<D / 64>(p.maps, p.B, kMapK, nb, nko, nt, p.total_kv, nh * D);
              prefetch_tile<D / 64>(p.maps, p.B, kMapV, nb, nko, nt, p.total_kv, nh * D);
            }
          }
        }
        if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      if (item_n > 0) drain_wait(&kv_full, (item_n - 1) & 1);
    }
   } else if (warp == 0) {
    // ------------------------------------------------------------ dO / Q ring producer
    if (lane == 0) {
      uint32_t ring_n = 0, qtile_n = 0, tn = 0;
      int acq_b = -1;
      bool ok = true;
      auto fill = [&](const TileMap& m, int col, const float* l2src, const float* dsrc) {
        const uint32_t e = ring_n % R, ph = (ring_n / R) & 1;
        if (m.tail) tmap_acquire(m.map);
        if (!mbar_wait(&ring_empty[e], ph ^ 1, abort_flag, kWaitTimeoutNs)) return false;
        trace_event(p.trace, kTraceProducer, tn, 2);
        mbar_arrive_expect_tx(&ring_full[e], C::kTileBytes + (l2src ? 2 * kBM * 4 : 0));
        load_tile<D>(sRing + e * C::kTileBytes, m.map, &ring_full[e], col, m.y);
        if (l2src) {
          float* v = sVec + (qtile_n % C::kVecSlots) * 256;
          bulk_load(v, l2src, kBM * 4, &ring_full[e]);
          bulk_load(v + 128, dsrc, kBM * 4, &ring_full[e]);
        }
        ++ring_n;
        return true;
      };
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
        if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
        const ItemMeta& wi = meta.e[item_k % kMetaSlots];
        if (wi.b < 0) break;  // end of this CTA's items
        const int Lq = wi.Lq, Lk = wi.Lk;
        acquire_seq_maps(p.maps, wi.b, kMapQ, kMapDO, acq_b, false);
        const int64_t vec0 = int64_t(wi.h) * p.qpad_cap + wi.qp;
        for (int kt = wi.u0; kt < wi.u1 && ok; ++kt) {
          int first, count;
          q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
          for (int i = 0; i < count && ok; ++i) {
            const int qt = first + i;
            const TileMap mdo = tile_map(p.maps, p.B, kMapDO, wi.b, wi.qo, qt, p.total_q);
            const TileMap mq = tile_map(p.maps, p.B, kMapQ, wi.b, wi.qo, qt, p.total_q);
            // Q first: it is released after dK, dO after dV, so with Q ahead the next Q's
            // slot frees up a tile pair earlier (S^T of the next query tile is not held up)
            if (!fill(mq, wi.h * D, p.lse2 + vec0 + qt * kBM, p.delta + vec0 + qt * kBM)) {
              ok = false;
              break;
            }
            if (!fill(mdo, wi.h * D, nullptr, nullptr)) { ok = false; break; }
            ++qtile_n;
          }
        }
        if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      const uint32_t f = ring_n > uint32_t(R) ? ring_n - R : 0;
      for (uint32_t n = f; n < ring_n; ++n) drain_wait(&ring_full[n % R], (n / R) & 1);
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, false, true);  // A K-major (TMEM), B MN-major
      constexpr uint32_t kIdDq = idesc_bf16_f32(128, D, true, true);    // A (dS) and B (K) MN-major
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aR = smem_u32(sRing), aDS = smem_u32(sDS);
      uint32_t ring_n = 0, item_n = 0, g = 0, acc_n = 0, tn = 0;
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        if (!mbar_wait(bar, par, abort_flag, kWaitTimeoutNs)) return false;
        tc_fence_after();
        return true;
      };
      auto wait_ring = [&](uint32_t n) { return wait(&ring_full[n % R], (n / R) & 1); };
      auto ra = [&](uint32_t n) { return aR + (n % R) * C::kTileBytes; };
      auto mma_nt = [&](uint32_t dcol, uint32_t a, uint32_t b) {  // (keys x queries) = A(keys x D) B(queries x D)^T
        const uint64_t ad = sdesc_sw128(a, 16, 1024), bd = sdesc_sw128(b, 16, 1024);
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ss(tmem + dcol, ad + o, bd + o, kIdS, kk > 0);
        }
      };
      auto mma_acc = [&](uint32_t dcol, uint32_t xcol, uint32_t b, bool acc) {  // acc(keys x D) += X^T B
        const uint64_t bd = sdesc_sw128(b, 16384, 1024);
#pragma unroll 1
        for (int kk = 0; kk < kBM / 16; ++kk)
          umma_ts(tmem + dcol, tmem + xcol + (kk >> 2) * 64 + (kk & 3) * 8, bd + uint32_t(kk * 2048 >> 4), kIdAcc,
                  (acc || kk > 0) ? 1u : 0u);
      };
      uint32_t item_k = 0;
      for (; ok; ++item_k) {
       if (!meta_wait(meta, item_k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[item_k % kMetaSlots];
       if (wi.b < 0) break;  // end of this CTA's items
       const int Lq = wi.Lq, Lk = wi.Lk;
       for (int kt = wi.u0; kt < wi.u1 && ok; ++kt) {
        int first, count;
        q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
        if (count == 0) continue;
        if (!wait(&kv_full, item_n & 1)) { ok = false; break; }
        ++item_n;
        trace_event(p.trace, kTraceMma, tn, 10);
        const uint32_t n0 = ring_n;  // Q_i at n0 + 2i, dO_i at n0 + 2i + 1
        if (!wait_ring(n0)) { ok = false; break; }
        mma_nt(C::kColS, aK, ra(n0));
        umma_commit(&st_full);
        // d = 128: dP^T's columns held the previous tile pair's dQ: wait for its drain
        if (kDqOverDp && !wait(&dq_empty, (g & 1) ^ 1)) { ok = false; break; }
        if (!wait_ring(n0 + 1)) { ok = false; break; }
        mma_nt(C::kColP, aV, ra(n0 + 1));
        umma_commit(&dpt_full);
        for (int i = 0; i < count && ok; ++i) {
          const uint32_t nq = n0 + 2 * i, nd = nq + 1;
          if (!wait(&p_full, g & 1)) { ok = false; break; }
          trace_event(p.trace, kTraceMma, tn, 11);
          if (i == 0 && !wait(&dv_empty, (acc_n & 1) ^ 1)) { ok = false; break; }
          mma_acc(C::kColA1, C::kColS, ra(nd), i > 0);  // dV += P^T dO
          umma_commit(&ring_empty[nd % R]);
          if (i + 1 == count) umma_commit(&dv_full);
          if (i + 1 < count) {
            if (!wait_ring(nq + 2)) { ok = false; break; }
            mma_nt(C::kColS, aK, ra(nq + 2));
            umma_commit(&st_full);
          }
          if (!wait(&ds_full, g & 1)) { ok = false; break; }
          trace_event(p.trace, kTraceMma, tn, 14);
          if (i == 0 && !wait(&dk_empty, (acc_n & 1) ^ 1)) { ok = false; break; }
          mma_acc(C::kColA0, C::kColP, ra(nq), i > 0);  // dK += dS^T Q
          umma_commit(&ring_empty[nq % R]);
          // dQ_ij = dS K_j: the staging read as an MN-major A (queries x keys), K MN-major
          if (!kDqOverDp && !wait(&dq_empty, (g & 1) ^ 1)) { ok = false; break; }
          {
            const uint64_t ad = sdesc_sw128(aDS, 16384, 1024), bd = sdesc_sw128(aK, 16384, 1024);
#pragma unroll 1
            for (int kk = 0; kk < kBN / 16; ++kk)
              umma_ss(tmem + C::kColNspDq, ad + uint32_t(kk * 2048 >> 4), bd + uint32_t(kk * 2048 >> 4), kIdDq,
                      kk > 0 ? 1u : 0u);
          }
          umma_commit(&dq_full);
          umma_commit(&dsm_empty);
          trace_event(p.trace, kTraceMma, tn, 15);
          if (i + 1 < count) {
            if (kDqOverDp && !wait(&dq_empty, g & 1)) { ok = false; break; }
            trace_event(p.trace, kTraceMma, tn, 16);
            if (!wait_ring(nd + 2)) { ok = false; break; }
            mma_nt(C::kColP, aV, ra(nd + 2));
            umma_commit(&dpt_full);
            trace_event(p.trace, kTraceMma, tn, 17);
          }
          ++g;
        }
        if (!ok) break;
        ring_n = n0 + 2 * count;
        ++acc_n;
        umma_commit(&dk_full);
        umma_commit(&kv_empty);  // K is read by S^T and dQ, V by dP^T
       }
       if (ok) meta_release(meta, item_k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      umma_commit(&mma_done);
      drain_wait(&mma_done, 0);
    }
   } else if (warp == 3) {
    // ------------------------------------------------------------ scheduler
    if (lane == 0 && !meta_publish(meta, p.items, n_items, p.claim, p.q_off, p.kv_off, p.qpad, p.jb_off, abort_flag))
      raise_status(p.status, JFA_ERR_TIMEOUT);
   }
  } else if (warp < kFirstEpilogueWarp) {
    setmaxnreg_inc<kRegsComputeNsp>();
    // ------------------------------------------------------------ compute warpgroups
    const int w = (warp - kFirstComputeWarp) >> 2;  // column half owned: queries [64w, 64w+64)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row within the tile
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kColS + 64 * w;
    const uint32_t tP = tmem + lane_addr + C::kColP + 64 * w;
    uint8_t* drow = sDS + w * 16384 + row * 128;  // this key's 64 queries in the dS^T staging
    const float sl2 = p.scale_log2;
    uint32_t ring_n = 0, tile_n = 0, qtile_n = 0, tn = 0;
    const bool leader = (warp & 3) == 0 && lane == 0;
    bool ok = true;
    uint32_t item_k = 0;
    for (; ok; ++item_k) {
     if (!meta_wait_warp(meta, item_k, abort_flag)) { ok = false; break; }
     const ItemMeta& it = meta.e[item_k % kMetaSlots];
     if (it.b < 0) break;  // end of this CTA's items
     const int Lq = it.Lq, Lk = it.Lk;
     for (int kt = it.u0; kt < it.u1 && ok; ++kt) {
      int first, count;
      q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
      const int j = kt * kBN + row;  // local key index
      if (count == 0) continue;  // rows of zeros: written by the epilogue warpgroup
      const int diag = Lk - Lq;  // key j visible to query i iff i >= j - diag
      const float* brow = kBias ? p.bias2 + size_t(it.h) * p.num_buckets : nullptr;
      for (int i = 0; i < count && ok; ++i) {
        const int qt = first + i;
        uint4 jbw[8];  // general bias for this tile (row order), loaded before the waits
        if (kJBias) {
          const int64_t pitch = (Lk + 7) / 8 * 8;
          const int qi0 = qt * kBM + 64 * w, kj0 = kt * kBN + quarter * 32;
          jbias_load_cols_vec(jbw, p.jbias + size_t(it.h) * p.jb_plane + it.jb + int64_t(qi0) * pitch + kj0, pitch,
                              Lq - qi0, Lk - kj0, lane);
        }
        // relative-position bias * log2(e) of this tile (bucket of column c: idx0 - c), loaded
        // before the waits so the loads overlap the MMAs
        float bw[kBias ? 64 : 1];
        if (kBias) {
          const int idx0 = j - (qt * kBM + 64 * w) + p.center;
          if (idx0 - 63 >= 0 && idx0 < p.num_buckets) {
#pragma unroll
            for (int c = 0; c < 64; ++c) bw[c] = __ldg(brow + idx0 - c);
          } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) bw[c] = __ldg(brow + min(max(idx0 - c, 0), p.num_buckets - 1));
          }
        }
        // Q_i's ring slot (the first of the pair) carries this tile's lse2 / D vectors
        const uint32_t nq = ring_n;
        if (!mbar_wait(&ring_full[nq % R], (nq / R) & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        ring_n += 2;
        const float* vec = sVec + (qtile_n % C::kVecSlots) * 256;
        ++qtile_n;
        const uint64_t* nlse2 = reinterpret_cast<const uint64_t*>(vec + 64 * w);        // -lse2 pairs
        const uint64_t* ndvec = reinterpret_cast<const uint64_t*>(vec + 128 + 64 * w);  // -D pairs
        if (!mbar_wait(&st_full, tile_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 20);
        float x[64];
        ld_cols64(tS, x);
        const int i0 = qt * kBM + 64 * w;  // local query index of column 0 of this half
        if (kJBias) {
          uint32_t jbk[32];
          jbias_col_transpose(jbk, jbw, jb_scratch + (warp - kFirstComputeWarp) * 128, j < Lk, lane);
          jbias_apply<64>(x, jbk, sl2, kLog2e);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)
            f2_unpack(f2_add(f2_pack(x[2 * c2], x[2 * c2 + 1]), nlse2[c2]), x[2 * c2], x[2 * c2 + 1]);
        } else if (kBias) {
          const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)  // packed: x*scale + bias - lse2, two columns per op
            f2_unpack(f2_add(f2_fma(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2, f2_pack(bw[2 * c2], bw[2 * c2 + 1])),
                             nlse2[c2]),
                      x[2 * c2], x[2 * c2 + 1]);
        } else {
          const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)
            f2_unpack(f2_fma(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2, nlse2[c2]), x[2 * c2], x[2 * c2 + 1]);
        }
        if (causal) {
          const int lim = j - diag - i0;  // columns c < lim are hidden
          if (lim > 0) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c < lim) x[c] = -INFINITY;
          }
        }
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = ex2_approx(x[c]);  // P^T
        st_bf16_64(tS, x);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full);
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 21);
        if (!mbar_wait(&dpt_full, tile_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 22);
        float dp[64];
        ld_cols64(tP, dp);
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2)  // dS^T = P^T o (dP^T - D)
          f2_unpack(f2_mul(f2_pack(x[2 * c2], x[2 * c2 + 1]), f2_add(f2_pack(dp[2 * c2], dp[2 * c2 + 1]), ndvec[c2])),
                    dp[2 * c2], dp[2 * c2 + 1]);
        uint32_t pk[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) pk[t] = pack_bf16x2(dp[2 * t], dp[2 * t + 1]);
        tmem_st32(tP, pk);  // for dK (TMEM operand)
        // and into the staging for dQ, once the previous tile pair's dQ MMA has read it
        if (!mbar_wait(&dsm_empty, (tile_n & 1) ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
#pragma unroll
        for (int chunk = 0; chunk < 8; ++chunk)
          *reinterpret_cast<uint4*>(drow + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * chunk], pk[4 * chunk + 1], pk[4 * chunk + 2], pk[4 * chunk + 3]);
        fence_proxy_async_smem();  // the MMAs read the staging through the async proxy
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_full);
        ++tile_n;
        if (leader) trace_event(p.trace, kTraceCompute0 + w, tn, 23);
        if (kJBias && p.jb_grad) {  // the general bias's gradient is dS itself
          const int64_t pitch = (Lk + 7) / 8 * 8;
          const int kj0 = kt * kBN + quarter * 32;
          jbias_store_cols(pk, jb_scratch + (warp - kFirstComputeWarp) * 128,
                           p.jb_grad + size_t(it.h) * p.jb_plane + it.jb + int64_t(i0) * pitch + kj0, pitch, Lq - i0,
                           Lk - kj0, j < Lk, lane);
        }
        if (kBias && p.bias_grad) {
          // dS^T of a padded key row is not zero (k = 0 but lse2 of the query is not), and
          // padded query columns only give 0 while their P^T stays finite: count neither
          const int ncols = j < Lk ? Lq - i0 : 0;
          if (ncols < 64) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c >= ncols) dp[c] = 0.f;
          }
          dbias_warp_tile(dp, p.bias_grad + size_t(it.h) * p.num_buckets, p.num_buckets,
                          kt * kBN + quarter * 32 - i0 - 63 + p.center, lane);
        }
      }
      if (!ok) break;
     }
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, item_k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  } else {
    setmaxnreg_dec<kRegsEpiNsp>();
    // ------------------------------------------------------------ epilogue warpgroup
    // Per tile pair: this thread's dQ_ij row (TMEM lane = query row) into the fp32 sum
    // (store, then additions, then the bf16 dq row at the query tile's last key tile).  Per
    // key tile: its dV and dK rows (TMEM lane = key row), as in the dK/dV pass.  Per item:
    // zero dq rows for query tiles that see no key.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    uint32_t acc_n = 0, g = 0, tn = 0;
    const bool leader = warp == kFirstEpilogueWarp && lane == 0;  // traces as role 4 in this pass
    bool ok = true;
    uint32_t item_k = 0;
    for (; ok; ++item_k) {
     if (!meta_wait_warp(meta, item_k, abort_flag)) { ok = false; break; }
     const ItemMeta& it = meta.e[item_k % kMetaSlots];
     if (it.b < 0) break;  // end of this CTA's items
     const int64_t ko = it.ko, qo = it.qo;
     const int Lq = it.Lq, Lk = it.Lk;
     const int nq = (Lq + kBM - 1) / kBM;
     for (int qt = 0; qt < nq; ++qt) {  // query tiles no key reaches: zero dq rows
       if (kv_tiles_for_q_tile(qt, Lq, Lk, causal) > 0) continue;
       const int qi = qt * kBM + row;
       store_acc_row_own<D>(0, 0.f, p.g2 + ((qo + qi) * p.H + it.h) * int64_t(D), qi < Lq, true);
     }
     for (int kt = it.u0; kt < it.u1 && ok; ++kt) {
      int first, count;
      q_tiles_for_kv_tile(kt, Lq, Lk, causal, &first, &count);
      const int j = kt * kBN + row;  // local key index
      const bool valid = j < Lk;
      __nv_bfloat16* dk_row = p.g0 + ((ko + j) * p.H + it.h) * int64_t(D);
      __nv_bfloat16* dv_row = p.g1 + ((ko + j) * p.H + it.h) * int64_t(D);
      if (count == 0) {  // no query sees these keys
        if (kt * kBN < Lk) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            store_acc_row<32>(0, 0.f, dk_row + c0, valid, true);
            store_acc_row<32>(0, 0.f, dv_row + c0, valid, true);
          }
        }
        continue;
      }
      for (int i = 0; i < count && ok; ++i) {
        const int qt = first + i;
        const int qi = qt * kBM + row;  // local query index of this thread's dQ row
        const bool qvalid = qi < Lq;
        const int jl = kv_tiles_for_q_tile(qt, Lq, Lk, causal) - 1;  // last key tile that sees qt
        float* acc = p.dqacc + ((qo + qi) * p.H + it.h) * int64_t(D);
        __nv_bfloat16* dq_row = p.g2 + ((qo + qi) * p.H + it.h) * int64_t(D);
        if (!mbar_wait(&dq_full, g & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        ++g;
        tc_fence_after();
        if (leader) trace_event(p.trace, kTraceLoader, tn, 30);
        // one thread per row: each chunk of 32 columns leaves as eight 16-byte operations
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_addr + C::kColNspDq + c0, r);
          tmem_ld_wait();
          if (c0 + 32 == D) {  // the whole row is in registers: the MMA may reuse the columns
            tc_fence_before();
            mbar_arrive(&dq_empty);
            if (leader) trace_event(p.trace, kTraceLoader, tn, 31);
          }
          if (!qvalid) continue;  // a padding query row
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float* a4 = acc + c0 + 4 * k;
            float v0 = __uint_as_float(r[4 * k]), v1 = __uint_as_float(r[4 * k + 1]),
                  v2 = __uint_as_float(r[4 * k + 2]), v3 = __uint_as_float(r[4 * k + 3]);
            if (kt == jl) {  // the last contribution: finish the row segment in bf16
              if (kt > 0) {  // add the sum of the earlier key tiles
                const float4 a = ld_global_cg_v4f(a4);
                v0 += a.x, v1 += a.y, v2 += a.z, v3 += a.w;
              }
              *reinterpret_cast<uint2*>(dq_row + c0 + 4 * k) =
                  make_uint2(pack_bf16x2(v0 * p.scale, v1 * p.scale), pack_bf16x2(v2 * p.scale, v3 * p.scale));
            } else if (kt == 0) {  // the first contribution: store
              st_global_v4f(a4, v0, v1, v2, v3);
            } else {  // in between: add (this row has one owner, so the order is the key tiles')
              red_add_global_v4(a4, v0, v1, v2, v3);
            }
          }
        }
      }
      if (!ok) break;
      if (leader) trace_event(p.trace, kTraceLoader, tn, 32);
      if (!mbar_wait(&dv_full, acc_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      tc_fence_after();
      drain_acc_rows<D>(tmem + lane_addr + C::kColA1, 1.f, dv_row, valid, &dv_empty);
      if (!mbar_wait(&dk_full, acc_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      ++acc_n;
      tc_fence_after();
      drain_acc_rows<D>(tmem + lane_addr + C::kColA0, p.scale, dk_row, valid, &dk_empty);
     }
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, item_k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

enum BwdPass { kPassDkdv = 0, kPassDq = 1, kPassFused = 2, kPassNsp = 3 };

BwdParams make_params(const Problem& pr, const float* lse, void* ws, const WsLayout& L, int pass) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  BwdParams bp;
  bp.q_off = pr.q_off;
  bp.kv_off = pr.kv_off;
  bp.B = pr.B;
  bp.H = pr.H;
  bp.total_q = pr.total_q;
  bp.total_kv = pr.total_kv;
  bp.scale = pr.scale;
  bp.scale_log2 = pr.scale * kLog2e;
  bp.causal = pr.causal;
  bp.bias2 = pr.bias_table ? reinterpret_cast<const float*>(w + L.bias2) : nullptr;
  // the dK/dV, fused and non-sequence-parallel passes together see every visible pair once:
  // they add the bias gradient
  bp.bias_grad = (pr.bias_table && pass != kPassDq) ? pr.bias_grad : nullptr;
  bp.num_buckets = pr.num_buckets;
  bp.center = pr.center;
  bp.jbias = static_cast<const __nv_bfloat16*>(pr.jbias);
  bp.jb_off = pr.jb_off;
  bp.jb_plane = pr.jb_plane;
  bp.jb_grad = pass != kPassDq ? static_cast<__nv_bfloat16*>(pr.jb_grad) : nullptr;
  bp.maps = reinterpret_cast<const CUtensorMap*>(w + L.maps);
  bp.items = reinterpret_cast<const WorkItem*>(
      w + (pass == kPassDq ? L.dq : pass == kPassFused ? L.fused : pass == kPassNsp ? L.nsp : L.dkv));
  const WsHeader* hdr = reinterpret_cast<const WsHeader*>(w);
  bp.n_items = pass == kPassDq ? &hdr->n_dq : pass == kPassFused ? &hdr->n_fused
                                           : pass == kPassNsp ? &hdr->n_nsp : &hdr->n_dkv;
  WsHeader* mh = reinterpret_cast<WsHeader*>(w);
  bp.claim = pass == kPassDq ? &mh->claim_dq : pass == kPassFused ? &mh->claim_fused
                                             : pass == kPassNsp ? &mh->claim_nsp : &mh->claim_dkv;
  bp.status = &reinterpret_cast<WsHeader*>(w)->status;
  // list kinds of the planner: forward 0, dQ 1, dK/dV 2, fused 3, non-sequence-parallel 4
  bp.wait_ns = &hdr->wait_ns[pass == kPassDq ? 1 : pass == kPassFused ? 3 : pass == kPassNsp ? 4 : 2];
  bp.dqacc = reinterpret_cast<float*>(w + L.dqacc);
  (void)lse;
  bp.lse2 = reinterpret_cast<const float*>(w + L.lse2);
  bp.delta = reinterpret_cast<const float*>(w + L.delta);
  bp.qpad = reinterpret_cast<const int64_t*>(w + L.qpad);
  bp.qpad_cap = L.qpad_cap;
  bp.g0 = nullptr;
  bp.g1 = nullptr;
  bp.g2 = nullptr;
  bp.trace = pr.trace[pass == kPassDq ? JFA_KERNEL_BWD_DQ : pass == kPassFused ? JFA_KERNEL_BWD_FUSED
                     : pass == kPassNsp ? JFA_KERNEL_BWD_NSP : JFA_KERNEL_BWD_DKDV];
  return bp;
}

}  // namespace

cudaError_t launch_bwd_preprocess(const Problem& pr, const void* dout, const void* out, const float* lse,
                                  void* ws, const WsLayout& L, int num_sms, cudaStream_t stream) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  PreParams pp;
  pp.q_off = pr.q_off;
  pp.B = pr.B;
  pp.H = pr.H;
  pp.total_q = pr.total_q;
  pp.items = reinterpret_cast<const WorkItem*>(w + L.dq);
  pp.n_items = &reinterpret_cast<const WsHeader*>(w)->n_dq;
  pp.items2 = reinterpret_cast<const WorkItem*>(w + L.fused);
  pp.n_items2 = &reinterpret_cast<const WsHeader*>(w)->n_fused;
  pp.items3 = reinterpret_cast<const WorkItem*>(w + L.nsp);
  pp.n_items3 = &reinterpret_cast<const WsHeader*>(w)->n_nsp;
  pp.qpad = reinterpret_cast<const int64_t*>(w + L.qpad);
  pp.total_qpad = &reinterpret_cast<const WsHeader*>(w)->total_qpad;
  pp.qpad_cap = L.qpad_cap;
  pp.dout = static_cast<const __nv_bfloat16*>(dout);
  pp.out = static_cast<const __nv_bfloat16*>(out);
  pp.lse = lse;
  pp.lse2 = reinterpret_cast<float*>(w + L.lse2);
  pp.delta = reinterpret_cast<float*>(w + L.delta);
  // row-parallel for wide token rows (every block resident at once, 4 per SM at <= 64
  // registers); per item otherwise
  const bool wide = int64_t(pr.H) * pr.d >= 1024;
  if (pr.d == 128)
    return wide ? launch_pdl(preprocess_kernel<128>, dim3(4 * num_sms), dim3(256), 0, stream, pp)
                : launch_pdl(preprocess_items_kernel<128>, dim3(8 * num_sms), dim3(256), 0, stream, pp);
  return wide ? launch_pdl(preprocess_kernel<64>, dim3(4 * num_sms), dim3(256), 0, stream, pp)
              : launch_pdl(preprocess_items_kernel<64>, dim3(8 * num_sms), dim3(256), 0, stream, pp);
}

template <typename K>
cudaError_t launch_dkdv_k(K kern, int smem, int grid, const BwdParams& bp, cudaStream_t stream) {
  cudaError_t e = check_launch_registers(kern, kLaunchRegsDkdv);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreadsDkdv), smem, stream, bp);
}

cudaError_t launch_bwd_dkdv(const Problem& pr, const float* lse, void* ws, const WsLayout& L, void* dk, void* dv,
                            int num_sms, cudaStream_t stream) {
  BwdParams bp = make_params(pr, lse, ws, L, kPassDkdv);
  bp.g0 = static_cast<__nv_bfloat16*>(dk);
  bp.g1 = static_cast<__nv_bfloat16*>(dv);
  const bool bias = pr.bias_table != nullptr, jb = pr.jbias != nullptr;
  if (pr.d == 128)
    return bias ? launch_dkdv_k(dkdv_kernel<128, true>, BwdCfg<128>::kSmemDkdv, num_sms, bp, stream)
                : jb ? launch_dkdv_k(dkdv_kernel<128, false, true>, BwdCfg<128>::kSmemDkdv, num_sms, bp, stream)
                     : launch_dkdv_k(dkdv_kernel<128, false>, BwdCfg<128>::kSmemDkdv, num_sms, bp, stream);
  return bias ? launch_dkdv_k(dkdv_kernel<64, true>, BwdCfg<64>::kSmemDkdv, num_sms, bp, stream)
              : jb ? launch_dkdv_k(dkdv_kernel<64, false, true>, BwdCfg<64>::kSmemDkdv, num_sms, bp, stream)
                   : launch_dkdv_k(dkdv_kernel<64, false>, BwdCfg<64>::kSmemDkdv, num_sms, bp, stream);
}

cudaError_t launch_bwd_fused(const Problem& pr, const float* lse, void* ws, const WsLayout& L, void* dq, void* dk,
                             void* dv, int num_sms, cudaStream_t stream) {
  BwdParams bp = make_params(pr, lse, ws, L, kPassFused);
  bp.g0 = static_cast<__nv_bfloat16*>(dk);
  bp.g1 = static_cast<__nv_bfloat16*>(dv);
  bp.g2 = static_cast<__nv_bfloat16*>(dq);
  const bool bias = pr.bias_table != nullptr, jb = pr.jbias != nullptr;
  if (pr.d == 128)
    return bias ? launch_dkdv_k(fused_kernel<128, true>, BwdCfg<128>::kSmemFused, num_sms, bp, stream)
                : jb ? launch_dkdv_k(fused_kernel<128, false, true>, BwdCfg<128>::kSmemFused, num_sms, bp, stream)
                     : launch_dkdv_k(fused_kernel<128, false>, BwdCfg<128>::kSmemFused, num_sms, bp, stream);
  return bias ? launch_dkdv_k(fused_kernel<64, true>, BwdCfg<64>::kSmemFused, num_sms, bp, stream)
              : jb ? launch_dkdv_k(fused_kernel<64, false, true>, BwdCfg<64>::kSmemFused, num_sms, bp, stream)
                   : launch_dkdv_k(fused_kernel<64, false>, BwdCfg<64>::kSmemFused, num_sms, bp, stream);
}

cudaError_t launch_bwd_dq(const Problem& pr, const float* lse, void* ws, const WsLayout& L, void* dq, int num_sms,
                          cudaStream_t stream) {
  BwdParams bp = make_params(pr, lse, ws, L, kPassDq);
  bp.g0 = static_cast<__nv_bfloat16*>(dq);
  const bool bias = pr.bias_table != nullptr, jb = pr.jbias != nullptr;
  if (pr.d == 128)
    return bias ? launch_dkdv_k(dq_kernel<128, true>, BwdCfg<128>::kSmemDq, num_sms, bp, stream)
                : jb ? launch_dkdv_k(dq_kernel<128, false, true>, BwdCfg<128>::kSmemDq, num_sms, bp, stream)
                     : launch_dkdv_k(dq_kernel<128, false>, BwdCfg<128>::kSmemDq, num_sms, bp, stream);
  return bias ? launch_dkdv_k(dq_kernel<64, true>, BwdCfg<64>::kSmemDq, num_sms, bp, stream)
              : jb ? launch_dkdv_k(dq_kernel<64, false, true>, BwdCfg<64>::kSmemDq, num_sms, bp, stream)
                   : launch_dkdv_k(dq_kernel<64, false>, BwdCfg<64>::kSmemDq, num_sms, bp, stream);
}

cudaError_t launch_bwd_nsp(const Problem& pr, const float* lse, void* ws, const WsLayout& L, void* dq, void* dk,
                           void* dv, int num_sms, cudaStream_t stream) {
  BwdParams bp = make_params(pr, lse, ws, L, kPassNsp);
  bp.g0 = static_cast<__nv_bfloat16*>(dk);
  bp.g1 = static_cast<__nv_bfloat16*>(dv);
  bp.g2 = static_cast<__nv_bfloat16*>(dq);
  const bool bias = pr.bias_table != nullptr, jb = pr.jbias != nullptr;
  if (pr.d == 128)
    return bias ? launch_dkdv_k(nsp_kernel<128, true>, BwdCfg<128>::kSmemNsp, num_sms, bp, stream)
                : jb ? launch_dkdv_k(nsp_kernel<128, false, true>, BwdCfg<128>::kSmemNsp, num_sms, bp, stream)
                     : launch_dkdv_k(nsp_kernel<128, false>, BwdCfg<128>::kSmemNsp, num_sms, bp, stream);
  return bias ? launch_dkdv_k(nsp_kernel<64, true>, BwdCfg<64>::kSmemNsp, num_sms, bp, stream)
              : jb ? launch_dkdv_k(nsp_kernel<64, false, true>, BwdCfg<64>::kSmemNsp, num_sms, bp, stream)
                   : launch_dkdv_k(nsp_kernel<64, false>, BwdCfg<64>::kSmemNsp, num_sms, bp, stream);
}

}  // namespace jfa
