// Jagged Flash Attention forward for sm_103a.
//
// What it computes: exact softmax attention per jagged sequence ("Jagged Flash
// Attention (JFA)", Definition), via tiling plus online softmax ("TLX-Optimized
// Jagged Flash Attention ...", section "Why Jagged Flash Attention Deserves
// Attention"), with the jagged boundary handled by the subtraction scheme ("Four
// generations" item 1): tile loads through per-sequence tensor maps deliver zero
// rows past the sequence end, so padded keys score exactly 0; their contribution
// n_pad * exp(0 - m) is subtracted from the row sum once, on the last key tile.
// No -inf mask pass touches jagged boundaries (causal masking of diagonal tiles is
// a real mask, not a jagged one).
//
// How (one persistent CTA per SM, "Four generations" item 3: warp specialisation
// plus persistent scheduling over a longest-first work list):
//   warp 0      K/V producer: K_j, V_j into a ring of smem stages (TMA)
//   warp 1      MMA issuer:   S_s = Q_s K_j^T (tcgen05, SS, fp32 in TMEM);
//                             O_s += P_s V_j (tcgen05, A = P from TMEM, B = V from smem)
//   warp 2      Q loader: the unit's pair of query tiles
//   warp 3      scheduler: work-item metadata into a shared-memory ring
//   warps 4-7   softmax for query tile 0 of the pair (one TMEM lane = one query row)
//   warps 8-11  softmax for query tile 1
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 [256+d, 256+2d).
// P (bf16, two per column) overwrites the first 64 columns of its S region.  At d = 64 the
// query tiles are copied into Q_0 [384,416), Q_1 [416,448) and feed the S MMAs from TMEM.
// The issue order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) lets one tile's softmax
// overlap the other tile's MMAs (ping-pong).  The running max is only raised (and O
// rescaled) when it grows by more than 2^8, which keeps exp2 arguments <= 8 in between.
#include <cuda_bf16.h>

#include "jfa_internal.h"
#include "sm100_ptx.cuh"
#include "jfa_sched.cuh"

namespace jfa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kRegsLoad = 120, kRegsCompute = 192;
static_assert(reg_split_fits(kRegsLoad, kRegsCompute), "register split exceeds the launch allocation");

struct FwdParams {
  const int64_t* q_off;
  const int64_t* kv_off;
  int B, H;
  int64_t total_q, total_kv;
  float scale_log2;      // scale * log2(e), > 0
  int causal;
  const float* bias2;    // [H][num_buckets] bias * log2(e), or nullptr
  int num_buckets, center;
  const __nv_bfloat16* jbias;  // general jagged bias [H][jb_plane], or nullptr
  const int64_t* jb_off;       // its block offsets [B+1]
  int64_t jb_plane;
  const CUtensorMap* maps;  // [B][kNumMapSlots]
  const WorkItem* items;
  const int* n_items;
  int* claim;  // the list's claim counter (zeroed by the planner)
  int* status;
  const uint64_t* wait_ns;  // the planner's item hand-off wait limit for this launch (ns)
  __nv_bfloat16* out;
  float* lse;
  TraceBuf trace;
};

template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kStages = D == 128 ? 4 : 8;
  static constexpr int kSmemBytes = 2 * kTileBytes + kStages * kTileBytes + 1024;
  static_assert(kSmemBytes + 1024 <= 232448, "shared memory per CTA (dynamic + static barriers)");
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  // d = 64: each query tile is also copied into TMEM ([384,416), [416,448)) by its softmax
  // warpgroup and read from there as the A operand of its S MMAs, so the shared-memory
  // pair buffer is free again as soon as both copies are done and the next unit's pair
  // loads a whole unit ahead
  static constexpr bool kQTmem = D == 64;
  static constexpr uint32_t kColQ0 = 384, kColQ1 = 416;
};

struct ItemInfo {
  int b, h, t0, t1;
  int64_t qo, ko;
  int64_t jb;  // general jagged bias: the sequence's block offset
  int Lq, Lk;
  int nkv0, nkv1, njt;
  bool has1;
};

// Unit u (query-tile pair {2u, 2u+1}) of work item `it`.
__device__ __forceinline__ ItemInfo decode(const FwdParams& p, const ItemMeta& it, int u) {
  ItemInfo r;
  r.b = it.b;
  r.h = it.h;
  r.t0 = 2 * u;
  r.t1 = r.t0 + 1;
  r.qo = it.qo;
  r.jb = it.jb;
  r.ko = it.ko;
  r.Lq = it.Lq;
  r.Lk = it.Lk;
  r.has1 = r.t1 * kBM < r.Lq;
  r.nkv0 = kv_tiles_for_q_tile(r.t0, r.Lq, r.Lk, p.causal != 0);
  r.nkv1 = r.has1 ? kv_tiles_for_q_tile(r.t1, r.Lq, r.Lk, p.causal != 0) : 0;
  r.njt = max(r.nkv0, r.nkv1);
  return r;
}

__device__ __forceinline__ void raise_status(int* status, int code) { atomicCAS(status, 0, code); }

// Wait that ignores the abort flag: used only to drain copies already in flight.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

template <int D, bool kBias, bool kJBias = false>
__global__ void __launch_bounds__(kThreads, 1) fwd_kernel(const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                          // 2 tiles
  uint8_t* sRing = smem + 2 * C::kTileBytes;   // kStages tiles

  __shared__ uint64_t q_full, q_empty, mma_done;
  __shared__ uint64_t kv_full[C::kStages], kv_empty[C::kStages];
  __shared__ uint64_t s_full[2], p_full[2], o_full[2], qt_full[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ MetaRing meta;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, C::kQTmem ? 256 : 1);  // both softmax warpgroups, else the last S MMA
    mbar_init(&mma_done, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 128);
      mbar_init(&o_full[s], 1);
      mbar_init(&qt_full[s], 128);
    }
    meta_init(meta, p.wait_ns);
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

  if (warp < kFirstComputeWarp) {
   setmaxnreg_dec<kRegsLoad>();
   if (warp == 2) {
    // ------------------------------------------------------------ Q loader
    // Its own warp, so the next pair's Q load starts the moment the buffer is free (after
    // the current pair's last S MMA; at d = 64 once both softmax warpgroups have copied
    // their tiles into TMEM), whatever the K/V producer is waiting on.
    if (lane == 0) {
      uint32_t item_n = 0, tn = 0;
      bool ok = true;
      uint32_t k = 0;
      // sequence whose Q map this thread has acquired: a map is acquired (and its
      // descriptor prefetched) once, an item ahead, not before every load -- an acquire
      // makes the next copy through the map wait for a fresh descriptor fetch
      int acq_b = -1;
      for (; ok; ++k) {
       if (!meta_wait(meta, k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[k % kMetaSlots];  // read in place, freed after the item
       if (wi.b < 0) break;  // end of this CTA's items
       for (int u = wi.u0; u < wi.u1 && ok; ++u) {
        const ItemInfo it = decode(p, wi, u);
        if (it.njt == 0) continue;
        const TileMap q0 = tile_map(p.maps, p.B, kMapQ, it.b, it.qo, it.t0, p.total_q);
        const TileMap q1 = it.has1 ? tile_map(p.maps, p.B, kMapQ, it.b, it.qo, it.t1, p.total_q) : q0;
        if (it.b != acq_b) {
          tmap_acquire(p.maps + size_t(it.b) * kNumMapSlots + kMapQ);
          acq_b = it.b;
        }
        if (q0.tail) tmap_acquire(q0.map);
        if (q1.tail && q1.map != q0.map) tmap_acquire(q1.map);
        if (!mbar_wait(&q_empty, (item_n & 1) ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        trace_event(p.trace, kTraceLoader, tn, 1);
        mbar_arrive_expect_tx(&q_full, (it.has1 ? 2 : 1) * C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kBoxes; ++c) {
          tma_load_2d(sQ + c * 16384, q0.map, &q_full, it.h * D + c * 64, q0.y);
          if (it.has1) tma_load_2d(sQ + C::kTileBytes + c * 16384, q1.map, &q_full, it.h * D + c * 64, q1.y);
        }
        ++item_n;
        // pull the next pair into L2 meanwhile: the next unit of this range, else the first
        // unit of this CTA's next item
        {
          int nb = -1, nh = 0, nu = 0;
          if (u + 1 < wi.u1) {
            nb = wi.b, nh = wi.h, nu = u + 1;
          } else if (const ItemMeta* wn = meta_peek_next(meta, k)) {
            nb = wn->b, nh = wn->h, nu = wn->u0;
          }
          if (nb >= 0) {
            const int64_t nqo = p.q_off[nb];
            const int nLq = int(p.q_off[nb + 1] - nqo);
            if (nb != acq_b) {
              const CUtensorMap* nm = p.maps + size_t(nb) * kNumMapSlots + kMapQ;
              tmap_acquire(nm);
              tmap_prefetch(nm);
              acq_b = nb;
            }
            for (int t = 2 * nu; t < 2 * nu + 2 && t * kBM < nLq; ++t)
              prefetch_tile<C::kBoxes>(p.maps, p.B, kMapQ, nb, nqo, t, p.total_q, nh * D);
          }
        }
       }
       if (ok) meta_release(meta, k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      if (item_n > 0) drain_wait(&q_full, (item_n - 1) & 1);
    }
   } else if (warp == 0) {
    // ------------------------------------------------------------ K/V producer
    if (lane == 0) {
      uint32_t ring_n = 0, tn = 0;
      bool ok = true;
      uint32_t k = 0;
      int acq_b = -1;  // sequence whose K / V maps this thread has acquired (see the Q loader)
      for (; ok; ++k) {
       if (!meta_wait(meta, k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[k % kMetaSlots];  // read in place, freed after the item
       if (wi.b < 0) break;  // end of this CTA's items
       for (int u = wi.u0; u < wi.u1 && ok; ++u) {
        const ItemInfo it = decode(p, wi, u);
        if (it.njt == 0) continue;
        if (it.b != acq_b) {
          tmap_acquire(p.maps + size_t(it.b) * kNumMapSlots + kMapK);
          tmap_acquire(p.maps + size_t(it.b) * kNumMapSlots + kMapV);
          acq_b = it.b;
        }
        // last unit of this item: pull the first key tiles of this CTA's next item into L2
        if (const ItemMeta* wnp = u + 1 == wi.u1 ? meta_peek_next(meta, k) : nullptr) {
          const ItemMeta& wn = *wnp;
          const int64_t nko = p.kv_off[wn.b];
          const int nLk = int(p.kv_off[wn.b + 1] - nko);
          if (wn.b != acq_b) {
            const CUtensorMap* nk = p.maps + size_t(wn.b) * kNumMapSlots + kMapK;
            tmap_acquire(nk);
            tmap_acquire(nk + (kMapV - kMapK));
            tmap_prefetch(nk);
            tmap_prefetch(nk + (kMapV - kMapK));
            acq_b = wn.b;
          }
          for (int t = 0; t < 2 && t * kBN < nLk; ++t) {
            prefetch_tile<C::kBoxes>(p.maps, p.B, kMapK, wn.b, nko, t, p.total_kv, wn.h * D);
            prefetch_tile<C::kBoxes>(p.maps, p.B, kMapV, wn.b, nko, t, p.total_kv, wn.h * D);
          }
        }
        for (int j = 0; j < it.njt && ok; ++j) {
          const TileMap mk = tile_map(p.maps, p.B, kMapK, it.b, it.ko, j, p.total_kv);
          const TileMap mv = tile_map(p.maps, p.B, kMapV, it.b, it.ko, j, p.total_kv);
          if (mk.tail) {
            tmap_acquire(mk.map);
            tmap_acquire(mv.map);
          }
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t e = ring_n % C::kStages, ph = (ring_n / C::kStages) & 1;
            if (!mbar_wait(&kv_empty[e], ph ^ 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
            trace_event(p.trace, kTraceProducer, tn, 2);
            mbar_arrive_expect_tx(&kv_full[e], C::kTileBytes);
            uint8_t* dst = sRing + e * C::kTileBytes;
#pragma unroll
            for (int c = 0; c < C::kBoxes; ++c)
              tma_load_2d(dst + c * 16384, kv ? mv.map : mk.map, &kv_full[e], it.h * D + c * 64, mk.y);
            ++ring_n;
          }
        }
       }
       if (ok) meta_release(meta, k);
      }
      if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
      // drain: every copy this thread started has landed before the CTA can exit
      const uint32_t first = ring_n > C::kStages ? ring_n - C::kStages : 0;
      for (uint32_t n = first; n < ring_n; ++n) drain_wait(&kv_full[n % C::kStages], (n / C::kStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp walks the schedule (its state stays warp-uniform); one elected lane
    // issues the tcgen05 instructions
    {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, false, true);
      const uint32_t colS[2] = {C::kColS0, C::kColS1};
      const uint32_t colO[2] = {C::kColO0, C::kColO1};
      const uint32_t sQ_addr = smem_u32(sQ), sR_addr = smem_u32(sRing);
      auto mma_commit = [&](uint64_t* bar) {
        if (elect_one()) umma_commit(bar);
      };
      uint32_t ring_n = 0, item_n = 0, p_n[2] = {0, 0}, qt_n[2] = {0, 0}, tn = 0;
      bool ok = true;
      uint32_t k = 0;
      for (; ok; ++k) {
       if (!meta_wait_warp(meta, k, abort_flag)) { ok = false; break; }
       const ItemMeta& wi = meta.e[k % kMetaSlots];  // read in place, freed after the item
       if (wi.b < 0) break;  // end of this CTA's items
       for (int u = wi.u0; u < wi.u1 && ok; ++u) {
        const ItemInfo it = decode(p, wi, u);
        if (it.njt == 0) continue;
        const int nkv[2] = {it.nkv0, it.nkv1};
        if (!C::kQTmem) {
          if (!__all_sync(0xffffffffu, mbar_wait(&q_full, item_n & 1, abort_flag, kWaitTimeoutNs))) { ok = false; break; }
          ++item_n;
          tc_fence_after();
        }
        if (lane == 0) trace_event(p.trace, kTraceMma, tn, 10);
        int s_left = it.nkv0 + it.nkv1;
        auto issue_S = [&](int s, uint32_t e) {
          // descriptor start addresses are in 16-byte units in the low bits: step by adding
          const uint64_t qd = sdesc_sw128(sQ_addr + s * C::kTileBytes, 16, 1024);
          const uint64_t kd = sdesc_sw128(sR_addr + e * C::kTileBytes, 16, 1024);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
              if (C::kQTmem)
                umma_ts(tmem + colS[s], tmem + (s ? C::kColQ1 : C::kColQ0) + kk * 8, kd + o, kIdS, kk > 0);
              else
                umma_ss(tmem + colS[s], qd + o, kd + o, kIdS, kk > 0);
            }
          }
          mma_commit(&s_full[s]);
          if (lane == 0) trace_event(p.trace, kTraceMma, tn, 16 + s);
          if (--s_left == 0 && !C::kQTmem) mma_commit(&q_empty);
        };
        // a tile's first S reads Q from TMEM once its softmax warpgroup has copied it there
        auto wait_qt = [&](int s) -> bool {
          if (!C::kQTmem) return true;
          const bool r =
              __all_sync(0xffffffffu, mbar_wait(&qt_full[s], qt_n[s] & 1, abort_flag, kWaitTimeoutNs));
          ++qt_n[s];
          tc_fence_after();
          return r;
        };
        auto issue_PV = [&](int s, uint32_t e, bool acc) {
          const uint64_t vd = sdesc_sw128(sR_addr + e * C::kTileBytes, 16384, 1024);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              umma_ts(tmem + colO[s], tmem + colS[s] + kk * 8, vd + uint32_t(kk * 2048 >> 4), kIdPV,
                      (acc || kk > 0) ? 1u : 0u);
          }
        };
        auto wait_full = [&](uint32_t n) -> bool {
          const bool r =
              __all_sync(0xffffffffu, mbar_wait(&kv_full[n % C::kStages], (n / C::kStages) & 1, abort_flag, kWaitTimeoutNs));
          tc_fence_after();
          return r;
        };
        const uint32_t n0 = ring_n;  // K_j at n0 + 2j, V_j at n0 + 2j + 1
        if (!wait_full(n0)) { ok = false; break; }
        if (it.nkv0 > 0) {
          if (!wait_qt(0)) { ok = false; break; }
          issue_S(0, n0 % C::kStages);
        }
        if (it.nkv1 > 0) {
          if (!wait_qt(1)) { ok = false; break; }
          issue_S(1, n0 % C::kStages);
        }
        mma_commit(&kv_empty[n0 % C::kStages]);
        for (int j = 0; j < it.njt && ok; ++j) {
          const uint32_t nv = n0 + 2 * j + 1, nk = n0 + 2 * j + 2;
          if (!wait_full(nv)) { ok = false; break; }
          bool k_ready = false;
          for (int s = 0; s < 2 && ok; ++s) {
            if (j < nkv[s]) {
              if (!__all_sync(0xffffffffu, mbar_wait(&p_full[s], p_n[s] & 1, abort_flag, kWaitTimeoutNs))) {
                ok = false;
                break;
              }
              ++p_n[s];
              tc_fence_after();
              if (lane == 0) trace_event(p.trace, kTraceMma, tn, 12 + s);
              issue_PV(s, nv % C::kStages, j > 0);
              if (lane == 0) trace_event(p.trace, kTraceMma, tn, 14 + s);
              if (j == nkv[s] - 1) mma_commit(&o_full[s]);
            }
            if (j + 1 < nkv[s]) {
              if (!k_ready) {
                if (!wait_full(nk)) { ok = false; break; }
                k_ready = true;
              }
              issue_S(s, nk % C::kStages);
            }
          }
          if (!ok) break;
          mma_commit(&kv_empty[nv % C::kStages]);
          if (j + 1 < it.njt) mma_commit(&kv_empty[nk % C::kStages]);
        }
        ring_n = n0 + 2 * it.njt;
       }
       if (ok) meta_release_warp(meta, k);
      }
      if (!ok && lane == 0) raise_status(p.status, JFA_ERR_TIMEOUT);
      mma_commit(&mma_done);
      drain_wait(&mma_done, 0);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ scheduler
    if (lane == 0 && !meta_publish(meta, p.items, n_items, p.claim, p.q_off, p.kv_off, nullptr, p.jb_off, abort_flag))
      raise_status(p.status, JFA_ERR_TIMEOUT);
  }
  } else {
    setmaxnreg_inc<kRegsCompute>();
    // ------------------------------------------------------------ softmax warpgroups
    const int s = (warp - kFirstComputeWarp) >> 2;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + (s ? C::kColS1 : C::kColS0);
    const uint32_t tO = tmem + lane_addr + (s ? C::kColO1 : C::kColO0);
    const uint32_t tQ = tmem + lane_addr + (s ? C::kColQ1 : C::kColQ0);
    const float sl2 = p.scale_log2;
    uint32_t s_n = 0, o_n = 0, q_n = 0, tn = 0;
    const bool leader = (warp & 3) == 0 && lane == 0;  // records this warpgroup's trace
    bool ok = true;
    uint32_t k = 0;
    for (; ok; ++k) {
     if (!meta_wait_warp(meta, k, abort_flag)) { ok = false; break; }
     const ItemMeta& wi = meta.e[k % kMetaSlots];  // read in place, freed after the item
     if (wi.b < 0) break;  // end of this CTA's items
     for (int u = wi.u0; u < wi.u1 && ok; ++u) {
      const ItemInfo it = decode(p, wi, u);
      const int t = s ? it.t1 : it.t0;
      const int nkv = s ? it.nkv1 : it.nkv0;
      if (C::kQTmem && it.njt > 0) {
        // every unit the Q loader fills: wait for the pair (so that neither warpgroup frees a
        // later unit's buffer early), copy this tile's rows into TMEM if its S MMAs run, free
        // the buffer.  Row `row` of the 128-byte-swizzled tile: 16-byte chunk c at chunk
        // position c ^ (row & 7).
        if (!mbar_wait(&q_full, q_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        ++q_n;
        if (nkv > 0) {
          const uint4* qrow = reinterpret_cast<const uint4*>(sQ + s * C::kTileBytes + row * 128);
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = qrow[c ^ (row & 7)];
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
          }
          tmem_st32(tQ, w);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&qt_full[s]);
        }
        mbar_arrive(&q_empty);
      }
      if (t * kBM >= it.Lq) continue;
      const int i = t * kBM + row;  // local query index
      const bool valid_row = i < it.Lq;
      __nv_bfloat16* orow = p.out + ((it.qo + i) * p.H + it.h) * int64_t(D);
      float* lrow = p.lse + int64_t(it.h) * p.total_q + it.qo + i;
      if (nkv == 0) {
        if (valid_row) {
          uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          *lrow = -INFINITY;
        }
        continue;
      }
      const int diag = it.Lk - it.Lq;  // causal: key j visible iff j <= i + diag
      const float* brow = kBias ? p.bias2 + size_t(it.h) * p.num_buckets : nullptr;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        uint32_t jbk[kJBias ? 64 : 1];  // general bias for this tile, loaded before the wait
        if (kJBias) {
          const int64_t pitch = (it.Lk + 7) / 8 * 8;  // rows of the sequence's block: bias[i][j] at i * pitch + j
          const int kvj = j * kBN;
          const __nv_bfloat16* brow_j = p.jbias + size_t(it.h) * p.jb_plane + it.jb + int64_t(i) * pitch;
          jbias_load_row<128>(jbk, valid_row ? brow_j + kvj : nullptr, min(kBN, it.Lk - kvj));
          if (valid_row && kvj + kBN < it.Lk) {  // the next key tile's row segment into L2 meanwhile
            prefetch_l2(brow_j + kvj + kBN);
            prefetch_l2(brow_j + kvj + kBN + 64);
          }
        }
        const int kv0 = j * kBN;
        const bool last = (j == nkv - 1);
        // relative-position bias * log2(e) of this tile's columns, loaded before the wait so the
        // loads overlap the MMAs (0 on padded key columns, which then score exactly 0)
        float bw[kBias ? 128 : 1];
        if (kBias) {
          const int n_real = min(kBN, it.Lk - kv0);
          const int idx0 = kv0 - i + p.center;  // bucket of column c: idx0 + c
          if (idx0 >= 0 && idx0 + kBN - 1 < p.num_buckets && n_real == kBN) {
#pragma unroll
            for (int c = 0; c < 128; ++c) bw[c] = __ldg(brow + idx0 + c);
          } else {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              bw[c] = c < n_real ? __ldg(brow + min(max(idx0 + c, 0), p.num_buckets - 1)) : 0.f;
          }
        }
        if (!mbar_wait(&s_full[s], s_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
        ++s_n;
        tc_fence_after();
        if (leader) trace_event(p.trace, kTraceCompute0 + s, tn, 20);
        float x[128];
        if (kBias) {
          // x = scale*log2e * (q.k) + bias*log2e, 32 columns at a time (the bias registers
          // become the scores', so at most 32 more are live)
          const uint64_t k_sl2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t r[32];
            tmem_ld32(tS + 32 * q, r);
            tmem_ld_wait();
#pragma unroll
            for (int c2 = 0; c2 < 16; ++c2) {
              const int c = 32 * q + 2 * c2;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * c2]), __uint_as_float(r[2 * c2 + 1])), k_sl2,
                               f2_pack(bw[c], bw[c + 1])),
                        x[c], x[c + 1]);
            }
          }
        } else {
          // all four loads in flight before a single wait
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(tS + 0, r0);
          tmem_ld32(tS + 32, r1);
          tmem_ld32(tS + 64, r2);
          tmem_ld32(tS + 96, r3);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            x[c] = __uint_as_float(r0[c]);
            x[32 + c] = __uint_as_float(r1[c]);
            x[64 + c] = __uint_as_float(r2[c]);
            x[96 + c] = __uint_as_float(r3[c]);
          }
        }
        if (kJBias) {
          // x = scale*log2e * (q.k) + bias*log2e from this row of the sequence's block
          jbias_apply<128>(x, jbk, sl2, kLog2e);
        }
        if (p.causal) {
          const int lim = i + diag - kv0;  // last visible column of this row in this tile
          if (lim < kBN - 1) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > lim) x[c] = -INFINITY;
          }
        }
        // row max: 4 chains of 3-input max over 32 columns each, then a short tree
        float mx4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float m0 = fmaxf(x[32 * k], x[32 * k + 1]);
#pragma unroll
          for (int c = 2; c < 32; c += 2) m0 = fmax3(m0, x[32 * k + c], x[32 * k + c + 1]);
          mx4[k] = m0;
        }
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        const float m_tile = (kBias || kJBias) ? mx : mx * sl2;
        // raise the reference max only when it grows by more than 2^8
        const bool need = m_tile > m + kRescaleThreshold;
        const float m_new = need ? m_tile : m;
        const float alpha = need ? ex2_approx(m - m_new) : 1.f;  // m = -inf gives 0
        l *= alpha;
        m = m_new;
        const float m_use = (m == -INFINITY) ? 0.f : m;
        // exponentials two columns per packed fp32x2 op; row sum in 4 packed chains
        uint64_t sum2[4] = {0, 0, 0, 0};
        {
          const uint64_t k_scale = f2_pack(sl2, sl2), k_negm = f2_pack(-m_use, -m_use);
          uint32_t pk[64];
#pragma unroll
          for (int t2 = 0; t2 < 64; ++t2) {
            const uint64_t xx = f2_pack(x[2 * t2], x[2 * t2 + 1]);
            const uint64_t arg = (kBias || kJBias) ? f2_add(xx, k_negm) : f2_fma(xx, k_scale, k_negm);
            float a, b;
            f2_unpack(arg, a, b);
            const float pa = ex2_approx(a), pb = ex2_approx(b);
            sum2[t2 & 3] = f2_add(sum2[t2 & 3], f2_pack(pa, pb));
            pk[t2] = pack_bf16x2(pa, pb);
          }
          tmem_st64(tS, pk);
        }
        float sum4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float lo, hi;
          f2_unpack(sum2[k], lo, hi);
          sum4[k] = lo + hi;
        }
        float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
        if (last && !p.causal && kv0 + kBN > it.Lk) {
          // subtraction scheme: padded keys scored exactly 0, each added exp2(0 - m_use)
          sum -= float(kv0 + kBN - it.Lk) * ex2_approx(-m_use);
        }
        l += sum;
        // O still holds the sum over earlier tiles (their PV MMAs completed before this
        // tile's S did); rescale it now that the S registers are free
        if (__any_sync(0xffffffffu, need) && j > 0) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(tO + cc * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
            tmem_st32(tO + cc * 32, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[s]);
        if (leader) trace_event(p.trace, kTraceCompute0 + s, tn, 21);
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, lse = ln(sum) = (m + log2 l) * ln 2
      if (!mbar_wait(&o_full[s], o_n & 1, abort_flag, kWaitTimeoutNs)) { ok = false; break; }
      ++o_n;
      tc_fence_after();
      if (leader) trace_event(p.trace, kTraceCompute0 + s, tn, 22);
      const bool live = l > 0.f;
      const float inv_l = live ? 1.f / l : 0.f;
      const float m_use = (m == -INFINITY) ? 0.f : m;
      // all of the row's O columns in flight before one wait
      uint32_t o_r[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tO + cc * 32, o_r[cc]);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int t2 = 0; t2 < 16; ++t2)
          pk[t2] = pack_bf16x2(__uint_as_float(o_r[cc][2 * t2]) * inv_l, __uint_as_float(o_r[cc][2 * t2 + 1]) * inv_l);
        if (valid_row) {
          st_global_v8(orow + cc * 32, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
          st_global_v8(orow + cc * 32 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
        }
      }
      if (valid_row) *lrow = live ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
      tc_fence_before();
      if (leader) trace_event(p.trace, kTraceCompute0 + s, tn, 23);
     }
     if (__all_sync(0xffffffffu, ok)) meta_release_warp(meta, k);
    }
    if (!ok) raise_status(p.status, JFA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D, bool kBias, bool kJBias = false>
cudaError_t launch_fwd_t(const FwdParams& fp, int grid, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fwd_kernel<D, kBias, kJBias>;
  cudaError_t e = check_launch_registers(kern);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, fp);
}

}  // namespace

cudaError_t launch_forward(const Problem& pr, void* ws, const WsLayout& L, void* out, float* lse, int num_sms,
                           cudaStream_t stream) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  FwdParams fp;
  fp.q_off = pr.q_off;
  fp.kv_off = pr.kv_off;
  fp.B = pr.B;
  fp.H = pr.H;
  fp.total_q = pr.total_q;
  fp.total_kv = pr.total_kv;
  fp.scale_log2 = pr.scale * kLog2e;
  fp.causal = pr.causal;
  fp.bias2 = pr.bias_table ? reinterpret_cast<const float*>(w + L.bias2) : nullptr;
  fp.num_buckets = pr.num_buckets;
  fp.center = pr.center;
  fp.jbias = static_cast<const __nv_bfloat16*>(pr.jbias);
  fp.jb_off = pr.jb_off;
  fp.jb_plane = pr.jb_plane;
  fp.maps = reinterpret_cast<const CUtensorMap*>(w + L.maps);
  fp.items = reinterpret_cast<const WorkItem*>(w + L.fwd);
  fp.n_items = &reinterpret_cast<const WsHeader*>(w)->n_fwd;
  fp.claim = &reinterpret_cast<WsHeader*>(w)->claim_fwd;
  fp.status = &reinterpret_cast<WsHeader*>(w)->status;
  fp.wait_ns = &reinterpret_cast<const WsHeader*>(w)->wait_ns[0];
  fp.out = static_cast<__nv_bfloat16*>(out);
  fp.lse = lse;
  fp.trace = pr.trace[JFA_KERNEL_FORWARD];
  const int grid = num_sms;
  const bool bias = pr.bias_table != nullptr;
  const bool jb = pr.jbias != nullptr;
  if (pr.d == 128)
    return bias ? launch_fwd_t<128, true>(fp, grid, stream)
                : (jb ? launch_fwd_t<128, false, true>(fp, grid, stream) : launch_fwd_t<128, false>(fp, grid, stream));
  return bias ? launch_fwd_t<64, true>(fp, grid, stream)
              : (jb ? launch_fwd_t<64, false, true>(fp, grid, stream) : launch_fwd_t<64, false>(fp, grid, stream));
}

}  // namespace jfa
