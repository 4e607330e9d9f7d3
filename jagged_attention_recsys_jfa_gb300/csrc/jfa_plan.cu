// Planner kernel: validates the jagged offsets, builds one TMA tensor map per
// (sequence, tensor) whose row extent is that sequence's length -- so tile loads
// past a sequence end arrive as zeros, which the subtraction scheme of "Jagged
// Flash Attention (JFA)", "Four generations" item 1, relies on -- and writes the
// persistent kernels' work lists sorted longest first (counting sort on cost), which
// the kernels' CTAs claim one at a time from a counter, the scheduling that keeps SMs busy
// when short sequences finish early (same page, "Why standard FlashAttention falls short"
// and item 3).
#include "jfa_internal.h"
#include "sm100_ptx.cuh"

namespace jfa {
namespace {

struct PlanParams {
  const int64_t* q_off;
  const int64_t* kv_off;
  int B, H;
  int64_t total_q, total_kv;
  int causal, backward;
  int grid;  // persistent CTAs of the kernels that consume the lists
  int nsp_max_tiles;  // query tiles up to which a sequence takes the non-sequence-parallel pass
  int d;              // head dimension
  uint8_t* ws;
  WsLayout L;
  const float* bias;  // [H][nb] or nullptr
  float* bias_grad;   // [H][nb] gradient table to clear before the backward passes add into it, or nullptr
  int nb;
  const int64_t* jb_off;  // general jagged bias block offsets [B+1], or nullptr
  int64_t jb_plane;
};

enum ListKind { kListFwd = 0, kListDq = 1, kListDkv = 2, kListFused = 3, kListNsp = 4 };

// Backward: a sequence whose queries fit one tile (Lq <= 128) is done by the fused pass
// (one CTA per sequence and head, every key tile once); one of 2 .. kNspMaxTiles query
// tiles by the non-sequence-parallel pass (one CTA per sequence and head, every tile pair
// once); the others by the split dK/dV and dQ passes.  Units: key tiles, except for the
// forward (query-tile pairs) and the dQ pass (query tiles); a sequence without keys still
// gets one unit in the fused and non-sequence-parallel lists (its dq rows are zeroed there).
__device__ __forceinline__ int list_units(int kind, int Lq, int Lk, int nsp_max) {
  const int nq = (Lq + kBM - 1) / kBM;
  const int nk = (Lk + kBN - 1) / kBN;
  if (kind == kListFwd) return (nq + 1) / 2;
  if (kind == kListFused) return Lq <= kBM ? (nk > 0 ? nk : (Lq > 0 ? 1 : 0)) : 0;
  if (kind == kListNsp) return nsp_path(Lq, nsp_max) ? (nk > 0 ? nk : 1) : 0;
  if (Lq <= kBM || nsp_path(Lq, nsp_max)) return 0;
  return kind == kListDq ? nq : nk;
}

__device__ __forceinline__ int unit_cost(int kind, int u, int Lq, int Lk, bool causal) {
  if (kind == kListFused) return 1;  // a key tile (its dK / dV rows are stored even when unseen)
  if (kind == kListNsp) {            // the query tiles that see key tile u (at least 1)
    int first, count;
    q_tiles_for_kv_tile(u, Lq, Lk, causal, &first, &count);
    return count > 0 ? count : 1;
  }
  if (kind == kListFwd)
    return kv_tiles_for_q_tile(2 * u, Lq, Lk, causal) + kv_tiles_for_q_tile(2 * u + 1, Lq, Lk, causal);
  if (kind == kListDq) return kv_tiles_for_q_tile(u, Lq, Lk, causal);
  int first, count;
  q_tiles_for_kv_tile(u, Lq, Lk, causal, &first, &count);
  return count;
}

// Block-wide inclusive scan of one 64-bit value per thread (blockDim.x == 1024).
__device__ long long block_scan_incl(long long v, long long* total) {
  __shared__ long long warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const long long w = warp_sums[lane];
    long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const long long r = warp_sums[warp] + incl;
  __syncthreads();
  return r;
}

// Exclusive scan of hist[] in descending cost order: base[c] = sum_{c' > c} hist[c'].
// 1024 threads, kCostBuckets = 2048 buckets (two per thread).  Returns the total.
__device__ int scan_desc(const int* hist, int* base) {
  __shared__ long long total;
  const int tid = threadIdx.x;
  // thread tid owns descending positions r = 2*tid, 2*tid+1  (bucket c = kCostBuckets-1-r)
  const int c0 = kCostBuckets - 1 - 2 * tid, c1 = c0 - 1;
  const int v0 = hist[c0], v1 = hist[c1];
  const long long incl = block_scan_incl(v0 + v1, &total);
  const int excl = int(incl) - (v0 + v1);
  base[c0] = excl;
  base[c1] = excl + v0;
  __syncthreads();
  return int(total);
}

// Walk the units of one sequence, cutting them into consecutive ranges whose summed
// cost stays <= cap (a unit costlier than cap forms its own range); calls f(u0, u1, cost).
template <typename F>
__device__ void for_each_range(int kind, int Lq, int Lk, bool causal, int nsp_max, long long cap, F&& f) {
  const int n = list_units(kind, Lq, Lk, nsp_max);
  int start = 0;
  long long acc = 0;
  for (int u = 0; u < n; ++u) {
    const int c = unit_cost(kind, u, Lq, Lk, causal);
    if (u > start && acc + c > cap) {
      f(start, u, acc);
      start = u;
      acc = 0;
    }
    acc += c;
  }
  if (n > 0) f(start, n, acc);
}

__device__ void emit_list(const PlanParams& p, int kind, WorkItem* items, int64_t cap, int* count_out,
                          int* hist, int* base) {
  __shared__ long long total_cost;
  const int tid = threadIdx.x;
  const bool causal = p.causal != 0;
  // total work, to cap range cost at about 1/kItemsPerCta of a CTA's share
  long long local = 0;
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int Lq = int(p.q_off[b + 1] - p.q_off[b]);
    const int Lk = int(p.kv_off[b + 1] - p.kv_off[b]);
    const int n = list_units(kind, Lq, Lk, p.nsp_max_tiles);
    for (int u = 0; u < n; ++u) local += unit_cost(kind, u, Lq, Lk, causal);
  }
  block_scan_incl(local, &total_cost);
  const long long share = (total_cost * p.H + (long long)kItemsPerCta * p.grid - 1) /
                          ((long long)kItemsPerCta * p.grid);
  // the fused and non-sequence-parallel passes own each sequence's dQ: their items are
  // never cut into ranges.  At d = 128 the dK/dV and dQ passes take one tile per item, and
  // a (sequence, head)'s items sit next to each other in the list (ordered by the group's
  // total cost, longest first): neighbouring CTAs claim them together and stream the
  // operand they share (Q / dO for dK/dV, K / V for dQ) at the same time, so more of it
  // comes from L2 (GEM-like shape: dK/dV 720 -> 699 us; long-tail causal 1172 -> 1122 us).
  // At d = 64 a tile is too short for the per-item cost (biased causal shape: dK/dV
  // 344 -> 398 us), so those lists keep capped ranges, and so does the forward (grouped
  // query-tile pairs: GEM-like forward 411 -> 447 us).
  const bool grouped = (kind == kListDkv || kind == kListDq) && p.d == 128;
  const long long range_cap =
      (kind == kListFused || kind == kListNsp) ? (1ll << 62) : (grouped ? 1 : (share > 1 ? share : 1));
  auto bucket = [](long long cost) { return cost < kCostBuckets - 1 ? int(cost) : kCostBuckets - 1; };

  for (int c = tid; c < kCostBuckets; c += blockDim.x) hist[c] = 0;
  __syncthreads();
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int Lq = int(p.q_off[b + 1] - p.q_off[b]);
    const int Lk = int(p.kv_off[b + 1] - p.kv_off[b]);
    if (grouped) {
      long long gcost = 0;
      int nr = 0;
      for_each_range(kind, Lq, Lk, causal, p.nsp_max_tiles, range_cap, [&](int, int, long long cost) {
        gcost += cost;
        ++nr;
      });
      if (nr) atomicAdd(&hist[bucket(gcost)], p.H * nr);
    } else {
      for_each_range(kind, Lq, Lk, causal, p.nsp_max_tiles, range_cap,
                     [&](int, int, long long cost) { atomicAdd(&hist[bucket(cost)], p.H); });
    }
  }
  __syncthreads();
  const int total = scan_desc(hist, base);
  if (total > cap) {  // cannot happen for valid offsets (capacities are upper bounds)
    if (tid == 0) {
      atomicCAS(&reinterpret_cast<WsHeader*>(p.ws)->status, 0, int(JFA_ERR_WORKSPACE));
      *count_out = 0;
    }
    return;
  }
  __shared__ unsigned long long max_item;
  if (tid == 0) max_item = 0;
  __syncthreads();
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int Lq = int(p.q_off[b + 1] - p.q_off[b]);
    const int Lk = int(p.kv_off[b + 1] - p.kv_off[b]);
    unsigned long long mx = 0;
    if (grouped) {
      long long gcost = 0;
      int nr = 0;
      for_each_range(kind, Lq, Lk, causal, p.nsp_max_tiles, range_cap, [&](int, int, long long cost) {
        gcost += cost;
        ++nr;
      });
      if (nr) {
        // head h's tiles at pos + h * nr + r, in tile order
        const int pos = atomicAdd(&base[bucket(gcost)], p.H * nr);
        int r = 0;
        for_each_range(kind, Lq, Lk, causal, p.nsp_max_tiles, range_cap, [&](int u0, int u1, long long cost) {
          for (int h = 0; h < p.H; ++h) items[pos + h * nr + r] = WorkItem{b, h, u0, u1};
          ++r;
          if ((unsigned long long)cost > mx) mx = (unsigned long long)cost;
        });
      }
    } else {
      for_each_range(kind, Lq, Lk, causal, p.nsp_max_tiles, range_cap, [&](int u0, int u1, long long cost) {
        const int pos = atomicAdd(&base[bucket(cost)], p.H);
        for (int h = 0; h < p.H; ++h) items[pos + h] = WorkItem{b, h, u0, u1};
        if ((unsigned long long)cost > mx) mx = (unsigned long long)cost;
      });
    }
    if (mx) atomicMax(&max_item, mx);
  }
  __syncthreads();
  if (tid == 0) {
    *count_out = total;
    // the bounded waits of the kernel that walks this list scale with the planned work
    reinterpret_cast<WsHeader*>(p.ws)->wait_ns[kind] =
        wait_limit_ns(total_cost * p.H, p.grid, (long long)max_item);
  }
  __syncthreads();
}

// Backward: offsets of each sequence in the 128-row-padded per-query vectors.
__device__ void write_qpad(const PlanParams& p) {
  __shared__ long long chunk_total;
  int64_t* qpad = reinterpret_cast<int64_t*>(p.ws + p.L.qpad);
  long long carry = 0;
  for (int b0 = 0; b0 < p.B; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    long long v = 0;
    if (b < p.B) v = ((p.q_off[b + 1] - p.q_off[b]) + kBM - 1) / kBM * kBM;
    const long long incl = block_scan_incl(v, &chunk_total);
    if (b < p.B) qpad[b] = carry + incl - v;
    carry += chunk_total;
  }
  if (threadIdx.x == 0) {
    qpad[p.B] = carry;
    reinterpret_cast<WsHeader*>(p.ws)->total_qpad = carry;
  }
}

// The first CTAs validate the offsets and write one work list each (block-wide scans: the
// forward list, or the dK/dV (with the padded query offsets), dQ and fused lists); the
// other CTAs write the bias table, the tail copies and the tensor maps in parallel.
__global__ void __launch_bounds__(1024, 1) plan_kernel(const __grid_constant__ PlanMaps maps, PlanParams p) {
  __shared__ int hist[kCostBuckets];
  __shared__ int base[kCostBuckets];
  const int tid = threadIdx.x;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
  grid_dependency_wait();    // the offsets and the workspace may come from earlier work
  grid_launch_dependents();  // the next kernel may start its prologue; it waits for this one

  const int list_ctas = p.backward ? 4 : 1;
  if (int(blockIdx.x) >= list_ctas) {
    const size_t gt = size_t(blockIdx.x - list_ctas) * blockDim.x + tid;
    const size_t gstride = size_t(gridDim.x - list_ctas) * blockDim.x;
    // ---- bias table pre-scaled to log2 units (the kernels work with exp2)
    if (p.bias) {
      float* b2 = reinterpret_cast<float*>(p.ws + p.L.bias2);
      for (size_t i = gt; i < size_t(p.H) * p.nb; i += gstride) b2[i] = p.bias[i] * 1.4426950408889634f;
    }
    if (p.bias_grad)
      for (size_t i = gt; i < size_t(p.H) * p.nb; i += gstride) p.bias_grad[i] = 0.f;
    // ---- tail copies: the last min(128, total) rows of each tensor, which the boxes that
    //      would otherwise read past the tensor's last row load from instead
    const size_t rb = p.L.row_bytes;
    for (int slot = 0; slot < kNumMapSlots; ++slot) {
      if (!maps.used[slot]) continue;
      const int64_t total = (slot == kMapQ || slot == kMapDO) ? p.total_q : p.total_kv;
      if (total <= 0) continue;
      const int64_t n = total < kBM ? total : kBM;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(maps.base[slot]) +
                                                        size_t(total - n) * rb);
      uint4* dst = reinterpret_cast<uint4*>(p.ws + p.L.tail + size_t(slot) * kTailRows * rb);
      const size_t nvec = size_t(n) * rb / 16;
      for (size_t i = gt; i < nvec; i += gstride) dst[i] = src[i];
    }
    // ---- per-sequence tensor maps: copy the template, point it at the sequence's first
    //      row and clip its row extent to the sequence length.  A sequence whose last tile
    //      would reach past the tensor's last row also gets a tail map over the tail copy,
    //      pointed at that tile's first row and clipped to the tile's rows.  (With invalid
    //      offsets CTA 0 leaves every list empty, so no map is used; a tail map is only
    //      written for a sequence inside its tensor, which keeps its index in range.)
    CUtensorMap* out_maps = reinterpret_cast<CUtensorMap*>(p.ws + p.L.maps);
    for (size_t idx = gt; idx < size_t(p.B) * kNumMapSlots; idx += gstride) {
      const int b = int(idx / kNumMapSlots), slot = int(idx % kNumMapSlots);
      if (!maps.used[slot]) continue;
      const bool is_q_side = (slot == kMapQ || slot == kMapDO);
      const int64_t row0 = is_q_side ? p.q_off[b] : p.kv_off[b];
      const int64_t len = (is_q_side ? p.q_off[b + 1] : p.kv_off[b + 1]) - row0;
      const uint4* src = reinterpret_cast<const uint4*>(&maps.tmpl[slot]);
      CUtensorMap* dst = out_maps + idx;
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int i = 0; i < 8; ++i) d4[i] = src[i];
      tmap_replace_address(dst, static_cast<const uint8_t*>(maps.base[slot]) + row0 * int64_t(rb));
      tmap_replace_dim1(dst, uint32_t(len > 0 ? len : 1));
      const int64_t total = is_q_side ? p.total_q : p.total_kv;
      if (len <= 0 || row0 < 0 || row0 + len > total) continue;
      const int64_t g0 = row0 + (len - 1) / kBM * kBM;  // first row of the sequence's last tile
      if (g0 + kBM > total) {
        const int64_t n = total < kBM ? total : kBM;  // rows in the tail copy; it starts at row total - n
        CUtensorMap* tdst =
            out_maps + size_t(p.B) * kNumMapSlots + size_t(slot) * kTailMaps + size_t(g0 + kBM - total);
        uint4* t4 = reinterpret_cast<uint4*>(tdst);
#pragma unroll
        for (int i = 0; i < 8; ++i) t4[i] = src[i];
        tmap_replace_address(tdst, p.ws + p.L.tail + size_t(slot) * kTailRows * rb + size_t(g0 - (total - n)) * rb);
        tmap_replace_dim1(tdst, uint32_t(row0 + len - g0));
      }
    }
    tmap_release();
    return;
  }

  // ---- list CTAs: validate offsets (each list CTA on its own, so all agree)
  int bad = 0;
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int64_t lq = p.q_off[b + 1] - p.q_off[b];
    const int64_t lk = p.kv_off[b + 1] - p.kv_off[b];
    if (lq < 0 || lk < 0 || lq > (int64_t(1) << 30) || lk > (int64_t(1) << 30)) bad = 1;
    // a general bias's blocks must hold exactly Lq x round_up(Lk, 8) elements each
    if (p.jb_off && !bad && p.jb_off[b + 1] - p.jb_off[b] != lq * ((lk + 7) / 8 * 8)) bad = 1;
  }
  if (tid == 0) {
    if (p.q_off[0] != 0 || p.kv_off[0] != 0 || p.q_off[p.B] != p.total_q || p.kv_off[p.B] != p.total_kv)
      bad = 1;
    if (p.jb_off && (p.jb_off[0] != 0 || p.jb_off[p.B] != p.jb_plane)) bad = 1;
  }
  if (blockIdx.x == 0 && tid == 0) hdr->claim_fwd = hdr->claim_dq = hdr->claim_dkv = hdr->claim_fused = hdr->claim_nsp = 0;
  bad = __syncthreads_or(bad);
  if (bad) {
    if (tid == 0) {
      atomicCAS(&hdr->status, 0, int(JFA_ERR_BAD_OFFSETS));
      hdr->n_fwd = hdr->n_dq = hdr->n_dkv = hdr->n_fused = hdr->n_nsp = 0;
      hdr->total_qpad = 0;  // the preprocess walks no rows
    }
    return;
  }

  // ---- work lists
  if (!p.backward) {
    emit_list(p, kListFwd, reinterpret_cast<WorkItem*>(p.ws + p.L.fwd), p.L.cap_fwd, &hdr->n_fwd, hist, base);
  } else if (blockIdx.x == 0) {
    write_qpad(p);
    emit_list(p, kListDkv, reinterpret_cast<WorkItem*>(p.ws + p.L.dkv), p.L.cap_dkv, &hdr->n_dkv, hist,
              base);
  } else if (blockIdx.x == 1) {
    emit_list(p, kListDq, reinterpret_cast<WorkItem*>(p.ws + p.L.dq), p.L.cap_dq, &hdr->n_dq, hist, base);
  } else if (blockIdx.x == 2) {
    emit_list(p, kListFused, reinterpret_cast<WorkItem*>(p.ws + p.L.fused), p.L.cap_fused, &hdr->n_fused, hist,
              base);
  } else {
    emit_list(p, kListNsp, reinterpret_cast<WorkItem*>(p.ws + p.L.nsp), p.L.cap_nsp, &hdr->n_nsp, hist, base);
  }
}

// Failure-detection self test: one thread waits on an mbarrier that nothing arrives on,
// through the same bounded wait the pipelines use; when the limit runs out it records
// JFA_ERR_TIMEOUT in the workspace status word and the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, &abort_flag, timeout_ns)) atomicCAS(status, 0, int(JFA_ERR_TIMEOUT));
  }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(void* ws, uint64_t timeout_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(&reinterpret_cast<WsHeader*>(ws)->status, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_plan(const Problem& pr, const PlanMaps& maps, void* ws, const WsLayout& L, bool backward,
                        int num_sms, cudaStream_t stream) {
  PlanParams p;
  p.q_off = pr.q_off;
  p.kv_off = pr.kv_off;
  p.B = pr.B;
  p.H = pr.H;
  p.total_q = pr.total_q;
  p.total_kv = pr.total_kv;
  p.causal = pr.causal;
  p.backward = backward ? 1 : 0;
  p.grid = num_sms;
  p.nsp_max_tiles = pr.nsp_max_tiles;
  p.d = pr.d;
  p.ws = static_cast<uint8_t*>(ws);
  p.L = L;
  p.bias = pr.bias_table;
  p.bias_grad = backward ? pr.bias_grad : nullptr;
  p.jb_off = pr.jb_off;
  p.jb_plane = pr.jb_plane;
  p.nb = pr.num_buckets;
  // one CTA per list; helpers for the maps (one thread each), tail copies and bias table
  const long long map_ctas = (static_cast<long long>(pr.B) * kNumMapSlots + 1023) / 1024;
  const int helpers = int(map_ctas < 1 ? 1 : (map_ctas > 32 ? 32 : map_ctas)) + 4;
  return launch_pdl(plan_kernel, dim3((backward ? 4 : 1) + helpers), dim3(1024), 0, stream, maps, p);
}

}  // namespace jfa
