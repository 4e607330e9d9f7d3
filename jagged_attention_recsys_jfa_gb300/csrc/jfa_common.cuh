// Shared definitions of the jagged attention kernels: tile sizes, the work-item
// format written by the planner, and the workspace layout.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>

#include "../../include/jfa.h"

namespace jfa {

constexpr int kBM = 128;  // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;  // key rows per tile
constexpr int kMaxBuckets = 8192;
constexpr int kCostBuckets = 2048;  // planner's counting-sort buckets (cost clamped)
// Bounded pipeline waits.  A wait that outlasts its limit ends the CTA with
// JFA_ERR_TIMEOUT, so the limit must exceed any wait a correct launch can have.  Waits
// inside an item's tile pipeline last at most a few units' time (a unit visits at most
// 2 x 128 tile pairs, well under a millisecond) and keep the fixed kWaitTimeoutNs.  The
// waits that scale with the launch are the item hand-offs of the scheduler ring: a CTA's
// scheduler waits for item k - 2 to be released, and its roles for item k to be
// published, i.e. for up to about a CTA's whole share of the launch.  The planner
// therefore sizes each list's hand-off limit from the work it planned: a 2 s floor plus a
// generous time per tile pair (kWaitNsPerTilePair, ~30x the measured ~1 us per 128x128
// tile pair on one SM) for one CTA's share of the pairs and the costliest single item.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // floor: 2 s
constexpr uint64_t kWaitNsPerTilePair = 32000ull;    // 32 us per planned tile pair
constexpr uint64_t kWaitLimitCapNs = 3600ull * 1000000000ull;  // an hour: no overflow
__host__ __device__ inline uint64_t wait_limit_ns(long long total_pairs, int ctas, long long max_item_pairs) {
  if (ctas < 1) ctas = 1;
  if (total_pairs < 0) total_pairs = 0;
  if (max_item_pairs < 0) max_item_pairs = 0;
  const unsigned long long per_cta = (unsigned long long)((total_pairs + ctas - 1) / ctas) + max_item_pairs;
  const unsigned long long cap_pairs = kWaitLimitCapNs / kWaitNsPerTilePair;
  const uint64_t extra = per_cta >= cap_pairs ? kWaitLimitCapNs : per_cta * kWaitNsPerTilePair;
  return kWaitTimeoutNs + extra;
}

// Persistent tensor-core kernels: 3 warpgroups.  Warpgroup 0 = TMA producer (warp 0),
// tcgen05 issuer and TMEM owner (warp 1), two idle warps; warpgroups 1 and 2 = the
// compute warps (one TMEM lane per thread).  Each kernel moves registers from warpgroup
// 0 to the compute warpgroups with setmaxnreg; 128*load + 256*compute must not exceed
// the launch allocation of 384 threads x 168 registers.
constexpr int kThreads = 384;
constexpr int kFirstComputeWarp = 4;
constexpr uint32_t kLaunchRegs = 168;
__host__ __device__ constexpr bool reg_split_fits(uint32_t load, uint32_t compute) {
  return load % 8 == 0 && compute % 8 == 0 && 128 * load + 256 * compute <= kLaunchRegs * kThreads;
}
// The dK/dV pass adds a fourth warpgroup (warps 12..15) that writes the dK / dV rows out
// while the compute warpgroups start the next key tile: 512 threads, 128 registers each
// at launch, split role / compute / epilogue with setmaxnreg.
constexpr int kThreadsDkdv = 512;
constexpr int kFirstEpilogueWarp = 12;
constexpr uint32_t kLaunchRegsDkdv = 128;
__host__ __device__ constexpr bool reg_split_fits_dkdv(uint32_t load, uint32_t compute, uint32_t epi) {
  return load % 8 == 0 && compute % 8 == 0 && epi % 8 == 0 &&
         128 * load + 256 * compute + 128 * epi <= kLaunchRegsDkdv * kThreadsDkdv;
}

// One unit of work for a persistent CTA: the consecutive units [u0, u1) of sequence b,
// head h, where a unit is
//   forward: the query-tile pair {2u, 2u+1}
//   dQ pass: query tile u
//   dK/dV  : key/value tile u
// The planner cuts each (sequence, head) into ranges whose cost (tile pairs visited) is
// capped, so one CTA walks neighbouring tiles of one sequence and the shared operand
// (K/V for the forward and dQ pass, Q/dO for dK/dV) is re-read from L2, not HBM.
struct WorkItem {
  int b, h, u0, u1;
};
constexpr int kItemsPerCta = 4;  // target items per CTA when capping range cost

// Backward paths by query length: one query tile (Lq <= 128) -> the fused short-query
// pass; 2 .. nsp_max_tiles query tiles -> the non-sequence-parallel pass (one CTA owns the
// sequence and head: every tile pair once, dQ summed over key tiles in fp32); longer ->
// the split dK/dV and dQ passes.  nsp_max_tiles is a process-wide setting
// (jfa_set_nsp_max_tiles), 0 .. kNspMaxTiles; below 2 no sequence takes the pass.
constexpr int kNspMaxTiles = 16;
constexpr int kNspDefaultMaxTiles = 0;
__host__ __device__ inline bool nsp_path(int Lq, int max_tiles) { return Lq > kBM && Lq <= max_tiles * kBM; }

// Tensor-map slots per sequence (per-sequence maps clip TMA boxes at the sequence end
// so rows past it arrive as zeros).
enum MapSlot { kMapQ = 0, kMapK = 1, kMapV = 2, kMapDO = 3, kNumMapSlots = 4 };

// A map whose row extent was shortened on the device still has the TMA unit READ every
// row of a box from memory (the rows past the extent are only zero-filled in shared
// memory), so a box at the tail of the last sequence would read up to 127 rows past the
// end of the caller's tensor.  Boxes that would cross a tensor's last row therefore load
// from a workspace copy of its last 128 rows followed by 128 rows of slack, through
// "tail maps": one per possible start row of such a box (start - (total - 128) is in
// [1, 127]), stored after the per-sequence maps.
constexpr int kTailRows = 2 * kBM;  // rows per tensor in the workspace tail copy
constexpr int kTailMaps = kBM;      // tail maps per tensor

// Header at the start of the workspace.
// Developer tracing (off unless a buffer is configured): one thread per warp role of
// CTA 0 records (SM clock << 16 | role << 8 | event) into its own region of `cap` entries.
enum TraceRole {
  kTraceProducer = 0,
  kTraceMma = 1,
  kTraceCompute0 = 2,
  kTraceCompute1 = 3,
  kTraceLoader = 4,
  kTraceRoles = 5
};
struct TraceBuf {
  unsigned long long* buf;  // nullptr: tracing off
  int cap;                  // entries per role
};
#ifdef __CUDACC__
__device__ __forceinline__ void trace_event(const TraceBuf& t, int role, uint32_t& n, int ev) {
  if (t.buf != nullptr && blockIdx.x == 0) {
    if (n < uint32_t(t.cap))
      t.buf[size_t(role) * t.cap + n] = (static_cast<unsigned long long>(clock64()) << 16) |
                                        (static_cast<unsigned long long>(role) << 8) | unsigned(ev);
    ++n;
  }
}
#endif

struct WsHeader {
  int status;      // jfa_status of device-side checks (0 = ok)
  int n_fwd;       // number of forward items
  int n_dq;        // number of dQ items
  int n_dkv;       // number of dK/dV items
  int64_t total_qpad;  // sum_b round_up(Lq_b, 128): rows of the padded per-query vectors
  int n_fused;     // number of fused short-query backward items
  // next unclaimed item of each list (forward, dQ, dK/dV, fused, non-sequence-parallel),
  // zeroed by the planner
  int claim_fwd, claim_dq, claim_dkv, claim_fused;
  int claim_nsp;
  // item hand-off wait limit of the kernel that walks each list (forward, dQ, dK/dV, fused,
  // non-sequence-parallel), in ns, from wait_limit_ns over the list's planned tile pairs
  // (written by the planner)
  uint64_t wait_ns[5];
  int n_nsp;       // number of non-sequence-parallel backward items
  int pad[41];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct WsLayout {
  size_t maps = 0;       // CUtensorMap[B][kNumMapSlots], then CUtensorMap[kNumMapSlots][kTailMaps]
  size_t tail = 0;       // per used slot: kTailRows rows of the tensor's row pitch (tail copies)
  size_t row_bytes = 0;  // H * d * 2, the row pitch of q, k, v, dout
  size_t fwd = 0;      // WorkItem[cap_fwd]
  size_t dq = 0;       // WorkItem[cap_dq]
  size_t dkv = 0;      // WorkItem[cap_dkv]
  size_t fused = 0;    // WorkItem[cap_fused]  backward: sequences whose queries fit one tile
  size_t nsp = 0;      // WorkItem[cap_nsp]    backward: sequences of 2 .. kNspMaxTiles query tiles
  size_t dqacc = 0;    // float[total_q][H][d] backward: their dQ sums over key tiles
  size_t bias2 = 0;    // float[H][num_buckets]  bias table pre-multiplied by log2(e)
  size_t qpad = 0;     // int64[B+1]  backward: offsets of each sequence in the padded vectors
  size_t lse2 = 0;     // float[H][qpad_cap]  backward: lse * log2(e) (+inf if -inf), 0 on padding
  size_t delta = 0;    // float[H][qpad_cap]  backward: D_i = rowsum(dO * O), 0 on padding
  size_t total = 0;
  int64_t cap_fwd = 0, cap_dq = 0, cap_dkv = 0, cap_fused = 0, cap_nsp = 0, qpad_cap = 0;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Capacities are upper bounds on the item counts for any offsets with these totals:
//   sum_b ceil(ceil(L_b/128)/2) <= total/256 + B,  sum_b ceil(L_b/128) <= total/128 + B.
// `nsp`: the backward may route sequences to the non-sequence-parallel pass, which needs its
// fp32 dQ sum buffer (4 * total_q * H * d bytes); without it the buffer is left out.
__host__ __device__ inline WsLayout make_layout(int B, int H, int d, int64_t total_q, int64_t total_kv,
                                                bool backward, bool nsp = false) {
  WsLayout L;
  size_t off = sizeof(WsHeader);
  L.maps = align_up(off, 128);
  off = L.maps + (size_t(B) + kTailMaps) * kNumMapSlots * 128;
  L.row_bytes = size_t(H) * size_t(d) * 2;
  L.tail = align_up(off, 1024);
  off = L.tail + size_t(backward ? 4 : 3) * kTailRows * L.row_bytes;
  L.cap_fwd = int64_t(H) * (total_q / 256 + B + 1);
  L.fwd = align_up(off, 16);
  off = L.fwd + size_t(L.cap_fwd) * sizeof(WorkItem);
  L.bias2 = align_up(off, 256);
  off = L.bias2 + size_t(H) * size_t(kMaxBuckets) * sizeof(float);
  if (backward) {
    L.cap_dq = int64_t(H) * (total_q / 128 + B + 1);
    L.dq = align_up(off, 16);
    off = L.dq + size_t(L.cap_dq) * sizeof(WorkItem);
    L.cap_dkv = int64_t(H) * (total_kv / 128 + B + 1);
    L.dkv = align_up(off, 16);
    off = L.dkv + size_t(L.cap_dkv) * sizeof(WorkItem);
    L.cap_fused = int64_t(H) * (B + 1);
    L.fused = align_up(off, 16);
    off = L.fused + size_t(L.cap_fused) * sizeof(WorkItem);
    L.cap_nsp = int64_t(H) * (B + 1);
    L.nsp = align_up(off, 16);
    off = L.nsp + size_t(L.cap_nsp) * sizeof(WorkItem);
    L.dqacc = align_up(off, 256);
    off = L.dqacc + (nsp ? size_t(total_q) * size_t(H) * size_t(d) * sizeof(float) : 0);
    L.qpad = align_up(off, 256);
    off = L.qpad + size_t(B + 1) * sizeof(int64_t);
    L.qpad_cap = int64_t(align_up(size_t(total_q) + size_t(kBM) * B, kBM));  // rows per head, 512-B aligned
    L.lse2 = align_up(off, 256);
    off = L.lse2 + size_t(H) * size_t(L.qpad_cap) * sizeof(float);
    L.delta = align_up(off, 256);
    off = L.delta + size_t(H) * size_t(L.qpad_cap) * sizeof(float);
  }
  L.total = align_up(off, 256);
  return L;
}

// Number of key tiles query tile t of a sequence visits (bottom-right causal).
__host__ __device__ inline int kv_tiles_for_q_tile(int t, int Lq, int Lk, bool causal) {
  if (Lk <= 0 || t * kBM >= Lq) return 0;
  if (!causal) return (Lk + kBN - 1) / kBN;
  const int i_max = min(t * kBM + kBM - 1, Lq - 1);
  const int last_j = min(Lk - 1, i_max + (Lk - Lq));
  return last_j < 0 ? 0 : last_j / kBN + 1;
}

// First query tile that sees any key of key tile t (causal), and the count of query tiles visited.
__host__ __device__ inline void q_tiles_for_kv_tile(int t, int Lq, int Lk, bool causal, int* first,
                                                    int* count) {
  const int nq = (Lq + kBM - 1) / kBM;
  if (Lq <= 0 || t * kBN >= Lk) {
    *first = 0;
    *count = 0;
    return;
  }
  if (!causal) {
    *first = 0;
    *count = nq;
    return;
  }
  // key j is seen by query i iff i >= j - (Lk - Lq); the smallest key of the tile is t*kBN
  const int i_min = max(0, t * kBN - (Lk - Lq));
  if (i_min >= Lq) {
    *first = 0;
    *count = 0;
    return;
  }
  *first = i_min / kBM;
  *count = nq - *first;
}

#ifdef __CUDACC__
// The tensor map and box row coordinate that load row tile `t` of a sequence starting at
// row `row0` of a tensor with `total` rows: the sequence's own map, or the tail map when
// the 128-row box would reach past the tensor's last row (such a tile is always the
// sequence's last; its tail map points at the tile's first row, so the box starts at 0).
struct TileMap {
  const CUtensorMap* map;
  int y;
  bool tail;
};
__device__ __forceinline__ TileMap tile_map(const CUtensorMap* maps, int B, int slot, int b, int64_t row0, int t,
                                            int64_t total) {
  const int64_t g0 = row0 + int64_t(t) * kBM;
  if (g0 + kBM > total)
    return {maps + size_t(B) * kNumMapSlots + size_t(slot) * kTailMaps + size_t(g0 + kBM - total), 0, true};
  return {maps + size_t(b) * kNumMapSlots + slot, t * kBM, false};
}

// Pull row tile `t` of a sequence (boxes of 64 columns from column col0) into L2 ahead of
// its load.  Tiles whose box would reach past the tensor's last row are skipped.
template <int kBoxes>
__device__ __forceinline__ void prefetch_tile(const CUtensorMap* maps, int B, int slot, int b, int64_t row0, int t,
                                              int64_t total, int col0) {
  const TileMap m = tile_map(maps, B, slot, b, row0, t, total);
  if (m.tail) return;
#pragma unroll
  for (int c = 0; c < kBoxes; ++c)
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(m.map), "r"(col0 + c * 64),
                 "r"(m.y)
                 : "memory");
}
#endif

}  // namespace jfa
