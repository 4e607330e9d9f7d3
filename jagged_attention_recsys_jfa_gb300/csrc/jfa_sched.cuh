// Work-item metadata staged in shared memory.  One scheduler thread per CTA claims items
// of the planner's longest-first list from a launch-wide counter, loads each item and
// its sequence's offsets from global memory, and publishes them into a small ring; every
// role of the CTA (loaders, MMA issuer, compute warps) takes item k from the ring.  Items
// are claimed one ahead of the one in progress, so the list is dealt out greedily, largest
// first, to whichever CTA frees up first, and the dependent global loads (item, then
// offsets) are still off the critical path at unit boundaries.
#pragma once
#include "jfa_common.cuh"
#include "sm100_ptx.cuh"

namespace jfa {

constexpr int kMetaSlots = 4;
// Arrivals that free an entry: the three single-thread roles of warpgroup 0 (streaming
// producer, MMA issuer, resident-tile loader) and one per compute warp.
constexpr int kMetaConsumers = 3 + (kThreads / 32 - kFirstComputeWarp);

struct ItemMeta {
  int b, h, u0, u1;   // the work item: sequence, head, unit range [u0, u1)
  int64_t qo, ko;     // first query / key row of the sequence
  int Lq, Lk;         // its lengths
  int64_t qp;         // backward: first row of the sequence in the 128-row-padded vectors
  int64_t jb;         // general jagged bias: the sequence's block offset in each head's plane
};

struct MetaRing {
  ItemMeta e[kMetaSlots];
  uint64_t full[kMetaSlots], empty[kMetaSlots];
  // the planner's hand-off wait limit for this launch (global memory; read only by a wait
  // that did not complete at once, so after griddepcontrol.wait)
  const uint64_t* wait_ns;
};

// One thread, before the CTA-wide barrier that publishes mbarrier initialisation.
__device__ __forceinline__ void meta_init(MetaRing& r, const uint64_t* wait_ns, int consumers = kMetaConsumers) {
  for (int i = 0; i < kMetaSlots; ++i) {
    mbar_init(&r.full[i], 1);
    mbar_init(&r.empty[i], consumers);
  }
  r.wait_ns = wait_ns;
}

// Scheduler (one thread).  Claims item k (idx = atomicAdd(claim, 1)) once item k - 2 is
// released by every role, i.e. while the CTA works on item k - 1, so a CTA never holds
// more than one claimed item it has not started.  After the list runs out it publishes an
// end marker (b = -1) that ends every role's loop.  Slot k % kMetaSlots was last used by
// item k - 4, which every role released before item k - 2.  False when a bounded wait ran
// out (the CTA is aborting).
__device__ __forceinline__ bool meta_publish(MetaRing& r, const WorkItem* items, int n_items, int* claim,
                                             const int64_t* q_off, const int64_t* kv_off, const int64_t* qpad,
                                             const int64_t* jb_off, volatile int* abort) {
  for (uint32_t k = 0;; ++k) {
    if (k >= 2) {
      const uint32_t kp = k - 2;
      if (!mbar_wait(&r.empty[kp % kMetaSlots], (kp / kMetaSlots) & 1, abort, r.wait_ns, kWaitTimeoutNs)) return false;
    }
    const int idx = atomicAdd(claim, 1);
    ItemMeta m;
    if (idx < n_items) {
      const WorkItem wi = items[idx];
      m.b = wi.b;
      m.h = wi.h;
      m.u0 = wi.u0;
      m.u1 = wi.u1;
      m.qo = q_off[wi.b];
      m.ko = kv_off[wi.b];
      m.Lq = int(q_off[wi.b + 1] - m.qo);
      m.Lk = int(kv_off[wi.b + 1] - m.ko);
      m.qp = qpad ? qpad[wi.b] : 0;
      m.jb = jb_off ? jb_off[wi.b] : 0;
    } else {
      m = ItemMeta{-1, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    }
    const uint32_t s = k % kMetaSlots;
    r.e[s] = m;
    mbar_arrive(&r.full[s]);  // release: the entry is visible to every thread that waits on it
    if (idx >= n_items) {
      grid_launch_dependents();  // nothing left to claim: the next kernel may take freed SMs
      return true;
    }
  }
}

// The CTA's item after k if the scheduler has already published it (nullptr if not yet,
// or if it is the end marker): a look ahead for L2 prefetches, never a wait.
__device__ __forceinline__ const ItemMeta* meta_peek_next(MetaRing& r, uint32_t k) {
  const uint32_t n = k + 1;
  if (!mbar_test_wait(&r.full[n % kMetaSlots], (n / kMetaSlots) & 1)) return nullptr;
  const ItemMeta* m = &r.e[n % kMetaSlots];
  return m->b >= 0 ? m : nullptr;
}

// Entry k for a single-thread role, read in place for the item's duration and then
// freed with meta_release.
__device__ __forceinline__ bool meta_wait(MetaRing& r, uint32_t k, volatile int* abort) {
  return mbar_wait(&r.full[k % kMetaSlots], (k / kMetaSlots) & 1, abort, r.wait_ns, kWaitTimeoutNs);
}
__device__ __forceinline__ void meta_release(MetaRing& r, uint32_t k) { mbar_arrive(&r.empty[k % kMetaSlots]); }

// Entry k for a whole warp (all 32 lanes call it), which reads the entry in place for
// the item's duration and then frees it with meta_release_warp.  The lanes agree on the
// outcome: a lane whose wait gave up has raised the abort flag, which ends the other
// lanes' waits too.
__device__ __forceinline__ bool meta_wait_warp(MetaRing& r, uint32_t k, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(&r.full[k % kMetaSlots], (k / kMetaSlots) & 1, abort, r.wait_ns, kWaitTimeoutNs));
}
__device__ __forceinline__ void meta_release_warp(MetaRing& r, uint32_t k) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[k % kMetaSlots]);
}

// Tensor maps are acquired once per sequence by each thread that loads through them (and
// an item ahead when possible, with their descriptors prefetched): an acquire makes the
// next copy through the map wait for a fresh descriptor fetch.  `acq_b` is the sequence
// whose maps of these two slots this thread holds.
__device__ __forceinline__ void acquire_seq_maps(const CUtensorMap* maps, int b, int slot_a, int slot_b, int& acq_b,
                                                 bool prefetch) {
  if (b == acq_b) return;
  const CUtensorMap* m = maps + size_t(b) * kNumMapSlots;
  tmap_acquire(m + slot_a);
  tmap_acquire(m + slot_b);
  if (prefetch) {
    tmap_prefetch(m + slot_a);
    tmap_prefetch(m + slot_b);
  }
  acq_b = b;
}

}  // namespace jfa
