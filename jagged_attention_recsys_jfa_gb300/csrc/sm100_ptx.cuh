// Thin inline-PTX wrappers for the Blackwell (sm_100 family, built for sm_103a)
// features the jagged attention kernels use: mbarriers with bounded waits, TMA
// tiled loads, per-sequence tensor-map patching, and tcgen05 tensor-core MMAs
// with their tensor-memory (TMEM) accumulators.  Written from the public PTX ISA.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace jfa {

// ---------------------------------------------------------------- addresses
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  A kernel launched with programmatic stream serialization
// may start while the previous kernel on its stream is still finishing; it must wait here
// before it reads or writes anything earlier work produced.  launch_dependents lets the next
// kernel launch once every CTA of this one has issued it (or exited).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Pull the line holding `p` into L2 (no value returned, never faults on a valid address).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Fire-and-forget fp32 addition into global memory (performed at L2, no value returned).
__device__ __forceinline__ void red_add_global(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Four consecutive fp32 values (16-byte aligned): added into global memory at L2; stored;
// loaded through L2 only (never from a possibly stale L1 line).
__device__ __forceinline__ void red_add_global_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ void st_global_v4f(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ float4 ld_global_cg_v4f(const float* p) {
  float4 r;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p)
               : "memory");
  return r;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Every wait in the
// kernels is bounded: after `timeout_ns` (or as soon as another warp of the CTA
// has raised `*abort`) it gives up, raises `*abort` and returns false, so a lost
// arrival turns into an error status instead of a hung GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// The same wait with its limit read from `*timeout_ns` (a per-launch value in global
// memory) only after the first test has failed, so the fast path loads nothing; never
// below `floor_ns`.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          const uint64_t* timeout_ns, uint64_t floor_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t = *timeout_ns;
  return mbar_wait(bar, parity, abort, t > floor_ns ? t : floor_ns);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// Pull a tile into L2 ahead of its load (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
               : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmap_acquire(const void* tmap) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(tmap) : "memory");
}
__device__ __forceinline__ void tmap_prefetch(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
// Patch a 128-byte tensor map that lives in global memory.
__device__ __forceinline__ void tmap_replace_address(void* tmap, const void* addr) {
  asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(tmap), "l"(addr)
               : "memory");
}
__device__ __forceinline__ void tmap_replace_dim1(void* tmap, uint32_t dim) {
  asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(tmap), "r"(dim)
               : "memory");
}
__device__ __forceinline__ void tmap_release() {
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05 / TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T  (both operands described by smem descriptors)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// True in exactly one lane (the lowest active one) of a converged warp.  The forward's MMA
// warp runs its issue loop with all 32 lanes, so loop state and descriptors stay
// warp-uniform, and issues each tcgen05 instruction from the elected lane (measured faster
// there than a lane-0-only loop; the backward passes measured slower that way and keep the
// single-lane loop).
__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r));
  return r != 0;
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle, for tcgen05 operands.
//   start address >> 4 in bits [0,14), leading byte offset >> 4 in [16,30),
//   stride byte offset >> 4 in [32,46), descriptor version 1 in [46,48),
//   base offset 0 (atoms are 1024-byte aligned), swizzle mode 2 (128B) in [61,64).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
//   D format f32 (bit 4), A bf16 (bits 7-9 = 1), B bf16 (bits 10-12 = 1),
//   A/B major (bits 15/16: 0 = K-major, 1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// 32 lanes x 32 bits, 32 consecutive columns: thread t of the warp receives
// columns [col, col+32) of lane (warp's lane quarter base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]),
      "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]),
      "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]),
      "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]),
      "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- math helpers
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Per-warpgroup register budget changes (all four warps of a warpgroup execute them).
// The sum over warpgroups must stay within the block's launch allocation.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Packed fp32x2 arithmetic (two lanes of math per instruction) and 3-input max.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 32 bytes (a full L2 sector) per thread in one store; 32-byte aligned address.
__device__ __forceinline__ void st_global_v8(void* ptr, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(ptr), "r"(a0), "r"(a1), "r"(a2), "r"(a3),
               "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// Stores one NB-byte row segment per lane (NB = 64 or 128; dst 16-byte aligned, nullptr
// skips the row) so that every store instruction writes whole segments rather than one
// 32-byte piece per row: within each group of NB/16 lanes the 16-byte chunks are transposed
// with xor-shuffles (afterwards lane base+i holds chunk i of the group's rows base..base+G-1),
// then the group writes one row segment per instruction.  All 32 lanes call it together.
template <int NB>
__device__ __forceinline__ void st_rows_coalesced(uint4 (&c)[NB / 16], void* dst) {
  constexpr int G = NB / 16;
  const int lane = threadIdx.x & 31;
  const int i = lane & (G - 1);
#pragma unroll
  for (int s = 1; s < G; s <<= 1) {
    const bool hi = (i & s) != 0;
#pragma unroll
    for (int k = 0; k < G; ++k) {
      if ((k & s) == 0) {
        const uint4 send = hi ? c[k] : c[k | s];
        uint4 got;
        got.x = __shfl_xor_sync(0xffffffffu, send.x, s);
        got.y = __shfl_xor_sync(0xffffffffu, send.y, s);
        got.z = __shfl_xor_sync(0xffffffffu, send.z, s);
        got.w = __shfl_xor_sync(0xffffffffu, send.w, s);
        if (hi) c[k] = got;
        else c[k | s] = got;
      }
    }
  }
  const unsigned long long mine = reinterpret_cast<unsigned long long>(dst);
  const int base = lane & ~(G - 1);
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const unsigned long long d = __shfl_sync(0xffffffffu, mine, base + k);
    if (d != 0ull)
      asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(d + 16ull * i), "r"(c[k].x), "r"(c[k].y),
                   "r"(c[k].z), "r"(c[k].w)
                   : "memory");
  }
}

// bf16 pair (packed in a 32-bit word, element 0 in the low half) -> two floats, exactly.
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Relative-position bias windows.  The bucket of (query i, key j) is j - i + center, so the
// 32 rows of a warp and n consecutive columns of a tile need only n + 31 consecutive table
// entries.  The warp stages them in a per-warp shared scratch with coalesced loads; each lane
// then reads its n values from there.  For a fixed column the lanes read consecutive words,
// so every read is one conflict-free wavefront, where the same gather straight from global
// memory touches two cache lines per instruction.  That pays where the gather bounds the
// pass (the dQ pass at d = 64, whose three GEMMs per tile pair are short); the forward and
// the key-row passes measured faster gathering straight from global memory.
// The window is fetched into registers a tile ahead (relbias_fetch: v = table[clamp(lo + k,
// 0, nb - 1)] for k = lane + 32 r < len, len <= 32 * kRounds, lo the same in every lane) and
// written to the scratch when its tile comes up (relbias_store), so the global loads' latency
// overlaps a whole tile's work.
template <int kRounds>
__device__ __forceinline__ void relbias_fetch(float (&v)[kRounds], const float* table, int lo, int len, int nb,
                                              int lane) {
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int k = lane + 32 * r;
    v[r] = k < len ? __ldg(table + min(max(lo + k, 0), nb - 1)) : 0.f;
  }
}
template <int kRounds>
__device__ __forceinline__ void relbias_store(float* scr, const float (&v)[kRounds], int len, int lane) {
  __syncwarp();  // every lane has read the previous window
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int k = lane + 32 * r;
    if (k < len) scr[k] = v[r];
  }
  __syncwarp();
}

// General jagged bias, split into loads and arithmetic so the loads can be issued before
// the wait for the scores they apply to.  Values are kept as packed bf16 pairs (0 where no
// bias applies).
//
// One query row: N columns from `src` (bf16, 16-byte aligned; the row is padded to a
// multiple of 8 elements, so every 8-column chunk that starts before n_real lies inside
// it); columns c >= n_real (keys past the sequence end) get 0.  src nullptr: all 0.
template <int N>
__device__ __forceinline__ void jbias_load_row(uint32_t* pk, const void* src, int n_real) {
#pragma unroll
  for (int c8 = 0; c8 < N / 8; ++c8) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (src != nullptr && 8 * c8 < n_real) w = __ldg(reinterpret_cast<const uint4*>(src) + c8);
    pk[4 * c8 + 0] = w.x;
    pk[4 * c8 + 1] = w.y;
    pk[4 * c8 + 2] = w.z;
    pk[4 * c8 + 3] = w.w;
  }
  if (n_real < N) {
#pragma unroll
    for (int c2 = 0; c2 < N / 2; ++c2) {
      if (2 * c2 >= n_real) pk[c2] = 0u;
      else if (2 * c2 + 1 >= n_real) pk[c2] &= 0xffffu;
    }
  }
}

// One key row j against N query rows: bias[i0 + c][j] at col[c * pitch] (bf16); the lanes
// of a warp hold consecutive keys, so each load instruction reads consecutive elements of
// one query row.  Query rows c >= n_q get 0; col nullptr (a key past the sequence end): all 0.
template <int N>
__device__ __forceinline__ void jbias_load_col(uint32_t* pk, const void* col, int64_t pitch, int n_q) {
  const uint16_t* c16 = reinterpret_cast<const uint16_t*>(col);
#pragma unroll
  for (int c2 = 0; c2 < N / 2; ++c2) {
    const uint32_t lo = (col != nullptr && 2 * c2 < n_q) ? uint32_t(__ldg(c16 + (2 * c2) * pitch)) : 0u;
    const uint32_t hi = (col != nullptr && 2 * c2 + 1 < n_q) ? uint32_t(__ldg(c16 + (2 * c2 + 1) * pitch)) : 0u;
    pk[c2] = lo | (hi << 16);
  }
}

// One warp's 32 consecutive key rows j0 + lane against 64 query rows, loaded with 16-byte
// loads: in pass p (0, 1) chunk q = lane + 32 k (k < 4) is query row 32 p + q / 4, keys
// j0 + 8 (q % 4) .. + 7 of the block (`rows` points at query row 0, key j0; rows `pitch`
// elements apart).  Chunks of query rows >= n_q or starting at a key >= n_k are 0.  The
// values are in row order; jbias_col_transpose hands each lane its key's column.
__device__ __forceinline__ void jbias_load_cols_vec(uint4 (&w)[8], const void* rows, int64_t pitch, int n_q, int n_k,
                                                    int lane) {
  const uint16_t* r16 = reinterpret_cast<const uint16_t*>(rows);
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const int q = lane + 32 * (t & 3), row = 32 * (t >> 2) + q / 4, part = q % 4;
    w[t] = make_uint4(0u, 0u, 0u, 0u);
    if (rows != nullptr && row < n_q && 8 * part < n_k)
      w[t] = __ldg(reinterpret_cast<const uint4*>(r16 + row * pitch + 8 * part));
  }
}

// The transpose through a 2 KB per-warp shared scratch (16-byte aligned): each pass writes
// its 32 rows x 32 keys, then lane l reads key l of every row (consecutive 2-byte elements
// of one row per instruction: no bank conflicts).  key_valid false (a key past the sequence
// end, whose padding holds no bias) gives 0.  Packs two query rows per register.
__device__ __forceinline__ void jbias_col_transpose(uint32_t* pk, const uint4 (&w)[8], uint4* scratch, bool key_valid,
                                                    int lane) {
  const uint16_t* s16 = reinterpret_cast<const uint16_t*>(scratch);
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
    for (int k = 0; k < 4; ++k) scratch[lane + 32 * k] = w[4 * pass + k];
    __syncwarp();
#pragma unroll
    for (int r2 = 0; r2 < 16; ++r2) {
      const uint32_t lo = key_valid ? uint32_t(s16[(2 * r2) * 32 + lane]) : 0u;
      const uint32_t hi = key_valid ? uint32_t(s16[(2 * r2 + 1) * 32 + lane]) : 0u;
      pk[16 * pass + r2] = lo | (hi << 16);
    }
    __syncwarp();
  }
}

// The reverse of the two helpers above, for the general bias's gradient: a warp's 32 key
// rows (lane) x 64 query rows, as packed bf16 pairs of query rows (pk[r2] = rows 2 r2,
// 2 r2 + 1 of this lane's key), written row-major to `rows` (query row 0, key j0; rows
// `pitch` elements apart) through the per-warp scratch, as 16-byte chunks: query rows >= n_q
// and chunks starting at a key >= n_k are not written; key_valid false writes 0 (the row
// padding past the sequence's keys).
__device__ __forceinline__ void jbias_store_cols(const uint32_t* pk, uint4* scratch, void* rows, int64_t pitch,
                                                 int n_q, int n_k, bool key_valid, int lane) {
  uint16_t* s16 = reinterpret_cast<uint16_t*>(scratch);
  uint16_t* r16 = reinterpret_cast<uint16_t*>(rows);
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
    for (int r2 = 0; r2 < 16; ++r2) {
      const uint32_t v = key_valid ? pk[16 * pass + r2] : 0u;
      s16[(2 * r2) * 32 + lane] = uint16_t(v & 0xffffu);
      s16[(2 * r2 + 1) * 32 + lane] = uint16_t(v >> 16);
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int q = lane + 32 * k, row = q / 4, part = q % 4;
      if (rows != nullptr && 32 * pass + row < n_q && 8 * part < n_k)
        *reinterpret_cast<uint4*>(r16 + (32 * pass + row) * pitch + 8 * part) = scratch[q];
    }
    __syncwarp();
  }
}

// x[c] = x[c] * sl2 + l2e * bias[c] for the N columns, bias from the packed pairs.
template <int N>
__device__ __forceinline__ void jbias_apply(float* x, const uint32_t* pk, float sl2, float l2e) {
  const uint64_t k_sl2 = f2_pack(sl2, sl2), k_l2e = f2_pack(l2e, l2e);
#pragma unroll
  for (int c2 = 0; c2 < N / 2; ++c2)
    f2_unpack(f2_fma(f2_pack(bf16lo(pk[c2]), bf16hi(pk[c2])), k_l2e, f2_mul(f2_pack(x[2 * c2], x[2 * c2 + 1]), k_sl2)),
              x[2 * c2], x[2 * c2 + 1]);
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace jfa
