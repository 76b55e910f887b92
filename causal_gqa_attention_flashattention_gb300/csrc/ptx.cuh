// Thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// bulk copies/reductions, tcgen05 (TMEM alloc, MMA, ld/st, commit, fences).
// Written from the PTX ISA description of each instruction; no library code.
#pragma once
#include <cuda.h>
#include <cstdint>

namespace ne {

// Upper bound on any single wait inside a kernel.  A wait that runs past it
// records NE_ERR_DEVICE_TIMEOUT in the device status word and gives up, so a
// broken pipeline returns an error instead of hanging the GPU.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One arrival per warp instead of 32 on the same shared-memory word: the warp
// barrier orders every lane's earlier work (including its tcgen05 wait and
// fence) before lane 0's release-arrive.  A barrier a whole group of threads
// signals this way is initialised with the group's number of warps.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
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

// Non-blocking test: has the phase of `bar` with parity `parity` completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
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

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or about `hint_ns` nanoseconds pass, instead of spinning and
// taking issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits until the phase of `bar` with parity `parity` has completed.
// Returns false if *abort becomes non-zero or the wait exceeds limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------------------ proxies / fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMA / bulk
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 4-D tiled load, coordinates innermost first; completes `bar` by the box bytes.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled load, coordinates innermost first; completes `bar` by the box bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Element-wise fp32 add of a shared-memory block into global memory.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, const void* src, uint32_t bytes) {
  asm volatile(
      "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
          reinterpret_cast<uint64_t>(gdst)),
      "r"(smem_u32(src)), "r"(bytes)
      : "memory");
}
// Tiled 4-D store shared -> global (rows outside the tensor are not written).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* m, const void* src, int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the sources of all but the newest N bulk groups have been read.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ tcgen05: TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMEM address: lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// 32 lanes x 32 bit, 16 consecutive columns per thread (thread i <-> lane base+i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// ------------------------------------------------------------------ tcgen05: MMA
// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), version 1 at bits 46..47, swizzle mode in
// bits 61..63 (0 none, 2 = 128-byte, 4 = 64-byte, 6 = 32-byte).
enum : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation.  A and B share
// one operand type: fp16 (format code 0) or bf16 (format code 1).
// a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool a_mn, bool b_mn, bool bf16) {
  return (1u << 4)                          // D format: f32
         | ((bf16 ? 1u : 0u) << 7)          // A format
         | ((bf16 ? 1u : 0u) << 10)         // B format
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return idesc_f16kind(M, N, a_mn, b_mn, true);
}
__host__ __device__ constexpr uint32_t idesc_fp16(int M, int N, bool a_mn, bool b_mn) {
  return idesc_f16kind(M, N, a_mn, b_mn, false);
}
// kind::f8f6f4 with both operands e4m3 (format code 0 in the same A / B fields)
// and fp32 accumulation: the same bit pattern as fp16 under kind::f16.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn, bool b_mn) {
  return idesc_f16kind(M, N, a_mn, b_mn, false);
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Chains of NK MMAs into one accumulator, operand k at base + k * step (step in
// 16-byte units, added to the descriptor's start-address field).  The first
// MMA accumulates if `acc`, the rest always do.  All NK instructions sit in one
// asm block with their predicates set once, so the issuing thread spends its
// time on the MMAs themselves.
template <int NK>
__device__ __forceinline__ void mma_ss_chain(uint32_t d, uint64_t a, uint32_t a_step, uint64_t b, uint32_t b_step,
                                             uint32_t idesc, uint32_t acc) {
  static_assert(NK == 2 || NK == 4 || NK == 8, "chain length");
  uint64_t ad[NK], bd[NK];
#pragma unroll
  for (int k = 0; k < NK; k++) {
    ad[k] = a + (uint64_t)(k * a_step);
    bd[k] = b + (uint64_t)(k * b_step);
  }
  if constexpr (NK == 2) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 q, %5, %5;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %3, %6, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %4, %6, q;\n\t}" ::"r"(d),
        "l"(ad[0]), "l"(ad[1]), "l"(bd[0]), "l"(bd[1]), "r"(acc), "r"(idesc)
        : "memory");
  } else if constexpr (NK == 4) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %9, 0;\n\tsetp.eq.b32 q, %9, %9;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %10, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %10, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %10, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %10, q;\n\t}" ::"r"(d),
        "l"(ad[0]), "l"(ad[1]), "l"(ad[2]), "l"(ad[3]), "l"(bd[0]), "l"(bd[1]), "l"(bd[2]), "l"(bd[3]),
        "r"(acc), "r"(idesc)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %17, 0;\n\tsetp.eq.b32 q, %17, %17;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %18, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %18, q;\n\t}" ::"r"(d),
        "l"(ad[0]), "l"(ad[1]), "l"(ad[2]), "l"(ad[3]), "l"(ad[4]), "l"(ad[5]), "l"(ad[6]), "l"(ad[7]),
        "l"(bd[0]), "l"(bd[1]), "l"(bd[2]), "l"(bd[3]), "l"(bd[4]), "l"(bd[5]), "l"(bd[6]), "l"(bd[7]),
        "r"(acc), "r"(idesc)
        : "memory");
  }
}

// Two MMAs of kind::f8f6f4 (8-bit operands, 32 values of K each) into one
// accumulator; operand k at base + k * step (16-byte units).
__device__ __forceinline__ void mma_ss_chain2_f8(uint32_t d, uint64_t a, uint32_t a_step, uint64_t b, uint32_t b_step,
                                                 uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 q, %5, %5;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %3, %6, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %2, %4, %6, q;\n\t}" ::"r"(d),
      "l"(a), "l"(a + (uint64_t)a_step), "l"(b), "l"(b + (uint64_t)b_step), "r"(acc), "r"(idesc)
      : "memory");
}

// Same with the A operand in tensor memory: A_k at TMEM column a + 8k (16
// bf16/fp16 values per k-step).  SPLIT places k-steps 4..7 at a + 64 + 8(k-4):
// an operand whose two 64-wide halves were written into separate column ranges.
template <int NK, bool SPLIT = false>
__device__ __forceinline__ void mma_ts_chain(uint32_t d, uint32_t a, uint64_t b, uint32_t b_step, uint32_t idesc,
                                             uint32_t acc) {
  static_assert(NK == 2 || NK == 4 || NK == 8, "chain length");
  uint32_t at[NK];
  uint64_t bd[NK];
#pragma unroll
  for (int k = 0; k < NK; k++) {
    at[k] = a + ((SPLIT && k >= 4) ? 64u + 8u * (k - 4) : 8u * k);
    bd[k] = b + (uint64_t)(k * b_step);
  }
  if constexpr (NK == 2) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 q, %5, %5;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %3, %6, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %4, %6, q;\n\t}" ::"r"(d),
        "r"(at[0]), "r"(at[1]), "l"(bd[0]), "l"(bd[1]), "r"(acc), "r"(idesc)
        : "memory");
  } else if constexpr (NK == 4) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %9, 0;\n\tsetp.eq.b32 q, %9, %9;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %10, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %10, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %10, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %10, q;\n\t}" ::"r"(d),
        "r"(at[0]), "r"(at[1]), "r"(at[2]), "r"(at[3]), "l"(bd[0]), "l"(bd[1]), "l"(bd[2]), "l"(bd[3]),
        "r"(acc), "r"(idesc)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %17, 0;\n\tsetp.eq.b32 q, %17, %17;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %9, %18, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %18, q;\n\t}" ::"r"(d),
        "r"(at[0]), "r"(at[1]), "r"(at[2]), "r"(at[3]), "r"(at[4]), "r"(at[5]), "r"(at[6]), "r"(at[7]),
        "l"(bd[0]), "l"(bd[1]), "l"(bd[2]), "l"(bd[3]), "l"(bd[4]), "l"(bd[5]), "l"(bd[6]), "l"(bd[7]),
        "r"(acc), "r"(idesc)
        : "memory");
  }
}

// Arrive once on `bar` when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ register budget
// Per-warpgroup register limits (all four warps of a warpgroup execute these):
// dec returns registers to the block's pool, inc takes them from it and waits
// until enough are free.  The warpgroups' shares must add up to at most the
// block's launch total (threads x registers per thread at launch).
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ misc math
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed pairs of fp32 (sm_100+ f32x2 arithmetic: one instruction handles two
// values, on the FMA pipe).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t w) {
  float f;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, a;\n\t}" : "=f"(f) : "r"(w));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  float f;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, b;\n\t}" : "=f"(f) : "r"(w));
  return f;
}

// Double-float helpers: a value carried as hi + lo (two fp32 numbers).
constexpr float kLn2Hi = 0.693147182464599609375f;       // fp32(ln 2)
constexpr float kLn2Lo = -1.904654299957768e-09f;        // ln 2 - kLn2Hi
constexpr float kLog2eHi = 1.44269502162933349609375f;   // fp32(log2 e)
constexpr float kLog2eLo = 1.925963033500011e-08f;       // log2 e - kLog2eHi
// hi + lo = a + b exactly (Knuth's two-sum).  The _rn intrinsics keep the
// compiler from fusing these operations into FMAs, which would break the
// exactness the algorithm relies on.
__device__ __forceinline__ void two_sum(float a, float b, float& hi, float& lo) {
  hi = __fadd_rn(a, b);
  const float bb = __fsub_rn(hi, a);
  lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(b, bb));
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile whose rows are
// `span` bytes (32, 64 or 128) and which uses the matching TMA/UMMA swizzle:
// the chunk index is XORed with address bits 7.. of the unswizzled offset.
__host__ __device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk, uint32_t span) {
  uint32_t lin = row * span + chunk * 16u;
  uint32_t mask = span / 16u - 1u;
  return lin ^ (((lin >> 7) & mask) << 4);
}

}  // namespace ne
