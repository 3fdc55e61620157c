// Thin inline-PTX wrappers for sm_103a: shared-memory barriers (mbarrier), TMA tensor
// loads, tcgen05 tensor-memory allocation / MMA / load / store, and the bounded waits the
// kernels use instead of unbounded spins.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace bw {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Called by a whole converged warp: one elected lane arrives (with the expected byte count).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
               "@pe mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n\t}\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the barrier phase with the given parity has completed. Gives up after
// `timeout_ns` of wall time or as soon as *abort is set; returns false then.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int* abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(a, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
  }
}

// Record a timed-out wait: CTA-local abort flag plus the device status word.
__device__ __forceinline__ void raise_timeout(volatile int* abort, unsigned int* status) {
  *abort = 1;
  atomicOr(status, kStatusTimeoutBit);
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled bulk tensor load global -> shared, completion counted in bytes on `bar`.
// Called by a whole converged warp: one elected lane issues the copy.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
      "@pe cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];\n\t}\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05 (TMEM + UMMA)

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

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B), in two 32-bit halves. Low word: start address >> 4 (bits 0-13) and
// leading-dimension byte offset >> 4 (bits 16-29); high word: stride-dimension byte offset >> 4
// (descriptor bits 32-45), version 1 (bits 46-47), base offset 0, swizzle mode 2 = 128B (bits
// 61-63). Within one swizzle-aligned tile, moving the start address only changes the low word.
//
// The MMA and commit wrappers below are called by a whole converged warp with warp-uniform
// operands: one lane, chosen by elect.sync (the same lane on every call of a full warp), issues
// the instructions. Keeping the issuing warp converged keeps the descriptor arithmetic on the
// warp-uniform datapath; issuing from a single-lane branch made every MMA about 100 cycles
// apart, against 64 cycles of tensor work for an M128 N128 K16 MMA.
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint32_t sdesc_hi(uint32_t sbo_bytes) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}

// Eight K=16 steps of D[tmem] (+)= A[smem] B[smem] over a 128-element-deep contraction held as
// two 128-byte swizzle atoms (K-major, 128 rows per atom): the start address advances by 32 B
// inside an atom and by one atom (`atom_bytes`) after four steps. acc0 = 0 overwrites D.
__device__ __forceinline__ void umma_ss_k128(uint32_t d_tmem, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi,
                                             uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, pe;\n\t.reg .b64 da, db;\n\t.reg .b32 xa, xb;\n\telect.sync _|pe, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %6, 0;\n\tsetp.eq.u32 p1, 0, 0;\n\t"
      "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p0;\n\t"
      "add.u32 xa, %1, 2;\n\tadd.u32 xb, %3, 2;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t"
      "add.u32 xa, %1, 4;\n\tadd.u32 xb, %3, 4;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t"
      "add.u32 xa, %1, 6;\n\tadd.u32 xb, %3, 6;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t"
      "add.u32 xa, %1, 1024;\n\tadd.u32 xb, %3, 1024;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t"
      "add.u32 xa, %1, 1026;\n\tadd.u32 xb, %3, 1026;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t"
      "add.u32 xa, %1, 1028;\n\tadd.u32 xb, %3, 1028;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t"
      "add.u32 xa, %1, 1030;\n\tadd.u32 xb, %3, 1030;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t}\n" ::"r"(d_tmem),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc0)
      : "memory");
}

// Same for a 64-element-deep contraction (one atom): four K=16 steps.
__device__ __forceinline__ void umma_ss_k64(uint32_t d_tmem, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi,
                                            uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, pe;\n\t.reg .b64 da, db;\n\t.reg .b32 xa, xb;\n\telect.sync _|pe, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %6, 0;\n\tsetp.eq.u32 p1, 0, 0;\n\t"
      "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p0;\n\t"
      "add.u32 xa, %1, 2;\n\tadd.u32 xb, %3, 2;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t"
      "add.u32 xa, %1, 4;\n\tadd.u32 xb, %3, 4;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t"
      "add.u32 xa, %1, 6;\n\tadd.u32 xb, %3, 6;\n\tmov.b64 da, {xa, %2};\n\tmov.b64 db, {xb, %4};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p1;\n\t}\n" ::"r"(d_tmem),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc0)
      : "memory");
}

// Eight K=16 steps of D[tmem] (+)= A[tmem] B[smem]: A advances 8 columns (16 bf16) per step,
// B (MN-major, 128-byte rows) advances 16 rows = 2048 B per step. acc0 = 0 overwrites D.
__device__ __forceinline__ void umma_ts_k128(uint32_t d_tmem, uint32_t a_tmem, uint32_t blo, uint32_t bhi,
                                             uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, pe;\n\t.reg .b64 db;\n\t.reg .b32 ta, xb;\n\telect.sync _|pe, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %5, 0;\n\tsetp.eq.u32 p1, 0, 0;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p0;\n\t"
      "add.u32 ta, %1, 8;\n\tadd.u32 xb, %2, 128;\n\tmov.b64 db, {xb, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 16;\n\tadd.u32 xb, %2, 256;\n\tmov.b64 db, {xb, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 24;\n\tadd.u32 xb, %2, 384;\n\tmov.b64 db, {xb, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 32;\n\tadd.u32 xb, %2, 512;\n\tmov.b64 db, {xb, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 40;\n\tadd.u32 xb, %2, 640;\n\tmov.b64 db, {xb, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 48;\n\tadd.u32 xb, %2, 768;\n\tmov.b64 db, {xb, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t"
      "add.u32 ta, %1, 56;\n\tadd.u32 xb, %2, 896;\n\tmov.b64 db, {xb, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p1;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc0)
      : "memory");
}

// Packed fp32 pairs (one instruction for two lanes of work): d = a * b + c, d = a + b.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\tmov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}\n"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

// 32 lanes x 16 columns store (thread t of the warp writes lane base + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Arrive once on `bar` when every tcgen05 async op issued so far by the warp's elected lane completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
               "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Registers written by tcgen05.ld may be read only after tcgen05.wait::ld. Passing them
// through an empty volatile asm placed after the wait makes every later use depend on it,
// so the compiler cannot hoist a use above the wait.
__device__ __forceinline__ void tmem_reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane (base lane + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9 = 1), B bf16
// (bits 10-12 = 1), A major (bit 15), B major (bit 16; 1 = MN-major), N >> 3 (bits 17-22),
// M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn_major & 1) << 15) |
         (static_cast<uint32_t>(b_mn_major & 1) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- scalar helpers

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` goes to the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace bw
