// hq_umma.cuh -- fifth-generation tensor-core helpers (tcgen05, sm_103a):
// tensor-memory allocation, shared-memory matrix descriptors, the tf32 and
// bf16 MMAs with an fp32 accumulator in tensor memory, completion through an
// mbarrier, and the 32-lane tensor-memory loads of the epilogue.
//
// Operands sit in shared memory as "core matrices" of 8 rows x 16 bytes
// (8 x 4 tf32 or 8 x 8 bf16 values, row-major inside the core), K-major, no
// swizzle: with E values per 16 bytes, the element (row, k) of an operand
// lives at
//   (row / 8) * SBO + (k / E) * LBO + (row % 8) * 16 + (k % E) * (16 / E)
// bytes from its base, so LBO is the distance between cores adjacent along K
// and SBO the distance between 8-row groups.  An MMA reads two cores along K
// (K = 8 for tf32, 16 for bf16); the next K step starts 2 * LBO further on.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace hq {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Shared-memory matrix descriptor: start address, LBO and SBO in 16-byte
// units, descriptor version 1 (bits 46-47), no swizzle, base offset 0.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::tf32: fp32 accumulator (bits 4-5 = 1),
// A and B tf32 (bits 7-9, 10-12 = 2), both K-major, N / 8 at bit 17,
// M / 16 at bit 24.
constexpr uint32_t umma_idesc_tf32(int m, int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// Instruction descriptor of kind::f16 with fp16 A and B (bits 7-9, 10-12 =
// 0), fp32 accumulator, both K-major.
constexpr uint32_t umma_idesc_f16(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// One warp allocates `ncols` (a power of two >= 32) tensor-memory columns
// and writes their base address to *dst; the permit is given up at once so
// that other blocks on the SM can allocate.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
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
// Makes this thread's ordinary shared-memory stores visible to the tensor
// core (the async proxy); each writing thread issues it before the barrier.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Waits for the completion of the barrier phase of parity `parity`, giving
// up after `limit` polls (false).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
  const uint32_t addr = smem_addr(bar);
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// D (tensor memory) = A * B^T (+ D when `accumulate`), issued by one thread.
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with 16-bit operands (kind::f16, K = 16 per instruction).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on the mbarrier once every MMA this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane (warp w
// reads lanes 32 (w % 4) .. +31; taddr carries the lane in bits 16-31).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// 8 consecutive fp32 columns of this thread's tensor-memory lane (the same
// lane rule as tmem_ld16).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float v[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}

// x = hi + lo with hi = x rounded to tf32 (nearest, ties away) and lo the
// rest, itself rounded to tf32: |x - hi - lo| <= 2^-22 |x|, so the four
// products of two split operands carry an fp32-level error.
__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo) {
  uint32_t h, l;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
  hi = __uint_as_float(h);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(__fsub_rn(x, hi)));
  lo = __uint_as_float(l);
}

// (x0, x1) = hi + lo as fp16 pairs (x0 in the low half of each word) for
// |x| < 1: hi = x rounded to fp16 (nearest even), lo = x - hi (exact in
// fp32) rounded the same way, so |x - hi - lo| <= 2^-22 |x| + 2^-25 (the
// second term from fp16's subnormal spacing 2^-24).
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(x1), "f"(x0));
  float h0, h1;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(h0), "=f"(h1)
      : "r"(hi));
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(__fsub_rn(x1, h1)), "f"(__fsub_rn(x0, h0)));
}

// Power-of-two scale for values of largest magnitude m: scale_of(m) * m lies
// in [1/2, 1) for 2^-126 <= m < 2^126 (below 1 for smaller m, below 4 for
// any finite m), inv_scale_of(m) = 1 / scale_of(m); multiplying by either
// changes no bit of a value that stays in the normal range.
__device__ __forceinline__ uint32_t exp_field_of(float m) {
  return min((__float_as_uint(m) >> 23) & 0xFFu, 252u);
}
__device__ __forceinline__ float scale_of(float m) {
  return __uint_as_float((253u - exp_field_of(m)) << 23);
}
__device__ __forceinline__ float inv_scale_of(float m) {
  return __uint_as_float((exp_field_of(m) + 1u) << 23);
}

}  // namespace hq
