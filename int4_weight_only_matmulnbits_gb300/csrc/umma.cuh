// Device helpers shared by the tcgen05 (TMEM) tensor-core kernels: shared-
// memory operand descriptors, tcgen05 fences and loads, TMA stores, bf16x2
// arithmetic and the exact hi + lo split of a dequantised weight pair.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "mnb_common.cuh"

namespace mnb {

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  // K-major operand, 128-byte swizzle: rows of 128 bytes, 8-row atoms of
  // 1024 bytes (stride dimension byte offset), descriptor version 1.
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFF) >> 4);         // start address
  d |= static_cast<uint64_t>(16 >> 4) << 16;                  // leading byte offset
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                        // version
  d |= static_cast<uint64_t>(2) << 61;                        // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled TMA store from this CTA's shared memory (bulk group).
__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(smem_addr(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk store has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// w = (q - z) * s for a bf16 pair holding 128 + q, returned as two bf16
// pairs whose sum is w: hi = w rounded to bf16, lo = (w - hi) rounded to
// bf16. The tensor core multiplies the activations by both (two MMAs into
// one accumulator), so no weight carries the 2^-8 relative error of a single
// bf16 rounding:
//  * bf16 scales: q - z is an integer of at most 4 bits and s has an 8-bit
//    significand, so w is exact in 12 bits; hi takes the leading 8 and the
//    fused multiply-add returns the remainder w - hi exactly (at most 5
//    significant bits). hi + lo == w.
//  * fp32 scales: w is formed in fp32 (relative error 2^-24), w - hi is exact
//    in fp32, and rounding it to bf16 leaves at most 2^-8 |w - hi| <=
//    2^-16 |w|.
template <bool SF32>
__device__ __forceinline__ void dequant_pair(uint32_t v, uint32_t zc, uint32_t sb, float sf,
                                             uint32_t &hi, uint32_t &lo) {
  const uint32_t dq = bf16x2_sub(v, zc);  // q - z, exact
  if (!SF32) {
    hi = bf16x2_mul(dq, sb);
    lo = bf16x2_fma(dq, sb, hi ^ 0x80008000u);  // w - hi, exact
    return;
  }
  const float w0 = bf16_bits_to_f32(dq & 0xFFFFu) * sf;
  const float w1 = bf16_bits_to_f32(dq >> 16) * sf;
  hi = f32x2_to_bf16x2(w0, w1);
  lo = f32x2_to_bf16x2(w0 - bf16_bits_to_f32(hi & 0xFFFFu), w1 - bf16_bits_to_f32(hi >> 16));
}

// Output column (within the CTA's 128) of B row / accumulator column c.
__host__ __device__ constexpr int out_col(int c) {
  return (c & ~15) + ((c & 1) ? 8 : 0) + ((c & 15) >> 1);
}

}  // namespace mnb
