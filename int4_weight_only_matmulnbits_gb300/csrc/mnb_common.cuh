// Internal definitions shared by the sm_103a kernels of the MatMulNBits
// library: the prepacked weight layout and small PTX wrappers.
//
// Prepacked layout (the "packed constant storage aligned for the selected
// kernel" of the page "Qwen3 CPU Inference Critical Path", section "Prepared
// weight-only plan"):
//
//  * Rows are grouped in tiles of 16 (N16 = ceil(N/16) tiles) and K in chunks
//    of 64 (K64 = ceil(K/64) chunks). Codes of rows >= N or k >= K are 0.
//  * packed_b holds N16*K64 chunks of 512 bytes, chunk (tile, c) at byte
//    (tile*K64 + c)*512. Inside a chunk, 32-bit word (lane*4 + j) holds the
//    codes lane `lane` of a warp feeds to the j-th 16-wide k step of the
//    chunk as the A operand of mma.m16n8k16: with g = lane/4, t = lane%4,
//    rows r0 = tile*16 + g and r1 = r0 + 8, and k0 = c*64 + 16*j + 4*t,
//    code (row r0+8*h, k0+e) sits at bit  16*(e&1) + 8*(e>>1) + 4*h.
//    A lop3 of (word >> 4*i) with 0x000F000F and 0x43004300 then yields the
//    bf16 pair (128+q, 128+q') the MMA fragment register i needs. The k
//    order inside each 16-wide step is permuted so that a lane's matching
//    activations A[m][k0 .. k0+3] are four consecutive elements.
//  * packed_scales holds, per (tile, block b), the 16 scales of the tile's
//    rows in the stored dtype: element ((tile*nb + b)*16 + r).
//  * packed_zp holds, per (tile, block b), one 64-bit word whose nibble r is
//    the zero point of row tile*16 + r; each tile has nbz = nb rounded up to
//    even words (element tile*nbz + b), so any even-aligned block range of a
//    tile is a 16-byte aligned span.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mnb {

constexpr int kTileN = 16;       // rows per tile
constexpr int kChunkK = 64;      // k per chunk
constexpr int kChunkBytes = 512; // packed bytes per (tile, chunk)

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) {
  return (a + b - 1) / b;
}

// Bit position of code (row r0 + 8*h, k0 + e) inside its packed word.
__host__ __device__ inline int code_shift(int e, int h) {
  return 16 * (e & 1) + 8 * (e >> 1) + 4 * h;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b,
                                                uint32_t c) {
  uint32_t d;
  // (a & b) | c : lut = (0xF0 & 0xCC) | 0xAA = 0xEA
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Eight packed codes -> four bf16x2 registers holding 128 + q (exact).
__device__ __forceinline__ void codes_to_bf16x2(uint32_t w, uint32_t (&r)[4]) {
  constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;
  r[0] = lop3_and_or(w, kMask, kMagic);
  r[1] = lop3_and_or(w >> 4, kMask, kMagic);
  r[2] = lop3_and_or(w >> 8, kMask, kMagic);
  r[3] = lop3_and_or(w >> 12, kMask, kMagic);
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4],
                                               const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same product into d, starting from zero sums.
__device__ __forceinline__ void mma_bf16_16816_zero(float (&d)[4],
                                                    const uint32_t (&a)[4],
                                                    uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

// Streaming 128-bit load of constant data (not kept in L1).
__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Programmatic dependent launch controls (no-ops without the launch
// attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block cluster helpers.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float *local_addr,
                                              uint32_t rank) {
  uint32_t src = static_cast<uint32_t>(__cvta_generic_to_shared(local_addr));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(src), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
  return v;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

}  // namespace mnb

namespace mnb {

// ---- mbarrier + bulk-copy (TMA, non-tensor) helpers ------------------------

// Iteration cap for every mbarrier wait: far beyond any legitimate wait
// (seconds), but finite, so a copy that never lands ends the kernel with a
// recorded fault instead of a hang.
constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n\t"
               "fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; returns false if the cap was reached.
template <uint32_t kLimit = kWaitLimit>
__device__ __forceinline__ bool mbar_wait_n(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  return mbar_wait_n<kWaitLimit>(bar, parity);
}

// 1-D bulk copy global -> this CTA's shared memory, completing on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src,
                                              uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled TMA load into this CTA's shared memory, completing on bar.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int x,
                                            int y, int z, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z),
      "r"(smem_addr(bar))
      : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory, completing on bar.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x,
                                            int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// Barrier among `count` threads (a multiple of 32) on hardware barrier `id`.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Each kernel file keeps a device fault word that a kernel sets when one of
// its bounded waits runs out; mnb_fault_status() reads and clears them.
__device__ __forceinline__ void record_fault(unsigned int *word,
                                             unsigned int code) {
  atomicOr(word, code);
}

constexpr unsigned int kFaultGemvWait = 1u;
constexpr unsigned int kFaultGemmWait = 2u;
constexpr unsigned int kFaultChainWait = 4u;

}  // namespace mnb
