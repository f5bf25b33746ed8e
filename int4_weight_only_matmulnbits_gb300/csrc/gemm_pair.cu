// Persistent CTA-pair tensor-core MatMulNBits kernel for prefill rows.
//
// The same product as the tile-per-CTA kernel in gemm.cu, Y[m,n] = sum_k
// A[m,k] (q[n,k] - z[n,b]) s[n,b] + bias[n] with bf16 activations on the
// prepacked layout (page "Qwen3 CPU Inference Critical Path", section
// "Prepared weight-only plan", int4_gemm: activation panels staged per tile,
// weight blocks reused across the rows of a tile, the weight matrix never
// expanded beyond one dequantised slice per pipeline stage), scheduled for
// GB300 as follows:
//  * A cluster of two CTAs on two SMs (a CTA pair) owns a 256-row x (32 NT)-
//    column output tile, NT = 4..8 sixteen-row weight tiles per CTA. CTA r
//    of the pair stages rows 128 r .. 128 r + 127 of the tile's A and
//    dequantises weight rows 16 NT r .. 16 NT r + 16 NT - 1 of its columns;
//    one thread of CTA 0 issues tcgen05.mma.cta_group::2 (M = 256, N = 32 NT,
//    K = 16), which reads both CTAs' operands and leaves rows 128 r .. of the
//    product in CTA r's tensor memory. Each SM so holds half the A rows and
//    half the weight columns of a tile twice as large as one CTA could feed.
//  * The pairs are persistent: pair i takes tiles i, i + P, i + 2P, ... (P
//    pairs, tiles ordered M fastest so that concurrent pairs share weight
//    columns in L2), with two TMEM accumulators (2 x 256 columns): the MMAs
//    of the next tile run while the epilogue warps drain the last one.
//  * Warp roles (24 warps per CTA): 0 A loads (TMA, 128-byte swizzle), 1
//    packed-weight loads (codes, scales, zero points), 2 the tensor memory
//    and, in CTA 0, the MMAs, 3 in CTA 1 the relay of its A stages, 4-7 the
//    epilogue (one TMEM lane quarter each), 8 .. 23 the dequantisation in
//    16 / NT groups of NT warps, one 16-row weight tile per warp, group i
//    taking the stages i, i + groups, ... (a warp's hand-off latency then
//    spreads over several stages), into B slots of hi and lo bf16 tiles
//    (each weight w = hi + lo exactly for bf16 scales, within 2^-16 |w| for
//    fp32 scales; the two tiles go through two MMAs into one accumulator).
//    The ring depths (A 4 to 9 stages, B and weights a multiple of the
//    group count) are planned per launch by pair_rings.
//  * Hand-offs across the pair go through CTA 0's mbarriers: both CTAs'
//    dequantisation warps arrive on CTA 0's bfull, CTA 1's A relay (warp 3)
//    on CTA 0's apeer once CTA 1's A stage has landed; the MMA completions
//    are committed to both CTAs' barriers at once (multicast commit).
// Every mbarrier wait is bounded; a wait that runs out records a fault bit,
// the CTA gives up its remaining tiles, waits (bounded) for its copies in
// flight and for the MMAs already issued, and exits through the same
// cluster barrier and TMEM release as a normal run.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "mnb_common.cuh"
#include "mnb_launch.h"
#include "umma.cuh"

namespace mnb {

__device__ unsigned int g_fault_pair = 0;

namespace {

constexpr int kPairThreads = 768;
constexpr int kWarpA = 0, kWarpW = 1, kWarpMma = 2, kWarpRelay = 3, kWarpEpi = 4, kWarpDq = 8;
constexpr int kDqWarps = 16;
constexpr int kMaxNT = 8;
constexpr int kCtaRows = 128;              // A rows per CTA (the pair tile has 256)
constexpr int kStageK = 64;                // one chunk of the packed layout
constexpr int kAccCols = 256;              // TMEM columns per accumulator
constexpr int kTmemCols = 2 * kAccCols;    // two accumulators
constexpr int kABytes = kCtaRows * kStageK * 2;      // 16 KB
constexpr int kMaxAStages = 10, kMaxBStages = 8, kMaxWStages = 8;
constexpr int kSmemBudget = 227 * 1024 - 1024;        // less the 1024-byte alignment slack

struct PairParams {
  CUtensorMap tma;            // A: {K, M} bf16, box {64, 128}, 128-byte swizzle
  CUtensorMap tmw, tms, tmz;  // codes, scales, zero points: boxes of nt tiles
  const float *bias;
  void *Y;
  int M, N, K64;
  int nt;                     // weight tiles per CTA (4..8): tile columns 32 nt
  int tiles_m, tiles;         // pair tiles: tiles_m along M (fastest), then N
  int w_bytes;                // bytes of one weight stage (codes + scales + zero points)
  int sc_off, zp_off;         // offsets of the scales and zero points in a weight stage
  int y_vec;                  // Y rows 16-byte aligned: 16-byte stores
  // Ring plan (host-computed, see pair_rings): depths, the dequantisation
  // groups, B slot and weight stage sizes, shared-memory offsets.
  int a_stages, b_stages, w_stages, groups;
  int b_slot, b_lo, w_stage;  // B slot bytes (hi tile, lo tile at b_lo), weight stage bytes
  int off_b, off_w, off_bar;
};

// Shared memory (offsets from a 1024-aligned base, the same in both CTAs of
// a pair, as the MMAs address the peer's operands at the issuing CTA's
// offsets): the A ring from 0, the B slots from off_b, the weight ring from
// off_w, the barriers from off_bar: afull, apeer, aempty (A ring); wfull,
// wempty (weights); bfull, bempty (B slots); acc_full[2],
// acc_empty[2]; done; then the TMEM address.
constexpr int kBarBytes = 8 * (3 * kMaxAStages + 2 * kMaxWStages + 2 * kMaxBStages + 5) + 16;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of this CTA's shared variable `p` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

// Arrival on a barrier of any CTA of the cluster, with the default
// semantics (release at CTA scope). What it publishes to CTA 0 is either
// shared memory that CTA 0's MMAs read through the async proxy (written,
// then fenced with fence.proxy.async, before the arrival) or the arriving
// CTA's own progress; cluster-scope release, which costs a memory barrier
// of over a thousand cycles per arrival, is not needed for either.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// D (TMEM, both CTAs) += A (both CTAs' 128 rows) x B (both CTAs' halves)^T.
__device__ __forceinline__ void umma_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(static_cast<int>(accumulate))
      : "memory");
}

// Arrival, once the MMAs issued so far have completed, on the barrier at
// `bar`'s offset in each CTA of `mask` (bit r: cluster rank r).
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// One warp's share of a stage's B operand: the 16 weight rows of tile
// `tile` dequantised over the stage's 64 k into the hi and lo bf16 tiles of
// a K-major, 128-byte-swizzled B slot (lo `lo` bytes after hi). Weight rows
// g and g + 8 go to B rows 2g and 2g + 1 (conflict-free stores); the
// epilogue maps the columns back with out_col.
template <int BS, bool HAS_ZP, bool SF32>
__device__ __forceinline__ void dequant_tile(const unsigned char *codes, const unsigned char *sc,
                                             const uint2 *zp, int tile, int blk0,
                                             unsigned char *bslot, int lo, int lane) {
  constexpr int kBpc = BS < kStageK ? kStageK / BS : 1;
  const int g = lane >> 2, t = lane & 3;
  const int r0 = tile * kTileN + 2 * g;
  const uint4 w4 = *reinterpret_cast<const uint4 *>(codes + tile * kChunkBytes + lane * 16);
  const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // Scales and zero points of weight rows g and g + 8 for the block of
    // this 16-wide k step.
    const int bi = BS < kStageK ? (16 * j) / BS : 0;
    uint32_t sb0 = 0, sb1 = 0;
    float sf0 = 0.f, sf1 = 0.f;
    if (SF32) {
      const float *s4 = reinterpret_cast<const float *>(sc) + (tile * kBpc + bi) * kTileN;
      sf0 = s4[g];
      sf1 = s4[g + 8];
    } else {
      const uint16_t *s2 = reinterpret_cast<const uint16_t *>(sc) + (tile * kBpc + bi) * kTileN;
      sb0 = s2[g] * 0x10001u;
      sb1 = s2[g + 8] * 0x10001u;
    }
    uint32_t zc0 = 0x43084308u, zc1 = 0x43084308u;  // bf16 136 = 128 + 8 (the default)
    if (HAS_ZP) {
      // 16 bytes per tile and pair of blocks: word (b & 1) of slot b / 2.
      const int b = blk0 + bi;
      const int pairs = BS < 32 ? 2 : 1;
      const uint2 zw = zp[(tile * pairs + (BS < 32 ? bi >> 1 : 0)) * 2 + (b & 1)];
      zc0 = (0x4300u | ((zw.x >> (4 * g)) & 15)) * 0x10001u;
      zc1 = (0x4300u | ((zw.y >> (4 * g)) & 15)) * 0x10001u;
    }
    uint32_t r[4];
    codes_to_bf16x2(wv[j], r);
    uint32_t h00, l00, h02, l02, h10, l10, h12, l12;
    dequant_pair<SF32>(r[0], zc0, sb0, sf0, h00, l00);  // row g
    dequant_pair<SF32>(r[2], zc0, sb0, sf0, h02, l02);
    dequant_pair<SF32>(r[1], zc1, sb1, sf1, h10, l10);  // row g + 8
    dequant_pair<SF32>(r[3], zc1, sb1, sf1, h12, l12);
    // 16-byte chunk (k / 8) XOR (row % 8) of the row's 128 bytes.
    const int k0 = 16 * j + 4 * t;
    const int inner = (k0 & 7) * 2;
    const int o0 = r0 * 128 + (((k0 >> 3) ^ (r0 & 7)) * 16) + inner;
    const int o1 = (r0 + 1) * 128 + (((k0 >> 3) ^ ((r0 + 1) & 7)) * 16) + inner;
    *reinterpret_cast<uint2 *>(bslot + o0) = make_uint2(h00, h02);
    *reinterpret_cast<uint2 *>(bslot + o1) = make_uint2(h10, h12);
    *reinterpret_cast<uint2 *>(bslot + lo + o0) = make_uint2(l00, l02);
    *reinterpret_cast<uint2 *>(bslot + lo + o1) = make_uint2(l10, l12);
  }
}

template <int BS, bool HAS_ZP, bool SF32>
__global__ void __launch_bounds__(kPairThreads, 1)
    gemm_pair_kernel(const __grid_constant__ PairParams p) {
  const int AS = p.a_stages, BST = p.b_stages, WS = p.w_stages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *afull = reinterpret_cast<uint64_t *>(smem + p.off_bar);
  uint64_t *apeer = afull + AS;
  uint64_t *aempty = apeer + AS;
  uint64_t *wfull = aempty + AS;
  uint64_t *wempty = wfull + WS;
  uint64_t *bfull = wempty + WS;
  uint64_t *bempty = bfull + BST;
  uint64_t *acc_full = bempty + BST;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *done = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
  const int nt = p.nt, cols = 2 * kTileN * nt;

  if (tid == 0) {
    for (int i = 0; i < AS; ++i) {
      mbar_init(afull + i, 1);
      mbar_init(apeer + i, 1);
      mbar_init(aempty + i, 1);
    }
    for (int i = 0; i < WS; ++i) {
      mbar_init(wfull + i, 1);
      mbar_init(wempty + i, nt);
    }
    for (int i = 0; i < BST; ++i) {
      mbar_init(bfull + i, 2 * nt);  // both CTAs' dequantisation warps
      mbar_init(bempty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, 8);  // both CTAs' four epilogue warps
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Dependents may launch once every CTA has started; A is the upstream
  // kernel's output.
  grid_dependents_launch();
  grid_dependency_wait();

  bool fault = false;
  if (warp == kWarpA) {
    if (lane == 0) {
      int it = 0;
      for (int t = pair; t < p.tiles && !fault; t += npairs) {
        const int m0 = (t % p.tiles_m) * (2 * kCtaRows) + static_cast<int>(rank) * kCtaRows;
        for (int kb = 0; kb < p.K64; ++kb, ++it) {
          const int s = it % AS;
          if (it >= AS && !mbar_wait(aempty + s, ((it / AS) - 1) & 1)) {
            fault = true;
            break;
          }
          mbar_arrive_expect_tx(afull + s, kABytes);
          tma_load_2d(smem + s * kABytes, &p.tma, kb * kStageK, m0, afull + s);
        }
      }
      // The last copy into each slot has landed (already true unless a wait
      // above ran out).
      for (int i = it > AS ? it - AS : 0; i < it; ++i) mbar_wait(afull + i % AS, (i / AS) & 1);
    }
  } else if (warp == kWarpW) {
    if (lane == 0) {
      int it = 0;
      for (int t = pair; t < p.tiles && !fault; t += npairs) {
        const int nt0 = (t / p.tiles_m) * 2 * nt + static_cast<int>(rank) * nt;
        for (int kb = 0; kb < p.K64; ++kb, ++it) {
          const int s = it % WS;
          if (it >= WS && !mbar_wait(wempty + s, ((it / WS) - 1) & 1)) {
            fault = true;
            break;
          }
          uint64_t *bar = wfull + s;
          unsigned char *dst = smem + p.off_w + s * p.w_stage;
          const int blk = (kb * kStageK) / BS;
          mbar_arrive_expect_tx(bar, p.w_bytes);
          tma_load_3d(dst, &p.tmw, 0, kb, nt0, bar);
          tma_load_3d(dst + p.sc_off, &p.tms, 0, blk, nt0, bar);
          if (HAS_ZP) tma_load_3d(dst + p.zp_off, &p.tmz, 0, blk >> 1, nt0, bar);
        }
      }
      for (int i = it > WS ? it - WS : 0; i < it; ++i) mbar_wait(wfull + i % WS, (i / WS) & 1);
    }
  } else if (warp == kWarpMma) {
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) |
                             (static_cast<uint32_t>(cols >> 3) << 17) |
                             (static_cast<uint32_t>((2 * kCtaRows) >> 4) << 24);
      int it = 0, j = 0;
      for (int t = pair; t < p.tiles && !fault; t += npairs, ++j) {
        const int ab = j & 1;
        if (j >= 2 && !mbar_wait(acc_empty + ab, ((j >> 1) - 1) & 1)) {
          fault = true;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + ab * kAccCols;
        for (int kb = 0; kb < p.K64; ++kb, ++it) {
          const int s = it % AS, b = it % BST;
          if (!mbar_wait(afull + s, (it / AS) & 1) ||
              !mbar_wait(apeer + s, (it / AS) & 1) ||
              !mbar_wait(bfull + b, (it / BST) & 1)) {
            fault = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(smem + s * kABytes);
          const uint32_t b_base = smem_addr(smem + p.off_b + b * p.b_slot);
#pragma unroll
          for (int kk = 0; kk < kStageK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_base + kk * 32);
            umma_pair(d, ad, smem_desc_sw128(b_base + kk * 32), idesc, kb > 0 || kk > 0);
            umma_pair(d, ad, smem_desc_sw128(b_base + p.b_lo + kk * 32), idesc, true);
          }
          umma_commit_pair(aempty + s, 3);
          umma_commit_pair(bempty + b, 3);
        }
        if (fault) break;
        umma_commit_pair(acc_full + ab, 3);
      }
      // Every MMA issued has completed before the tensor memory is released.
      umma_commit_pair(done, 1);
      if (!mbar_wait(done, 0)) fault = true;
    }
  } else if (warp == kWarpRelay) {
    if (rank == 1 && lane == 0) {
      const uint32_t peer_apeer = cluster_addr(apeer, 0);
      int it = 0;
      for (int t = pair; t < p.tiles && !fault; t += npairs)
        for (int kb = 0; kb < p.K64; ++kb, ++it) {
          const int s = it % AS;
          if (!mbar_wait(afull + s, (it / AS) & 1)) {
            fault = true;
            break;
          }
          mbar_arrive_cluster(peer_apeer + 8 * s);
        }
    }
  } else if (warp >= kWarpEpi && warp < kWarpDq) {
    // ---- epilogue: TMEM -> registers -> Y ----------------------------------
    const int q = warp & 3;  // TMEM lanes 32 q .. 32 q + 31
    const uint32_t peer_acc_empty = cluster_addr(acc_empty, 0);
    int j = 0;
    for (int t = pair; t < p.tiles; t += npairs, ++j) {
      const int ab = j & 1;
      const bool ok = mbar_wait(acc_full + ab, (j >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        fault = true;
        break;
      }
      tc_fence_after();
      const int m = (t % p.tiles_m) * (2 * kCtaRows) + static_cast<int>(rank) * kCtaRows +
                    q * 32 + lane;
      const int n_base = (t / p.tiles_m) * cols;
      uint16_t *yrow = static_cast<uint16_t *>(p.Y) + static_cast<int64_t>(m) * p.N;
#pragma unroll 1
      for (int c = 0; c < cols / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + ab * kAccCols + c * 32, v);
        if (m < p.M) {
        // Accumulator columns 32 c .. 32 c + 31: two 16-column groups, each
        // permuted within itself; CTA 0's weight rows first, then CTA 1's, so
        // the group's output columns start at n_base + its first column.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n0 = n_base + c * 32 + h * 16;
          float o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = n0 + out_col(i);
            o[out_col(i)] = v[16 * h + i] + ((p.bias && n < p.N) ? __ldg(p.bias + n) : 0.f);
          }
          if (p.y_vec && n0 + 16 <= p.N) {
#pragma unroll
            for (int i = 0; i < 16; i += 8) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = bf16_bits(o[i + 2 * e]) | (bf16_bits(o[i + 2 * e + 1]) << 16);
              *reinterpret_cast<uint4 *>(yrow + n0 + i) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            for (int i = 0; i < 16; ++i)
              if (n0 + i < p.N) yrow[n0 + i] = static_cast<uint16_t>(bf16_bits(o[i]));
          }
        }
        }
      }
      // The accumulator may be overwritten once both CTAs have read theirs.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(peer_acc_empty + 8 * ab);
    }
  } else if (warp < kWarpDq + p.groups * nt) {
    // ---- dequantisation ----------------------------------------------------
    const int groups = p.groups;
    const int tile = (warp - kWarpDq) % nt, grp = (warp - kWarpDq) / nt;
    const uint32_t peer_bfull = cluster_addr(bfull, 0);
    int it = 0;
    for (int t = pair; t < p.tiles && !fault; t += npairs)
      for (int kb = 0; kb < p.K64; ++kb, ++it) {
        if (it % groups != grp) continue;
        const int s = it % WS, b = it % BST;
        const bool ok = mbar_wait(wfull + s, (it / WS) & 1) &&
                        (it < BST || mbar_wait(bempty + b, ((it / BST) - 1) & 1));
        if (!__all_sync(0xffffffffu, ok)) {
          fault = true;
          break;
        }
        const unsigned char *w = smem + p.off_w + s * p.w_stage;
        dequant_tile<BS, HAS_ZP, SF32>(w, w + p.sc_off, reinterpret_cast<const uint2 *>(w + p.zp_off),
                                       tile, (kb * kStageK) / BS, smem + p.off_b + b * p.b_slot,
                                       p.b_lo, lane);
        fence_async_smem();  // the tile, to the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(peer_bfull + 8 * b);
          mbar_arrive(wempty + s);
        }
      }
  }

  if (fault) record_fault(&g_fault_pair, kFaultGemmWait);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA releases the tensor memory while the pair uses it
  if (warp == kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// The ring plan for nt weight tiles per CTA. The dequantisation warps form
// groups = 16 / nt groups; group g takes the stages g, g + groups, ..., so
// the B and weight rings hold a multiple of `groups` slots and each group
// always returns to its own slots: no warp then waits on a barrier more
// than one phase ahead of it (the parity of a wait two phases ahead would
// name a phase already completed). The A ring takes the rest of the shared
// memory, four to ten stages.
PairParams pair_rings(PairParams p, int bs, bool sf32, bool zp) {
  const int nt = p.nt;
  const int bpc = bs < kStageK ? kStageK / bs : 1;
  const int ppc = bs < 32 ? 2 : 1;
  p.groups = kDqWarps / nt;
  const int code_bytes = nt * kChunkBytes;
  const int sc_bytes = nt * bpc * kTileN * (sf32 ? 4 : 2);
  const int zp_bytes = zp ? nt * ppc * 16 : 0;
  p.sc_off = code_bytes;  // a multiple of 512
  p.zp_off = code_bytes + (sc_bytes + 127) / 128 * 128;
  p.w_bytes = code_bytes + sc_bytes + zp_bytes;
  p.w_stage = p.zp_off + 256;  // room for the largest zero-point box
  p.b_lo = nt * kTileN * 128;  // a multiple of 1024
  p.b_slot = 2 * p.b_lo;
  p.w_stages = p.groups * ((4 + p.groups - 1) / p.groups);
  p.b_stages = p.groups * ((3 + p.groups - 1) / p.groups);
  for (;;) {
    const int room = kSmemBudget - kBarBytes - p.b_stages * p.b_slot - p.w_stages * p.w_stage;
    p.a_stages = std::min(kMaxAStages, room / kABytes);
    if (p.a_stages >= 4 || p.b_stages <= p.groups) break;
    p.b_stages -= p.groups;
  }
  p.off_b = p.a_stages * kABytes;
  p.off_w = p.off_b + p.b_stages * p.b_slot;
  p.off_bar = p.off_w + p.w_stages * p.w_stage;
  return p;
}

int pair_smem_bytes(const PairParams &p) { return p.off_bar + kBarBytes + 1024; }

template <int BS, bool HAS_ZP, bool SF32>
cudaError_t pair_launch_one(const PairParams &p, int pairs, bool pdl, cudaStream_t stream) {
  auto kernel = gemm_pair_kernel<BS, HAS_ZP, SF32>;
  const int smem = pair_smem_bytes(p);
  static std::atomic<unsigned long long> configured{0};
  if (const cudaError_t e = ensure_smem_limit(kernel, kSmemBudget + 1024, configured);
      e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = 2;
  attrs[na].val.clusterDim.y = 1;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int BS>
cudaError_t pair_launch_flags(const PairParams &p, int pairs, bool zp, bool sf32, bool pdl,
                              cudaStream_t stream) {
  if (zp)
    return sf32 ? pair_launch_one<BS, true, true>(p, pairs, pdl, stream)
                : pair_launch_one<BS, true, false>(p, pairs, pdl, stream);
  return sf32 ? pair_launch_one<BS, false, true>(p, pairs, pdl, stream)
              : pair_launch_one<BS, false, false>(p, pairs, pdl, stream);
}

// CTA pairs resident at once on the current device (one CTA per SM), from
// the occupancy of the launch configuration; looked up once per device.
int resident_pairs() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  }
  auto kernel = gemm_pair_kernel<128, false, false>;
  const int smem = kSmemBudget + 1024;  // the largest plan
  static std::atomic<unsigned long long> configured{0};
  if (ensure_smem_limit(kernel, smem, configured) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

}  // namespace

cudaError_t pair_take_fault(unsigned int *out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fault_pair, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fault_pair, &zero, sizeof(unsigned int));
  return e;
}

bool pair_supports(const MatmulArgs &a) {
  return gemm_supports(a) && !a.a_f32 && !a.paired && !a.norm && !a.code;
}

PairPlan plan_pair(const MatmulArgs &a, int pairs) {
  // Columns per tile 32 nt: the fewest rounds of tiles over the pairs, each
  // round costing in proportion to nt (the MMA work per k stage), plus a
  // small fixed cost per k stage that favours wider tiles at equal work.
  PairPlan r;
  if (pairs <= 0) return r;
  const int64_t tiles_m = ceil_div(a.M, int64_t(2 * kCtaRows));
  double best = 0.0;
  for (int nt = kMaxNT; nt >= 4; --nt) {
    const int64_t tiles = tiles_m * ceil_div(a.N, int64_t(2 * kTileN * nt));
    const int64_t rounds = ceil_div(tiles, int64_t(pairs));
    const double cost = double(rounds) * (double(nt) + 0.5);
    if (r.nt == 0 || cost < best - 1e-9) {
      best = cost;
      r.nt = nt;
      r.tiles = tiles;
      r.pairs = static_cast<int>(std::min<int64_t>(tiles, pairs));
    }
  }
  return r;
}

int pair_slots() { return resident_pairs(); }

cudaError_t launch_gemm_pair(const MatmulArgs &a, cudaStream_t stream) {
  if (!pair_supports(a)) return cudaErrorNotSupported;
  const int slots = resident_pairs();
  if (slots <= 0) return cudaErrorNotSupported;
  const PairPlan plan = plan_pair(a, slots);
  if (plan.nt == 0) return cudaErrorNotSupported;
  const int nt = plan.nt;
  PairParams p{};
  const uint64_t N16 = ceil_div(a.N, kTileN), K64 = ceil_div(a.K, kStageK);
  const uint64_t nb = ceil_div(a.K, a.bs), nbz = ceil_div(nb, 2) * 2;
  const uint64_t es = a.scale_f32 ? 4 : 2;
  const uint32_t bpc = a.bs < kStageK ? kStageK / a.bs : 1;
  const uint32_t ppc = a.bs < 32 ? 2 : 1;
  cudaError_t e;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.K) * 2};
    const uint32_t box[2] = {kStageK, kCtaRows};
    e = make_tmap(&p.tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.A, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  {
    const uint64_t dims[3] = {kChunkBytes / 4, K64, N16};
    const uint64_t strides[2] = {kChunkBytes, K64 * kChunkBytes};
    const uint32_t box[3] = {kChunkBytes / 4, 1, static_cast<uint32_t>(nt)};
    e = make_tmap(&p.tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.packed_b, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  {
    const uint64_t words = kTileN * es / 4;
    const uint64_t dims[3] = {words, nb, N16};
    const uint64_t strides[2] = {kTileN * es, nb * kTileN * es};
    const uint32_t box[3] = {static_cast<uint32_t>(words), bpc, static_cast<uint32_t>(nt)};
    e = make_tmap(&p.tms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.scales, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  if (a.zp) {
    const uint64_t dims[3] = {4, nbz / 2, N16};
    const uint64_t strides[2] = {16, nbz * 8};
    const uint32_t box[3] = {4, ppc, static_cast<uint32_t>(nt)};
    e = make_tmap(&p.tmz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.zp, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  p.bias = a.bias;
  p.Y = a.Y;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K64 = static_cast<int>(K64);
  p.nt = nt;
  p.tiles_m = static_cast<int>(ceil_div(a.M, int64_t(2 * kCtaRows)));
  p.tiles = static_cast<int>(plan.tiles);
  p.y_vec = (a.N % 8) == 0 && (reinterpret_cast<uintptr_t>(a.Y) % 16) == 0;
  p = pair_rings(p, a.bs, a.scale_f32, a.zp != nullptr);
  if (p.a_stages < 4 || p.b_stages > kMaxBStages || p.w_stages > kMaxWStages ||
      pair_smem_bytes(p) > kSmemBudget + 1024)
    return cudaErrorNotSupported;
  switch (a.bs) {
    case 16: return pair_launch_flags<16>(p, plan.pairs, a.zp, a.scale_f32, a.pdl, stream);
    case 32: return pair_launch_flags<32>(p, plan.pairs, a.zp, a.scale_f32, a.pdl, stream);
    case 64: return pair_launch_flags<64>(p, plan.pairs, a.zp, a.scale_f32, a.pdl, stream);
    case 128: return pair_launch_flags<128>(p, plan.pairs, a.zp, a.scale_f32, a.pdl, stream);
    case 256: return pair_launch_flags<256>(p, plan.pairs, a.zp, a.scale_f32, a.pdl, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace mnb
