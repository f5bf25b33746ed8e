// Small-M (decode) MatMulNBits kernel for sm_103a.
//
// Computes Y[m,n] = sum_k A[m,k] (q[n,k] - z[n,b]) s[n,b] + bias[n] for
// M <= 16 on the prepacked layout of mnb_common.cuh, for one weight or for a
// group of weights that share the same activations (fused-N projections such
// as q/k/v or gate/up). It follows the page "Qwen3 CPU Inference Critical
// Path", section "Prepared weight-only plan": weights stay compressed, are
// unpacked in registers, zero points and scales are applied per block and
// accumulation is fp32; int4_gemv streams every weight byte once,
// partitioned over output channels, and int4_small_m reuses the unpacked
// codes across a few activation rows.
//
// GB300 mapping:
//  * Warp-specialised, persistent CTAs: 16 consumer warps and one producer
//    warp. Output rows form 16-row tiles; a CTA works on a tile group of
//    `tpc` tiles, each consumer warp owning one tile and one of `ksw`
//    interleaved k slices: in stage j it takes `cpw` consecutive chunks,
//    starting at chunk (j*ksw + ks)*cpw of the CTA's k range (a cluster of
//    CTAs splits K further). CTAs walk the tile groups with a fixed stride.
//  * Per pipeline stage the producer moves the next ksw*cpw chunks of all
//    tpc tiles with one 3-D TMA tensor copy (8 KB per chunk per warp), plus
//    one copy each for their scales and zero points, into a ring of
//    shared-memory stages guarded by full/empty mbarriers. Several chunks
//    per warp and stage spread the ring bookkeeping over more weights. TMA
//    zero fill covers ragged N, K and blocks.
//    The weights are constant, so the producer starts before the upstream
//    kernel has finished, and the kernel lets its own dependents launch at
//    once: consecutive launches overlap their weight streams.
//  * Activations are staged once per CTA in shared memory as bf16 (fp32
//    activations as a pair hi + lo exact to 2^-16). Codes become bf16
//    128 + q (exact) with one lop3 per pair; they feed mma.m16n8k16 as the
//    16-row operand, the activations (8 rows per MMA) as the 8-column
//    operand: no per-weight zero-point or scale arithmetic.
//  * Per block (or block piece) the fp32 correction
//      acc += s * (D - (128 + z) * S),   S = sum of the block's staged
//    activations, applies zero point and scale.
//  * Split-K partials are reduced in fixed order: consumer warps of a CTA
//    through shared memory, CTAs of a cluster through distributed shared
//    memory; a warp that owns all of K stores its tile directly. No global
//    workspace, no atomics on results: outputs are bitwise reproducible.
//  * Gated-MLP pairs (page "Qwen3 CPU Inference Critical Path", the
//    graph-level fusion "gate projection, SiLU, and gate/up multiplication"):
//    a tile group holds tpc/2 tiles of the gate weight and the same rows of
//    the up weight, and the epilogue stores silu(gate) * up, with
//    silu(x) = x * sigmoid(x) in fp32.
#include <cuda_bf16.h>

#include <algorithm>

#include "mnb_common.cuh"
#include "mnb_launch.h"

namespace mnb {

__device__ unsigned int g_fault_gemv = 0;

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kBarConsumers = 1;           // named barrier id for consumers
// Shared memory per CTA small enough that a CTA of the next launch fits
// beside a running one on the same SM.
constexpr int kSmemBudget = 112 * 1024;
constexpr int kSmemMax = 227 * 1024;  // one CTA per SM
constexpr int kMaxStages = 8;
constexpr int kStageBatch = 4;  // activation pieces a thread loads before converting
constexpr int kPrefetchStages = 1;  // weight stages issued before the upstream kernel ends

struct GemvParams {
  CUtensorMap tmw[kMaxGroup];  // codes: {128 words, K64 chunks, N16 tiles}
  CUtensorMap tms[kMaxGroup];  // scales: {16 scales as words, nb, N16}
  CUtensorMap tmz[kMaxGroup];  // zero points: {4 words, nbz/2 pairs, N16}
  const void *A;
  const float *bias[kMaxGroup];
  void *Y[kMaxGroup];
  int N[kMaxGroup], N16[kMaxGroup], tg_begin[kMaxGroup];
  int nprob, tg_total;
  int M, K, K64, nb;
  int a_f32, a_vec;
  int a_bulk;  // bf16 rows TMA can copy (16-byte aligned, K % 8 == 0)
  int paired;  // gate (weight 0) and up (weight 1) tiles share each tile group
  int sc_up, zp_up;  // paired: offsets of the up halves of a stage's scales / zero points
  int ksw, tpc, cluster, R;  // k slices per CTA, tiles per group, stages per tile group
  int cpw, scs;              // chunks per warp and stage; chunks per stage and tile (ksw*cpw)
  int krp, sg;               // staged activation row stride, block sums per row
  int nst, stage_bytes, stage_tx;  // ring depth, stage stride, bytes per stage
  // Failure-detection test (mnb_test_wait_fault; the PROBE instantiation
  // only): the stage at which CTA 0's producer stops issuing.
  int stop_stage;
  // RMS-normalized activations (the fusion "RMSNorm into packed projection
  // input"): the staged row is A * gamma and every output is scaled by
  // r[m] = 1 / sqrt(mean_k A[m,k]^2 + eps). norm = 0: plain A.
  int norm;
  const float *gamma;  // [K] or null (1)
  float eps;
  // Greedy ArgMax over the outputs of weight 0 (the fusion "final RMSNorm,
  // LM-head GEMV, and greedy ArgMax"): keys [M], or null. Y[0] may then be
  // null (logits not stored).
  unsigned long long *amax;
  // Code-book weights (the bitsandbytes-style format): the 16 fp32 values,
  // or null for the affine codes. Each CTA turns them into a 256-entry table
  // indexed by two codes: the bf16 pair (code[lo], code[hi]) rounded, and the
  // pair of their remainders, so that each value is hi + lo.
  const float *code;
  int st_sc, st_zp;  // offsets of scales and zero points in a stage (128-aligned)
  int nbs, nps;      // blocks and zero-point word pairs per stage and tile
  int off_alo, off_s, off_red, off_part, off_bar, off_ring;
  int off_nrm;  // r[m] and the ArgMax keys (norm or amax)
  int off_lut;  // the code-book pair table (code)
};

// Four bf16x2 registers of eight codes through the pair table: register i
// takes the codes at bits 4i and 16 + 4i, as codes_to_bf16x2 does; r holds
// the rounded code-book values, rl their remainders.
__device__ __forceinline__ void codes_to_lut(uint32_t w, const uint2 *pair, uint32_t (&r)[4],
                                             uint32_t (&rl)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = w >> (4 * i);
    const uint2 e = pair[(x & 0xFu) | ((x >> 12) & 0xF0u)];
    r[i] = e.x;
    rl[i] = e.y;
  }
}

// ArgMax key of output (v, n): larger keys for larger v (an order-preserving
// map of the fp32 bits) and, among equal v, for smaller n.
__device__ __forceinline__ unsigned long long argmax_key(float v, int n) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(n));
}

template <int BS>
struct BlockGeom {
  static constexpr int kLog2 = BS == 16 ? 4 : BS == 32 ? 5 : BS == 64 ? 6 : BS == 128 ? 7 : 8;
};

// Problem of global tile group gi (the group table is tiny: linear scan).
__device__ __forceinline__ int problem_of(const GemvParams &p, int gi) {
  int q = 0;
#pragma unroll
  for (int i = 1; i < kMaxGroup; ++i)
    if (i < p.nprob && gi >= p.tg_begin[i]) q = i;
  return q;
}

// Eight activations A[m][k..k+7] as fp32 (zeros past K).
__device__ __forceinline__ void load8(const GemvParams &p, int m, int64_t k,
                                      float (&v)[8]) {
  if (p.a_f32) {
    const float *a = static_cast<const float *>(p.A) + (int64_t)m * p.K;
    if (p.a_vec && k + 8 <= p.K) {
      const float4 x = *reinterpret_cast<const float4 *>(a + k);
      const float4 y = *reinterpret_cast<const float4 *>(a + k + 4);
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
      v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = (k + q < p.K) ? a[k + q] : 0.f;
    }
  } else {
    const uint16_t *a = static_cast<const uint16_t *>(p.A) + (int64_t)m * p.K;
    if (p.a_vec && k + 8 <= p.K) {
      const uint4 x = *reinterpret_cast<const uint4 *>(a + k);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[2 * q] = bf16_bits_to_f32(w[q] & 0xFFFFu);
        v[2 * q + 1] = bf16_bits_to_f32(w[q] >> 16);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = (k + q < p.K) ? bf16_bits_to_f32(a[k + q]) : 0.f;
    }
  }
}

// Y[m][n] = r[m] v + bias[n], in A's dtype (bf16 rounded to nearest even);
// with the ArgMax epilogue the fp32 value also competes for the row's key
// (sNrm: r[m] in the first 16 floats, then the rows' best keys as 64-bit
// words).
__device__ __forceinline__ void store_y(const GemvParams &p, int q, int m, int n, float v,
                                        float *sNrm) {
  if (p.norm) v *= sNrm[m];
  if (p.bias[q]) v += __ldg(p.bias[q] + n);
  if (p.amax && q == 0) {
    // Only a value above the CTA's current best pays for the atomic.
    unsigned long long *best = reinterpret_cast<unsigned long long *>(sNrm + kGemvMaxM) + m;
    const unsigned long long key = argmax_key(v, n);
    if (key > *reinterpret_cast<volatile unsigned long long *>(best)) atomicMax(best, key);
  }
  if (!p.Y[q]) return;
  if (p.a_f32)
    static_cast<float *>(p.Y[q])[(int64_t)m * p.N[q] + n] = v;
  else
    static_cast<uint16_t *>(p.Y[q])[(int64_t)m * p.N[q] + n] =
        static_cast<uint16_t>(bf16_bits(v));
}

// Gated-MLP output: with g = gate + bias_g and u = up + bias_u,
// Y[m][n] = g * sigmoid(g) * u, in fp32, stored in A's dtype.
__device__ __forceinline__ void store_gate_up(const GemvParams &p, int m, int n, float g,
                                              float u, const float *sNrm) {
  if (p.norm) {
    g *= sNrm[m];
    u *= sNrm[m];
  }
  if (p.bias[0]) g += __ldg(p.bias[0] + n);
  if (p.bias[1]) u += __ldg(p.bias[1] + n);
  const float v = g / (1.f + expf(-g)) * u;
  if (p.a_f32)
    static_cast<float *>(p.Y[0])[(int64_t)m * p.N[0] + n] = v;
  else
    static_cast<uint16_t *>(p.Y[0])[(int64_t)m * p.N[0] + n] =
        static_cast<uint16_t>(bf16_bits(v));
}

// PROBE: the failure-detection test's instantiation (a short wait cap and a
// producer that stops); every other launch compiles without it.
template <int MT, int BS, bool HAS_ZP, bool SF32, bool CODE, bool PROBE = false>
__global__ void __launch_bounds__(kThreads, MT == 1 ? 2 : 1)
    gemv_kernel(const __grid_constant__ GemvParams p) {
  constexpr uint32_t kLimit = PROBE ? (1u << 16) : kWaitLimit;
  using G = BlockGeom<BS>;
  constexpr int kEs = SF32 ? 4 : 2;
  extern __shared__ __align__(128) unsigned char smem[];
  uint16_t *sA = reinterpret_cast<uint16_t *>(smem);
  uint16_t *sAlo = reinterpret_cast<uint16_t *>(smem + p.off_alo);
  float *sS = reinterpret_cast<float *>(smem + p.off_s);
  float *sRed = reinterpret_cast<float *>(smem + p.off_red);
  float *sPart = reinterpret_cast<float *>(smem + p.off_part);
  float *sNrm = reinterpret_cast<float *>(smem + p.off_nrm);
  uint2 *sPair = reinterpret_cast<uint2 *>(smem + p.off_lut);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
  uint64_t *empty = full + kMaxStages;
  uint64_t *abar = empty + kMaxStages;  // activation copy
  unsigned char *ring = smem + p.off_ring;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int crank = static_cast<int>(blockIdx.x) % p.cluster;
  const int gstride = static_cast<int>(gridDim.x) / p.cluster;
  const int gfirst = static_cast<int>(blockIdx.x) / p.cluster;
  const int clo = crank * p.scs * p.R;  // first chunk of this CTA's k range

  if (tid == 0) {
    for (int i = 0; i < p.nst; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsumerWarps);
    }
    mbar_init(abar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Dependents may launch now: before waiting on this grid they only touch
  // their own constant weights.
  grid_dependents_launch();

  if (warp == kConsumerWarps) {
    // ---- producer: one stage per chunk step of the tile group ----------------
    // The whole warp runs the loop (converged, as cluster barriers need);
    // lane 0 issues. In cluster mode the producer joins the two cluster
    // barriers of each tile group right after issuing its last stage, and
    // only then prefetches the next group, so it never waits on a slot that
    // only a later group would free.
    // Only the first kPrefetchStages stages go out before the upstream
    // kernel has finished; the activation copy follows them, so it does
    // not queue behind the whole weight stream, then the rest.
    // Ring position: slot, its use count parity, and whether it was used.
    int slot = 0;
    uint32_t phase = 0;
    bool wrapped = false;
    bool ok = true;
    int issued = 0;
    bool a_issued = false;
    auto issue_a = [&] {
      grid_dependency_wait();
      if (p.a_bulk && lane == 0) {
        const int64_t k0 = int64_t(clo) * kChunkK;
        const int kr = p.scs * p.R * kChunkK;
        const int n = p.K - k0 < kr ? static_cast<int>(p.K - k0) : kr;
        mbar_arrive_expect_tx(abar, static_cast<uint32_t>(p.M) * n * 2);
        for (int m = 0; m < p.M; ++m)
          bulk_copy_g2s(sA + m * p.krp,
                        static_cast<const uint16_t *>(p.A) + int64_t(m) * p.K + k0,
                        static_cast<uint32_t>(n) * 2, abar);
      }
      __syncwarp();
      a_issued = true;
    };
    for (int u = 0;; ++u) {
      const int gi = gfirst + u * gstride;
      if (gi >= p.tg_total) break;
      const int q = problem_of(p, gi);
      const int tile0 = (gi - p.tg_begin[q]) * p.tpc;
      for (int j = 0; j < p.R && ok; ++j) {
        if (!a_issued && issued == kPrefetchStages) issue_a();
        // Test-only stop (launches without a cluster): the stage is never
        // issued, so CTA 0's consumers give up waiting for it; every copy
        // issued before it is consumed first, so none is left in flight.
        if (PROBE && issued == p.stop_stage && blockIdx.x == 0 && p.cluster == 1) {
          ok = false;
          break;
        }
        ++issued;
        if (wrapped && !mbar_wait_n<kLimit>(empty + slot, phase ^ 1)) {
          if (lane == 0) record_fault(&g_fault_gemv, kFaultGemvWait);
          ok = false;
          break;
        }
        if (lane == 0) {
          uint64_t *bar = full + slot;
          unsigned char *st = ring + slot * p.stage_bytes;
          const int c = clo + j * p.scs;  // first chunk of the stage
          const int b = (c * kChunkK) >> G::kLog2;
          mbar_arrive_expect_tx(bar, p.stage_tx);
          if (p.paired) {
            // Gate tiles fill the first half of the stage, up tiles (same rows)
            // the second.
            const int h = p.tpc / 2, t0 = (gi - p.tg_begin[0]) * h;
            tma_load_3d(st, &p.tmw[0], 0, c, t0, bar);
            tma_load_3d(st + h * p.scs * kChunkBytes, &p.tmw[1], 0, c, t0, bar);
            tma_load_3d(st + p.st_sc, &p.tms[0], 0, b, t0, bar);
            tma_load_3d(st + p.st_sc + p.sc_up, &p.tms[1], 0, b, t0, bar);
            if (HAS_ZP) {
              tma_load_3d(st + p.st_zp, &p.tmz[0], 0, b >> 1, t0, bar);
              tma_load_3d(st + p.st_zp + p.zp_up, &p.tmz[1], 0, b >> 1, t0, bar);
            }
          } else {
            tma_load_3d(st, &p.tmw[q], 0, c, tile0, bar);
            tma_load_3d(st + p.st_sc, &p.tms[q], 0, b, tile0, bar);
            if (HAS_ZP) tma_load_3d(st + p.st_zp, &p.tmz[q], 0, b >> 1, tile0, bar);
          }
        }
        __syncwarp();
        if (++slot == p.nst) {
          slot = 0;
          phase ^= 1;
          wrapped = true;
        }
      }
      if (p.cluster > 1) {
        // The consumers reach these barriers only after the activations.
        if (!a_issued) issue_a();
        cluster_sync_all();
        cluster_sync_all();
      }
    }
    if (!a_issued) issue_a();
  } else {
    // ---- consumers ---------------------------------------------------------------
    const int g = lane >> 2, t = lane & 3;
    const int tau = warp / p.ksw, ks = warp - tau * p.ksw;
    // This warp's chunks in stage j are cbase + j*scs + i, i < cpw.
    const int cbase = clo + ks * p.cpw;

    // From here on the upstream kernel's results (A) are visible.
    grid_dependency_wait();

    // Stage A rows [0, M) over the CTA's k range as bf16 (fp32 activations
    // as hi + lo) and the sum of every block of the staged values, so the
    // code offset 128 cancels exactly up to fp32 rounding.
    const int ppr = p.scs * p.R * (kChunkK / 8);  // 8-element pieces per row
    const int npieces = p.M * ppr;
    constexpr int gp = BS / 8;  // pieces per block, consecutive lanes
    bool fault = false;
    if (p.amax && tid < kGemvMaxM)
      reinterpret_cast<unsigned long long *>(sNrm + kGemvMaxM)[tid] = 0ull;
    if (CODE && tid < 256) {
      // Each code-book value c as bf16 hi = round(c) and lo = round(c - hi)
      // (c - hi is exact in fp32): hi + lo is within 2^-16 |c| of c, where
      // hi alone could be 2^-8 |c| off.
      const float c0 = __ldg(p.code + (tid & 15)), c1 = __ldg(p.code + (tid >> 4));
      const uint32_t h0 = bf16_bits(c0), h1 = bf16_bits(c1);
      const uint32_t l0 = bf16_bits(c0 - bf16_bits_to_f32(h0));
      const uint32_t l1 = bf16_bits(c1 - bf16_bits_to_f32(h1));
      sPair[tid] = make_uint2(h0 | (h1 << 16), l0 | (l1 << 16));
    }
    if (p.norm) {
      // r[m] from the whole row (this CTA may stage only part of K): per-warp
      // partial sums of squares, then a fixed-order sum over the warps.
      const int pr = (p.K + 7) / 8;
      for (int m = 0; m < p.M; ++m) {
        float ss = 0.f;
#pragma unroll 2
        for (int pc = tid; pc < pr; pc += kConsumers) {
          float v[8];
          load8(p, m, int64_t(pc) * 8, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) sRed[warp * kGemvMaxM + m] = ss;
      }
      named_barrier_sync(kBarConsumers, kConsumers);
      if (tid < p.M) {
        float ss = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) ss += sRed[w * kGemvMaxM + tid];
        sNrm[tid] = 1.f / sqrtf(ss / static_cast<float>(p.K) + p.eps);
      }
    }
    if (p.a_bulk) {
      // bf16 rows: the producer copies the part inside K with one bulk copy
      // per row; zeros past K.
      const int64_t k0 = int64_t(clo) * kChunkK;
      const int kr = ppr * 8;
      const int n = p.K - k0 < kr ? static_cast<int>(p.K - k0) : kr;
      for (int e = n + tid; e < kr; e += kConsumers)
        for (int m = 0; m < p.M; ++m) sA[m * p.krp + e] = 0;
      if (!mbar_wait_n<kLimit>(abar, 0)) {
        record_fault(&g_fault_gemv, kFaultGemvWait);
        fault = true;
      }
      named_barrier_sync(kBarConsumers, kConsumers);  // zero tails visible
      for (int base = 0; base < npieces; base += kConsumers) {
        const int pc2 = base + tid;
        const bool ok = pc2 < npieces;
        const int m = ok ? pc2 / ppr : 0;
        const int kp = pc2 - m * ppr;
        float part = 0.f;
        if (ok) {
          const uint4 x = *reinterpret_cast<const uint4 *>(sA + m * p.krp + kp * 8);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            part += bf16_bits_to_f32(w[e] & 0xFFFFu) + bf16_bits_to_f32(w[e] >> 16);
        }
#pragma unroll
        for (int o = 1; o < gp; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (ok && (kp % gp) == 0) sS[m * p.sg + kp / gp] = part;
      }
    } else {
      // Each thread first issues the loads of up to kStageBatch pieces,
      // then converts them.
      for (int base = 0; base < npieces; base += kConsumers * kStageBatch) {
        float v[kStageBatch][8];
#pragma unroll
        for (int q = 0; q < kStageBatch; ++q) {
          const int pc2 = base + q * kConsumers + tid;
          if (pc2 < npieces) {
            const int m = pc2 / ppr;
            const int64_t k = (int64_t)clo * kChunkK + (pc2 - m * ppr) * 8;
            load8(p, m, k, v[q]);
            if (p.norm && p.gamma) {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                v[q][e] *= (k + e < p.K) ? __ldg(p.gamma + k + e) : 0.f;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[q][e] = 0.f;
          }
        }
#pragma unroll
        for (int q = 0; q < kStageBatch; ++q) {
          const int pc2 = base + q * kConsumers + tid;
          if (base + q * kConsumers >= npieces) break;  // warp-uniform
          const bool ok = pc2 < npieces;
          const int m = ok ? pc2 / ppr : 0;
          const int kp = pc2 - m * ppr;
          float part = 0.f;
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t h0 = bf16_bits(v[q][2 * e]), h1 = bf16_bits(v[q][2 * e + 1]);
            hi[e] = h0 | (h1 << 16);
            const float f0 = bf16_bits_to_f32(h0), f1 = bf16_bits_to_f32(h1);
            const uint32_t l0 = bf16_bits(v[q][2 * e] - f0), l1 = bf16_bits(v[q][2 * e + 1] - f1);
            lo[e] = l0 | (l1 << 16);
            // The block sums cover exactly what the MMAs see: hi + lo for fp32
            // activations, hi alone otherwise (a normalized bf16 row is
            // rounded to bf16 here).
            part += p.a_f32 ? (f0 + bf16_bits_to_f32(l0)) + (f1 + bf16_bits_to_f32(l1))
                            : f0 + f1;
          }
          if (ok) {
            const int off = m * p.krp + kp * 8;
            *reinterpret_cast<uint4 *>(sA + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            if (p.a_f32)
              *reinterpret_cast<uint4 *>(sAlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
#pragma unroll
          for (int o = 1; o < gp; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
          if (ok && (kp % gp) == 0) sS[m * p.sg + kp / gp] = part;
        }
      }
    }
    named_barrier_sync(kBarConsumers, kConsumers);

    constexpr int MC = MT * 8;
    const int rows = p.tpc * kTileN;
    // Activation fragments this lane reads (rows >= M stay zero) and the
    // block sums its accumulator columns need (rows >= M read row 0 and
    // meet zero activations).
    const bool mok0 = g < p.M, mok1 = 8 + g < p.M;
    const uint16_t *arow0 = sA + (mok0 ? g : 0) * p.krp + 4 * t - clo * kChunkK;
    const uint16_t *arow1 = sA + (mok1 ? 8 + g : 0) * p.krp + 4 * t - clo * kChunkK;
    const int lo_off = static_cast<int>(sAlo - sA);
    const bool two = p.a_f32 != 0;
    const int blo = (clo * kChunkK) >> G::kLog2;  // first block of the CTA's k range
    const float *srow[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = mt * 8 + 2 * t + h;
        srow[mt][h] = sS + (m < p.M ? m : 0) * p.sg - blo;
      }
    const bool direct = p.ksw == 1 && p.cluster == 1 && !p.paired;
    // This warp's slices of a stage: its chunks, and its tile's scales and
    // zero-point pairs (stage block b0s = first block of the stage).
    const int cofs = (tau * p.scs + ks * p.cpw) * kChunkBytes + lane * 16;
    // A pair keeps the up tiles' scales and zero points in 128-byte-aligned
    // halves of their stage regions.
    const int ht = p.tpc / 2;
    const bool up_half = p.paired && tau >= ht;
    const int sofs = p.st_sc + (up_half ? p.sc_up + (tau - ht) * p.nbs * kTileN * kEs
                                        : tau * p.nbs * kTileN * kEs);
    const int zofs = p.st_zp + (up_half ? p.zp_up + (tau - ht) * p.nps * 16 : tau * p.nps * 16);
    uint2 bfrag0 = make_uint2(0, 0), bfrag1 = make_uint2(0, 0);
    int slot = 0;
    uint32_t phase = 0;

    for (int u = 0;; ++u) {
      const int gi = gfirst + u * gstride;
      if (gi >= p.tg_total) break;
      const int q = problem_of(p, gi);
      float acc[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;

      for (int j = 0; j < p.R && !fault; ++j) {
        if (!mbar_wait_n<kLimit>(full + slot, phase)) {
          record_fault(&g_fault_gemv, kFaultGemvWait);
          fault = true;
          break;
        }
        const unsigned char *st = ring + slot * p.stage_bytes;
        const int cst = cbase + j * p.scs;                            // warp's first chunk
        const int b0s = ((cst - ks * p.cpw) * kChunkK) >> G::kLog2;  // stage's first block
        const unsigned char *wp = st + cofs;
        const uint16_t *ap0 = arow0 + cst * kChunkK;
        const uint16_t *ap1 = arow1 + cst * kChunkK;

        // Applies scale and zero point of block b to its MMA sums d.
        // Blocks past the last real one arrive zero-filled: scale 0.
        auto correct = [&](int b, float (&d)[MT][4]) {
          const int bi = b - b0s;
          // Affine codes arrive as 128 + q: remove (128 + z) S. Code-book
          // values are the weights themselves: nothing to remove.
          float s0, s1, z0 = CODE ? 0.f : 136.f, z1 = z0;
          if (SF32) {
            const float *sc = reinterpret_cast<const float *>(st + sofs) + bi * kTileN + g;
            s0 = sc[0];
            s1 = sc[8];
          } else {
            const uint16_t *sc = reinterpret_cast<const uint16_t *>(st + sofs) + bi * kTileN + g;
            s0 = bf16_bits_to_f32(sc[0]);
            s1 = bf16_bits_to_f32(sc[8]);
          }
          if (HAS_ZP) {
            // b's word in the staged word pairs (the first pair holds b0s).
            const uint2 zw = reinterpret_cast<const uint2 *>(st + zofs)[b - (b0s & ~1)];
            z0 = static_cast<float>(128 + ((zw.x >> (4 * g)) & 15));
            z1 = static_cast<float>(128 + ((zw.y >> (4 * g)) & 15));
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const float S0 = srow[mt][0][b], S1 = srow[mt][1][b];
            acc[mt][0] = fmaf(s0, fmaf(-z0, S0, d[mt][0]), acc[mt][0]);
            acc[mt][1] = fmaf(s0, fmaf(-z0, S1, d[mt][1]), acc[mt][1]);
            acc[mt][2] = fmaf(s1, fmaf(-z1, S0, d[mt][2]), acc[mt][2]);
            acc[mt][3] = fmaf(s1, fmaf(-z1, S1, d[mt][3]), acc[mt][3]);
          }
        };

        // One 16-wide k step of chunk ci (relative to cst): convert the
        // lane's codes, multiply with the activation fragments; the first
        // step of a block starts its sums from zero.
        // Code-book values are hi + lo: a second MMA with the remainders
        // (their product with the activations' fp32 remainder is below
        // 2^-16 of the term and left out).
        auto kstep = [&](uint32_t w, int ci, int jj, bool first, float (&d)[MT][4]) {
          uint32_t wf[4], wl[4];
          if (CODE) codes_to_lut(w, sPair, wf, wl);
          else codes_to_bf16x2(w, wf);
          const int ko = ci * kChunkK + 16 * jj;
          if (mok0) bfrag0 = *reinterpret_cast<const uint2 *>(ap0 + ko);
          if (first) mma_bf16_16816_zero(d[0], wf, bfrag0.x, bfrag0.y);
          else mma_bf16_16816(d[0], wf, bfrag0.x, bfrag0.y);
          if (CODE) mma_bf16_16816(d[0], wl, bfrag0.x, bfrag0.y);
          if (two) {
            if (mok0) bfrag0 = *reinterpret_cast<const uint2 *>(ap0 + lo_off + ko);
            mma_bf16_16816(d[0], wf, bfrag0.x, bfrag0.y);
          }
          if (MT == 2) {
            if (mok1) bfrag1 = *reinterpret_cast<const uint2 *>(ap1 + ko);
            if (first) mma_bf16_16816_zero(d[MT - 1], wf, bfrag1.x, bfrag1.y);
            else mma_bf16_16816(d[MT - 1], wf, bfrag1.x, bfrag1.y);
            if (CODE) mma_bf16_16816(d[MT - 1], wl, bfrag1.x, bfrag1.y);
            if (two) {
              if (mok1) bfrag1 = *reinterpret_cast<const uint2 *>(ap1 + lo_off + ko);
              mma_bf16_16816(d[MT - 1], wf, bfrag1.x, bfrag1.y);
            }
          }
        };

        if (BS >= kChunkK) {
          // The warp's chunks of a stage are whole blocks of BS/64 chunks.
          constexpr int kCpb = BS >= kChunkK ? BS / kChunkK : 1;
          const int cb0 = (cst * kChunkK) >> G::kLog2;
#pragma unroll 1
          for (int ub = 0; ub < p.cpw / kCpb; ++ub) {
            float d[MT][4];
#pragma unroll
            for (int cc = 0; cc < kCpb; ++cc) {
              const int ci = ub * kCpb + cc;
              const uint4 w4 = *reinterpret_cast<const uint4 *>(wp + ci * kChunkBytes);
              kstep(w4.x, ci, 0, cc == 0, d);
              kstep(w4.y, ci, 1, false, d);
              kstep(w4.z, ci, 2, false, d);
              kstep(w4.w, ci, 3, false, d);
            }
            correct(cb0 + ub, d);
          }
        } else {
          constexpr int kSpb = BS / 16;  // k steps per block
#pragma unroll 1
          for (int ci = 0; ci < p.cpw; ++ci) {
            const uint4 w4 = *reinterpret_cast<const uint4 *>(wp + ci * kChunkBytes);
            const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
            const int cb0 = ((cst + ci) * kChunkK) >> G::kLog2;
#pragma unroll
            for (int bb = 0; bb < 4 / kSpb; ++bb) {
              float d[MT][4];
#pragma unroll
              for (int jj = 0; jj < kSpb; ++jj)
                kstep(wv[bb * kSpb + jj], ci, bb * kSpb + jj, jj == 0, d);
              correct(cb0 + bb, d);
            }
          }
        }
        // The stage slice is consumed: release it to the producer.
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);
        if (++slot == p.nst) {
          slot = 0;
          phase ^= 1;
        }
      }

      if (direct) {
        // The warp owns all of K for its tile: store straight from registers.
        const int n0 = (gi - p.tg_begin[q]) * rows + tau * kTileN + g;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = mt * 8 + 2 * t + (e & 1);
            const int nn = n0 + 8 * (e >> 1);
            if (m < p.M && nn < p.N[q]) store_y(p, q, m, nn, acc[mt][e], sNrm);
          }
        continue;
      }

      // Fixed-order split-K reduction of this tile group.
      {
        float *red = sRed + warp * (kTileN * MC);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int col = mt * 8 + 2 * t;
          red[g * MC + col] = acc[mt][0];
          red[g * MC + col + 1] = acc[mt][1];
          red[(g + 8) * MC + col] = acc[mt][2];
          red[(g + 8) * MC + col + 1] = acc[mt][3];
        }
      }
      named_barrier_sync(kBarConsumers, kConsumers);
      if (p.paired) {
        // Rows r < rows/2 are gate rows, r + rows/2 the same rows of up.
        const int half = rows / 2, ht = p.tpc / 2;
        const int n_base = (gi - p.tg_begin[0]) * half;
        const int total = p.M * half;
        for (int e = tid; e < total; e += kConsumers) {
          const int m = e / half, r = e - m * half;
          const int tt = r >> 4, row = r & 15;
          float vg = 0.f, vu = 0.f;
          for (int k2 = 0; k2 < p.ksw; ++k2) {
            vg += sRed[((tt * p.ksw + k2) * kTileN + row) * MC + m];
            vu += sRed[(((tt + ht) * p.ksw + k2) * kTileN + row) * MC + m];
          }
          if (p.cluster == 1) {
            if (n_base + r < p.N[0]) store_gate_up(p, m, n_base + r, vg, vu, sNrm);
          } else {
            sPart[e] = vg;
            sPart[total + e] = vu;
          }
        }
        if (p.cluster > 1) {
          cluster_sync_all();
          for (int e = tid * p.cluster + crank; e < total; e += kConsumers * p.cluster) {
            float vg = 0.f, vu = 0.f;
            for (int r = 0; r < p.cluster; ++r) {
              vg += ld_dsmem_f32(sPart + e, r);
              vu += ld_dsmem_f32(sPart + total + e, r);
            }
            const int m = e / half, r = e - m * half;
            if (n_base + r < p.N[0]) store_gate_up(p, m, n_base + r, vg, vu, sNrm);
          }
          cluster_sync_all();
        } else {
          named_barrier_sync(kBarConsumers, kConsumers);
        }
        continue;
      }
      const int n_base = (gi - p.tg_begin[q]) * rows;
      const int total = p.M * rows;
      for (int e = tid; e < total; e += kConsumers) {
        const int m = e / rows, r = e - m * rows;
        const int tt = r >> 4, row = r & 15;
        float v = 0.f;
        for (int k2 = 0; k2 < p.ksw; ++k2)
          v += sRed[((tt * p.ksw + k2) * kTileN + row) * MC + m];
        if (p.cluster == 1) {
          if (n_base + r < p.N[q]) store_y(p, q, m, n_base + r, v, sNrm);
        } else {
          sPart[e] = v;
        }
      }
      if (p.cluster > 1) {
        // Combine the cluster's partials in rank order, then let every CTA
        // reuse its buffers.
        cluster_sync_all();
        for (int e = tid * p.cluster + crank; e < total; e += kConsumers * p.cluster) {
          float v = 0.f;
          for (int r = 0; r < p.cluster; ++r) v += ld_dsmem_f32(sPart + e, r);
          const int m = e / rows, r = e - m * rows;
          if (n_base + r < p.N[q]) store_y(p, q, m, n_base + r, v, sNrm);
        }
        cluster_sync_all();
      } else {
        named_barrier_sync(kBarConsumers, kConsumers);
      }
    }
    if (p.amax) {
      // This CTA's best key of each row joins the grid-wide maximum.
      named_barrier_sync(kBarConsumers, kConsumers);
      if (tid < p.M) {
        const unsigned long long key =
            reinterpret_cast<const unsigned long long *>(sNrm + kGemvMaxM)[tid];
        if (key) atomicMax(p.amax + tid, key);
      }
    }
  }
}

// Clears the ArgMax keys. The decode kernel launched after it (programmatic
// dependent launch) starts streaming weights at once and reaches its first
// atomic only after its dependency wait, i.e. after this kernel.
__global__ void argmax_init_kernel(unsigned long long *amax, int M) {
  grid_dependents_launch();
  for (int m = threadIdx.x; m < M; m += blockDim.x) amax[m] = 0ull;
}

// Turns the ArgMax keys into indices in place (a thread per row, striding
// over the rows); launched as a programmatic dependent of the decode kernel,
// it is resident before that kernel ends and waits for its results.
__global__ void argmax_finalize_kernel(unsigned long long *amax, int M) {
  grid_dependency_wait();
  for (int m = threadIdx.x; m < M; m += blockDim.x) {
    const unsigned long long key = amax[m];
    amax[m] = static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(key));
  }
}

struct Choice {
  int KS, ksw, cluster, tpc, R, nst, cpw;
  int64_t tg;
  size_t smem;
  GemvParams layout;
};

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }
size_t align128(size_t x) { return (x + 127) & ~size_t(127); }

// Chunks a warp takes per stage at least: whole blocks for blocks of a
// chunk or more.
int min_cpw(int bs) { return bs > kChunkK ? bs / kChunkK : 1; }

bool layout_for(const GroupArgs &a, int ksw, int cluster, int cpw, Choice &ch) {
  const int64_t K64 = ceil_div(a.K, kChunkK);
  const int KS = ksw * cluster;  // k ranges per tile group
  // More chunks per warp than blocks need only while the split still
  // covers K with them.
  if (cpw < min_cpw(a.bs) || (cpw > min_cpw(a.bs) && int64_t(KS) * cpw > K64)) return false;
  const int tpc = kConsumerWarps / ksw;
  if (a.paired && tpc < 2) return false;  // a gate and an up tile per group
  const int scs = ksw * cpw;
  // Every CTA of a cluster starts inside K.
  if (int64_t(cluster - 1) * scs * ceil_div(K64, int64_t(KS) * cpw) >= K64) return false;
  int64_t tg = 0;
  if (a.paired)
    tg = ceil_div(ceil_div(a.N[0], kTileN), tpc / 2);
  else
    for (int i = 0; i < a.count; ++i) tg += ceil_div(ceil_div(a.N[i], kTileN), tpc);
  const int MT = a.M <= 8 ? 1 : 2;
  const int R = static_cast<int>(ceil_div(K64, int64_t(KS) * cpw));
  const int64_t kr = int64_t(scs) * R * kChunkK;  // staged activations per row
  const int krp = static_cast<int>(kr) + 16;
  const int sg = static_cast<int>(kr / a.bs);  // block sums per staged row
  const int es = a.scale_f32 ? 4 : 2;
  // A stage holds scs consecutive chunks (scs * 64 k) of tpc tiles, the
  // nbs blocks they touch (stage starts are multiples of scs chunks, so for
  // blocks of at least scs chunks a stage lies inside one block) and the
  // nps zero-point pairs holding those blocks.
  const int nbs = std::max<int>(1, scs * kChunkK / a.bs);
  const int nps = std::max(1, nbs / 2);
  GemvParams L{};
  L.nbs = nbs;
  L.nps = nps;
  L.st_sc = scs * tpc * kChunkBytes;  // cpw * 8 KB: 128-byte aligned
  // Every TMA destination starts on 128 bytes: a pair's up halves of the
  // scale and zero-point regions start at aligned offsets.
  const size_t sc_all = size_t(tpc) * nbs * kTileN * es;
  const size_t zp_all = a.has_zp ? size_t(tpc) * nps * 16 : 0;
  L.sc_up = a.paired ? static_cast<int>(align128(sc_all / 2)) : 0;
  L.zp_up = a.paired ? static_cast<int>(align128(zp_all / 2)) : 0;
  L.st_zp = static_cast<int>(align128(L.st_sc + (a.paired ? L.sc_up + sc_all / 2 : sc_all)));
  L.stage_bytes = static_cast<int>(align128(L.st_zp + (a.paired ? L.zp_up + zp_all / 2 : zp_all)));
  L.stage_tx = tpc * (scs * kChunkBytes + nbs * kTileN * es + (a.has_zp ? nps * 16 : 0));
  size_t off = align16(size_t(a.M) * krp * 2);
  L.off_alo = static_cast<int>(off);
  if (a.a_f32) off += align16(size_t(a.M) * krp * 2);
  L.off_s = static_cast<int>(off);
  off += align16(size_t(a.M) * sg * 4);
  L.off_red = static_cast<int>(off);
  off += align16(size_t(kConsumerWarps) * kTileN * MT * 8 * 4);
  L.off_part = static_cast<int>(off);
  if (cluster > 1) off += align16(size_t(tpc) * kTileN * a.M * 4);
  L.off_nrm = static_cast<int>(off);
  off += align16(kGemvMaxM * 4 + kGemvMaxM * 8);  // r[m], then the ArgMax keys
  L.off_lut = static_cast<int>(off);
  off += a.code ? 256 * 8 : 0;  // code-book pair table (rounded values and remainders)
  L.off_bar = static_cast<int>(off);
  off += (2 * kMaxStages + 1) * 8;
  off = align128(off);
  L.off_ring = static_cast<int>(off);
  // Ring depth: as many stages as fit, at most kMaxStages, at least 2; stay
  // within the two-CTAs-per-SM budget when the layout allows it.
  size_t cap = kSmemBudget;
  if (MT == 2 || off + 2 * size_t(L.stage_bytes) > cap) cap = kSmemMax;
  if (off + 2 * size_t(L.stage_bytes) > cap) return false;
  int nst = static_cast<int>((cap - off) / L.stage_bytes);
  nst = std::min(nst, kMaxStages);
  // Do not hold more stages than the whole k range needs.
  nst = std::max(2, std::min<int>(nst, R * 2));
  off += size_t(nst) * L.stage_bytes;
  L.krp = krp;
  L.sg = sg;
  L.nst = nst;
  ch.KS = KS;
  ch.ksw = ksw;
  ch.cluster = cluster;
  ch.tpc = tpc;
  ch.R = R;
  ch.nst = nst;
  ch.cpw = cpw;
  ch.tg = tg;
  ch.smem = off;
  ch.layout = L;
  return true;
}

template <int MT, int BS, bool HAS_ZP, bool SF32, bool CODE = false, bool PROBE = false>
cudaError_t launch_one(const GemvParams &p, const Choice &ch, int grid, bool pdl,
                       cudaStream_t stream) {
  auto kernel = gemv_kernel<MT, BS, HAS_ZP, SF32, CODE, PROBE>;
  static std::atomic<unsigned long long> configured{0};
  if (const cudaError_t e = ensure_smem_limit(kernel, kSmemMax, configured); e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = ch.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (ch.cluster > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = ch.cluster;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int MT, int BS>
cudaError_t launch_flags(const GemvParams &p, const Choice &ch, int grid, bool has_zp,
                         bool sf32, bool pdl, cudaStream_t stream) {
  if (p.code) {  // code-book weights carry no zero points; up to 8 rows per launch
    if constexpr (MT == 1)
      return sf32 ? launch_one<MT, BS, false, true, true>(p, ch, grid, pdl, stream)
                  : launch_one<MT, BS, false, false, true>(p, ch, grid, pdl, stream);
    else
      return cudaErrorNotSupported;
  }
  if (has_zp)
    return sf32 ? launch_one<MT, BS, true, true>(p, ch, grid, pdl, stream)
                : launch_one<MT, BS, true, false>(p, ch, grid, pdl, stream);
  return sf32 ? launch_one<MT, BS, false, true>(p, ch, grid, pdl, stream)
              : launch_one<MT, BS, false, false>(p, ch, grid, pdl, stream);
}

template <int MT>
cudaError_t launch_bs(const GemvParams &p, const Choice &ch, int grid, int bs,
                      bool has_zp, bool sf32, bool pdl, cudaStream_t stream) {
  switch (bs) {
    case 16: return launch_flags<MT, 16>(p, ch, grid, has_zp, sf32, pdl, stream);
    case 32: return launch_flags<MT, 32>(p, ch, grid, has_zp, sf32, pdl, stream);
    case 64: return launch_flags<MT, 64>(p, ch, grid, has_zp, sf32, pdl, stream);
    case 128: return launch_flags<MT, 128>(p, ch, grid, has_zp, sf32, pdl, stream);
    case 256: return launch_flags<MT, 256>(p, ch, grid, has_zp, sf32, pdl, stream);
    default: return cudaErrorNotSupported;
  }
}

// Tensor maps of one prepacked weight (see the layout in mnb_common.cuh).
cudaError_t weight_maps(const GroupArgs &a, int i, int tpc, int scs, GemvParams &p) {
  const uint64_t N16 = ceil_div(a.N[i], kTileN), K64 = ceil_div(a.K, kChunkK);
  const uint64_t nb = ceil_div(a.K, a.bs), nbz = ceil_div(nb, 2) * 2;
  const uint64_t es = a.scale_f32 ? 4 : 2;
  const uint32_t nbs = static_cast<uint32_t>(p.nbs), nps = static_cast<uint32_t>(p.nps);
  {
    const uint64_t dims[3] = {kChunkBytes / 4, K64, N16};
    const uint64_t strides[2] = {kChunkBytes, K64 * kChunkBytes};
    const uint32_t box[3] = {kChunkBytes / 4, static_cast<uint32_t>(scs),
                             static_cast<uint32_t>(a.paired ? tpc / 2 : tpc)};
    cudaError_t e = make_tmap(&p.tmw[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.packed_b[i],
                              dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  {
    const uint64_t words = kTileN * es / 4;
    const uint64_t dims[3] = {words, nb, N16};
    const uint64_t strides[2] = {kTileN * es, nb * kTileN * es};
    const uint32_t box[3] = {static_cast<uint32_t>(words), nbs,
                             static_cast<uint32_t>(a.paired ? tpc / 2 : tpc)};
    cudaError_t e = make_tmap(&p.tms[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.scales[i],
                              dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  if (a.has_zp) {
    const uint64_t dims[3] = {4, nbz / 2, N16};
    const uint64_t strides[2] = {16, nbz * 8};
    const uint32_t box[3] = {4, nps, static_cast<uint32_t>(a.paired ? tpc / 2 : tpc)};
    cudaError_t e = make_tmap(&p.tmz[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.zp[i], dims,
                              strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

std::atomic<int> g_test_stop_stage{-1};

void gemv_set_wait_fault(int stop_stage) { g_test_stop_stage.store(stop_stage < 0 ? -1 : stop_stage); }

cudaError_t gemv_take_fault(unsigned int *out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fault_gemv, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fault_gemv, &zero, sizeof(unsigned int));
  return e;
}

cudaError_t launch_gemv_group(const GroupArgs &a, cudaStream_t stream) {
  if (a.M < 1 || a.M > kGemvMaxM || a.count < 1 || a.count > kMaxGroup)
    return cudaErrorNotSupported;
  const int sms = sm_count();
  const int MT = a.M <= 8 ? 1 : 2;
  // Pick the k split and the chunks per warp and stage by a small cost
  // model: rounds of resident CTAs times the chunks each warp streams per
  // tile group, plus a per-stage cost for the ring bookkeeping and a
  // per-round cost for the split-K reduction.
  Choice best{}, ch{};
  bool have = false;
  double best_cost = 0.0;
  for (int ksw = 1; ksw <= kConsumerWarps; ksw *= 2)
    for (int cluster = 1; cluster <= 8; cluster *= 2)
      for (int cpw = 1; cpw <= 4; cpw *= 2) {
        if (!layout_for(a, ksw, cluster, cpw, ch)) continue;
        const int per_sm = (MT == 1 && ch.smem <= static_cast<size_t>(kSmemBudget)) ? 2 : 1;
        const int64_t resident = std::max<int64_t>(1, int64_t(sms) * per_sm / cluster);
        const int64_t rounds = ceil_div(ch.tg, resident);
        const double per_round = double(ch.R) * (cpw + 0.6) + (ksw * cluster > 1 ? 2.0 : 0.0) +
                                 (cluster > 1 ? 1.0 : 0.0);
        const double cost = double(rounds) * per_round;
        if (!have || cost < best_cost - 1e-9) {
          best = ch;
          best_cost = cost;
          have = true;
        }
      }
  if (!have) return cudaErrorNotSupported;

  GemvParams p = best.layout;
  p.A = a.A;
  p.nprob = a.paired ? 1 : a.count;  // a pair walks the gate's tile groups
  p.paired = a.paired;
  int64_t tg = 0;
  for (int i = 0; i < a.count; ++i) {
    const cudaError_t e = weight_maps(a, i, best.tpc, best.ksw * best.cpw, p);
    if (e != cudaSuccess) return e;
    p.bias[i] = a.bias[i];
    p.Y[i] = a.Y[i];
    p.N[i] = static_cast<int>(a.N[i]);
    p.N16[i] = static_cast<int>(ceil_div(a.N[i], kTileN));
    p.tg_begin[i] = static_cast<int>(tg);
    if (!a.paired) tg += ceil_div(p.N16[i], best.tpc);
  }
  if (a.paired) tg = ceil_div(p.N16[0], best.tpc / 2);
  p.tg_total = static_cast<int>(tg);
  p.M = static_cast<int>(a.M);
  p.K = static_cast<int>(a.K);
  p.K64 = static_cast<int>(ceil_div(a.K, kChunkK));
  p.nb = static_cast<int>(ceil_div(a.K, a.bs));
  p.a_f32 = a.a_f32;
  const int vec_elems = a.a_f32 ? 4 : 8;
  p.a_vec = (reinterpret_cast<uintptr_t>(a.A) % 16 == 0) && (a.K % vec_elems == 0);
  p.code = a.code;
  p.norm = a.norm ? 1 : 0;
  p.gamma = a.gamma;
  p.eps = a.eps;
  p.amax = a.amax;
  // A normalized row is scaled by gamma while it is staged: not a raw copy.
  p.a_bulk = !a.a_f32 && p.a_vec && !a.norm;
  p.ksw = best.ksw;
  p.tpc = best.tpc;
  p.cluster = best.cluster;
  p.R = best.R;
  p.cpw = best.cpw;
  p.scs = best.ksw * best.cpw;
  p.stop_stage = g_test_stop_stage.load();

  // Persistent grid: every tile group gets a CTA (cluster) when they fit in
  // the CTAs resident at once; otherwise CTAs walk the groups.
  const int per_sm = (MT == 1 && best.smem <= static_cast<size_t>(kSmemBudget)) ? 2 : 1;
  const int64_t resident = int64_t(sms) * per_sm / best.cluster;
  const int64_t clusters = tg < resident ? tg : resident;
  const int grid = static_cast<int>(clusters) * best.cluster;

  if (p.stop_stage >= 0 && MT == 1 && a.bs == 128 && !a.has_zp && !a.scale_f32 && !a.code)
    return launch_one<1, 128, false, false, false, true>(p, best, grid, a.pdl, stream);
  return MT == 2 ? launch_bs<2>(p, best, grid, a.bs, a.has_zp, a.scale_f32, a.pdl, stream)
                 : launch_bs<1>(p, best, grid, a.bs, a.has_zp, a.scale_f32, a.pdl, stream);
}

cudaError_t launch_argmax_init(unsigned long long *amax, int M, cudaStream_t stream) {
  argmax_init_kernel<<<1, 256, 0, stream>>>(amax, M);
  return cudaGetLastError();
}

cudaError_t launch_argmax_finalize(unsigned long long *amax, int M, bool pdl,
                                   cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, argmax_finalize_kernel, amax, M);
}

cudaError_t launch_gemv(const MatmulArgs &a, cudaStream_t stream) {
  GroupArgs g{};
  g.A = a.A;
  g.count = 1;
  g.packed_b[0] = a.packed_b;
  g.scales[0] = a.scales;
  g.zp[0] = a.zp;
  g.bias[0] = a.bias;
  g.Y[0] = a.Y;
  g.N[0] = a.N;
  g.M = a.M;
  g.K = a.K;
  g.bs = a.bs;
  g.a_f32 = a.a_f32;
  g.scale_f32 = a.scale_f32;
  g.has_zp = a.zp != nullptr;
  g.pdl = a.pdl;
  return launch_gemv_group(g, stream);
}

}  // namespace mnb
