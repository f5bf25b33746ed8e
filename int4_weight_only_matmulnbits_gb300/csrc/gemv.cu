// Small-M (decode) MatMulNBits kernel for sm_103a.
//
// Computes Y[m,n] = sum_k A[m,k] (q[n,k] - z[n,b]) s[n,b] + bias[n] for
// M <= 16 on the prepacked layout of mnb_common.cuh. It follows the page
// "Qwen3 CPU Inference Critical Path", section "Prepared weight-only plan":
// weights stay compressed, are unpacked in registers, zero points and scales
// are applied per block and accumulation is fp32; int4_gemv streams every
// weight byte once, partitioned over output channels, and int4_small_m reuses
// the unpacked codes across a few activation rows.
//
// GB300 mapping:
//  * A warp owns one 16-row tile and a contiguous range of <= 8 64-wide k
//    chunks. It issues all its 128-bit weight loads at once, before waiting
//    on the upstream kernel (the weights are constant), so each launch puts
//    its whole weight stream in flight immediately.
//  * Codes become bf16 (128 + q) with one lop3 per pair and feed
//    mma.m16n8k16 as the 16-row operand, with the activations (8 rows per
//    MMA) as the 8-column operand. Products and sums are exact up to fp32
//    accumulation; no per-weight subtract or multiply is needed.
//  * Per block (or block piece) the fp32 correction
//      acc += s * (D - (128 + z) * S),   S = sum of the block's activations,
//    applies zero point and scale. fp32 activations are split into bf16
//    hi + lo (two MMAs), and S is summed from hi + lo so the offset cancels.
//  * Split-K partials are reduced in fixed order: warps of a CTA through
//    shared memory, CTAs of a cluster through distributed shared memory.
//    No global workspace, no atomics: results are bitwise reproducible.
#include <cuda_bf16.h>

#include "mnb_common.cuh"
#include "mnb_launch.h"

namespace mnb {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxChunks = 8;  // k chunks per warp (registers: 4 per chunk)
constexpr int kSmemLimit = 160 * 1024;

struct GemvParams {
  const void *A;
  const uint4 *wq;
  const void *scales;
  const uint2 *zp;
  const float *bias;
  void *Y;
  int M, N, K;
  int K64, N16, nb;
  int bs, bs_log2;
  int scale_f32, has_zp;
  int ksplit, tiles_per_cta, cluster, KS;
  int a_vec;
  int krp;      // row stride (elements) of the staged activations
  int sg;       // activation-sum granules per staged row
  int granule;  // min(bs, 64)
  int nbr;      // block slots per tile in the staged scales
  int off_alo, off_s, off_sc, off_zp, off_red, off_part;
};

template <bool AF32>
__device__ __forceinline__ void load8(const GemvParams &p, int m, int64_t k,
                                      float (&v)[8]) {
  if (AF32) {
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

template <int MT, bool AF32>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t *sAhi = reinterpret_cast<uint16_t *>(smem);
  uint16_t *sAlo = reinterpret_cast<uint16_t *>(smem + p.off_alo);
  float *sS = reinterpret_cast<float *>(smem + p.off_s);
  unsigned char *sSc = smem + p.off_sc;
  uint2 *sZp = reinterpret_cast<uint2 *>(smem + p.off_zp);
  float *sRed = reinterpret_cast<float *>(smem + p.off_red);
  float *sPart = reinterpret_cast<float *>(smem + p.off_part);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int crank = static_cast<int>(blockIdx.x) % p.cluster;
  const int tgroup = static_cast<int>(blockIdx.x) / p.cluster;
  const int tau = warp / p.ksplit, ks = warp - tau * p.ksplit;
  const int tile = tgroup * p.tiles_per_cta + tau;
  const bool tile_ok = tile < p.N16;
  const int kidx = crank * p.ksplit + ks;
  const int c0 = static_cast<int>((int64_t)kidx * p.K64 / p.KS);
  const int c1 = static_cast<int>((int64_t)(kidx + 1) * p.K64 / p.KS);
  const int clo = static_cast<int>((int64_t)crank * p.K64 / p.cluster);
  const int chi = static_cast<int>((int64_t)(crank + 1) * p.K64 / p.cluster);
  const int blo = (clo * kChunkK) >> p.bs_log2;
  const int bhi = min(p.nb, (chi * kChunkK + p.bs - 1) >> p.bs_log2);

  // 1. The warp's whole constant weight stream goes in flight first.
  uint4 wreg[kMaxChunks];
  {
    const uint4 *src = p.wq + ((int64_t)tile * p.K64 + c0) * 32 + lane;
#pragma unroll
    for (int i = 0; i < kMaxChunks; ++i)
      wreg[i] = (tile_ok && c0 + i < c1) ? ldg_stream(src + i * 32)
                                         : make_uint4(0, 0, 0, 0);
  }

  // 2. Scales and zero points of the CTA's tiles over its block range.
  {
    const int nbl = bhi - blo;
    const int per_tile = nbl * kTileN;
    const int total = p.tiles_per_cta * per_tile;
    for (int i = tid; i < total; i += kThreads) {
      const int tt = i / per_tile, e = i - tt * per_tile;
      const int tl = tgroup * p.tiles_per_cta + tt;
      if (tl >= p.N16) continue;
      const int64_t src = ((int64_t)tl * p.nb + blo) * kTileN + e;
      const int dst = tt * p.nbr * kTileN + e;
      if (p.scale_f32)
        reinterpret_cast<float *>(sSc)[dst] =
            __ldg(static_cast<const float *>(p.scales) + src);
      else
        reinterpret_cast<uint16_t *>(sSc)[dst] =
            __ldg(static_cast<const uint16_t *>(p.scales) + src);
    }
    if (p.has_zp) {
      const int totz = p.tiles_per_cta * nbl;
      for (int i = tid; i < totz; i += kThreads) {
        const int tt = i / nbl, e = i - tt * nbl;
        const int tl = tgroup * p.tiles_per_cta + tt;
        if (tl < p.N16)
          sZp[tt * p.nbr + e] = __ldg(p.zp + (int64_t)tl * p.nb + blo + e);
      }
    }
  }

  // 3. From here on the upstream kernel's results (A) are visible.
  grid_dependency_wait();

  // 4. Stage A rows [0, M) over the CTA's k range as bf16 (hi, lo) and the
  //    activation sum of every granule (block, or 64-wide piece of a block).
  {
    const int kr = (chi - clo) * kChunkK;
    const int ppr = kr >> 3;  // 8-element pieces per row
    const int total = p.M * ppr;
    const int gp = p.granule >> 3;
    for (int base = 0; base < total; base += kThreads) {
      const int pc = base + tid;
      const bool ok = pc < total;
      float part = 0.f;
      int m = 0, kp = 0;
      if (ok) {
        m = pc / ppr;
        kp = pc - m * ppr;
        float v[8];
        load8<AF32>(p, m, (int64_t)clo * kChunkK + kp * 8, v);
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t h0 = bf16_bits(v[2 * q]), h1 = bf16_bits(v[2 * q + 1]);
          hi[q] = h0 | (h1 << 16);
          if (AF32) {
            const float r0 = v[2 * q] - bf16_bits_to_f32(h0);
            const float r1 = v[2 * q + 1] - bf16_bits_to_f32(h1);
            const uint32_t l0 = bf16_bits(r0), l1 = bf16_bits(r1);
            lo[q] = l0 | (l1 << 16);
            part += (bf16_bits_to_f32(h0) + bf16_bits_to_f32(l0)) +
                    (bf16_bits_to_f32(h1) + bf16_bits_to_f32(l1));
          } else {
            part += v[2 * q] + v[2 * q + 1];
          }
        }
        const int off = m * p.krp + kp * 8;
        *reinterpret_cast<uint4 *>(sAhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (AF32)
          *reinterpret_cast<uint4 *>(sAlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      for (int o = 1; o < gp; o <<= 1)
        part += __shfl_xor_sync(0xffffffffu, part, o);
      if (ok && (kp % gp) == 0) sS[m * p.sg + kp / gp] = part;
    }
  }
  __syncthreads();
  grid_dependents_launch();

  // 5. Convert, multiply and correct per block.
  float acc[MT][4], d[MT][4], srun[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[mt][q] = d[mt][q] = 0.f;
    srun[mt][0] = srun[mt][1] = 0.f;
  }
  if (tile_ok) {
    const bool big_blocks = p.bs >= kChunkK;
    const int spb_mask = (p.bs >> 4) - 1;
#pragma unroll
    for (int i = 0; i < kMaxChunks; ++i) {
      const int c = c0 + i;
      if (c < c1) {
        const int cl = c - clo;
        if (big_blocks) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int m0 = mt * 8 + 2 * t;
            if (m0 < p.M) srun[mt][0] += sS[m0 * p.sg + cl];
            if (m0 + 1 < p.M) srun[mt][1] += sS[(m0 + 1) * p.sg + cl];
          }
        }
        const uint32_t wv[4] = {wreg[i].x, wreg[i].y, wreg[i].z, wreg[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t wf[4];
          codes_to_bf16x2(wv[j], wf);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int m = mt * 8 + g;
            uint2 bh = make_uint2(0, 0), bl = make_uint2(0, 0);
            if (m < p.M) {
              const int off = m * p.krp + cl * kChunkK + 16 * j + 4 * t;
              bh = *reinterpret_cast<const uint2 *>(sAhi + off);
              if (AF32) bl = *reinterpret_cast<const uint2 *>(sAlo + off);
            }
            mma_bf16_16816(d[mt], wf, bh.x, bh.y);
            if (AF32) mma_bf16_16816(d[mt], wf, bl.x, bl.y);
          }
          const int s = c * 4 + j;
          const bool block_end = ((s + 1) & spb_mask) == 0;
          const bool range_end = (j == 3) && (c + 1 == c1);
          if (block_end || range_end) {
            // Blocks past the last real one (k >= nb*bs, chunk padding) hold
            // no codes and no activations: their slot is never staged, so
            // they contribute scale 0.
            const int bglob = (s * 16) >> p.bs_log2;
            const int bl = bglob - blo;
            const int si = tau * p.nbr * kTileN + bl * kTileN + g;
            float s0 = 0.f, s1 = 0.f;
            float z0 = 136.f, z1 = 136.f;
            if (bglob < p.nb) {
              if (p.scale_f32) {
                s0 = reinterpret_cast<const float *>(sSc)[si];
                s1 = reinterpret_cast<const float *>(sSc)[si + 8];
              } else {
                s0 = bf16_bits_to_f32(reinterpret_cast<const uint16_t *>(sSc)[si]);
                s1 = bf16_bits_to_f32(reinterpret_cast<const uint16_t *>(sSc)[si + 8]);
              }
              if (p.has_zp) {
                const uint2 zw = sZp[tau * p.nbr + bl];
                z0 = static_cast<float>(128 + ((zw.x >> (4 * g)) & 15));
                z1 = static_cast<float>(128 + ((zw.y >> (4 * g)) & 15));
              }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              float S0, S1;
              if (big_blocks) {
                S0 = srun[mt][0];
                S1 = srun[mt][1];
                srun[mt][0] = srun[mt][1] = 0.f;
              } else {
                const int gl = (cl * kChunkK + 16 * j) >> p.bs_log2;
                const int m0 = mt * 8 + 2 * t;
                S0 = m0 < p.M ? sS[m0 * p.sg + gl] : 0.f;
                S1 = m0 + 1 < p.M ? sS[(m0 + 1) * p.sg + gl] : 0.f;
              }
              acc[mt][0] = fmaf(s0, fmaf(-z0, S0, d[mt][0]), acc[mt][0]);
              acc[mt][1] = fmaf(s0, fmaf(-z0, S1, d[mt][1]), acc[mt][1]);
              acc[mt][2] = fmaf(s1, fmaf(-z1, S0, d[mt][2]), acc[mt][2]);
              acc[mt][3] = fmaf(s1, fmaf(-z1, S1, d[mt][3]), acc[mt][3]);
#pragma unroll
              for (int q = 0; q < 4; ++q) d[mt][q] = 0.f;
            }
          }
        }
      }
    }
  }

  // 6. Fixed-order split-K reduction and epilogue.
  constexpr int MC = MT * 8;
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
  __syncthreads();

  const int rows = p.tiles_per_cta * kTileN;
  const int total = p.M * rows;
  const int n_base = tgroup * p.tiles_per_cta * kTileN;
  auto store = [&](int e, float v) {
    const int m = e / rows, r = e - m * rows;
    const int n = n_base + r;
    if (n < p.N) {
      if (p.bias) v += __ldg(p.bias + n);
      if (AF32)
        static_cast<float *>(p.Y)[(int64_t)m * p.N + n] = v;
      else
        static_cast<uint16_t *>(p.Y)[(int64_t)m * p.N + n] =
            static_cast<uint16_t>(bf16_bits(v));
    }
  };
  for (int e = tid; e < total; e += kThreads) {
    const int m = e / rows, r = e - m * rows;
    const int tt = r >> 4, row = r & 15;
    float v = 0.f;
    for (int q = 0; q < p.ksplit; ++q)
      v += sRed[((tt * p.ksplit + q) * kTileN + row) * MC + m];
    if (p.cluster == 1)
      store(e, v);
    else
      sPart[e] = v;
  }
  if (p.cluster > 1) {
    cluster_sync_all();
    for (int e = tid * p.cluster + crank; e < total; e += kThreads * p.cluster) {
      float v = 0.f;
      for (int r = 0; r < p.cluster; ++r) v += ld_dsmem_f32(sPart + e, r);
      store(e, v);
    }
    cluster_sync_all();
  }
}

struct Choice {
  int KS, ksplit, cluster, tiles_per_cta, ctas;
  size_t smem;
  GemvParams layout;
};

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

bool layout_for(const MatmulArgs &a, int KS, Choice &ch) {
  const int64_t K64 = ceil_div(a.K, kChunkK), N16 = ceil_div(a.N, kTileN);
  if (ceil_div(K64, KS) > kMaxChunks) return false;
  if (KS > 1 && KS > K64) return false;
  const int ksplit = KS < kWarps ? KS : kWarps;
  const int cluster = KS / ksplit;
  if (cluster > 8) return false;
  const int tpc = kWarps / ksplit;
  const int MT = a.M <= 8 ? 1 : 2;
  const int64_t krmax = ceil_div(K64, cluster) * kChunkK;
  const int krp = static_cast<int>(krmax) + 16;
  const int granule = a.bs < kChunkK ? a.bs : kChunkK;
  const int sg = static_cast<int>(krmax / granule);
  const int nbr = static_cast<int>(ceil_div(krmax, a.bs)) + 1;
  const int es = a.scale_f32 ? 4 : 2;
  GemvParams L{};
  size_t off = align16(size_t(a.M) * krp * 2);
  L.off_alo = static_cast<int>(off);
  if (a.a_f32) off += align16(size_t(a.M) * krp * 2);
  L.off_s = static_cast<int>(off);
  off += align16(size_t(a.M) * sg * 4);
  L.off_sc = static_cast<int>(off);
  off += align16(size_t(tpc) * nbr * kTileN * es);
  L.off_zp = static_cast<int>(off);
  if (a.zp) off += align16(size_t(tpc) * nbr * 8);
  L.off_red = static_cast<int>(off);
  off += align16(size_t(kWarps) * kTileN * MT * 8 * 4);
  L.off_part = static_cast<int>(off);
  if (cluster > 1) off += align16(size_t(tpc) * kTileN * a.M * 4);
  if (off > static_cast<size_t>(kSmemLimit)) return false;
  L.krp = krp;
  L.sg = sg;
  L.granule = granule;
  L.nbr = nbr;
  ch.KS = KS;
  ch.ksplit = ksplit;
  ch.cluster = cluster;
  ch.tiles_per_cta = tpc;
  ch.ctas = static_cast<int>(ceil_div(N16, tpc)) * cluster;
  ch.smem = off;
  ch.layout = L;
  return true;
}

template <int MT, bool AF32>
cudaError_t launch_one(const GemvParams &p, const Choice &ch, bool pdl,
                       cudaStream_t stream) {
  auto kernel = gemv_kernel<MT, AF32>;
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ch.ctas, 1, 1);
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

}  // namespace

cudaError_t launch_gemv(const MatmulArgs &a, cudaStream_t stream) {
  if (a.M < 1 || a.M > kGemvMaxM) return cudaErrorNotSupported;
  const int target = 2 * sm_count();
  Choice best{}, ch{};
  bool have = false;
  for (int KS = 1; KS <= 64; KS *= 2) {
    if (!layout_for(a, KS, ch)) continue;
    if (!have || (best.ctas < target && ch.ctas > best.ctas)) {
      best = ch;
      have = true;
    }
    if (best.ctas >= target) break;
  }
  if (!have) return cudaErrorNotSupported;

  GemvParams p = best.layout;
  p.A = a.A;
  p.wq = static_cast<const uint4 *>(a.packed_b);
  p.scales = a.scales;
  p.zp = static_cast<const uint2 *>(a.zp);
  p.bias = a.bias;
  p.Y = a.Y;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.K64 = static_cast<int>(ceil_div(a.K, kChunkK));
  p.N16 = static_cast<int>(ceil_div(a.N, kTileN));
  p.nb = static_cast<int>(ceil_div(a.K, a.bs));
  p.bs = a.bs;
  p.bs_log2 = 31 - __builtin_clz(static_cast<unsigned>(a.bs));
  p.scale_f32 = a.scale_f32;
  p.has_zp = a.zp != nullptr;
  p.ksplit = best.ksplit;
  p.tiles_per_cta = best.tiles_per_cta;
  p.cluster = best.cluster;
  p.KS = best.KS;
  const int vec_elems = a.a_f32 ? 4 : 8;
  p.a_vec = (reinterpret_cast<uintptr_t>(a.A) % 16 == 0) && (a.K % vec_elems == 0);

  const bool mt2 = a.M > 8;
  if (a.a_f32)
    return mt2 ? launch_one<2, true>(p, best, a.pdl, stream)
               : launch_one<1, true>(p, best, a.pdl, stream);
  return mt2 ? launch_one<2, false>(p, best, a.pdl, stream)
             : launch_one<1, false>(p, best, a.pdl, stream);
}

}  // namespace mnb
