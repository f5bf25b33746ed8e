// Decode chain: a sequence of MatMulNBits projections with declared data
// dependencies, executed by one persistent cooperative kernel.
//
// Every op computes Y[m,n] = sum_k A[m,k] (q[n,k] - z[n,b]) s[n,b] + bias[n]
// (or, for a gated-MLP pair, silu(gate) * up of two such projections) on the
// prepacked layout of mnb_common.cuh, with the arithmetic of the decode
// kernel: codes become bf16 128 + q with one lop3 per pair, feed
// mma.m16n8k16 as the 16-row operand against the staged activations, and
// per block the fp32 correction acc += s * (D - (128 + z) * S) applies the
// zero point and scale (page "Qwen3 CPU Inference Critical Path", section
// "Prepared weight-only plan": compressed weights unpacked in registers,
// per-block zero point and scale, fp32 accumulation; the gated pair follows
// that page's graph-level fusion "gate projection, SiLU, and gate/up
// multiplication").
//
// What the chain adds is the schedule. A decode step runs hundreds of small
// projections in a row; launched one by one, each pays a fixed start, a
// staging round trip and a drain. Here:
//  * One CTA per resident slot of every SM (cooperative launch: all CTAs run
//    at once, so CTAs may wait on one another). The host splits every op
//    into 16-row tiles (a gated pair: a gate tile and the up tile of the
//    same rows) and assigns contiguous tile ranges ("segments", at most
//    `tmax` tiles each) to CTAs by list scheduling: each tile goes to the
//    CTA that would finish it first, given when that CTA is free and when
//    the op's dependencies are expected to be complete.
//  * A CTA's work is one stream of groups (a group = one quantisation block
//    of one tile, or one 64-wide k chunk for blocks under 64) in op order.
//    A producer warp copies 16 groups per pipeline stage (codes, scales,
//    zero points: three bulk copies per group) into a ring of shared-memory
//    stages, straight across segment and op boundaries: the weights of the
//    next op are already in flight while the CTA waits for that op's inputs.
//  * Consumer warp w takes group w of every stage. At a segment's end each
//    warp leaves its partial sums per tile in shared memory, and the
//    consumers add them in a fixed warp order (bitwise reproducible) and
//    store Y with the bias (and SiLU for a pair).
//  * Completion: after a segment's stores, one thread releases (device
//    scope) an increment of the op's counter; an op completes when its
//    counter reaches its segment count. Before reading an op's activations
//    a CTA acquires the counters of the op's deps. Activations are then
//    loaded with L2-coherent loads into shared memory (bf16; fp32 as hi + lo
//    exact to 2^-16) with the per-block sums S.
//  * Every wait is bounded; a wait that runs out sets the launch's abort
//    word, after which every other wait gives up at once. The last CTA to
//    finish resets the counters, so the next launch on the stream starts
//    from zero (a plan is reusable and graph-capturable).
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "mnb_common.cuh"
#include "mnb_launch.h"

namespace mnb {

__device__ unsigned int g_fault_chain = 0;

namespace {

constexpr int kCW = 16;                   // consumer warps = groups per stage
constexpr int kCT = kCW * 32;             // consumer threads
constexpr int kThreadsChain = kCT + 32;   // + one producer warp
constexpr int kBarCons = 1;               // named barrier of the consumers
constexpr int kMaxStagesChain = 16;
constexpr int kBudget2 = 112 * 1024;      // two CTAs per SM
constexpr int kBudget1 = 226 * 1024;      // one CTA per SM (static shared memory beside it)
constexpr uint32_t kDepSpinLimit = 1u << 22;  // polls of a dependency counter
constexpr int kSegWait = 1;   // wait for the op's deps and stage its activations

struct alignas(16) OpDev {
  const unsigned char *b[2], *s[2], *z[2];
  const float *bias[2];
  const void *A;
  void *Y;
  int N, K, K64, nb, nbz;
  int paired;  // 1: virtual tile v is tile v/2 of weight v%2 (gate, up)
  int gpt;     // groups per (virtual) tile
  int target;  // segments of this op: complete when its counter reaches this
  int a_vec;   // activation rows allow 16-byte loads
  int dep[kChainMaxDeps];
};

struct ChainParams {
  const OpDev *ops;
  const int *cta_seg;    // [grid + 1]: first segment of each CTA
  const int4 *segs;      // {op, first virtual tile, virtual tiles, flags}
  unsigned int *count;   // [n_ops] completion counters
  unsigned int *ctl;     // [0] CTAs finished, [1] abort
  int n_ops, M, a_f32;
  int kp, sg;            // staged activation row stride (elements), block sums per row
  int nst, stage_bytes, sc_off, zp_off;
  int off_alo, off_s, off_red, off_opc, off_bar, off_ring;
};

// The consumers read their segment and op descriptors from a small
// shared-memory cache that warp 0 fills one segment ahead with cp.async
// (an L1 miss after every barrier would otherwise cost an L2 round trip).
static_assert(sizeof(OpDev) % 16 == 0, "op descriptors are copied in 16-byte pieces");
constexpr int kOpChunks = static_cast<int>(sizeof(OpDev) / 16);
constexpr int kOpCacheBytes = 2 * static_cast<int>(sizeof(OpDev)) + 4 * 16;

template <int BS>
struct Geo {
  static constexpr int kCpg = BS >= kChunkK ? BS / kChunkK : 1;  // chunks per group
  static constexpr int kBpg = BS >= kChunkK ? 1 : kChunkK / BS;  // blocks per group
  static constexpr int kSpb = BS / 16;                           // k steps per block
};

// Polls read with relaxed loads (an acquire load would invalidate the L1
// on every poll); one acquire fence follows the last successful poll.
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const unsigned int *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void red_release_gpu_add(unsigned int *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile(const unsigned int *p) {
  return *reinterpret_cast<const volatile unsigned int *>(p);
}

__device__ __forceinline__ void chain_abort(const ChainParams &p) {
  record_fault(&g_fault_chain, kFaultChainWait);
  atomicExch(p.ctl + 1, 1u);
}

// Bounded mbarrier wait that also gives up once the launch was aborted.
__device__ __forceinline__ bool chain_wait(const ChainParams &p, uint64_t *bar,
                                           uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023u) == 1023u && ld_volatile(p.ctl + 1)) return false;
  }
  chain_abort(p);
  return false;
}

// Eight activations A[m][k..k+7] as fp32 (zeros past K), through L2: an
// earlier op of this launch may have written them.
__device__ __forceinline__ void load8_cg(const void *A, int K, bool a_vec, bool a_f32, int m,
                                         int k, float (&v)[8]) {
  if (a_f32) {
    const float *a = static_cast<const float *>(A) + (size_t)m * K;
    if (a_vec && k + 8 <= K) {
      const float4 x = __ldcg(reinterpret_cast<const float4 *>(a + k));
      const float4 y = __ldcg(reinterpret_cast<const float4 *>(a + k + 4));
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
      v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = (k + q < K) ? __ldcg(a + k + q) : 0.f;
    }
  } else {
    const uint16_t *a = static_cast<const uint16_t *>(A) + (size_t)m * K;
    if (a_vec && k + 8 <= K) {
      const uint4 x = __ldcg(reinterpret_cast<const uint4 *>(a + k));
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[2 * q] = bf16_bits_to_f32(w[q] & 0xFFFFu);
        v[2 * q + 1] = bf16_bits_to_f32(w[q] >> 16);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = (k + q < K) ? bf16_bits_to_f32(__ldcg(a + k + q)) : 0.f;
    }
  }
}

__device__ __forceinline__ void store_out(void *Y, int N, bool a_f32, int m, int n, float v) {
  if (a_f32)
    static_cast<float *>(Y)[(size_t)m * N + n] = v;
  else
    static_cast<uint16_t *>(Y)[(size_t)m * N + n] = static_cast<uint16_t>(bf16_bits(v));
}

// The fields of an op the producer needs, cached in registers per segment.
struct ProdOp {
  const unsigned char *b[2], *s[2], *z[2];
  int K64, nb, nbz, paired;
};

__device__ __forceinline__ void load_prod_op(const OpDev *o, ProdOp &c) {
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    c.b[w] = o->b[w];
    c.s[w] = o->s[w];
    c.z[w] = o->z[w];
  }
  c.K64 = o->K64;
  c.nb = o->nb;
  c.nbz = o->nbz;
  c.paired = o->paired;
}

// Stages activation rows [0, M) of an op (zeros past K) as bf16 (fp32 rows
// as hi + lo) and the sum of every block of the staged values. Each thread
// first issues the loads of NB 8-element pieces, then converts them; the
// pieces of one block sit in consecutive lanes of one row (rows are padded
// to multiples of 256 elements).
template <int NB, bool F32, int BS>
__device__ __forceinline__ void stage_rows(const void *A, int K, bool a_vec, int M, int ppr,
                                           int kp, int sg, uint16_t *sA, int lo_off, float *sS,
                                           int tid) {
  const int npieces = M * ppr;
  constexpr int gp = BS / 8;  // pieces per block
  for (int base = 0; base < npieces; base += kCT * NB) {
    float v[NB][8];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int pc = base + b * kCT + tid;
      if (pc < npieces) {
        const int m = pc / ppr;
        load8_cg(A, K, a_vec, F32, m, (pc - m * ppr) * 8, v[b]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[b][e] = 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (base + b * kCT >= npieces) break;  // warp-uniform
      const int pc = base + b * kCT + tid;
      const bool ok = pc < npieces;
      const int m = ok ? pc / ppr : 0;
      const int kq = pc - m * ppr;
      float part = 0.f;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t h0 = bf16_bits(v[b][2 * e]), h1 = bf16_bits(v[b][2 * e + 1]);
        hi[e] = h0 | (h1 << 16);
        const float f0 = bf16_bits_to_f32(h0), f1 = bf16_bits_to_f32(h1);
        if (F32) {
          const uint32_t l0 = bf16_bits(v[b][2 * e] - f0);
          const uint32_t l1 = bf16_bits(v[b][2 * e + 1] - f1);
          lo[e] = l0 | (l1 << 16);
          part += (f0 + bf16_bits_to_f32(l0)) + (f1 + bf16_bits_to_f32(l1));
        } else {
          part += f0 + f1;
        }
      }
      if (ok) {
        const int off = m * kp + kq * 8;
        *reinterpret_cast<uint4 *>(sA + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (F32)
          *reinterpret_cast<uint4 *>(sA + lo_off + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
#pragma unroll
      for (int o = 1; o < gp; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (ok && (kq % gp) == 0) sS[m * sg + kq / gp] = part;
    }
  }
}

template <int BS, bool HAS_ZP, bool SF32>
__global__ void __launch_bounds__(kThreadsChain, 2)
    chain_kernel(const __grid_constant__ ChainParams p) {
  using G = Geo<BS>;
  constexpr int kEs = SF32 ? 4 : 2;
  constexpr int kCB = G::kCpg * kChunkBytes;        // codes per group slot
  constexpr int kSCB = G::kBpg * kTileN * kEs;      // scales per group slot
  constexpr int kZPB = BS >= kChunkK ? 16 : G::kBpg * 8;  // zero-point words per group slot
  extern __shared__ __align__(128) unsigned char smem[];
  uint16_t *sA = reinterpret_cast<uint16_t *>(smem);
  float *sS = reinterpret_cast<float *>(smem + p.off_s);
  float *sRed = reinterpret_cast<float *>(smem + p.off_red);
  OpDev *sOpc = reinterpret_cast<OpDev *>(smem + p.off_opc);
  int4 *sSegc = reinterpret_cast<int4 *>(smem + p.off_opc + 2 * sizeof(OpDev));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
  uint64_t *empty = full + kMaxStagesChain;
  unsigned char *ring = smem + p.off_ring;
  __shared__ int sh_fault;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg_lo = p.cta_seg[blockIdx.x], seg_hi = p.cta_seg[blockIdx.x + 1];

  if (tid == 0) {
    for (int i = 0; i < p.nst; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kCW);
    }
    sh_fault = 0;
    fence_barrier_init();
  }
  if (warp == 0 && seg_lo < seg_hi) {
    // The consumers' descriptor cache: the first two segments, the first op.
    if (lane < 2 && seg_lo + lane < seg_hi) sSegc[lane] = p.segs[seg_lo + lane];
    if (lane < kOpChunks)
      reinterpret_cast<uint4 *>(sOpc)[lane] =
          reinterpret_cast<const uint4 *>(p.ops + p.segs[seg_lo].x)[lane];
  }
  __syncthreads();

  if (warp == kCW) {
    // ---- producer: lane l < 16 copies group 16*q + l of stage q -------------
    int s = seg_lo, gs = 0, gpt = 1, ng = 0;
    int4 sg = make_int4(0, 0, 0, 0);
    ProdOp po{};
    if (s < seg_hi) {
      sg = p.segs[s];
      gpt = p.ops[sg.x].gpt;
      ng = sg.z * gpt;
      load_prod_op(p.ops + sg.x, po);
    }
    int x = lane, q = 0, slot = 0;
    int i = 0, gi = lane;  // x's tile in the segment and group in the tile
    uint32_t phase = 0;
    bool ok = true;
    for (;;) {
      if (lane < kCW && s < seg_hi) {
        if (x < gs + ng && q > 0) {
          // Same segment: step 16 groups without a division.
          gi += kCW;
          while (gi >= gpt) {
            gi -= gpt;
            ++i;
          }
        } else {
          while (s < seg_hi && x >= gs + ng) {
            gs += ng;
            if (++s < seg_hi) {
              sg = p.segs[s];
              gpt = p.ops[sg.x].gpt;
              ng = sg.z * gpt;
              load_prod_op(p.ops + sg.x, po);
            }
          }
          if (s < seg_hi) {
            i = (x - gs) / gpt;
            gi = x - gs - i * gpt;
          }
        }
      }
      const bool valid = lane < kCW && s < seg_hi;
      if (__ballot_sync(0xffffffffu, valid) == 0u) break;
      const unsigned char *src_c = nullptr, *src_s = nullptr, *src_z = nullptr;
      uint32_t nc = 0, ns = 0, nz = 0;
      if (valid) {
        const ProdOp &op = po;
        const int vt = sg.y + i;
        const int wsel = op.paired ? (vt & 1) : 0;
        const int t = op.paired ? (vt >> 1) : vt;
        int c0, nch, b0, nbr;
        if (BS >= kChunkK) {
          c0 = gi * G::kCpg;
          nch = min(G::kCpg, op.K64 - c0);
          b0 = gi;
          nbr = 1;
        } else {
          c0 = gi;
          nch = 1;
          b0 = gi * G::kBpg;
          nbr = min(G::kBpg, op.nb - b0);
        }
        src_c = (wsel ? op.b[1] : op.b[0]) + ((size_t)t * op.K64 + c0) * kChunkBytes;
        nc = nch * kChunkBytes;
        src_s = (wsel ? op.s[1] : op.s[0]) + ((size_t)t * op.nb + b0) * kTileN * kEs;
        ns = nbr * kTileN * kEs;
        if (HAS_ZP) {
          // Whole 16-byte word pairs: the pair holding b0 (blocks of 64 and
          // more), or the even-aligned words of the chunk's blocks.
          const int zb = b0 & ~1;
          src_z = (wsel ? op.z[1] : op.z[0]) + ((size_t)t * op.nbz + zb) * 8;
          nz = (BS >= kChunkK ? 2 : min(G::kBpg, op.nbz - zb)) * 8;
        }
      }
      uint32_t bytes = nc + ns + nz;
#pragma unroll
      for (int o = 16; o; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      if (q >= p.nst) {
        int w = 1;
        if (lane == 0) w = chain_wait(p, empty + slot, phase ^ 1) ? 1 : 0;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
      }
      if (lane == 0) mbar_arrive_expect_tx(full + slot, bytes);
      __syncwarp();
      if (valid) {
        unsigned char *st = ring + slot * p.stage_bytes;
        bulk_copy_g2s(st + lane * kCB, src_c, nc, full + slot);
        bulk_copy_g2s(st + p.sc_off + lane * kSCB, src_s, ns, full + slot);
        if (HAS_ZP) bulk_copy_g2s(st + p.zp_off + lane * kZPB, src_z, nz, full + slot);
      }
      x += kCW;
      ++q;
      if (++slot == p.nst) {
        slot = 0;
        phase ^= 1;
      }
    }
    // Copies still in flight (only after an abort) land before the CTA
    // exits: wait, bounded, for the last stages issued.
    if (lane == 0) {
      const int first = q > p.nst ? q - p.nst : 0;
      for (int qq = first; qq < q; ++qq) {
        const int sl = qq % p.nst;
        if (!mbar_wait(full + sl, static_cast<uint32_t>((qq / p.nst) & 1)))
          record_fault(&g_fault_chain, kFaultChainWait);
      }
    }
    (void)ok;
  } else {
    // ---- consumers ---------------------------------------------------------------
    const int g = lane >> 2, t = lane & 3;
    const int M = p.M;
    const bool mok = g < M;
    const bool two = p.a_f32 != 0;
    const int lo_off = p.off_alo / 2;  // hi -> lo activations, in elements
    const uint16_t *arow = sA + (mok ? g : 0) * p.kp + 4 * t;
    const float *S0row = sS + (2 * t < M ? 2 * t : 0) * p.sg;
    const float *S1row = sS + (2 * t + 1 < M ? 2 * t + 1 : 0) * p.sg;
    bool fault = false;
    int x = warp, slot = 0, gs = 0;
    uint32_t phase = 0;
    uint2 bfrag = make_uint2(0, 0);

    for (int s = seg_lo; s < seg_hi; ++s) {
      const int r = s - seg_lo;
      // Descriptor fields are read from the cache where used, not held in
      // registers across the group loop.
      const int4 *sgp = sSegc + (r & 3);
      const OpDev *opp = sOpc + (r & 1);
      if (warp == 0) {
        // Prefetch: segment s + 2, and the op of segment s + 1 (its segment
        // arrived one step earlier). Each slot's previous reader finished
        // before the last barrier.
        if (lane == 0 && s + 2 < seg_hi) cp_async16(sSegc + ((r + 2) & 3), p.segs + s + 2);
        if (lane < kOpChunks && s + 1 < seg_hi)
          cp_async16(reinterpret_cast<uint4 *>(sOpc + ((r + 1) & 1)) + lane,
                     reinterpret_cast<const uint4 *>(p.ops + sSegc[(r + 1) & 3].x) + lane);
        cp_async_commit();
      }
      // Op fields live in registers: the barriers' memory clobbers would
      // otherwise reload them from global memory after every barrier.
      const int gpt = opp->gpt, ng = sgp->z * gpt;

      if (sgp->w & kSegWait) {
        // Dependencies, then the op's activations and block sums.
        if (tid == 0 && !fault) {
          for (int k = 0; k < kChainMaxDeps && !sh_fault; ++k) {
            const int d = opp->dep[k];
            if (d < 0) continue;
            const uint32_t target = static_cast<uint32_t>(p.ops[d].target);
            uint32_t it = 0;
            while (ld_relaxed_gpu(p.count + d) < target) {
              if (++it > kDepSpinLimit) {
                chain_abort(p);
                sh_fault = 1;
                break;
              }
              if ((it & 255u) == 0u && ld_volatile(p.ctl + 1)) {
                sh_fault = 1;
                break;
              }
            }
          }
          fence_acq_rel_gpu();
        }
        named_barrier_sync(kBarCons, kCT);
        fault = fault || sh_fault;
        const void *opA = opp->A;
        const int opK = opp->K;
        const bool avec = opp->a_vec != 0;
        const int ppr = ((opp->K64 * kChunkK + 255) / 256) * 32;  // 8-element pieces per row
        if (two)
          stage_rows<2, true, BS>(opA, opK, avec, M, ppr, p.kp, p.sg, sA, lo_off, sS, tid);
        else
          stage_rows<3, false, BS>(opA, opK, avec, M, ppr, p.kp, p.sg, sA, lo_off, sS, tid);
        named_barrier_sync(kBarCons, kCT);
      }

      // ---- this warp's groups of the segment ----
      int cur = -1;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      auto flush = [&](int i) {
        float *r = sRed + ((i * kCW + warp) * kTileN) * M;
        if (2 * t < M) {
          r[g * M + 2 * t] = acc[0];
          r[(g + 8) * M + 2 * t] = acc[2];
        }
        if (2 * t + 1 < M) {
          r[g * M + 2 * t + 1] = acc[1];
          r[(g + 8) * M + 2 * t + 1] = acc[3];
        }
      };
      int i = 0, gi = 0;  // x's tile in the segment and group in the tile
      if (x < gs + ng) {
        i = (x - gs) / gpt;
        gi = x - gs - i * gpt;
      }
      for (; x < gs + ng; x += kCW) {
        if (i != cur) {
          if (cur >= 0) flush(cur);
          acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
          cur = i;
        }
        // A warp that gave up (abort) neither computes nor releases slots:
        // the producer then stops at the first slot it cannot get, and every
        // copy it issued still lands before the CTA exits.
        if (!fault) fault = !__all_sync(0xffffffffu, chain_wait(p, full + slot, phase));
        if (!fault) {
          const unsigned char *st = ring + slot * p.stage_bytes;
          const unsigned char *wp = st + warp * kCB + lane * 16;
          const unsigned char *scp = st + p.sc_off + warp * kSCB;
          const unsigned char *zpp = st + p.zp_off + warp * kZPB;

          // Scale and zero point of block b (its slot bi in the group) on
          // the MMA sums d.
          auto correct = [&](int b, int bi, int zi, const float (&d)[4]) {
            float s0, s1, z0 = 136.f, z1 = 136.f;
            if (SF32) {
              const float *sc = reinterpret_cast<const float *>(scp) + bi * kTileN + g;
              s0 = sc[0];
              s1 = sc[8];
            } else {
              const uint16_t *sc = reinterpret_cast<const uint16_t *>(scp) + bi * kTileN + g;
              s0 = bf16_bits_to_f32(sc[0]);
              s1 = bf16_bits_to_f32(sc[8]);
            }
            if (HAS_ZP) {
              const uint2 zw = reinterpret_cast<const uint2 *>(zpp)[zi];
              z0 = static_cast<float>(128 + ((zw.x >> (4 * g)) & 15));
              z1 = static_cast<float>(128 + ((zw.y >> (4 * g)) & 15));
            }
            const float S0 = S0row[b], S1 = S1row[b];
            acc[0] = fmaf(s0, fmaf(-z0, S0, d[0]), acc[0]);
            acc[1] = fmaf(s0, fmaf(-z0, S1, d[1]), acc[1]);
            acc[2] = fmaf(s1, fmaf(-z1, S0, d[2]), acc[2]);
            acc[3] = fmaf(s1, fmaf(-z1, S1, d[3]), acc[3]);
          };
          // One 16-wide k step at absolute k offset ko.
          auto kstep = [&](uint32_t w, int ko, bool first, float (&d)[4]) {
            uint32_t wf[4];
            codes_to_bf16x2(w, wf);
            if (mok) bfrag = *reinterpret_cast<const uint2 *>(arow + ko);
            if (first) mma_bf16_16816_zero(d, wf, bfrag.x, bfrag.y);
            else mma_bf16_16816(d, wf, bfrag.x, bfrag.y);
            if (two) {
              if (mok) bfrag = *reinterpret_cast<const uint2 *>(arow + lo_off + ko);
              mma_bf16_16816(d, wf, bfrag.x, bfrag.y);
            }
          };

          if (BS >= kChunkK) {
            const int c0 = gi * G::kCpg;
            const int nch = min(G::kCpg, opp->K64 - c0);
            float d[4];
#pragma unroll
            for (int cc = 0; cc < G::kCpg; ++cc) {
              if (cc < nch) {
                const uint4 w4 = *reinterpret_cast<const uint4 *>(wp + cc * kChunkBytes);
                const int ko = (c0 + cc) * kChunkK;
                kstep(w4.x, ko, cc == 0, d);
                kstep(w4.y, ko + 16, false, d);
                kstep(w4.z, ko + 32, false, d);
                kstep(w4.w, ko + 48, false, d);
              }
            }
            correct(gi, 0, gi & 1, d);
          } else {
            const uint4 w4 = *reinterpret_cast<const uint4 *>(wp);
            const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
            const int b0 = gi * G::kBpg;
#pragma unroll
            for (int bb = 0; bb < G::kBpg; ++bb) {
              float d[4];
#pragma unroll
              for (int jj = 0; jj < G::kSpb; ++jj)
                kstep(wv[bb * G::kSpb + jj], gi * kChunkK + 16 * (bb * G::kSpb + jj), jj == 0,
                      d);
              if (b0 + bb < opp->nb) correct(b0 + bb, bb, bb, d);
            }
          }
        }
        __syncwarp();
        if (lane == 0 && !fault) mbar_arrive(empty + slot);
        if (++slot == p.nst) {
          slot = 0;
          phase ^= 1;
        }
        gi += kCW;
        while (gi >= gpt) {
          gi -= gpt;
          ++i;
        }
      }
      if (cur >= 0) flush(cur);
      named_barrier_sync(kBarCons, kCT);
      const int opN = opp->N, paired = opp->paired;
      void *opY = opp->Y;
      const float *bias0 = opp->bias[0], *bias1 = opp->bias[1];

      // ---- fixed-order reduction over the warps, bias, store ----
      if (!fault) {
        const int outs_t = paired ? sgp->z / 2 : sgp->z;  // output tiles of the segment
        const int t_first = paired ? sgp->y / 2 : sgp->y;
        const int total = outs_t * kTileN * M;
        for (int e = tid; e < total; e += kCT) {
          const int m = e % M, r = (e / M) % kTileN, io = e / (M * kTileN);
          const int n = (t_first + io) * kTileN + r;
          if (n >= opN) continue;
          auto sum_tile = [&](int i) {
            const float *rr = sRed + (i * kCW * kTileN + r) * M + m;
            float v = 0.f;
            if (gpt >= kCW) {
              for (int w = 0; w < kCW; ++w) v += rr[w * kTileN * M];
            } else {
              const int f = gs + i * gpt;  // the tile's first group in the stream
              for (int k = 0; k < gpt; ++k) v += rr[((f + k) & (kCW - 1)) * kTileN * M];
            }
            return v;
          };
          if (paired) {
            float vg = sum_tile(2 * io), vu = sum_tile(2 * io + 1);
            if (bias0) vg += __ldg(bias0 + n);
            if (bias1) vu += __ldg(bias1 + n);
            store_out(opY, opN, two, m, n, vg / (1.f + expf(-vg)) * vu);
          } else {
            float v = sum_tile(io);
            if (bias0) v += __ldg(bias0 + n);
            store_out(opY, opN, two, m, n, v);
          }
        }
      }
      if (warp == 0) cp_async_wait_all();  // the next segment's descriptors
      named_barrier_sync(kBarCons, kCT);
      // The barrier orders every consumer's stores before thread 0's
      // device-scope release (barrier, then release: cumulative).
      if (tid == 0) {
        red_release_gpu_add(p.count + sgp->x, 1u);
      }
      gs += ng;
    }
  }

  // The last CTA to finish resets the counters for the next launch.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned int done = atomicAdd(p.ctl, 1u);
    if (done == gridDim.x - 1) {
      for (int i = 0; i < p.n_ops; ++i) p.count[i] = 0u;
      p.ctl[1] = 0u;
      __threadfence();
      p.ctl[0] = 0u;
    }
  }
}

// ---- host: layout, schedule, launch ------------------------------------------------

size_t a16(size_t x) { return (x + 15) & ~size_t(15); }
size_t a128(size_t x) { return (x + 127) & ~size_t(127); }

struct SmemLayout {
  int kp, sg, tmax, stage_bytes, sc_off, zp_off;
  int off_alo, off_s, off_red, off_opc, off_bar, off_ring;
};

// Shared-memory layout for the shape and the largest K; nst stages follow.
SmemLayout smem_layout(const ChainShape &sh, int kmax) {
  SmemLayout L{};
  const int es = sh.scale_f32 ? 4 : 2;
  const int cpg = sh.bs >= kChunkK ? sh.bs / kChunkK : 1;
  const int bpg = sh.bs >= kChunkK ? 1 : kChunkK / sh.bs;
  const int cb = cpg * kChunkBytes, scb = bpg * kTileN * es;
  const int zpb = sh.bs >= kChunkK ? 16 : bpg * 8;
  const int64_t staged = ceil_div(ceil_div(kmax, kChunkK) * kChunkK, 256) * 256;
  L.kp = static_cast<int>(staged) + 16;
  L.sg = static_cast<int>(staged / sh.bs);
  L.tmax = std::max(2, (8 / sh.M) & ~1);
  L.sc_off = kCW * cb;
  L.zp_off = static_cast<int>(a16(L.sc_off + size_t(kCW) * scb));
  L.stage_bytes = static_cast<int>(a128(L.zp_off + (sh.has_zp ? size_t(kCW) * zpb : 0)));
  size_t off = a16(size_t(sh.M) * L.kp * 2);
  L.off_alo = static_cast<int>(off);
  if (sh.a_f32) off += a16(size_t(sh.M) * L.kp * 2);
  L.off_s = static_cast<int>(off);
  off += a16(size_t(sh.M) * L.sg * 4);
  L.off_red = static_cast<int>(off);
  off += a16(size_t(L.tmax) * kCW * kTileN * sh.M * 4);
  L.off_opc = static_cast<int>(off);
  off += kOpCacheBytes;
  L.off_bar = static_cast<int>(off);
  off += 2 * kMaxStagesChain * 8;
  L.off_ring = static_cast<int>(a128(off));
  return L;
}

// Ring depth and CTAs per SM for a layout: two CTAs per SM when three
// stages fit in half the SM, else one with a deeper ring.
bool ring_for(const SmemLayout &L, int &per_sm, int &nst) {
  if (L.off_ring + 3 * L.stage_bytes <= kBudget2) {
    per_sm = 2;
    nst = std::min(8, (kBudget2 - L.off_ring) / L.stage_bytes);
    return true;
  }
  per_sm = 1;
  nst = std::min(kMaxStagesChain, (kBudget1 - L.off_ring) / L.stage_bytes);
  return nst >= 2;
}

template <int BS, bool HAS_ZP, bool SF32>
cudaError_t configure_one(int smem, int *occ) {
  auto kernel = chain_kernel<BS, HAS_ZP, SF32>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kBudget1);
  if (e != cudaSuccess) return e;
  if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kernel, kThreadsChain, smem);
  return cudaSuccess;
}

template <int BS, bool HAS_ZP, bool SF32>
cudaError_t launch_chain_one(const ChainParams &p, const ChainGeom &g, cudaStream_t stream) {
  static std::atomic<unsigned long long> configured{0};
  if (const cudaError_t e =
          ensure_smem_limit(chain_kernel<BS, HAS_ZP, SF32>, kBudget1, configured);
      e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid, 1, 1);
  cfg.blockDim = dim3(kThreadsChain, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chain_kernel<BS, HAS_ZP, SF32>, p);
}

template <int BS>
cudaError_t dispatch_flags(const ChainShape &sh, const ChainParams *p, const ChainGeom &g,
                           cudaStream_t stream, int *occ) {
  if (sh.has_zp) {
    if (sh.scale_f32)
      return p ? launch_chain_one<BS, true, true>(*p, g, stream)
               : configure_one<BS, true, true>(g.smem, occ);
    return p ? launch_chain_one<BS, true, false>(*p, g, stream)
             : configure_one<BS, true, false>(g.smem, occ);
  }
  if (sh.scale_f32)
    return p ? launch_chain_one<BS, false, true>(*p, g, stream)
             : configure_one<BS, false, true>(g.smem, occ);
  return p ? launch_chain_one<BS, false, false>(*p, g, stream)
           : configure_one<BS, false, false>(g.smem, occ);
}

// Launches (p != nullptr) or queries occupancy (p == nullptr).
cudaError_t dispatch(const ChainShape &sh, const ChainParams *p, const ChainGeom &g,
                     cudaStream_t stream, int *occ) {
  switch (sh.bs) {
    case 16: return dispatch_flags<16>(sh, p, g, stream, occ);
    case 32: return dispatch_flags<32>(sh, p, g, stream, occ);
    case 64: return dispatch_flags<64>(sh, p, g, stream, occ);
    case 128: return dispatch_flags<128>(sh, p, g, stream, occ);
    case 256: return dispatch_flags<256>(sh, p, g, stream, occ);
    default: return cudaErrorNotSupported;
  }
}

void plan_offsets(ChainGeom &g) {
  size_t off = a16(size_t(g.n_ops) * sizeof(OpDev));
  g.off_ctaseg = off;
  off = a16(off + size_t(g.grid + 1) * sizeof(int));
  g.off_segs = off;
  off = a16(off + size_t(g.n_segs) * sizeof(int4));
  g.off_count = off;
  off = a16(off + size_t(g.n_ops) * sizeof(unsigned int));
  g.off_ctl = off;
  g.plan_bytes = off + 4 * sizeof(unsigned int);
}

// Cost model of the list schedule, in units of one 64-wide chunk streamed
// and multiplied by one consumer warp.
constexpr double kDepLatency = 4.0;   // release -> acquire -> activations staged
constexpr double kSegOverhead = 1.0;  // reduction, stores, release

struct Seg {
  int op, tile0, ntiles, flags;
};

}  // namespace

// Plan storage owned by the library, for callers that cannot allocate
// device memory (mnb_chain_run_noalloc). Every GPU that loads the library
// holds this array until the process exits; every call shares it.
constexpr size_t kChainScratchBytes = size_t(1) << 20;
constexpr int kScratchDevices = 64;
static __device__ __align__(256) unsigned char g_chain_scratch[kChainScratchBytes];

cudaError_t chain_scratch(void **ptr, size_t *bytes) {
  // The array's host-side name is not a device address: look the address
  // up once per device, with that device current.
  static std::mutex mu;
  static void *addr[kScratchDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *a = nullptr;
    e = cudaGetSymbolAddress(&a, g_chain_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = a;
  }
  *ptr = addr[dev];
  *bytes = kChainScratchBytes;
  return cudaSuccess;
}

cudaError_t chain_take_fault(unsigned int *out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fault_chain, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fault_chain, &zero, sizeof(unsigned int));
  return e;
}

bool chain_geom(const ChainShape &sh, int n_ops, int kmax, int grid, int per_sm, int nst,
                int n_segs, ChainGeom &g) {
  if (sh.M < 1 || sh.M > kChainMaxM || kmax < 1 || grid < 1 || n_ops < 1 || n_segs < 0)
    return false;
  const SmemLayout L = smem_layout(sh, kmax);
  int ps = 0, ns = 0;
  // The occupancy query may have granted fewer CTAs per SM than the layout
  // allows; the ring depth is the layout's.
  if (!ring_for(L, ps, ns) || per_sm < 1 || per_sm > ps || ns != nst) return false;
  g.grid = grid;
  g.per_sm = per_sm;
  g.nst = nst;
  g.tmax = L.tmax;
  g.kmax = kmax;
  g.smem = L.off_ring + nst * L.stage_bytes;
  g.n_ops = n_ops;
  g.n_segs = n_segs;
  plan_offsets(g);
  return true;
}

cudaError_t chain_plan(const ChainOp *ops, int n, const ChainShape &sh, ChainGeom &g,
                       std::vector<unsigned char> *image) {
  int64_t kmax = 0;
  for (int j = 0; j < n; ++j) kmax = std::max(kmax, ops[j].K);
  const SmemLayout L = smem_layout(sh, static_cast<int>(kmax));
  int per_sm = 0, nst = 0;
  if (!ring_for(L, per_sm, nst)) return cudaErrorNotSupported;
  g.per_sm = per_sm;
  g.nst = nst;
  g.tmax = L.tmax;
  g.kmax = static_cast<int>(kmax);
  g.smem = L.off_ring + nst * L.stage_bytes;
  g.n_ops = n;
  int occ = 0;
  cudaError_t e = dispatch(sh, nullptr, g, nullptr, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorNotSupported;
  g.per_sm = std::min(per_sm, occ);
  g.grid = sm_count() * g.per_sm;
  chain_schedule(ops, n, sh, g, image);
  return cudaSuccess;
}

void chain_schedule(const ChainOp *ops, int n, const ChainShape &sh, ChainGeom &g,
                    std::vector<unsigned char> *image) {
  const int G = g.grid;

  // List schedule: tiles of op j go, one unit at a time (a pair's gate and
  // up tile together), to the CTA that would finish the unit first.
  const int cpg = sh.bs >= kChunkK ? sh.bs / kChunkK : 1;
  std::vector<double> avail(G, 0.0), done(n, 0.0);
  std::vector<std::vector<Seg>> per_cta(G);
  std::vector<const void *> staged_a(G, nullptr);
  std::vector<int> staged_op(G, -1);
  std::vector<int> target(n, 0), cnt(G);
  using Item = std::pair<double, int>;
  for (int j = 0; j < n; ++j) {
    const ChainOp &o = ops[j];
    double ready = 0.0;
    for (int k = 0; k < kChainMaxDeps; ++k)
      if (o.dep[k] >= 0) ready = std::max(ready, done[o.dep[k]] + kDepLatency);
    const int64_t N16 = ceil_div(o.N, kTileN), K64 = ceil_div(o.K, kChunkK);
    const int gpt = static_cast<int>(sh.bs >= kChunkK ? ceil_div(o.K, sh.bs) : K64);
    const int vpu = o.paired ? 2 : 1;  // virtual tiles per unit
    const double cost = double(vpu) * gpt * std::min<int64_t>(cpg, K64) / kCW;
    std::priority_queue<Item, std::vector<Item>, std::greater<Item>> pq;
    for (int c = 0; c < G; ++c) {
      cnt[c] = 0;
      pq.push({std::max(avail[c], ready) + cost, c});
    }
    for (int64_t u = 0; u < N16; ++u) {
      const Item it = pq.top();
      pq.pop();
      ++cnt[it.second];
      pq.push({it.first + cost, it.second});
    }
    const int tmax_units = std::max(1, g.tmax / vpu);
    int64_t next = 0;  // next unit
    double fin = 0.0;
    for (int c = 0; c < G; ++c) {
      if (cnt[c] == 0) continue;
      // Same activations and same deps as the op staged last: no new wait.
      bool same = staged_op[c] >= 0 && staged_a[c] == o.A && ops[staged_op[c]].K == o.K;
      if (same)
        for (int k = 0; k < kChainMaxDeps; ++k) same = same && ops[staged_op[c]].dep[k] == o.dep[k];
      double tc = std::max(avail[c], ready);
      for (int left = cnt[c]; left > 0;) {
        const int take = std::min(left, tmax_units);
        Seg sgm{j, static_cast<int>(next * vpu), take * vpu, same ? 0 : kSegWait};
        same = true;
        per_cta[c].push_back(sgm);
        ++target[j];
        next += take;
        left -= take;
        tc += take * cost + kSegOverhead;
      }
      staged_op[c] = j;
      staged_a[c] = o.A;
      avail[c] = tc;
      fin = std::max(fin, tc);
    }
    done[j] = fin;
  }
  int n_segs = 0;
  for (int c = 0; c < G; ++c) n_segs += static_cast<int>(per_cta[c].size());
  g.n_segs = n_segs;
  plan_offsets(g);
  if (!image) return;

  image->assign(g.plan_bytes, 0);
  unsigned char *base = image->data();
  OpDev *od = reinterpret_cast<OpDev *>(base);
  for (int j = 0; j < n; ++j) {
    const ChainOp &o = ops[j];
    OpDev d{};
    for (int w = 0; w < 2; ++w) {
      d.b[w] = static_cast<const unsigned char *>(o.b[w]);
      d.s[w] = static_cast<const unsigned char *>(o.s[w]);
      d.z[w] = static_cast<const unsigned char *>(o.z[w]);
      d.bias[w] = o.bias[w];
    }
    d.A = o.A;
    d.Y = o.Y;
    d.N = static_cast<int>(o.N);
    d.K = static_cast<int>(o.K);
    d.K64 = static_cast<int>(ceil_div(o.K, kChunkK));
    d.nb = static_cast<int>(ceil_div(o.K, sh.bs));
    d.nbz = static_cast<int>(ceil_div(d.nb, 2) * 2);
    d.paired = o.paired ? 1 : 0;
    d.gpt = sh.bs >= kChunkK ? d.nb : d.K64;
    d.target = target[j];
    const int vec = sh.a_f32 ? 4 : 8;
    d.a_vec = (reinterpret_cast<uintptr_t>(o.A) % 16 == 0) && (o.K % vec == 0);
    for (int k = 0; k < kChainMaxDeps; ++k) d.dep[k] = o.dep[k];
    std::memcpy(od + j, &d, sizeof d);
  }
  int *cta_seg = reinterpret_cast<int *>(base + g.off_ctaseg);
  int4 *segs = reinterpret_cast<int4 *>(base + g.off_segs);
  int at = 0;
  for (int c = 0; c < G; ++c) {
    cta_seg[c] = at;
    for (const Seg &s : per_cta[c]) segs[at++] = make_int4(s.op, s.tile0, s.ntiles, s.flags);
  }
  cta_seg[G] = at;
}

cudaError_t chain_launch(const void *plan, const ChainShape &sh, const ChainGeom &g,
                         cudaStream_t stream) {
  const SmemLayout L = smem_layout(sh, g.kmax);
  unsigned char *b = static_cast<unsigned char *>(const_cast<void *>(plan));
  ChainParams p{};
  p.ops = reinterpret_cast<const OpDev *>(b);
  p.cta_seg = reinterpret_cast<const int *>(b + g.off_ctaseg);
  p.segs = reinterpret_cast<const int4 *>(b + g.off_segs);
  p.count = reinterpret_cast<unsigned int *>(b + g.off_count);
  p.ctl = reinterpret_cast<unsigned int *>(b + g.off_ctl);
  p.n_ops = g.n_ops;
  p.M = sh.M;
  p.a_f32 = sh.a_f32 ? 1 : 0;
  p.kp = L.kp;
  p.sg = L.sg;
  p.nst = g.nst;
  p.stage_bytes = L.stage_bytes;
  p.sc_off = L.sc_off;
  p.zp_off = L.zp_off;
  p.off_alo = L.off_alo;
  p.off_s = L.off_s;
  p.off_red = L.off_red;
  p.off_opc = L.off_opc;
  p.off_bar = L.off_bar;
  p.off_ring = L.off_ring;
  return dispatch(sh, &p, g, stream, nullptr);
}

}  // namespace mnb
