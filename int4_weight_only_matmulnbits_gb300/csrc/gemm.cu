// Tensor-core (tcgen05 / TMEM) MatMulNBits kernel for larger M (prefill).
//
// Computes Y[m,n] = sum_k A[m,k] (q[n,k] - z[n,b]) s[n,b] + bias[n] with
// bf16 activations on the prepacked layout of mnb_common.cuh. It follows
// the page "Qwen3 CPU Inference Critical Path", section "Prepared weight-only
// plan", int4_gemm: activation panels are packed (here: TMA-staged tiles),
// weight blocks are reused across the rows of a tile, and the full weight
// matrix is never expanded: only one 128 x 64 bf16 slice per pipeline stage
// exists, in shared memory.
//
// GB300 mapping (one CTA per (128*MH) x 128 output tile, MH = 1 or 2 halves
// of 128 rows; two CTAs per SM so one CTA's epilogue overlaps the other's
// main loop):
//  * warp 0, one thread: TMA producer. Per 64-wide k stage it loads the A
//    tile ((128*MH) x 64 bf16, 128-byte swizzle), the 128 x 64 packed codes
//    of the stage and their scales and zero points into the input ring,
//    completing on full[s].
//  * warps 2-9, one 16-row weight tile each: dequantise the stage's codes,
//    w = (q - z) * s, into two bf16 B tiles, hi = w rounded and lo = the
//    remainder (hi + lo == w for bf16 scales, within 2^-16 |w| for fp32
//    scales), in the K-major, 128-byte-swizzled layout tcgen05.mma reads;
//    fence the writes to the async proxy and arrive on bfull[b]. Weight rows
//    g and g+8 of a 16-row tile go to B rows 2g and 2g+1, which keeps every
//    warp's stores free of bank conflicts; the epilogue maps the columns
//    back.
//  * warp 1: allocates the TMEM accumulators (128 lanes x 128*MH fp32
//    columns); one thread issues 8*MH tcgen05.mma (M=128, N=128, K=16) per
//    stage, the MH halves of A sharing the hi and the lo tile, and commits
//    each stage to empty[s] and bempty[b], the last one to acc_full.
//  * warps 2-9 then read the accumulators with tcgen05.ld (each warp its
//    TMEM lane quarter and half of the columns), add the bias (staged in
//    shared memory), round to bf16 and store Y.
//  * Gated-MLP pairs (the fusion "gate projection, SiLU, and gate/up
//    multiplication"): a CTA covers 64 output columns; its B tile holds 64
//    rows of the gate weight and the same 64 rows of the up weight, and the
//    epilogue stores silu(g) * u from accumulator columns c and 64 + c.
//  * Shapes with too few output tiles to fill the GPU split K over a
//    cluster of up to 8 CTAs (128-row tiles): each CTA accumulates its k
//    range, parks the accumulator in its own shared memory (the drained
//    operand rings), and after a cluster barrier each CTA reduces one column
//    slice of the tile over all ranks through distributed shared memory, in
//    rank order (bitwise reproducible), then adds the bias and stores.
// Every mbarrier wait is bounded; a wait that runs out records a fault bit
// and the kernel abandons the tile.
#include <cuda_bf16.h>

#include <algorithm>

#include "mnb_common.cuh"
#include "mnb_launch.h"
#include "umma.cuh"

namespace mnb {

__device__ unsigned int g_fault_gemm = 0;

namespace {

constexpr int kBH = 128;  // rows of one A half (the MMA's M)
constexpr int kBN = 128;
constexpr int kBK = 64;  // one chunk of the packed layout
constexpr int kBStagesTf32 = 2;  // dequantised B tiles of the tf32 kernel
constexpr int kDqWarps = 8;
constexpr int kThreads = 32 * (2 + kDqWarps);
constexpr int kTilesN = kBN / kTileN;
constexpr int kAHalfBytes = kBH * kBK * 2;  // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;  // 16 KB: one bf16 B tile
// A B slot of the bf16 kernels holds two tiles, hi and lo (see dequant_pair).
constexpr int kBSlotBytes = 2 * kBTileBytes;
constexpr int kCodeBytes = kTilesN * kChunkBytes;  // 4 KB
constexpr int kBarEpi = 1;  // named barrier of the dequantisation/epilogue warps

struct GemmParams {
  CUtensorMap tma;  // A: {K, M} bf16, box {64, 128*MH}, 128-byte swizzle
  CUtensorMap tmw;  // codes: {128 words, K64, N16}, box {128, 1, 8}
  CUtensorMap tms;  // scales: {16 scales as words, nb, N16}, box {.., bpc, 8}
  CUtensorMap tmz;  // zero points: {4 words, nbz/2, N16}, box {4, ppc, 8}
  CUtensorMap tmw2, tms2, tmz2;  // a pair's up weight (boxes of 4 tiles, as the gate's)
  CUtensorMap tmy;  // Y: {N, M} bf16, box {64, 128*MH}, 128-byte swizzle (when y_tma)
  // Stream-K schedule (gemm_sk_kernel): units = tiles * K64 (tile, k stage)
  // pairs split evenly over sk_ctas CTAs; tiles_n output tiles along N; ws
  // holds two 256 x 128 fp32 partial tiles per CTA (its first and its last
  // piece), count one arrival counter per CTA (for the split tile it heads).
  int64_t units;
  int sk_ctas, tiles_n;
  float *ws;
  unsigned int *count;
  const float *bias, *bias2;
  void *Y;
  int M, N, K64;
  int y_tma;  // the epilogue stages the tile in shared memory and stores it with TMA
  int has_zp;
  int y_vec;  // Y rows are 16-byte aligned: 16-byte stores
  int sc_bytes, zp_bytes;  // per stage
  int ksplit, kps;  // CTAs splitting K (cluster along z), k stages per CTA
  int paired;       // gate (tiles 0-3 of the B tile) and up (tiles 4-7)
  // RMS-normalized activations (the fusion "RMSNorm into packed projection
  // input"): gamma[k] multiplies the dequantised weights (in fp32, before the
  // hi + lo split) and each output row is scaled by r[m] = 1 / sqrt(mean_k
  // A[m,k]^2 + eps), summed over the whole row from the staged tiles (needs
  // ksplit == 1).
  int norm;
  const float *gamma;  // [K] or null (1)
  float eps;
  int K;
  // Code-book weights (the bitsandbytes-style form; the CB instantiation):
  // w = code[q] * s with the 16 fp32 values here, no zero points.
  const float *code;
  int sc_up, zp_up;  // paired: byte offsets of the up halves in a stage's scales / zero points
};

// Shared-memory plan (offsets from a 1024-aligned base). The A tiles and the
// packed weights of a stage travel in separate rings: the small weight
// stream (codes, scales, zero points) runs further ahead, so a stage's B tile
// is dequantised while its A tile is still in flight.
// Two CTAs share an SM: each may use at most half of its 228 KB, less the
// 1 KB the runtime reserves per CTA and the 1 KB alignment slack.
constexpr int kSmemLimit2 = (228 * 1024) / 2 - 1024;

template <int MH, int BS, bool SF32>
struct Smem {
  static constexpr int kAStages = MH == 1 ? 3 : 2;  // A ring depth
  // Dequantised B slots (hi and lo tiles, 32 KB each): one. The dequantisation
  // of stage i + 1 then waits for the MMAs of stage i; the SM's other CTA
  // keeps the tensor core busy meanwhile.
  static constexpr int kBStages = 1;
  static constexpr int kATileBytes = MH * kAHalfBytes;
  static constexpr int kBpcS = BS < kBK ? kBK / BS : 1;
  // 8 tiles x the stage's blocks x 16 scales (a multiple of 128 bytes).
  static constexpr int kScBytes = kTilesN * kBpcS * kTileN * (SF32 ? 4 : 2);
  static constexpr int kZpBytes = 256;  // 8 tiles x up to 2 pairs x 16 bytes, or a pair's halves
  // Weight ring depth: 3 where it fits beside the A and B rings, else 2.
  static constexpr int kWBytes = kCodeBytes + kScBytes + kZpBytes;
  static constexpr int kFixed =
      kAStages * kATileBytes + kBStages * kBSlotBytes + kBN * 4 + 256 + 1024;
  static constexpr int kWStages = kFixed + 3 * kWBytes <= kSmemLimit2 ? 3 : 2;
  static constexpr int kA = 0;
  static constexpr int kB = kA + kAStages * kATileBytes;
  static constexpr int kCodes = kB + kBStages * kBSlotBytes;
  static constexpr int kSc = kCodes + kWStages * kCodeBytes;
  static constexpr int kZp = kSc + kWStages * kScBytes;
  static constexpr int kBias = kZp + kWStages * kZpBytes;
  static constexpr int kCodeTab = kBias + kBN * 4;  // 16 fp32 code-book values
  static constexpr int kBar = kCodeTab + 64;
  // ... + acc_full, and acc_empty (the stream-K kernel's drained accumulator)
  static constexpr int kNumBars = 2 * kAStages + 2 * kWStages + 2 * kBStages + 2;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kTotal = kTmemSlot + 16;
};
static_assert(Smem<1, 16, true>::kTotal + 1024 <= kSmemLimit2, "two CTAs per SM");
static_assert(Smem<2, 16, true>::kTotal + 1024 <= kSmemLimit2, "two CTAs per SM");
static_assert(Smem<2, 128, false>::kWStages == 3, "three weight stages for the common case");
// A split-K CTA parks its 128 x 128 fp32 accumulator in the drained A and B rings.
static_assert(Smem<1, 16, true>::kCodes >= kBH * kBN * 4, "split-K parking space");

// Instruction descriptor: D fp32, A and B bf16, both K-major, M = 128, N = kBN.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBH >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(static_cast<int>(accumulate))
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

template <int BS, bool HAS_ZP, bool SF32, int MH, bool CB = false>
__global__ void __launch_bounds__(kThreads, 2) gemm_kernel(const __grid_constant__ GemmParams p) {
  using S = Smem<MH, BS, SF32>;
  static_assert(!(CB && HAS_ZP), "code-book weights carry no zero points");
  constexpr int kAStages = S::kAStages, kWStages = S::kWStages, kBStages = S::kBStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles. The offset is added
  // to the shared array itself (not through an integer cast) so that every
  // access below stays a shared-memory access rather than a generic one.
  unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *afull = reinterpret_cast<uint64_t *>(smem + S::kBar);
  uint64_t *aempty = afull + kAStages;
  uint64_t *wfull = aempty + kAStages;
  uint64_t *wempty = wfull + kWStages;
  uint64_t *bfull = wempty + kWStages;
  uint64_t *bempty = bfull + kBStages;
  uint64_t *acc_full = bempty + kBStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::kTmemSlot);
  float *sBias = reinterpret_cast<float *>(smem + S::kBias);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * (kBH * MH);
  const int nt0 = blockIdx.x * kTilesN;  // first 16-row weight tile
  constexpr int kBpc = BS < kBK ? kBK / BS : 1;
  // This CTA's k stages (its rank in the K-splitting cluster is blockIdx.z).
  const int kb0 = blockIdx.z * p.kps;
  const int nk = min(p.K64 - kb0, p.kps);

  if (tid == 0) {
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(afull + i, 1);
      // Normalized rows: the dequantisation warps' sum-of-squares pass reads
      // the A tile too, and arrives when done.
      mbar_init(aempty + i, p.norm ? 1 + kDqWarps : 1);
    }
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(wfull + i, 1);
      mbar_init(wempty + i, kDqWarps);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(bfull + i, kDqWarps);
      mbar_init(bempty + i, 1);
    }
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kBN * MH)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Dependents may launch once every CTA of this grid has started; A is the
  // upstream kernel's output.
  grid_dependents_launch();
  grid_dependency_wait();

  bool fault = false;
  if (warp == 0) {
    if (lane == 0) {
      // A tiles.
      for (int i = 0; i < nk; ++i) {
        const int s = i % kAStages, kb = kb0 + i;
        if (i >= kAStages && !mbar_wait(aempty + s, ((i / kAStages) - 1) & 1)) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          break;
        }
        mbar_arrive_expect_tx(afull + s, S::kATileBytes);
        tma_load_2d(smem + S::kA + s * S::kATileBytes, &p.tma, kb * kBK, m0, afull + s);
      }
    } else if (lane == 1) {
      // Packed weights: codes, scales and zero points of the stage.
      for (int i = 0; i < nk; ++i) {
        const int s = i % kWStages, kb = kb0 + i;
        if (i >= kWStages && !mbar_wait(wempty + s, ((i / kWStages) - 1) & 1)) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          break;
        }
        uint64_t *bar = wfull + s;
        mbar_arrive_expect_tx(bar, kCodeBytes + p.sc_bytes + p.zp_bytes);
        const int blk = (kb * kBK) / BS;
        unsigned char *cd = smem + S::kCodes + s * kCodeBytes;
        unsigned char *sd = smem + S::kSc + s * S::kScBytes;
        unsigned char *zd = smem + S::kZp + s * S::kZpBytes;
        if (p.paired) {
          const int t0 = blockIdx.x * (kTilesN / 2);  // 4 tiles of each weight
          tma_load_3d(cd, &p.tmw, 0, kb, t0, bar);
          tma_load_3d(cd + (kTilesN / 2) * kChunkBytes, &p.tmw2, 0, kb, t0, bar);
          tma_load_3d(sd, &p.tms, 0, blk, t0, bar);
          tma_load_3d(sd + p.sc_up, &p.tms2, 0, blk, t0, bar);
          if (HAS_ZP) {
            tma_load_3d(zd, &p.tmz, 0, blk >> 1, t0, bar);
            tma_load_3d(zd + p.zp_up, &p.tmz2, 0, blk >> 1, t0, bar);
          }
        } else {
          tma_load_3d(cd, &p.tmw, 0, kb, nt0, bar);
          tma_load_3d(sd, &p.tms, 0, blk, nt0, bar);
          if (HAS_ZP) tma_load_3d(zd, &p.tmz, 0, blk >> 1, nt0, bar);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % kAStages, b = i % kBStages;
        if (!mbar_wait(afull + s, (i / kAStages) & 1) ||
            !mbar_wait(bfull + b, (i / kBStages) & 1)) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          fault = true;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_addr(smem + S::kA + s * S::kATileBytes);
        const uint32_t b_base = smem_addr(smem + S::kB + b * kBSlotBytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
          for (int h = 0; h < MH; ++h) {
            const uint64_t ad = smem_desc_sw128(a_base + h * kAHalfBytes + kk * 32);
            umma_bf16(tmem + h * kBN, ad, smem_desc_sw128(b_base + kk * 32), i > 0 || kk > 0);
            umma_bf16(tmem + h * kBN, ad, smem_desc_sw128(b_base + kBTileBytes + kk * 32), true);
          }
        umma_commit(aempty + s);
        umma_commit(bempty + b);
      }
      if (!fault) umma_commit(acc_full);
    }
  } else {
    // ---- dequantisation warps (2..9), then the epilogue --------------------
    const int tile = warp - 2;  // this warp's 16-row weight tile of the stage
    const int g = lane >> 2, t = lane & 3;
    // Weight rows g and g + 8 of the tile go to B rows 2g and 2g + 1.
    const int r0 = tile * kTileN + 2 * g;
    {
      const int e = tid - 64;  // 0..255
      if (e < kBN) {
        if (p.paired) {  // gate biases, then up biases, of the CTA's 64 columns
          const int n = blockIdx.x * (kBN / 2) + (e & (kBN / 2 - 1));
          const float *b = e < kBN / 2 ? p.bias : p.bias2;
          sBias[e] = (b && n < p.N) ? __ldg(b + n) : 0.f;
        } else {
          const int n = nt0 * kTileN + e;
          sBias[e] = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.f;
        }
      }
    }
    // RMS normalization: thread e of the dequantisation warps takes A row
    // nrow of the tile (two threads a row for 128-row tiles), chunks nc0 ..
    // nc0 + kNormChunks - 1 of every stage.
    constexpr int kNormChunks = MH == 1 ? 4 : 8;
    const int ne = tid - 64;
    const int nrow = MH == 1 ? (ne >> 1) : ne, nc0 = MH == 1 ? (ne & 1) * 4 : 0;
    float nss = 0.f;
    float *sCode = reinterpret_cast<float *>(smem + S::kCodeTab);
    if (CB) {
      // Every dequantisation warp writes the same 16 values (identical
      // stores), so its own reads after __syncwarp need no CTA barrier.
      if (lane < 16) sCode[lane] = __ldg(p.code + lane);
      __syncwarp();
    }
    for (int i = 0; i < nk; ++i) {
      const int s = i % kWStages, bslot = i % kBStages, kb = kb0 + i;
      if (!mbar_wait(wfull + s, (i / kWStages) & 1) ||
          (i >= kBStages && !mbar_wait(bempty + bslot, ((i / kBStages) - 1) & 1))) {
        record_fault(&g_fault_gemm, kFaultGemmWait);
        fault = true;
        break;
      }
      const unsigned char *codes = smem + S::kCodes + s * kCodeBytes;
      const unsigned char *sc = smem + S::kSc + s * S::kScBytes;
      const uint2 *zp = reinterpret_cast<const uint2 *>(smem + S::kZp + s * S::kZpBytes);
      unsigned char *btile = smem + S::kB + bslot * kBSlotBytes;
      const int blk0 = (kb * kBK) / BS;
      // Scales and zero points of weight rows g, g + 8 for the stage's
      // blocks (zero-filled past the last block).
      uint32_t sb0[kBpc], sb1[kBpc], zc0[kBpc], zc1[kBpc];
      float sf0[kBpc], sf1[kBpc];
#pragma unroll
      for (int bi = 0; bi < kBpc; ++bi) {
        if (SF32) {
          const float *s4 = reinterpret_cast<const float *>(sc) + (tile * kBpc + bi) * kTileN;
          sf0[bi] = s4[g];
          sf1[bi] = s4[g + 8];
          sb0[bi] = sb1[bi] = 0;
        } else {
          const uint16_t *s2 = reinterpret_cast<const uint16_t *>(sc) + (tile * kBpc + bi) * kTileN;
          sb0[bi] = s2[g] * 0x10001u;
          sb1[bi] = s2[g + 8] * 0x10001u;
          sf0[bi] = sf1[bi] = 0.f;
        }
        zc0[bi] = zc1[bi] = 0x43084308u;  // bf16 136 = 128 + 8
        if (HAS_ZP) {
          const int b = blk0 + bi;
          const int pairs = BS < 32 ? 2 : 1;
          // A pair's up tiles (4-7) start at zp_up bytes.
          const int zt = (p.paired && tile >= kTilesN / 2)
                             ? p.zp_up / 16 + (tile - kTilesN / 2) * pairs
                             : tile * pairs;
          const uint2 zw = zp[(zt + (BS < 32 ? bi >> 1 : 0)) * 2 + (b & 1)];
          zc0[bi] = (0x4300u | ((zw.x >> (4 * g)) & 15)) * 0x10001u;
          zc1[bi] = (0x4300u | ((zw.y >> (4 * g)) & 15)) * 0x10001u;
        }
      }
      // Normalized rows: gamma of this lane's 16 k positions of the stage
      // (k = 16 j + 4 t + e), folded into the weights below.
      float gm[4][4];
      if (p.norm) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = kb * kBK + 16 * j + 4 * t + e;
            gm[j][e] = p.gamma ? (k < p.K ? __ldg(p.gamma + k) : 0.f) : 1.f;
          }
      }
      const uint4 w4 = *reinterpret_cast<const uint4 *>(codes + tile * kChunkBytes + lane * 16);
      const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int bi = BS < kBK ? (16 * j) / BS : 0;  // block of this k step
        uint32_t h00, l00, h02, l02, h10, l10, h12, l12;
        if (CB) {
          // Register i of the affine path holds the codes at bits 4i and
          // 16 + 4i (rows g for even i, g + 8 for odd i): here their code-book
          // values times the row's scale, in fp32, split hi + lo.
          const float s0 = SF32 ? sf0[bi] : bf16_bits_to_f32(sb0[bi] & 0xFFFFu);
          const float s1 = SF32 ? sf1[bi] : bf16_bits_to_f32(sb1[bi] & 0xFFFFu);
          uint32_t hv[4], lv[4];
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) {
            const uint32_t x = wv[j] >> (4 * ii);
            const float sc2 = (ii & 1) ? s1 : s0;
            const float w0 = sCode[x & 15u] * sc2, w1 = sCode[(x >> 16) & 15u] * sc2;
            hv[ii] = f32x2_to_bf16x2(w0, w1);
            lv[ii] = f32x2_to_bf16x2(w0 - bf16_bits_to_f32(hv[ii] & 0xFFFFu),
                                     w1 - bf16_bits_to_f32(hv[ii] >> 16));
          }
          h00 = hv[0], l00 = lv[0], h02 = hv[2], l02 = lv[2];
          h10 = hv[1], l10 = lv[1], h12 = hv[3], l12 = lv[3];
        } else if (p.norm) {
          // (q - z) * s * gamma[k] in fp32, split hi + lo (within 2^-16):
          // gamma rides on the weights, so the A tile stays as staged.
          uint32_t r[4];
          codes_to_bf16x2(wv[j], r);
          const float s0 = SF32 ? sf0[bi] : bf16_bits_to_f32(sb0[bi] & 0xFFFFu);
          const float s1 = SF32 ? sf1[bi] : bf16_bits_to_f32(sb1[bi] & 0xFFFFu);
          uint32_t hv[4], lv[4];
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) {
            const uint32_t dq = bf16x2_sub(r[ii], (ii & 1) ? zc1[bi] : zc0[bi]);
            const float sc2 = (ii & 1) ? s1 : s0;
            const int e0 = (ii >> 1) * 2;  // registers 0, 1: k steps e 0, 1; 2, 3: e 2, 3
            const float w0 = bf16_bits_to_f32(dq & 0xFFFFu) * sc2 * gm[j][e0];
            const float w1 = bf16_bits_to_f32(dq >> 16) * sc2 * gm[j][e0 + 1];
            hv[ii] = f32x2_to_bf16x2(w0, w1);
            lv[ii] = f32x2_to_bf16x2(w0 - bf16_bits_to_f32(hv[ii] & 0xFFFFu),
                                     w1 - bf16_bits_to_f32(hv[ii] >> 16));
          }
          h00 = hv[0], l00 = lv[0], h02 = hv[2], l02 = lv[2];
          h10 = hv[1], l10 = lv[1], h12 = hv[3], l12 = lv[3];
        } else {
          uint32_t r[4];
          codes_to_bf16x2(wv[j], r);
          dequant_pair<SF32>(r[0], zc0[bi], sb0[bi], sf0[bi], h00, l00);  // row g
          dequant_pair<SF32>(r[2], zc0[bi], sb0[bi], sf0[bi], h02, l02);
          dequant_pair<SF32>(r[1], zc1[bi], sb1[bi], sf1[bi], h10, l10);  // row g + 8
          dequant_pair<SF32>(r[3], zc1[bi], sb1[bi], sf1[bi], h12, l12);
        }
        // K-major 128-byte swizzle: 16-byte chunk (k / 8) XOR (row % 8); the
        // lo tile sits kBTileBytes after the hi tile.
        const int k0 = 16 * j + 4 * t;
        const int inner = (k0 & 7) * 2;
        const int o0 = r0 * 128 + (((k0 >> 3) ^ (r0 & 7)) * 16) + inner;
        const int o1 = (r0 + 1) * 128 + (((k0 >> 3) ^ ((r0 + 1) & 7)) * 16) + inner;
        *reinterpret_cast<uint2 *>(btile + o0) = make_uint2(h00, h02);
        *reinterpret_cast<uint2 *>(btile + o1) = make_uint2(h10, h12);
        *reinterpret_cast<uint2 *>(btile + kBTileBytes + o0) = make_uint2(l00, l02);
        *reinterpret_cast<uint2 *>(btile + kBTileBytes + o1) = make_uint2(l10, l12);
      }
      fence_async_smem();  // make the tile visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bfull + bslot);
        mbar_arrive(wempty + s);  // this warp is done with the stage's weights
      }
      if (p.norm) {
        // Sum of squares of this thread's row and chunks of the stage's A
        // tile (swizzled rows of 128 bytes), read only, beside the MMAs that
        // read the same tile; then this warp lets the slot go.
        const int sa = i % kAStages;
        if (!mbar_wait(afull + sa, (i / kAStages) & 1)) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          fault = true;
          break;
        }
        const unsigned char *arow = smem + S::kA + sa * S::kATileBytes + nrow * 128;
#pragma unroll
        for (int c = nc0; c < nc0 + kNormChunks; ++c) {
          const uint4 x = *reinterpret_cast<const uint4 *>(arow + ((c ^ (nrow & 7)) * 16));
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const float a0 = bf16_bits_to_f32(w[e2] & 0xFFFFu), a1 = bf16_bits_to_f32(w[e2] >> 16);
            nss = fmaf(a0, a0, nss);
            nss = fmaf(a1, a1, nss);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(aempty + sa);
      }
    }

    // ---- epilogue: TMEM -> registers -> Y ----------------------------------
    if (!fault && !mbar_wait(acc_full, 0)) {
      record_fault(&g_fault_gemm, kFaultGemmWait);
      fault = true;
    }
    // r[m] of every row of the tile, in the B slot the MMAs have drained.
    float *sNorm = reinterpret_cast<float *>(smem + S::kB);
    if (p.norm) {
      const float ss = MH == 1 ? nss + __shfl_xor_sync(0xffffffffu, nss, 1) : nss;
      if (!fault && (MH == 2 || (ne & 1) == 0))
        sNorm[nrow] = 1.f / sqrtf(ss / static_cast<float>(p.K) + p.eps);
    }
    named_barrier_sync(kBarEpi, 32 * kDqWarps);  // bias and r staged
    if (!fault && MH == 1 && p.ksplit > 1) {
      // Park the accumulator, column-major [col][row], in the drained
      // operand rings.
      tc_fence_after();
      float *part = reinterpret_cast<float *>(smem);
      const int quarter = warp & 3, half = (warp - 2) >> 2;
      const int row = quarter * 32 + lane;
#pragma unroll 1
      for (int c = half * (kBN / 64); c < (half + 1) * (kBN / 64); ++c) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) part[(c * 32 + i) * kBH + row] = v[i];
      }
    } else if (!fault && p.paired) {
      // Output columns 32 h .. 32 h + 31 of the CTA's 64: gate sums in
      // accumulator columns 32 h + i, up sums in 64 + 32 h + i.
      tc_fence_after();
      const int quarter = warp & 3, h = (warp - 2) >> 2;
      const int n0 = blockIdx.x * (kBN / 2) + 32 * h;
#pragma unroll 1
      for (int mh = 0; mh < MH; ++mh) {
        const int m = m0 + mh * kBH + quarter * 32 + lane;
        float vg[32], vu[32];
        const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
        tmem_ld32(tmem + lanes + mh * kBN + 32 * h, vg);
        tmem_ld32(tmem + lanes + mh * kBN + kBN / 2 + 32 * h, vu);
        if (m < p.M) {
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int j = out_col(i);
            const float gg = vg[i] + sBias[32 * h + j];
            o[j] = gg / (1.f + expf(-gg)) * (vu[i] + sBias[kBN / 2 + 32 * h + j]);
          }
          uint16_t *yrow = static_cast<uint16_t *>(p.Y) + static_cast<int64_t>(m) * p.N;
          if (n0 + 32 <= p.N && p.y_vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = bf16_bits(o[i + 2 * e]) | (bf16_bits(o[i + 2 * e + 1]) << 16);
              *reinterpret_cast<uint4 *>(yrow + n0 + i) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            for (int i = 0; i < 32; ++i)
              if (n0 + i < p.N) yrow[n0 + i] = static_cast<uint16_t>(bf16_bits(o[i]));
          }
        }
      }
    } else if (!fault && p.y_tma) {
      // Stage the bf16 tile in the drained A ring (two 64-column boxes, each
      // rows x 128 bytes with the 128-byte swizzle: 16-byte chunk c of row r
      // at chunk c ^ (r % 8)), then one thread stores both boxes with TMA;
      // rows past M and columns past N are clipped by the tensor map.
      tc_fence_after();
      const int quarter = warp & 3;
      const int half = (warp - 2) >> 2;
      unsigned char *stage = smem + S::kA;
      constexpr int kBoxBytes = kBH * MH * 128;
#pragma unroll 1
      for (int h = 0; h < MH; ++h) {
        const int row = h * kBH + quarter * 32 + lane;
#pragma unroll 1
        for (int c = half * (kBN / 64); c < (half + 1) * (kBN / 64); ++c) {
          float v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + h * kBN + c * 32, v);
          float o[32];
          const float rn = p.norm ? sNorm[row] : 1.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) o[out_col(i)] = v[i] * rn + sBias[c * 32 + out_col(i)];
          unsigned char *box = stage + (c >> 1) * kBoxBytes + row * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = bf16_bits(o[8 * q + 2 * e]) | (bf16_bits(o[8 * q + 2 * e + 1]) << 16);
            const int chunk = ((c & 1) * 4 + q) ^ (row & 7);
            *reinterpret_cast<uint4 *>(box + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_async_smem();  // the staged tile, to the TMA engine
      named_barrier_sync(kBarEpi, 32 * kDqWarps);
      if (tid == 64) {
        const int n_base = nt0 * kTileN;
#pragma unroll
        for (int b = 0; b < kBN / 64; ++b)
          if (n_base + 64 * b < p.N) tma_store_2d(&p.tmy, stage + b * kBoxBytes, n_base + 64 * b, m0);
        bulk_commit();
        bulk_wait_read_all();  // the source stays valid until the CTA exits
      }
      __syncwarp();
    } else if (!fault) {
      tc_fence_after();
      const int quarter = warp & 3;          // TMEM lanes this warp may read
      const int half = (warp - 2) >> 2;      // which half of the columns
      const int n_base = nt0 * kTileN;
#pragma unroll 1
      for (int h = 0; h < MH; ++h) {
        const int m = m0 + h * kBH + quarter * 32 + lane;
#pragma unroll 1
        for (int c = half * (kBN / 64); c < (half + 1) * (kBN / 64); ++c) {
          float v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + h * kBN + c * 32, v);
          if (m < p.M) {
            // Accumulator columns c*32 + i hold output columns out_col(c*32 + i):
            // two whole 16-column tiles, permuted within each.
            const int n0 = n_base + c * 32;
            uint16_t *yrow = static_cast<uint16_t *>(p.Y) + static_cast<int64_t>(m) * p.N;
            float o[32];
            const float rn = p.norm ? sNorm[h * kBH + quarter * 32 + lane] : 1.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) o[out_col(i)] = v[i] * rn + sBias[c * 32 + out_col(i)];
            if (n0 + 32 <= p.N && p.y_vec) {
#pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  w[e] = bf16_bits(o[i + 2 * e]) | (bf16_bits(o[i + 2 * e + 1]) << 16);
                *reinterpret_cast<uint4 *>(yrow + n0 + i) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
              for (int i = 0; i < 32; ++i)
                if (n0 + i < p.N) yrow[n0 + i] = static_cast<uint16_t>(bf16_bits(o[i]));
            }
          }
        }
      }
    }
  }

  if (MH == 1 && p.ksplit > 1) {
    // Split-K reduction: this CTA's slice of the tile's columns, summed over
    // the cluster's partials in rank order.
    cluster_sync_all();
    if (warp >= 2 && p.paired) {
      // Gate column groups only (16, 32 or 64 columns per CTA); the up sums
      // sit 64 columns further.
      const float *part = reinterpret_cast<const float *>(smem);
      const int cols = (kBN / 2) / p.ksplit;
      const int items = kBH * (cols / 16);
      const int n_base = blockIdx.x * (kBN / 2);
      for (int it = tid - 64; it < items; it += 32 * kDqWarps) {
        const int row = it % kBH, c0 = blockIdx.z * cols + (it / kBH) * 16;
        float vg[16], vu[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) vg[i] = vu[i] = 0.f;
        for (int q = 0; q < p.ksplit; ++q)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            vg[i] += ld_dsmem_f32(part + (c0 + i) * kBH + row, q);
            vu[i] += ld_dsmem_f32(part + (kBN / 2 + c0 + i) * kBH + row, q);
          }
        const int m = m0 + row;
        if (m < p.M) {
          float o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = out_col(i);
            const float gg = vg[i] + sBias[c0 + j];
            o[j] = gg / (1.f + expf(-gg)) * (vu[i] + sBias[kBN / 2 + c0 + j]);
          }
          uint16_t *yrow = static_cast<uint16_t *>(p.Y) + static_cast<int64_t>(m) * p.N;
          const int n0 = n_base + c0;
          if (n0 + 16 <= p.N && p.y_vec) {
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
    } else if (warp >= 2) {
      const float *part = reinterpret_cast<const float *>(smem);
      const int cols = kBN / p.ksplit;  // 16, 32, 64 or 128
      const int items = kBH * (cols / 16);
      const int n_base = nt0 * kTileN;
      for (int it = tid - 64; it < items; it += 32 * kDqWarps) {
        const int row = it % kBH, c0 = blockIdx.z * cols + (it / kBH) * 16;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
        for (int q = 0; q < p.ksplit; ++q)
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] += ld_dsmem_f32(part + (c0 + i) * kBH + row, q);
        const int m = m0 + row;
        if (m < p.M) {
          // Accumulator columns c0..c0+15 are output columns c0..c0+15,
          // permuted within the 16.
          float o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) o[out_col(i)] = acc[i] + sBias[c0 + out_col(i)];
          uint16_t *yrow = static_cast<uint16_t *>(p.Y) + static_cast<int64_t>(m) * p.N;
          const int n0 = n_base + c0;
          if (n0 + 16 <= p.N && p.y_vec) {
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
    cluster_sync_all();  // peers are done reading this CTA's partials
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kBN * MH)
                 : "memory");
  }
}

// ---- stream-K schedule for 256-row tiles -----------------------------------
//
// A product with few output tiles (or a tile count just above a multiple of
// the CTA slots) leaves SMs idle in the kernel above: a CTA alone on its SM
// runs a k stage little faster than two CTAs sharing it. Here the product's
// T x K64 (tile, k stage) units are split evenly over two CTAs per SM: CTA c
// takes units [c U / C, (c + 1) U / C) in tile-major order. Its range falls
// into segments, one per tile it touches:
//  * a whole tile is stored as the kernel above stores it;
//  * a tile split over several CTAs has a head (the CTA holding k stage 0,
//    whose segment is the last of its range) and contributors (CTAs whose
//    ranges start inside the tile: their first segments). Each piece parks
//    its fp32 partial tile in the workspace and counts itself in on the
//    tile's counter (the word of its head CTA; acq_rel); the piece that
//    arrives last adds all partial tiles in k order (the head's first),
//    adds the bias, stores the tile and clears the counter. A head that finds every contribution already in
//    (the usual case: it reaches its last segment late) adds them to its
//    accumulators directly and parks nothing.
// The sums run in one fixed order whichever piece completes the tile, so
// results are bitwise reproducible. No CTA ever waits for another. Between
// segments the MMA thread waits until the epilogue has drained the TMEM
// accumulators.

__device__ __forceinline__ uint32_t count_load_acquire(const unsigned int *f) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t atom_add_acq_rel(unsigned int *f, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(f), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void count_store_relaxed(unsigned int *f, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

struct SkSeg {
  int t, kb0, kb1;  // tile, k stages [kb0, kb1)
};
__device__ __forceinline__ int64_t sk_lo(const GemmParams &p, int c) {
  return int64_t(c) * p.units / p.sk_ctas;
}
// The segment of the range [u, hi) that starts at unit u.
__device__ __forceinline__ SkSeg sk_seg(const GemmParams &p, int64_t u, int64_t hi) {
  SkSeg g;
  g.t = static_cast<int>(u / p.K64);
  g.kb0 = static_cast<int>(u - int64_t(g.t) * p.K64);
  const int64_t e = hi - int64_t(g.t) * p.K64;
  g.kb1 = e < p.K64 ? static_cast<int>(e) : p.K64;
  return g;
}
__device__ __forceinline__ int64_t sk_next(const GemmParams &p, const SkSeg &g) {
  return int64_t(g.t) * p.K64 + g.kb1;
}

// 32 output values of row m (output columns n0 .. n0 + 31) as bf16.
__device__ __forceinline__ void store_row32(const GemmParams &p, int m, int n0, const float (&o)[32]) {
  uint16_t *yrow = static_cast<uint16_t *>(p.Y) + static_cast<int64_t>(m) * p.N;
  if (n0 + 32 <= p.N && p.y_vec) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = bf16_bits(o[i + 2 * e]) | (bf16_bits(o[i + 2 * e + 1]) << 16);
      *reinterpret_cast<uint4 *>(yrow + n0 + i) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    for (int i = 0; i < 32; ++i)
      if (n0 + i < p.N) yrow[n0 + i] = static_cast<uint16_t>(bf16_bits(o[i]));
  }
}

template <int BS, bool HAS_ZP, bool SF32>
__global__ void __launch_bounds__(kThreads, 2) gemm_sk_kernel(const __grid_constant__ GemmParams p) {
  constexpr int MH = 2;
  constexpr int kTileRows = kBH * MH;
  using S = Smem<MH, BS, SF32>;
  constexpr int kAStages = S::kAStages, kWStages = S::kWStages, kBStages = S::kBStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *afull = reinterpret_cast<uint64_t *>(smem + S::kBar);
  uint64_t *aempty = afull + kAStages;
  uint64_t *wfull = aempty + kAStages;
  uint64_t *wempty = wfull + kWStages;
  uint64_t *bfull = wempty + kWStages;
  uint64_t *bempty = bfull + kBStages;
  uint64_t *acc_full = bempty + kBStages;
  uint64_t *acc_empty = acc_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::kTmemSlot);
  uint32_t *sh_fault = tmem_slot + 1;  // a wait ran out (epilogue warps)
  uint32_t *sh_mode = tmem_slot + 2;   // a head parks its piece (1) or completes the tile (0)
  uint32_t *sh_last = tmem_slot + 3;   // this CTA's piece was the tile's last
  float *sBias = reinterpret_cast<float *>(smem + S::kBias);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int64_t lo = sk_lo(p, c), hi = sk_lo(p, c + 1);

  if (tid == 0) {
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(afull + i, 1);
      mbar_init(aempty + i, 1);
    }
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(wfull + i, 1);
      mbar_init(wempty + i, kDqWarps);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(bfull + i, kDqWarps);
      mbar_init(bempty + i, 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 1);
    *sh_fault = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kBN * MH)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool fault = false;
  if (warp == 0) {
    if (lane == 0) {
      // A tiles of every stage of every segment.
      int i = 0;
      for (int64_t u = lo; u < hi && !fault;) {
        const SkSeg g = sk_seg(p, u, hi);
        const int m0 = (g.t / p.tiles_n) * kTileRows;
        for (int kb = g.kb0; kb < g.kb1; ++kb, ++i) {
          const int s = i % kAStages;
          if (i >= kAStages && !mbar_wait(aempty + s, ((i / kAStages) - 1) & 1)) {
            record_fault(&g_fault_gemm, kFaultGemmWait);
            fault = true;
            break;
          }
          mbar_arrive_expect_tx(afull + s, S::kATileBytes);
          tma_load_2d(smem + S::kA + s * S::kATileBytes, &p.tma, kb * kBK, m0, afull + s);
        }
        u = sk_next(p, g);
      }
    } else if (lane == 1) {
      // Packed weights of every stage of every segment.
      int i = 0;
      for (int64_t u = lo; u < hi && !fault;) {
        const SkSeg g = sk_seg(p, u, hi);
        const int nt0 = (g.t % p.tiles_n) * kTilesN;
        for (int kb = g.kb0; kb < g.kb1; ++kb, ++i) {
          const int s = i % kWStages;
          if (i >= kWStages && !mbar_wait(wempty + s, ((i / kWStages) - 1) & 1)) {
            record_fault(&g_fault_gemm, kFaultGemmWait);
            fault = true;
            break;
          }
          uint64_t *bar = wfull + s;
          mbar_arrive_expect_tx(bar, kCodeBytes + p.sc_bytes + p.zp_bytes);
          const int blk = (kb * kBK) / BS;
          tma_load_3d(smem + S::kCodes + s * kCodeBytes, &p.tmw, 0, kb, nt0, bar);
          tma_load_3d(smem + S::kSc + s * S::kScBytes, &p.tms, 0, blk, nt0, bar);
          if (HAS_ZP) tma_load_3d(smem + S::kZp + s * S::kZpBytes, &p.tmz, 0, blk >> 1, nt0, bar);
        }
        u = sk_next(p, g);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int i = 0, j = 0;
      for (int64_t u = lo; u < hi && !fault; ++j) {
        const SkSeg g = sk_seg(p, u, hi);
        // The epilogue has read the previous segment's accumulators.
        if (j > 0 && !mbar_wait(acc_empty, (j - 1) & 1)) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          fault = true;
          break;
        }
        for (int kb = g.kb0; kb < g.kb1; ++kb, ++i) {
          const int s = i % kAStages, b = i % kBStages;
          if (!mbar_wait(afull + s, (i / kAStages) & 1) ||
              !mbar_wait(bfull + b, (i / kBStages) & 1)) {
            record_fault(&g_fault_gemm, kFaultGemmWait);
            fault = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(smem + S::kA + s * S::kATileBytes);
          const uint32_t b_base = smem_addr(smem + S::kB + b * kBSlotBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
            for (int h = 0; h < MH; ++h) {
              const uint64_t ad = smem_desc_sw128(a_base + h * kAHalfBytes + kk * 32);
              umma_bf16(tmem + h * kBN, ad, smem_desc_sw128(b_base + kk * 32),
                        kb > g.kb0 || kk > 0);
              umma_bf16(tmem + h * kBN, ad, smem_desc_sw128(b_base + kBTileBytes + kk * 32),
                        true);
            }
          umma_commit(aempty + s);
          umma_commit(bempty + b);
        }
        if (fault) break;
        umma_commit(acc_full);
        u = sk_next(p, g);
      }
    }
  } else {
    // ---- dequantisation warps (2..9) and each segment's epilogue ----------
    // Every warp walks the same segments and passes the same named barriers
    // whatever happens; after a fault it only skips the work.
    const int tile = warp - 2;
    const int quarter = warp & 3;          // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;      // which half of the columns
    const int dg = lane >> 2, dt = lane & 3;
    // Weight rows g and g + 8 of the tile go to B rows 2g and 2g + 1.
    const int r0 = tile * kTileN + 2 * dg;
    constexpr int kBpc = BS < kBK ? kBK / BS : 1;
    int i = 0, j = 0;
    for (int64_t u = lo; u < hi; ++j) {
      const SkSeg g = sk_seg(p, u, hi);
      u = sk_next(p, g);
      for (int kb = g.kb0; kb < g.kb1; ++kb, ++i) {
        if (fault) continue;
        const int s = i % kWStages, bslot = i % kBStages;
        if (!mbar_wait(wfull + s, (i / kWStages) & 1) ||
            (i >= kBStages && !mbar_wait(bempty + bslot, ((i / kBStages) - 1) & 1))) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          fault = true;
          continue;
        }
        // As in gemm_kernel (single weight), every pointer taken from the
        // shared array in this scope so that the accesses stay shared ones.
        const unsigned char *codes = smem + S::kCodes + s * kCodeBytes;
        const unsigned char *sc = smem + S::kSc + s * S::kScBytes;
        const uint2 *zp = reinterpret_cast<const uint2 *>(smem + S::kZp + s * S::kZpBytes);
        unsigned char *btile = smem + S::kB + bslot * kBSlotBytes;
        const int blk0 = (kb * kBK) / BS;
        uint32_t sb0[kBpc], sb1[kBpc], zc0[kBpc], zc1[kBpc];
        float sf0[kBpc], sf1[kBpc];
#pragma unroll
        for (int bi = 0; bi < kBpc; ++bi) {
          if (SF32) {
            const float *s4 = reinterpret_cast<const float *>(sc) + (tile * kBpc + bi) * kTileN;
            sf0[bi] = s4[dg];
            sf1[bi] = s4[dg + 8];
            sb0[bi] = sb1[bi] = 0;
          } else {
            const uint16_t *s2 =
                reinterpret_cast<const uint16_t *>(sc) + (tile * kBpc + bi) * kTileN;
            sb0[bi] = s2[dg] * 0x10001u;
            sb1[bi] = s2[dg + 8] * 0x10001u;
            sf0[bi] = sf1[bi] = 0.f;
          }
          zc0[bi] = zc1[bi] = 0x43084308u;  // bf16 136 = 128 + 8
          if (HAS_ZP) {
            const int b = blk0 + bi;
            const int pairs = BS < 32 ? 2 : 1;
            const uint2 zw = zp[(tile * pairs + (BS < 32 ? bi >> 1 : 0)) * 2 + (b & 1)];
            zc0[bi] = (0x4300u | ((zw.x >> (4 * dg)) & 15)) * 0x10001u;
            zc1[bi] = (0x4300u | ((zw.y >> (4 * dg)) & 15)) * 0x10001u;
          }
        }
        const uint4 w4 = *reinterpret_cast<const uint4 *>(codes + tile * kChunkBytes + lane * 16);
        const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int bi = BS < kBK ? (16 * q) / BS : 0;
          uint32_t r[4];
          codes_to_bf16x2(wv[q], r);
          uint32_t h00, l00, h02, l02, h10, l10, h12, l12;
          dequant_pair<SF32>(r[0], zc0[bi], sb0[bi], sf0[bi], h00, l00);  // row g
          dequant_pair<SF32>(r[2], zc0[bi], sb0[bi], sf0[bi], h02, l02);
          dequant_pair<SF32>(r[1], zc1[bi], sb1[bi], sf1[bi], h10, l10);  // row g + 8
          dequant_pair<SF32>(r[3], zc1[bi], sb1[bi], sf1[bi], h12, l12);
          const int k0 = 16 * q + 4 * dt;
          const int inner = (k0 & 7) * 2;
          const int o0 = r0 * 128 + (((k0 >> 3) ^ (r0 & 7)) * 16) + inner;
          const int o1 = (r0 + 1) * 128 + (((k0 >> 3) ^ ((r0 + 1) & 7)) * 16) + inner;
          *reinterpret_cast<uint2 *>(btile + o0) = make_uint2(h00, h02);
          *reinterpret_cast<uint2 *>(btile + o1) = make_uint2(h10, h12);
          *reinterpret_cast<uint2 *>(btile + kBTileBytes + o0) = make_uint2(l00, l02);
          *reinterpret_cast<uint2 *>(btile + kBTileBytes + o1) = make_uint2(l10, l12);
        }
        fence_async_smem();  // make the tile visible to the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bfull + bslot);
          mbar_arrive(wempty + s);
        }
      }

      // ---- epilogue of the segment -----------------------------------------
      const int m0 = (g.t / p.tiles_n) * kTileRows;
      const int n_base = (g.t % p.tiles_n) * kBN;
      const bool head = g.kb0 == 0, whole = head && g.kb1 == p.K64;
      // A split tile: its head CTA (the one holding k stage 0) and the CTAs
      // after it whose ranges start inside the tile, in the order of their
      // k stages.
      int ch = c, ncontrib = 0;
      if (!whole) {
        const int64_t t0 = int64_t(g.t) * p.K64, tend = t0 + p.K64;
        while (sk_lo(p, ch) > t0) --ch;
        while (ch + 1 + ncontrib < p.sk_ctas && sk_lo(p, ch + 1 + ncontrib) < tend) ++ncontrib;
      }
      {
        const int e = tid - 64;
        if (e < kBN) {
          const int n = n_base + e;
          sBias[e] = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.f;
        }
      }
      // A head whose contributions have all arrived completes the tile from
      // its accumulators; any other piece of a split tile is parked.
      if (head && !whole && warp == 2) {
        if (lane == 0)
          *sh_mode = (!fault && count_load_acquire(p.count + c) == uint32_t(ncontrib)) ? 0u : 1u;
        __syncwarp();
      }
      if (!fault && !mbar_wait(acc_full, j & 1)) {
        record_fault(&g_fault_gemm, kFaultGemmWait);
        fault = true;
      }
      if (fault) *sh_fault = 1;
      named_barrier_sync(kBarEpi, 32 * kDqWarps);  // bias staged, mode decided
      fault = fault || *sh_fault != 0;
      const bool park = !whole && (!head || *sh_mode != 0u);
      float *own = p.ws + (2 * int64_t(c) + (head ? 1 : 0)) * (kTileRows * kBN);
      if (!fault) {
        if (!whole && !park) fence_acq_rel_gpu();  // the contributions the acquire saw
        tc_fence_after();
#pragma unroll 1
        for (int h = 0; h < MH; ++h) {
          const int row = h * kBH + quarter * 32 + lane;  // row of the tile
          const int m = m0 + row;
#pragma unroll 1
          for (int cc = half * (kBN / 64); cc < (half + 1) * (kBN / 64); ++cc) {
            float v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + h * kBN + cc * 32, v);
            if (park) {
              // Column-major [accumulator column][row]: each store
              // instruction writes 32 consecutive rows.
#pragma unroll
              for (int x = 0; x < 32; ++x) __stcg(own + (cc * 32 + x) * kTileRows + row, v[x]);
            } else {
              for (int q = 1; q <= ncontrib; ++q) {
                const float *part = p.ws + 2 * int64_t(c + q) * (kTileRows * kBN);
#pragma unroll
                for (int x = 0; x < 32; ++x)
                  v[x] += __ldcg(part + (cc * 32 + x) * kTileRows + row);
              }
              if (m < p.M) {
                float o[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) o[out_col(x)] = v[x] + sBias[cc * 32 + out_col(x)];
                store_row32(p, m, n_base + cc * 32, o);
              }
            }
          }
        }
        if (!whole && !park && tid == 64) count_store_relaxed(p.count + c, 0u);
      }
      if (park) {
        // Count this piece in; the last of the tile's pieces completes it,
        // adding the parked partial tiles in the order of their k stages
        // (the head's first), as a head completing from its accumulators
        // does: the result does not depend on which piece came last.
        __threadfence();
        named_barrier_sync(kBarEpi, 32 * kDqWarps);  // the partial tile is written
        if (tid == 64)
          *sh_last = (!fault && atom_add_acq_rel(p.count + ch, 1u) == uint32_t(ncontrib)) ? 1u : 0u;
        __syncwarp();
        named_barrier_sync(kBarEpi, 32 * kDqWarps);
        if (*sh_last != 0u && !fault) {
          fence_acq_rel_gpu();
#pragma unroll 1
          for (int h = 0; h < MH; ++h) {
            const int row = h * kBH + quarter * 32 + lane;
            const int m = m0 + row;
#pragma unroll 1
            for (int cc = half * (kBN / 64); cc < (half + 1) * (kBN / 64); ++cc) {
              float v[32];
              const float *hp = p.ws + (2 * int64_t(ch) + 1) * (kTileRows * kBN);
#pragma unroll
              for (int x = 0; x < 32; ++x) v[x] = __ldcg(hp + (cc * 32 + x) * kTileRows + row);
              for (int q = 1; q <= ncontrib; ++q) {
                const float *part = p.ws + 2 * int64_t(ch + q) * (kTileRows * kBN);
#pragma unroll
                for (int x = 0; x < 32; ++x)
                  v[x] += __ldcg(part + (cc * 32 + x) * kTileRows + row);
              }
              if (m < p.M) {
                float o[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) o[out_col(x)] = v[x] + sBias[cc * 32 + out_col(x)];
                store_row32(p, m, n_base + cc * 32, o);
              }
            }
          }
          if (tid == 64) count_store_relaxed(p.count + ch, 0u);
        }
      }
      // The accumulators are drained: the MMA thread may start the next segment.
      tc_fence_before();
      named_barrier_sync(kBarEpi, 32 * kDqWarps);
      if (tid == 64 && !fault) mbar_arrive(acc_empty);
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kBN * MH)
                 : "memory");
  }
}

// ---- fp32 activations: tf32 tensor-core products ---------------------------
//
// The same pipeline for fp32 activations, one 128 x 128 output tile per CTA:
// TMA stages the fp32 A tile as is (two 32-wide, 128-byte-swizzled boxes per
// 64-wide k stage), the dequantisation warps write (q - z) * s as fp32
// rounded to tf32 (nearest, ties away) into two K-major swizzled halves of
// the B tile, and tcgen05.mma kind::tf32 (K = 8 per instruction) multiplies
// them into the TMEM accumulator. The tensor core reads A with a tf32
// significand, so a product carries at most 2^-10 + 2^-11 relative error;
// with fp32 accumulation the stated bound 2e-3 * sum|a w| + 1e-5 holds. One
// CTA per SM (the fp32 tiles need about 180 KB of shared memory).
struct SmemT {
  static constexpr int kAStages = 3;  // A ring
  static constexpr int kWStages = 4;  // packed-weight ring, further ahead
  static constexpr int kATile = kBH * kBK * 4;  // 32 KB: two 16 KB halves
  static constexpr int kBTile = kBN * kBK * 4;  // 32 KB: two 16 KB halves
  static constexpr int kHalf = 16 * 1024;
  static constexpr int kA = 0;
  static constexpr int kB = kA + kAStages * kATile;
  static constexpr int kCodes = kB + kBStagesTf32 * kBTile;
  static constexpr int kSc = kCodes + kWStages * kCodeBytes;
  static constexpr int kScBytes = 2048;
  static constexpr int kZp = kSc + kWStages * kScBytes;
  static constexpr int kZpBytes = 256;
  static constexpr int kBias = kZp + kWStages * kZpBytes;
  static constexpr int kBar = kBias + kBN * 4;
  static constexpr int kTmemSlot = kBar + (2 * kAStages + 2 * kWStages + 2 * kBStagesTf32 + 1) * 8;
  static constexpr int kTotal = kTmemSlot + 16;
};
static_assert(SmemT::kTotal + 1024 <= 227 * 1024, "one CTA per SM");

// D fp32, A and B tf32, both K-major, M = 128, N = kBN.
constexpr uint32_t kIdescTf32 = (1u << 4) | (2u << 7) | (2u << 10) |
                                (static_cast<uint32_t>(kBN >> 3) << 17) |
                                (static_cast<uint32_t>(kBH >> 4) << 24);

__device__ __forceinline__ void umma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdescTf32), "r"(static_cast<int>(accumulate))
      : "memory");
}

// B row (within a 16-row tile) of weight row g < 8 in the tf32 tile: rows
// g = 2p and 2p + 1 (the lanes of one 8-lane store phase) go to rows p and
// p + 4, whose swizzle phases differ in bit 2, so the phase's two rows write
// disjoint halves of the 128-byte row: conflict-free 16-byte stores. Weight
// row g + 8 goes 8 rows further.
__host__ __device__ constexpr int tf32_row(int g) { return ((g & 1) << 2) | (g >> 1); }
// Output column (within the CTA's 128) of tf32 accumulator column c.
__host__ __device__ constexpr int out_col_tf32(int c) {
  return (c & ~7) + 2 * (c & 3) + ((c >> 2) & 1);
}

// fp32 -> tf32, round to nearest (ties away from zero), as fp32 bits.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

template <int BS, bool HAS_ZP, bool SF32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tf32_kernel(const __grid_constant__ GemmParams p) {
  using S = SmemT;
  constexpr int kAStages = S::kAStages, kWStages = S::kWStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *afull = reinterpret_cast<uint64_t *>(smem + S::kBar);
  uint64_t *aempty = afull + kAStages;
  uint64_t *wfull = aempty + kAStages;
  uint64_t *wempty = wfull + kWStages;
  uint64_t *bfull = wempty + kWStages;
  uint64_t *bempty = bfull + kBStagesTf32;
  uint64_t *acc_full = bempty + kBStagesTf32;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::kTmemSlot);
  float *sBias = reinterpret_cast<float *>(smem + S::kBias);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * kBH;
  const int nt0 = blockIdx.x * kTilesN;
  constexpr int kBpc = BS < kBK ? kBK / BS : 1;
  // This CTA's k stages (its rank in the K-splitting cluster is blockIdx.z).
  const int kb0 = blockIdx.z * p.kps;
  const int nk = min(p.K64 - kb0, p.kps);

  if (tid == 0) {
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(afull + i, 1);
      mbar_init(aempty + i, 1);
    }
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(wfull + i, 1);
      mbar_init(wempty + i, kDqWarps);
    }
    for (int i = 0; i < kBStagesTf32; ++i) {
      mbar_init(bfull + i, kDqWarps);
      mbar_init(bempty + i, 1);
    }
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kBN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependents_launch();
  grid_dependency_wait();

  bool fault = false;
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {  // A tiles
        const int s = i % kAStages, kb = kb0 + i;
        if (i >= kAStages && !mbar_wait(aempty + s, ((i / kAStages) - 1) & 1)) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          break;
        }
        mbar_arrive_expect_tx(afull + s, S::kATile);
        unsigned char *ad = smem + S::kA + s * S::kATile;
        tma_load_2d(ad, &p.tma, kb * kBK, m0, afull + s);
        tma_load_2d(ad + S::kHalf, &p.tma, kb * kBK + kBK / 2, m0, afull + s);
      }
    } else if (lane == 1) {
      for (int i = 0; i < nk; ++i) {  // packed weights
        const int s = i % kWStages, kb = kb0 + i;
        if (i >= kWStages && !mbar_wait(wempty + s, ((i / kWStages) - 1) & 1)) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          break;
        }
        uint64_t *bar = wfull + s;
        mbar_arrive_expect_tx(bar, kCodeBytes + p.sc_bytes + p.zp_bytes);
        const int blk = (kb * kBK) / BS;
        tma_load_3d(smem + S::kCodes + s * kCodeBytes, &p.tmw, 0, kb, nt0, bar);
        tma_load_3d(smem + S::kSc + s * S::kScBytes, &p.tms, 0, blk, nt0, bar);
        if (HAS_ZP) tma_load_3d(smem + S::kZp + s * S::kZpBytes, &p.tmz, 0, blk >> 1, nt0, bar);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % kAStages, b = i % kBStagesTf32;
        if (!mbar_wait(afull + s, (i / kAStages) & 1) ||
            !mbar_wait(bfull + b, (i / kBStagesTf32) & 1)) {
          record_fault(&g_fault_gemm, kFaultGemmWait);
          fault = true;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_addr(smem + S::kA + s * S::kATile);
        const uint32_t b_base = smem_addr(smem + S::kB + b * S::kBTile);
#pragma unroll
        for (int kk = 0; kk < kBK / 8; ++kk) {
          const uint32_t off = (kk >> 2) * S::kHalf + (kk & 3) * 32;
          umma_tf32(tmem, smem_desc_sw128(a_base + off), smem_desc_sw128(b_base + off),
                    i > 0 || kk > 0);
        }
        umma_commit(aempty + s);
        umma_commit(bempty + b);
      }
      if (!fault) umma_commit(acc_full);
    }
  } else {
    const int tile = warp - 2;
    const int g = lane >> 2, t = lane & 3;
    const int r0 = tile * kTileN + tf32_row(g);  // weight row g; g + 8 is r0 + 8
    {
      const int e = tid - 64;
      if (e < kBN) {
        const int n = nt0 * kTileN + e;
        sBias[e] = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.f;
      }
    }
    for (int i = 0; i < nk; ++i) {
      const int s = i % kWStages, bslot = i % kBStagesTf32;
      if (!mbar_wait(wfull + s, (i / kWStages) & 1) ||
          (i >= kBStagesTf32 && !mbar_wait(bempty + bslot, ((i / kBStagesTf32) - 1) & 1))) {
        record_fault(&g_fault_gemm, kFaultGemmWait);
        fault = true;
        break;
      }
      const unsigned char *codes = smem + S::kCodes + s * kCodeBytes;
      const unsigned char *sc = smem + S::kSc + s * S::kScBytes;
      const uint2 *zp = reinterpret_cast<const uint2 *>(smem + S::kZp + s * S::kZpBytes);
      unsigned char *btile = smem + S::kB + bslot * S::kBTile;
      const int blk0 = ((kb0 + i) * kBK) / BS;
      float s0[kBpc], s1[kBpc], z0[kBpc], z1[kBpc];
#pragma unroll
      for (int bi = 0; bi < kBpc; ++bi) {
        if (SF32) {
          const float *s4 = reinterpret_cast<const float *>(sc) + (tile * kBpc + bi) * kTileN;
          s0[bi] = s4[g];
          s1[bi] = s4[g + 8];
        } else {
          const uint16_t *s2 = reinterpret_cast<const uint16_t *>(sc) + (tile * kBpc + bi) * kTileN;
          s0[bi] = bf16_bits_to_f32(s2[g]);
          s1[bi] = bf16_bits_to_f32(s2[g + 8]);
        }
        z0[bi] = z1[bi] = 136.f;  // 128 + 8
        if (HAS_ZP) {
          const int b = blk0 + bi;
          const int pairs = BS < 32 ? 2 : 1;
          const uint2 zw = zp[(tile * pairs + (BS < 32 ? bi >> 1 : 0)) * 2 + (b & 1)];
          z0[bi] = static_cast<float>(128 + ((zw.x >> (4 * g)) & 15));
          z1[bi] = static_cast<float>(128 + ((zw.y >> (4 * g)) & 15));
        }
      }
      const uint4 w4 = *reinterpret_cast<const uint4 *>(codes + tile * kChunkBytes + lane * 16);
      const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int bi = BS < kBK ? (16 * j) / BS : 0;
        uint32_t r[4];
        codes_to_bf16x2(wv[j], r);
        // r[0], r[2]: row g at k0 .. k0 + 3; r[1], r[3]: row g + 8.
        auto w = [&](uint32_t pair, int hi, float z, float sc1) {
          const float v = bf16_bits_to_f32(hi ? (pair >> 16) : (pair & 0xFFFFu));
          return to_tf32((v - z) * sc1);  // q - z exact, one rounding in the product
        };
        const uint4 row0 = make_uint4(w(r[0], 0, z0[bi], s0[bi]), w(r[0], 1, z0[bi], s0[bi]),
                                      w(r[2], 0, z0[bi], s0[bi]), w(r[2], 1, z0[bi], s0[bi]));
        const uint4 row1 = make_uint4(w(r[1], 0, z1[bi], s1[bi]), w(r[1], 1, z1[bi], s1[bi]),
                                      w(r[3], 0, z1[bi], s1[bi]), w(r[3], 1, z1[bi], s1[bi]));
        // K-major 128-byte swizzle over 32 fp32 per row: 16-byte chunk
        // ((k % 32) / 4) XOR (row % 8), in the half holding k.
        const int k0 = 16 * j + 4 * t;
        unsigned char *half = btile + (k0 >> 5) * S::kHalf;
        const int c = (k0 & 31) >> 2;
        *reinterpret_cast<uint4 *>(half + r0 * 128 + ((c ^ (r0 & 7)) * 16)) = row0;
        *reinterpret_cast<uint4 *>(half + (r0 + 8) * 128 + ((c ^ (r0 & 7)) * 16)) = row1;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bfull + bslot);
        mbar_arrive(wempty + s);
      }
    }

    if (!fault && !mbar_wait(acc_full, 0)) {
      record_fault(&g_fault_gemm, kFaultGemmWait);
      fault = true;
    }
    named_barrier_sync(kBarEpi, 32 * kDqWarps);  // bias staged
    if (!fault && p.ksplit > 1) {
      // Park the accumulator, column-major [col][row], in the drained A ring.
      tc_fence_after();
      float *part = reinterpret_cast<float *>(smem + S::kA);
      const int quarter = warp & 3, half = (warp - 2) >> 2;
      const int row = quarter * 32 + lane;
#pragma unroll 1
      for (int c = half * (kBN / 64); c < (half + 1) * (kBN / 64); ++c) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + c * 32, v);
#pragma unroll
        for (int q = 0; q < 32; ++q) part[(c * 32 + q) * kBH + row] = v[q];
      }
    } else if (!fault) {
      tc_fence_after();
      const int quarter = warp & 3, half = (warp - 2) >> 2;
      const int m = m0 + quarter * 32 + lane;
      const int n_base = nt0 * kTileN;
      const bool y4 = (p.N % 4) == 0 && (reinterpret_cast<uintptr_t>(p.Y) % 16) == 0;
#pragma unroll 1
      for (int c = half * (kBN / 64); c < (half + 1) * (kBN / 64); ++c) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + c * 32, v);
        if (m < p.M) {
          const int n0 = n_base + c * 32;
          float *yrow = static_cast<float *>(p.Y) + static_cast<int64_t>(m) * p.N;
          float o[32];
#pragma unroll
          for (int q = 0; q < 32; ++q)
            o[out_col_tf32(q)] = v[q] + sBias[c * 32 + out_col_tf32(q)];
          if (n0 + 32 <= p.N && y4) {
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              *reinterpret_cast<float4 *>(yrow + n0 + q) =
                  make_float4(o[q], o[q + 1], o[q + 2], o[q + 3]);
          } else {
            for (int q = 0; q < 32; ++q)
              if (n0 + q < p.N) yrow[n0 + q] = o[q];
          }
        }
      }
    }
  }

  if (p.ksplit > 1) {
    // Split-K reduction: this CTA's slice of the tile's columns, summed over
    // the cluster's partials in rank order (bitwise reproducible).
    cluster_sync_all();
    if (warp >= 2) {
      const float *part = reinterpret_cast<const float *>(smem + S::kA);
      const int cols = kBN / p.ksplit;  // 16, 32, 64 or 128
      const int items = kBH * (cols / 16);
      const int n_base = nt0 * kTileN;
      for (int it = tid - 64; it < items; it += 32 * kDqWarps) {
        const int row = it % kBH, c0 = blockIdx.z * cols + (it / kBH) * 16;
        float acc[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] = 0.f;
        for (int r = 0; r < p.ksplit; ++r)
#pragma unroll
          for (int q = 0; q < 16; ++q) acc[q] += ld_dsmem_f32(part + (c0 + q) * kBH + row, r);
        const int m = m0 + row;
        if (m < p.M) {
          float *yrow = static_cast<float *>(p.Y) + static_cast<int64_t>(m) * p.N;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int n = n_base + c0 + out_col_tf32(q);
            if (n < p.N) yrow[n] = acc[q] + sBias[c0 + out_col_tf32(q)];
          }
        }
      }
    }
    cluster_sync_all();  // peers are done reading this CTA's partials
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kBN)
                 : "memory");
  }
}

template <int BS, bool HAS_ZP, bool SF32>
cudaError_t launch_tf32_one(const GemmParams &p, dim3 grid, bool pdl, cudaStream_t stream) {
  auto kernel = gemm_tf32_kernel<BS, HAS_ZP, SF32>;
  const int smem = SmemT::kTotal + 1024;
  static std::atomic<unsigned long long> configured{0};
  if (const cudaError_t e = ensure_smem_limit(kernel, smem, configured); e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (p.ksplit > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = p.ksplit;
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

template <int BS>
cudaError_t launch_tf32_flags(const GemmParams &p, dim3 grid, bool sf32, bool pdl,
                              cudaStream_t stream) {
  if (p.has_zp)
    return sf32 ? launch_tf32_one<BS, true, true>(p, grid, pdl, stream)
                : launch_tf32_one<BS, true, false>(p, grid, pdl, stream);
  return sf32 ? launch_tf32_one<BS, false, true>(p, grid, pdl, stream)
              : launch_tf32_one<BS, false, false>(p, grid, pdl, stream);
}

template <int BS, bool HAS_ZP, bool SF32, int MH, bool CB = false>
cudaError_t launch_one(const GemmParams &p, dim3 grid, bool pdl, cudaStream_t stream) {
  auto kernel = gemm_kernel<BS, HAS_ZP, SF32, MH, CB>;
  const int smem = Smem<MH, BS, SF32>::kTotal + 1024;
  static std::atomic<unsigned long long> configured{0};
  if (const cudaError_t e = ensure_smem_limit(kernel, smem, configured); e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (p.ksplit > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = p.ksplit;
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

template <int BS, int MH>
cudaError_t launch_flags(const GemmParams &p, dim3 grid, bool sf32, bool pdl,
                         cudaStream_t stream) {
  if (p.code)  // code-book weights: no zero points
    return sf32 ? launch_one<BS, false, true, MH, true>(p, grid, pdl, stream)
                : launch_one<BS, false, false, MH, true>(p, grid, pdl, stream);
  if (p.has_zp)
    return sf32 ? launch_one<BS, true, true, MH>(p, grid, pdl, stream)
                : launch_one<BS, true, false, MH>(p, grid, pdl, stream);
  return sf32 ? launch_one<BS, false, true, MH>(p, grid, pdl, stream)
              : launch_one<BS, false, false, MH>(p, grid, pdl, stream);
}

template <int BS>
cudaError_t launch_mh(const GemmParams &p, dim3 grid, int mh, bool sf32, bool pdl,
                      cudaStream_t stream) {
  return mh == 2 ? launch_flags<BS, 2>(p, grid, sf32, pdl, stream)
                 : launch_flags<BS, 1>(p, grid, sf32, pdl, stream);
}

struct GemmPlan {
  int mh = 1, ksplit = 1;  // tile height in halves of 128 rows; cluster K split
  bool sk = false;         // stream-K schedule
  int64_t sk_ctas = 0, units = 0;
};

// Stream-K workspace: a page of per-CTA arrival counters, then two
// 256 x 128 fp32 partial tiles per CTA.
constexpr size_t kSkCountBytes = 4096;
constexpr size_t kSkPartBytes = size_t(2 * kBH) * kBN * 4;
constexpr size_t kSkCtaBytes = 2 * kSkPartBytes;
constexpr int64_t kSkMaxCtas = kSkCountBytes / 4;
constexpr int64_t kSkMinStages = 4;  // fewer k stages per CTA do not pay for the fix-up

template <int BS, bool HAS_ZP, bool SF32>
cudaError_t sk_run(const GemmParams &p, cudaStream_t stream) {
  auto kernel = gemm_sk_kernel<BS, HAS_ZP, SF32>;
  const int smem = Smem<2, BS, SF32>::kTotal + 1024;
  static std::atomic<unsigned long long> configured{0};
  if (const cudaError_t e = ensure_smem_limit(kernel, smem, configured); e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.sk_ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int BS>
cudaError_t sk_flags(const GemmParams &p, bool sf32, cudaStream_t stream) {
  if (p.has_zp)
    return sf32 ? sk_run<BS, true, true>(p, stream) : sk_run<BS, true, false>(p, stream);
  return sf32 ? sk_run<BS, false, true>(p, stream) : sk_run<BS, false, false>(p, stream);
}

cudaError_t sk_bs(const GemmParams &p, int bs, bool sf32, cudaStream_t stream) {
  switch (bs) {
    case 16: return sk_flags<16>(p, sf32, stream);
    case 32: return sk_flags<32>(p, sf32, stream);
    case 64: return sk_flags<64>(p, sf32, stream);
    case 128: return sk_flags<128>(p, sf32, stream);
    case 256: return sk_flags<256>(p, sf32, stream);
    default: return cudaErrorNotSupported;
  }
}

// CTAs resident at once for a split-K cluster size: two per SM; clusters
// pack per GPC, which on GB300 (152 SMs) leaves 8 CTA slots unused with
// clusters of 4 and 16 with clusters of 8 (occupancy query for this kernel's
// shared memory and 320 threads: 152, 74 and 36 clusters of 2, 4 and 8).
int64_t resident_ctas(int c, int sms) {
  const int64_t two = 2 * int64_t(sms);
  return c <= 2 ? two : c == 4 ? two - two / 38 : two - two / 19;
}

}  // namespace

cudaError_t gemm_take_fault(unsigned int *out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fault_gemm, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fault_gemm, &zero, sizeof(unsigned int));
  return e;
}

size_t gemm_workspace_bytes() {
  return kSkCountBytes + size_t(2) * size_t(sm_count()) * kSkCtaBytes;
}

bool gemm_supports(const MatmulArgs &a) {
  // Activations whose rows TMA can address (16-byte row stride and base):
  // bf16 (any weight), or fp32 on the tf32 kernel (single weights).
  if (reinterpret_cast<uintptr_t>(a.A) % 16 != 0) return false;
  if (a.a_f32) return (a.K % 4) == 0 && !a.paired;
  return (a.K % 8) == 0;
}

// K split of the tf32 kernel (fp32 activations) on a GPU with `sms` SMs.
int plan_gemm_tf32(const MatmulArgs &a, int sms) {
  // K split (cluster of 1..8 CTAs) when the output tiles cannot fill the
  // GPU: a CTA spends about 0.75 us per 64-wide k stage (the tf32 tensor
  // rate of one SM), plus the split's fixed cost; one CTA per SM, clusters
  // packing per GPC.
  const uint64_t K64 = ceil_div(a.K, kChunkK);
  const int64_t tiles = ceil_div(a.M, int64_t(kBH)) * ceil_div(a.N, int64_t(kBN));
  int ksplit = 1;
  {
    double best = 0.0;
    for (int c = 1; c <= 8; c *= 2) {
      const int64_t kps = ceil_div(int64_t(K64), int64_t(c));
      if (c > 1 && (kps < 4 || (c - 1) * kps >= int64_t(K64))) continue;
      const int64_t slots = c <= 2 ? sms - (c == 2 ? 8 : 0) : sms - 24;
      if (slots <= 0) continue;
      const double fixed = c == 1 ? 2.0 : c == 2 ? 4.0 : c == 4 ? 6.0 : 13.0;
      const double cost = double(ceil_div(tiles * c, slots)) * (double(kps) * 0.75 + fixed);
      if (c == 1 || cost < best - 1e-9) {
        best = cost;
        ksplit = c;
      }
    }
  }
  return ksplit;
}

// fp32 activations: the tf32 kernel, 128 x 128 tiles, one CTA per SM.
cudaError_t launch_gemm_tf32(const MatmulArgs &a, cudaStream_t stream) {
  GemmParams p{};
  const uint64_t N16 = ceil_div(a.N, kTileN), K64 = ceil_div(a.K, kChunkK);
  const uint64_t nb = ceil_div(a.K, a.bs), nbz = ceil_div(nb, 2) * 2;
  const uint64_t es = a.scale_f32 ? 4 : 2;
  const uint32_t bpc = a.bs < kBK ? kBK / a.bs : 1;
  const uint32_t ppc = a.bs < 32 ? 2 : 1;
  cudaError_t e;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.K) * 4};
    const uint32_t box[2] = {kBK / 2, kBH};  // 32 fp32 = 128 bytes per row
    e = make_tmap(&p.tma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.A, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  {
    const uint64_t dims[3] = {kChunkBytes / 4, K64, N16};
    const uint64_t strides[2] = {kChunkBytes, K64 * kChunkBytes};
    const uint32_t box[3] = {kChunkBytes / 4, 1, kTilesN};
    e = make_tmap(&p.tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.packed_b, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  {
    const uint64_t words = kTileN * es / 4;
    const uint64_t dims[3] = {words, nb, N16};
    const uint64_t strides[2] = {kTileN * es, nb * kTileN * es};
    const uint32_t box[3] = {static_cast<uint32_t>(words), bpc, kTilesN};
    e = make_tmap(&p.tms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.scales, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  if (a.zp) {
    const uint64_t dims[3] = {4, nbz / 2, N16};
    const uint64_t strides[2] = {16, nbz * 8};
    const uint32_t box[3] = {4, ppc, kTilesN};
    e = make_tmap(&p.tmz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a.zp, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  p.sc_bytes = static_cast<int>(kTilesN * bpc * kTileN * es);
  p.zp_bytes = a.zp ? static_cast<int>(kTilesN * ppc * 16) : 0;
  p.bias = a.bias;
  p.Y = a.Y;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K64 = static_cast<int>(K64);
  p.has_zp = a.zp != nullptr;
  const int ksplit = plan_gemm_tf32(a, sm_count());
  p.ksplit = ksplit;
  p.kps = static_cast<int>(ceil_div(int64_t(K64), int64_t(ksplit)));
  p.norm = a.norm ? 1 : 0;
  p.K = static_cast<int>(a.K);
  p.code = a.code;
  p.gamma = a.gamma;
  p.eps = a.eps;
  const dim3 grid(static_cast<unsigned>(ceil_div(a.N, int64_t(kBN))),
                  static_cast<unsigned>(ceil_div(a.M, int64_t(kBH))),
                  static_cast<unsigned>(ksplit));
  switch (a.bs) {
    case 16: return launch_tf32_flags<16>(p, grid, a.scale_f32, a.pdl, stream);
    case 32: return launch_tf32_flags<32>(p, grid, a.scale_f32, a.pdl, stream);
    case 64: return launch_tf32_flags<64>(p, grid, a.scale_f32, a.pdl, stream);
    case 128: return launch_tf32_flags<128>(p, grid, a.scale_f32, a.pdl, stream);
    case 256: return launch_tf32_flags<256>(p, grid, a.scale_f32, a.pdl, stream);
    default: return cudaErrorNotSupported;
  }
}

// Tile height, K split and schedule of the bf16 kernel for a product on a
// GPU with `sms` SMs: pure host arithmetic, shared by the launch and by
// mnb_matmul_plan.
// Stage costs of the planner's model, us per 64-wide k stage of one CTA.
constexpr double kStage128 = 1.17, kStage256 = 1.6;

GemmPlan plan_gemm(const MatmulArgs &a, int sms) {
  const uint64_t K64 = ceil_div(a.K, kChunkK);
  const int64_t cols = a.paired ? kBN / 2 : kBN;
  // Tile height (128 or 256 rows) and K split (cluster of 1..8 CTAs, 128-row
  // tiles only) by a cost model fitted to GB300 measurements of the Qwen3-4B
  // shapes at M = 512, 2048 and 4096 (each dequantised weight as a hi + lo
  // pair, two MMAs per k step): a CTA spends about 1.17 us per 64-wide k
  // stage with 128 rows and 1.6 us with 256 rows (two CTAs share the SM's
  // tensor core), plus a fixed cost that grows with the split (the partial
  // tiles' reduction through distributed shared memory); CTAs run in rounds
  // of what can be resident at once, clusters packing per GPC.
  GemmPlan r;
  int &mh = r.mh, &ksplit = r.ksplit;
  double best = 0.0;
  {
    bool have = false;
    for (int h = 1; h <= 2; ++h)
      // A normalized row needs its whole K in one CTA: no K split.
      for (int c = 1; c <= (h == 1 ? (a.norm ? 1 : a.paired ? 4 : 8) : 1); c *= 2) {
        const int64_t kps = ceil_div(int64_t(K64), int64_t(c));
        if (c > 1 && (kps < 4 || (c - 1) * kps >= int64_t(K64))) continue;
        const int64_t ctas = ceil_div(a.M, int64_t(kBH) * h) * ceil_div(a.N, cols) * c;
        if (h == 2 && ctas < sms) continue;  // a lone 256-row CTA per SM is slower
        const int64_t slots = resident_ctas(c, sms);
        if (slots <= 0) continue;
        const double fixed = c == 1 ? 2.0 : c == 2 ? 4.0 : c == 4 ? 6.0 : 13.0;
        const double cost = double(ceil_div(ctas, slots)) *
                            (double(kps) * (h == 2 ? kStage256 : kStage128) + fixed);
        if (!have || cost < best - 1e-9) {
          best = cost;
          mh = h;
          ksplit = c;
          have = true;
        }
      }
  }
  // Stream-K over 256-row tiles (single weights, with a workspace): every
  // CTA takes an equal share of the (tile, k stage) units, at the 256-row
  // stage cost, plus what GB300 measurements of the split tiles show (Qwen3
  // prefill shapes, M = 512 to 4096): about 28 us fixed (parking partial
  // tiles through L2, the arrival counters, the accumulator drain between
  // segments), about 2.5 us for each further piece of a tile and about 1 us
  // for each further tile a CTA's range touches. It wins where whole tiles
  // leave half the CTA slots idle for long (down and o projections with
  // M >= 2048, 4096) and loses where tiles are few or short.
  if (a.ws && !a.paired && !a.norm && !a.code && a.ws_bytes > kSkCountBytes) {
    const int64_t tiles_n = ceil_div(a.N, int64_t(kBN));
    const int64_t units = ceil_div(a.M, int64_t(2 * kBH)) * tiles_n * int64_t(K64);
    const int64_t room = static_cast<int64_t>((a.ws_bytes - kSkCountBytes) / kSkCtaBytes);
    const int64_t ctas = std::min(std::min(2 * int64_t(sms), room),
                                  std::min(units / kSkMinStages, kSkMaxCtas));
    if (ctas >= 1) {
      const int64_t L = ceil_div(units, ctas);
      const int64_t segs = ceil_div(L - 1, int64_t(K64)) + 1;
      const int64_t parts = ceil_div(int64_t(K64), L);
      const double cost =
          double(L) * kStage256 + 28.0 + double(segs - 1) + 2.5 * double(parts - 1);
      if (a.sk_only || cost < best - 1e-9) {
        r.sk = true;
        r.sk_ctas = ctas;
        r.units = units;
        mh = 2;
        ksplit = 1;
      }
    }
  }
  return r;
}

cudaError_t launch_gemm(const MatmulArgs &a, cudaStream_t stream) {
  if (!gemm_supports(a)) return cudaErrorNotSupported;
  if (a.sk_only && (a.a_f32 || a.paired || a.norm || !a.ws)) return cudaErrorNotSupported;
  if (a.norm && (a.a_f32 || a.paired)) return cudaErrorNotSupported;
  if (a.code && (a.a_f32 || a.paired || a.norm || a.zp || a.sk_only)) return cudaErrorNotSupported;
  if (a.a_f32) return launch_gemm_tf32(a, stream);
  GemmParams p{};
  const uint64_t N16 = ceil_div(a.N, kTileN), K64 = ceil_div(a.K, kChunkK);
  // Output columns per CTA: 128, or 64 for a gated-MLP pair (64 gate and 64
  // up rows fill the B tile).
  const int64_t cols = a.paired ? kBN / 2 : kBN;
  const GemmPlan plan = plan_gemm(a, sm_count());
  const int mh = plan.mh, ksplit = plan.ksplit;
  const bool sk = plan.sk;
  const int64_t sk_ctas = plan.sk_ctas, units = plan.units;
  const int64_t tiles_n = ceil_div(a.N, int64_t(kBN));
  if (a.sk_only && !sk) return cudaErrorNotSupported;
  const uint64_t nb = ceil_div(a.K, a.bs), nbz = ceil_div(nb, 2) * 2;
  const uint64_t es = a.scale_f32 ? 4 : 2;
  const uint32_t bpc = a.bs < kBK ? kBK / a.bs : 1;
  const uint32_t ppc = a.bs < 32 ? 2 : 1;
  cudaError_t e;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.K) * 2};
    const uint32_t box[2] = {kBK, static_cast<uint32_t>(kBH * mh)};
    e = make_tmap(&p.tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.A, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  // Weight maps: one weight in boxes of 8 tiles, or each of a pair in boxes
  // of 4 tiles.
  const uint32_t bt = a.paired ? kTilesN / 2 : kTilesN;
  auto weight_maps = [&](const void *pb, const void *sc, const void *zp, CUtensorMap *mw,
                         CUtensorMap *ms, CUtensorMap *mz) -> cudaError_t {
    {
      const uint64_t dims[3] = {kChunkBytes / 4, K64, N16};
      const uint64_t strides[2] = {kChunkBytes, K64 * kChunkBytes};
      const uint32_t box[3] = {kChunkBytes / 4, 1, bt};
      const cudaError_t r = make_tmap(mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, pb, dims, strides,
                                      box, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (r != cudaSuccess) return r;
    }
    {
      const uint64_t words = kTileN * es / 4;
      const uint64_t dims[3] = {words, nb, N16};
      const uint64_t strides[2] = {kTileN * es, nb * kTileN * es};
      const uint32_t box[3] = {static_cast<uint32_t>(words), bpc, bt};
      const cudaError_t r = make_tmap(ms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, sc, dims, strides,
                                      box, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (r != cudaSuccess) return r;
    }
    if (zp) {
      const uint64_t dims[3] = {4, nbz / 2, N16};
      const uint64_t strides[2] = {16, nbz * 8};
      const uint32_t box[3] = {4, ppc, bt};
      const cudaError_t r = make_tmap(mz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, zp, dims, strides,
                                      box, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  };
  e = weight_maps(a.packed_b, a.scales, a.zp, &p.tmw, &p.tms, &p.tmz);
  if (e != cudaSuccess) return e;
  p.sc_bytes = static_cast<int>(kTilesN * bpc * kTileN * es);
  p.zp_bytes = a.zp ? static_cast<int>(kTilesN * ppc * 16) : 0;
  if (a.paired) {
    e = weight_maps(a.packed_b2, a.scales2, a.zp2, &p.tmw2, &p.tms2, &p.tmz2);
    if (e != cudaSuccess) return e;
    p.paired = 1;
    // The up halves start where tile 4 would (a multiple of 128 bytes for the
    // scales); zero points start at 128 bytes at least.
    p.sc_up = static_cast<int>((kTilesN / 2) * bpc * kTileN * es);
    p.zp_up = static_cast<int>(std::max<uint64_t>(128, (kTilesN / 2) * ppc * 16));
  }
  p.bias = a.bias;
  p.bias2 = a.bias2;
  p.Y = a.Y;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K64 = static_cast<int>(K64);
  p.has_zp = a.zp != nullptr;
  p.y_vec = (a.N % 8) == 0 && (reinterpret_cast<uintptr_t>(a.Y) % 16) == 0;
  p.ksplit = ksplit;
  p.kps = static_cast<int>(ceil_div(int64_t(K64), int64_t(ksplit)));
  p.norm = a.norm ? 1 : 0;
  p.K = static_cast<int>(a.K);
  p.code = a.code;
  p.gamma = a.gamma;
  p.eps = a.eps;
  // TMA stores of the output tile: single weight, no K split, rows of Y a
  // multiple of 16 bytes from a 16-byte aligned base.
  if (!sk && !a.paired && ksplit == 1 && (a.N % 8) == 0 &&
      (reinterpret_cast<uintptr_t>(a.Y) % 16) == 0) {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(kBH * mh)};
    e = make_tmap(&p.tmy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.Y, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    p.y_tma = 1;
  }
  if (sk) {
    p.units = units;
    p.sk_ctas = static_cast<int>(sk_ctas);
    p.tiles_n = static_cast<int>(tiles_n);
    p.count = static_cast<unsigned int *>(a.ws);
    p.ws = reinterpret_cast<float *>(static_cast<unsigned char *>(a.ws) + kSkCountBytes);
    return sk_bs(p, a.bs, a.scale_f32, stream);
  }
  const dim3 grid(static_cast<unsigned>(ceil_div(a.N, cols)),
                  static_cast<unsigned>(ceil_div(a.M, int64_t(kBH) * mh)),
                  static_cast<unsigned>(ksplit));
  switch (a.bs) {
    case 16: return launch_mh<16>(p, grid, mh, a.scale_f32, a.pdl, stream);
    case 32: return launch_mh<32>(p, grid, mh, a.scale_f32, a.pdl, stream);
    case 64: return launch_mh<64>(p, grid, mh, a.scale_f32, a.pdl, stream);
    case 128: return launch_mh<128>(p, grid, mh, a.scale_f32, a.pdl, stream);
    case 256: return launch_mh<256>(p, grid, mh, a.scale_f32, a.pdl, stream);
    default: return cudaErrorNotSupported;
  }
}

GemmPlanInfo gemm_plan_info(const MatmulArgs &a, int sms) {
  GemmPlanInfo o;
  if (a.a_f32) {
    o.tf32 = true;
    o.tile_rows = kBH;
    o.k_split = plan_gemm_tf32(a, sms);
    o.ctas = ceil_div(a.M, int64_t(kBH)) * ceil_div(a.N, int64_t(kBN)) * o.k_split;
    return o;
  }
  const GemmPlan pl = plan_gemm(a, sms);
  o.tile_rows = kBH * pl.mh;
  o.k_split = pl.ksplit;
  o.stream_k = pl.sk;
  o.ctas = pl.sk ? pl.sk_ctas
                 : ceil_div(a.M, int64_t(kBH) * pl.mh) *
                       ceil_div(a.N, int64_t(a.paired ? kBN / 2 : kBN)) * pl.ksplit;
  // As launch_gemm decides it.
  o.tma_store = !pl.sk && !a.paired && pl.ksplit == 1 && (a.N % 8) == 0 &&
                (reinterpret_cast<uintptr_t>(a.Y) % 16) == 0;
  return o;
}

}  // namespace mnb
