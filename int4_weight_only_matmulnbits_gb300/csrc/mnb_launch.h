// Host-side launch interfaces between the C ABI (api.cu) and the kernels.
// Arguments arrive here already validated.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <vector>

#include "../../include/mnb.h"

namespace mnb {

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device: `done` (one per kernel instantiation) holds a bit
// for each device ordinal below 64 already configured; higher ordinals are
// configured on every call. Two host threads may both set it the first
// time, which is harmless (the call is idempotent).
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kernel, int bytes, std::atomic<unsigned long long> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

struct PrepackArgs {
  const uint8_t *B;
  const void *scales;
  const uint8_t *zp;  // may be null
  int64_t N, K;
  int bs;
  bool scale_f32;
  void *packed_b, *packed_scales, *packed_zp;
  int qdq_axis = -1;  // -1: MatMulNBits storage; 0 / 1: QDQ UINT4 [K,N] / [N,K]
  // The bitsandbytes-style storage (flattened N x K codes, first of a pair
  // high; absmax [N * K / bs] read as [N, nb] scales, K a multiple of bs).
  bool bnb4 = false;
  // The packed-weight header, written by the last kernel to header_dst (the
  // end of packed_b).
  mnb_packed_header header{};
  void *header_dst = nullptr;
};

struct UnprepackArgs {
  const void *packed_b, *packed_scales, *packed_zp;  // packed_zp may be null
  int64_t N, K;
  int bs;
  bool scale_f32;
  uint8_t *B;
  void *scales;
  uint8_t *zp;
};

struct MatmulArgs {
  const void *A;
  const void *packed_b, *scales, *zp;  // zp may be null
  const float *bias;                   // may be null
  void *Y;
  int64_t M, N, K;
  int bs;
  bool a_f32, scale_f32;
  bool pdl;  // programmatic dependent launch
  // Gated-MLP pair for the tensor-core kernel: the "up" weight (same shape);
  // Y = silu(A gate^T + bias) * (A up^T + bias2).
  bool paired = false;
  const void *packed_b2 = nullptr, *scales2 = nullptr, *zp2 = nullptr;
  const float *bias2 = nullptr;
  // Caller-owned workspace for the tensor-core kernel's stream-K schedule
  // (null: not used); see gemm_workspace_bytes().
  void *ws = nullptr;
  size_t ws_bytes = 0;
  bool sk_only = false;  // the stream-K schedule or cudaErrorNotSupported
  // RMS-normalized activations (bf16, single weight, tensor-core kernel):
  // A * gamma staged, outputs scaled by 1 / sqrt(mean A^2 + eps).
  bool norm = false;
  const float *gamma = nullptr;
  float eps = 0.f;
  // Code-book weights (bf16 activations, tensor-core kernel): w = code[q] * s
  // with the 16 fp32 values here, no zero points.
  const float *code = nullptr;
};

// What launch_gemm would launch for a product on a GPU with `sms` SMs (host
// arithmetic only; `a.A`, `a.Y` and `a.ws` are only tested for alignment or
// presence).
struct GemmPlanInfo {
  bool tf32 = false, stream_k = false, tma_store = false;
  int tile_rows = 0, k_split = 1;
  int64_t ctas = 0;
};
GemmPlanInfo gemm_plan_info(const MatmulArgs &a, int sms);

// Workspace bytes that let launch_gemm use its stream-K schedule on the
// current device: a flag page plus one 256 x 128 fp32 partial tile for each
// CTA the cooperative grid can hold.
size_t gemm_workspace_bytes();

cudaError_t launch_prepack(const PrepackArgs &a, cudaStream_t stream);
// Test-only failure injection for the decode kernel (mnb_test_wait_fault).
void gemv_set_wait_fault(int stop_stage);
cudaError_t launch_unprepack(const UnprepackArgs &a, cudaStream_t stream);

// Up to kMaxGroup weights that share one activation matrix A (fused-N
// projections), each with its own N, output and optional bias.
constexpr int kMaxGroup = 4;
struct GroupArgs {
  const void *A;
  int count;
  const void *packed_b[kMaxGroup], *scales[kMaxGroup], *zp[kMaxGroup];
  const float *bias[kMaxGroup];
  void *Y[kMaxGroup];
  int64_t N[kMaxGroup];
  int64_t M, K;
  int bs;
  bool a_f32, scale_f32, has_zp;
  bool pdl;
  // Gated-MLP pair: weight 0 = gate, weight 1 = up (same N), one output
  // Y[0] = silu(gate) * up; bias[0] / bias[1] apply before the product.
  bool paired = false;
  // RMS-normalized activations: A * gamma staged, outputs scaled by
  // 1 / sqrt(mean(A^2) + eps) (gamma null: 1).
  bool norm = false;
  const float *gamma = nullptr;
  float eps = 0.f;
  // Greedy ArgMax keys [M] over weight 0's outputs (zeroed by the caller;
  // launch_argmax_finalize turns them into indices). Y[0] may be null.
  unsigned long long *amax = nullptr;
  // Code-book weights (the bitsandbytes-style format): w = code[q] * s with
  // code the 16 fp32 values here (each held as a bf16 hi + lo pair for the
  // products), no zero points. Null: the affine MatMulNBits codes.
  const float *code = nullptr;
};
cudaError_t launch_argmax_init(unsigned long long *amax, int M, cudaStream_t stream);
cudaError_t launch_argmax_finalize(unsigned long long *amax, int M, bool pdl,
                                   cudaStream_t stream);

// Small-M split-K kernel (M <= kGemvMaxM). Returns cudaErrorNotSupported when
// no launch configuration fits this shape.
constexpr int kGemvMaxM = 16;
cudaError_t launch_gemv(const MatmulArgs &a, cudaStream_t stream);
cudaError_t launch_gemv_group(const GroupArgs &a, cudaStream_t stream);

// tcgen05/TMEM tensor-core kernel for larger M: bf16 activations whose rows
// are 16-byte aligned (K % 8 == 0). Returns cudaErrorNotSupported otherwise.
bool gemm_supports(const MatmulArgs &a);
cudaError_t launch_gemm(const MatmulArgs &a, cudaStream_t stream);

// Persistent CTA-pair tensor-core kernel (gemm_pair.cu): bf16 activations,
// single affine weights (no gated pair, normalization or code book).
struct PairPlan {
  int nt = 0;         // 16-row weight tiles per CTA (tile columns 32 nt); 0: none
  int pairs = 0;      // CTA pairs launched
  int64_t tiles = 0;  // 256-row output tiles
};
bool pair_supports(const MatmulArgs &a);
// The tile width and grid for `pairs` resident CTA pairs (host arithmetic).
PairPlan plan_pair(const MatmulArgs &a, int pairs);
// CTA pairs the current device holds at once (0 if the query fails).
int pair_slots();
cudaError_t launch_gemm_pair(const MatmulArgs &a, cudaStream_t stream);
cudaError_t pair_take_fault(unsigned int *out);

// Decode chain (chain.cu): ops validated by the C ABI.
constexpr int kChainMaxDeps = 4;
constexpr int kChainMaxOps = 4096;
constexpr int kChainMaxM = 8;
struct ChainOp {
  const void *A;
  void *Y;
  const void *b[2], *s[2], *z[2];  // [1] = up weight of a gated-MLP pair
  const float *bias[2];
  int64_t N, K;
  bool paired;
  int dep[kChainMaxDeps];
};
struct ChainShape {
  int M, bs;
  bool a_f32, scale_f32, has_zp;
};
// Launch geometry and plan-buffer layout of a chain (a pure function of the
// shape, the largest K, the grid and the schedule's size).
struct ChainGeom {
  int grid, per_sm, nst, tmax, kmax, smem;
  int n_ops, n_segs;
  size_t off_ctaseg, off_segs, off_count, off_ctl, plan_bytes;
};
// Plans the chain: fills g and, if image != nullptr, the plan's host image
// (g.plan_bytes bytes). cudaErrorNotSupported if no layout fits.
cudaError_t chain_plan(const ChainOp *ops, int n, const ChainShape &sh, ChainGeom &g,
                       std::vector<unsigned char> *image);
// The schedule part of chain_plan for a fixed g.grid, g.tmax (host only).
void chain_schedule(const ChainOp *ops, int n, const ChainShape &sh, ChainGeom &g,
                    std::vector<unsigned char> *image);
// Recomputes the geometry of a built plan from its recorded sizes; false if
// they are inconsistent.
bool chain_geom(const ChainShape &sh, int n_ops, int kmax, int grid, int per_sm, int nst,
                int n_segs, ChainGeom &g);
cudaError_t chain_launch(const void *plan, const ChainShape &sh, const ChainGeom &g,
                         cudaStream_t stream);
cudaError_t chain_take_fault(unsigned int *out);
// Device address and size of the library-owned plan array (looked up once
// per device, with that device current).
cudaError_t chain_scratch(void **ptr, size_t *bytes);

int sm_count();

// Tiled tensor map over `rank` dims (dims[0] innermost; strides_bytes[i] is
// the stride of dim i+1). cudaErrorInvalidValue if the driver rejects it.
cudaError_t make_tmap(CUtensorMap *map, CUtensorMapDataType dtype, int rank,
                      const void *base, const uint64_t *dims,
                      const uint64_t *strides_bytes, const uint32_t *box,
                      CUtensorMapSwizzle swizzle);

// Read and clear the fault word of each kernel file (0 = no fault).
cudaError_t gemv_take_fault(unsigned int *out);
cudaError_t gemm_take_fault(unsigned int *out);

}  // namespace mnb
