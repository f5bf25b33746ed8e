// Host-side launch interfaces between the C ABI (api.cu) and the kernels.
// Arguments arrive here already validated.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mnb {

struct PrepackArgs {
  const uint8_t *B;
  const void *scales;
  const uint8_t *zp;  // may be null
  int64_t N, K;
  int bs;
  bool scale_f32;
  void *packed_b, *packed_scales, *packed_zp;
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
};

cudaError_t launch_prepack(const PrepackArgs &a, cudaStream_t stream);
cudaError_t launch_unprepack(const UnprepackArgs &a, cudaStream_t stream);

// Small-M split-K kernel (M <= kGemvMaxM). Returns cudaErrorNotSupported when
// no launch configuration fits this shape.
constexpr int kGemvMaxM = 16;
cudaError_t launch_gemv(const MatmulArgs &a, cudaStream_t stream);

// tcgen05/TMEM tensor-core kernel for larger M. Returns
// cudaErrorNotSupported for combinations it does not serve.
cudaError_t launch_gemm(const MatmulArgs &a, cudaStream_t stream);

int sm_count();

}  // namespace mnb
