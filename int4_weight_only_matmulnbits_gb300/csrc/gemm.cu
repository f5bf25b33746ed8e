// Tensor-core (tcgen05 / TMEM) MatMulNBits kernel for larger M.
#include "mnb_common.cuh"
#include "mnb_launch.h"

namespace mnb {

__device__ unsigned int g_fault_gemm = 0;

cudaError_t gemm_take_fault(unsigned int *out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fault_gemm, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fault_gemm, &zero, sizeof(unsigned int));
  return e;
}

cudaError_t launch_gemm(const MatmulArgs &, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mnb
