// Tensor-core (tcgen05 / TMEM) MatMulNBits kernel for larger M.
#include "mnb_common.cuh"
#include "mnb_launch.h"

namespace mnb {

cudaError_t launch_gemm(const MatmulArgs &, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mnb
