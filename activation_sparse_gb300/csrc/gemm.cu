// gemm.cu -- tcgen05 activation GEMM (in progress).
#include "common.cuh"
#include "internal.h"

namespace si {
cudaError_t launch_act_gemm(const ActGemmParams&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace si
