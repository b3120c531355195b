// Tensor-core phase 1 (filled in below as shapes are covered).
#include "kvq_internal.cuh"

namespace kvq {

bool mma_supported(const AttendArgs &) { return false; }

cudaError_t launch_attend_mma(const AttendArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kvq
