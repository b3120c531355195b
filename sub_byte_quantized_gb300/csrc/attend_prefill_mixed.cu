// Row-side tensor-core phase 1 for mixed K/V precision (the kernel template is in
// attend_prefill_kernel.cuh): lower-precision keys with 8-bit values, and a 2-bit Hadamard key body
// with a 4-bit value body (value errors reach the output directly, key errors pass through the
// softmax: Open-TQ-Metal, Section 5).
#include "attend_prefill_kernel.cuh"

namespace kvq {

cudaError_t launch_attend_prefill_mixed(const AttendArgs &a, cudaStream_t st) {
  const int kl = a.cache.layout, vl = a.cache.v_layout;
  if (kl == KVQ_Q4_0 && vl == KVQ_Q8_0) return launch_pair<KVQ_Q4_0, KVQ_Q8_0>(a, st);
  if (kl == KVQ_ASYM4_G32 && vl == KVQ_Q8_0) return launch_pair<KVQ_ASYM4_G32, KVQ_Q8_0>(a, st);
  if (kl == KVQ_HAD_INT2 && vl == KVQ_HAD_INT4) return launch_pair<KVQ_HAD_INT2, KVQ_HAD_INT4>(a, st);
  return cudaErrorNotSupported;
}

}  // namespace kvq
