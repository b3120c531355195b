// Row-side tensor-core phase 1 (the kernel template is in attend_prefill_kernel.cuh): which calls it
// takes, and the launches of the layout pairs with one layout in both planes. The mixed K/V pairs
// are instantiated in attend_prefill_mixed.cu (a translation unit of their own, so the two build in
// parallel).
#include "attend_prefill_kernel.cuh"

namespace kvq {

bool prefill_supported(const AttendArgs &a) {
  // block layouts: the query must be exact in f16 after a power-of-two prescale (bf16, f16)
  const bool q_ok = is_hadamard(a.cache.layout) || a.q_dtype != KVQ_F32;
  return prefill_shape(a.cache.layout, a.cache.v_layout, a.cache.D, a.gqa * a.n_q) && q_ok && a.n_body > 0 &&
         a.chunk % kStage == 0;
}

cudaError_t launch_attend_prefill(const AttendArgs &a, cudaStream_t st) {
  if (a.cache.layout != a.cache.v_layout) return launch_attend_prefill_mixed(a, st);
  switch (a.cache.layout) {
    case KVQ_HAD_INT4: return launch_pair<KVQ_HAD_INT4, KVQ_HAD_INT4>(a, st);
    case KVQ_HAD_INT2: return launch_pair<KVQ_HAD_INT2, KVQ_HAD_INT2>(a, st);
    case KVQ_ASYM4_G32: return launch_pair<KVQ_ASYM4_G32, KVQ_ASYM4_G32>(a, st);
    case KVQ_Q8_0: return launch_pair<KVQ_Q8_0, KVQ_Q8_0>(a, st);
    case KVQ_Q4_0: return launch_pair<KVQ_Q4_0, KVQ_Q4_0>(a, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kvq
