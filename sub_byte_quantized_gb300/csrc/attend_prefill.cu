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

// Many-row Hadamard calls: the query preparation (int8 codes and scales, and the rotated f32 rows
// when there is a window), then one tcgen05 grid for the body chunks and the window chunks. Launch
// chaining: the preparation waits for the preceding kernel (a plain launch); every tcgen05 CTA waits
// for the preparation. Score capture runs the window chunks on the row-side kernel afterwards (its
// first CTA waits for the tcgen05 grid, and every CTA of a prepared-query window chunk waits).
cudaError_t launch_prefill_tc(const AttendArgs &a, cudaStream_t st) {
  cudaError_t e = launch_had_prep(a, st, a.n_wchunks > 0);   // f32 rotated rows for the window chunks
  if (e == cudaSuccess) e = launch_attend_prefill_tc_body(a, st);
  if (e != cudaSuccess || a.n_wchunks == 0 || !a.cap_scores) return e;
  AttendArgs w = a;
  w.y_base = a.n_chunks;                                 // window chunks only
  w.q_prepped = 1;
  w.cap_scores = nullptr;
  return a.cache.layout == KVQ_HAD_INT2 ? launch_pair<KVQ_HAD_INT2, KVQ_HAD_INT2>(w, st)
                                        : launch_pair<KVQ_HAD_INT4, KVQ_HAD_INT4>(w, st);
}

cudaError_t launch_attend_prefill(const AttendArgs &a, cudaStream_t st) {
  if (tc_prefill_shape(a.cache.layout, a.cache.v_layout, a.cache.D, a.gqa * a.n_q)) return launch_prefill_tc(a, st);
  if (a.cache.layout != a.cache.v_layout) return launch_attend_prefill_mixed(a, st);
  switch (a.cache.layout) {
    case KVQ_HAD_INT4: return launch_pair<KVQ_HAD_INT4, KVQ_HAD_INT4>(a, st);
    case KVQ_HAD_INT2: return launch_pair<KVQ_HAD_INT2, KVQ_HAD_INT2>(a, st);
    case KVQ_ASYM4_G32: return launch_pair<KVQ_ASYM4_G32, KVQ_ASYM4_G32>(a, st);
    case KVQ_Q8_0: return launch_pair<KVQ_Q8_0, KVQ_Q8_0>(a, st);
    case KVQ_Q4_0: return launch_pair<KVQ_Q4_0, KVQ_Q4_0>(a, st);
    case KVQ_Q6_0: return launch_pair<KVQ_Q6_0, KVQ_Q6_0>(a, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kvq
