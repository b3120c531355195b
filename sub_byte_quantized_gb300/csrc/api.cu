// C ABI of the library: host-side validation, workspace layout and kernel launches.
// Nothing here allocates, synchronises or prints; failures return a kvq_status and record a
// one-line reason readable through kvq_last_error().
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kvq_internal.cuh"

namespace {

thread_local char g_last_error[256] = "";
thread_local cudaEvent_t g_ev_begin = nullptr, g_ev_end = nullptr;

kvq_status fail(kvq_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t row_bytes_of(int layout, int D) {
  if (D != 128 && D != 256) return 0;
  const int nb = D / kvq::kBlock;
  switch (layout) {
    case KVQ_Q4_0: return 16 * (size_t)nb;
    case KVQ_Q6_0: return 24 * (size_t)nb;
    case KVQ_HAD_INT4: return (size_t)D / 2;
    case KVQ_HAD_INT2: return (size_t)D / 4;
    case KVQ_Q8_0: return 32 * (size_t)nb;
    case KVQ_ASYM4_G32: return 16 * (size_t)nb;
    default: return 0;
  }
}

// The K and V layouts of a cache's layout field (plain, or KVQ_MIXED(k, v)); false when invalid.
bool split_layout(int32_t layout, int &k, int &v) {
  k = layout & 0xFF;
  v = (layout >> 8) ? (layout >> 8) - 1 : k;
  if ((layout >> 8) > kvq::kLastLayout + 1 || layout < 0) return false;
  if (k > kvq::kLastLayout || v > kvq::kLastLayout) return false;
  return kvq::is_hadamard(k) == kvq::is_hadamard(v);
}

// Layout checks shared by the contiguous and paged caches: both planes' layouts, head_dim, the
// window option and the plane pointers each plane's layout needs.
kvq_status check_planes(int32_t layout, int32_t head_dim, int32_t n_recent, const void *k_zero, const void *v_zero,
                        const float *k_recent, const float *v_recent, kvq::CacheView &v) {
  int kl, vl;
  if (!split_layout(layout, kl, vl)) return fail(KVQ_EINVAL, "unknown layout %d (or a rotated/unrotated mix)", layout);
  if (head_dim != 128 && head_dim != 256) return fail(KVQ_ESHAPE, "head_dim %d not 128/256", head_dim);
  if (n_recent < 0) return fail(KVQ_EINVAL, "n_recent < 0");
  if (!kvq::is_hadamard(kl) && n_recent != 0) return fail(KVQ_EUNSUPPORTED, "n_recent is an option of the Hadamard layouts");
  if (kl == KVQ_ASYM4_G32 && !k_zero) return fail(KVQ_EINVAL, "zero-point planes are NULL");
  if (vl == KVQ_ASYM4_G32 && !v_zero) return fail(KVQ_EINVAL, "zero-point planes are NULL");
  if ((k_zero && !aligned(k_zero, 16)) || (v_zero && !aligned(v_zero, 16)))
    return fail(KVQ_EALIGN, "zero plane not 16-byte aligned");
  if (kvq::is_hadamard(kl) && n_recent > 0) {
    if (!k_recent || !v_recent) return fail(KVQ_EINVAL, "recent-window planes are NULL");
    if (!aligned(k_recent, 16) || !aligned(v_recent, 16)) return fail(KVQ_EALIGN, "window plane not 16-byte aligned");
  }
  v.layout = kl;
  v.v_layout = vl;
  v.row_bytes = (int)row_bytes_of(kl, head_dim);
  v.v_row_bytes = (int)row_bytes_of(vl, head_dim);
  v.n_recent = kvq::is_hadamard(kl) ? n_recent : 0;
  return KVQ_OK;
}

kvq_status check_cache(const kvq_cache *c, kvq::CacheView &v) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  kvq_status st = check_planes(c->layout, c->head_dim, c->n_recent, c->k_zero, c->v_zero, c->k_recent, c->v_recent, v);
  if (st != KVQ_OK) return st;
  if (c->batch < 1 || c->n_kv_heads < 1 || c->capacity < 1)
    return fail(KVQ_EINVAL, "batch, n_kv_heads and capacity must be >= 1");
  const void *ptrs[] = {c->k_payload, c->v_payload, c->k_scale, c->v_scale};
  for (const void *p : ptrs) {
    if (!p) return fail(KVQ_EINVAL, "payload/scale pointer is NULL");
    if (!aligned(p, 16)) return fail(KVQ_EALIGN, "payload/scale pointer not 16-byte aligned");
  }
  v.B = c->batch; v.H = c->n_kv_heads; v.D = c->head_dim; v.cap = c->capacity;
  v.payload[0] = static_cast<uint8_t *>(c->k_payload);
  v.payload[1] = static_cast<uint8_t *>(c->v_payload);
  v.scale[0] = c->k_scale; v.scale[1] = c->v_scale;
  v.zero[0] = static_cast<__half *>(c->k_zero);
  v.zero[1] = static_cast<__half *>(c->v_zero);
  v.ring[0] = c->k_recent; v.ring[1] = c->v_recent;
  v.page_shift = -1; v.table_stride = 0; v.n_pages = 0; v.table = nullptr;
  return KVQ_OK;
}

// Validation of a paged pool and its block table.
kvq_status check_paged_cache(const kvq_paged_cache *c, kvq::CacheView &v) {
  if (!c) return fail(KVQ_EINVAL, "cache is NULL");
  kvq_status st = check_planes(c->layout, c->head_dim, c->n_recent, c->k_zero, c->v_zero, c->k_recent, c->v_recent, v);
  if (st != KVQ_OK) return st;
  if (c->batch < 1 || c->n_kv_heads < 1 || c->n_pages < 1 || c->max_pages_per_seq < 1)
    return fail(KVQ_EINVAL, "batch, n_kv_heads, n_pages and max_pages_per_seq must be >= 1");
  int shift = -1;
  for (int k = kvq::kMinPageShift; k <= 20; ++k)
    if (c->page_size == (1 << k)) shift = k;
  if (shift < 0) return fail(KVQ_ESHAPE, "page_size %d is not a power of two in [64, 2^20]", c->page_size);
  if ((long long)c->max_pages_per_seq * c->page_size > INT_MAX)
    return fail(KVQ_ECAPACITY, "max_pages_per_seq * page_size exceeds INT_MAX tokens");
  const void *ptrs[] = {c->k_payload, c->v_payload, c->k_scale, c->v_scale, c->block_table};
  for (const void *p : ptrs) {
    if (!p) return fail(KVQ_EINVAL, "payload/scale/block_table pointer is NULL");
    if (!aligned(p, 16)) return fail(KVQ_EALIGN, "payload/scale/block_table pointer not 16-byte aligned");
  }
  v.B = c->batch; v.H = c->n_kv_heads; v.D = c->head_dim;
  v.cap = c->max_pages_per_seq * c->page_size;
  v.payload[0] = static_cast<uint8_t *>(c->k_payload);
  v.payload[1] = static_cast<uint8_t *>(c->v_payload);
  v.scale[0] = c->k_scale; v.scale[1] = c->v_scale;
  v.zero[0] = static_cast<__half *>(c->k_zero);
  v.zero[1] = static_cast<__half *>(c->v_zero);
  v.ring[0] = c->k_recent; v.ring[1] = c->v_recent;
  v.page_shift = shift; v.table_stride = c->max_pages_per_seq; v.n_pages = c->n_pages;
  v.table = c->block_table;
  return KVQ_OK;
}

// Validation of an append (no launch). want_layout < 0 accepts the cache's own layout.
kvq_status check_store(int want_layout, const kvq_cache *cache, const void *k_new, const void *v_new, int dtype,
                       int n_new, int pos0, kvq::CacheView &v) {
  kvq_status st = check_cache(cache, v);
  if (st != KVQ_OK) return st;
  if (want_layout >= 0 && (v.layout != want_layout || v.v_layout != want_layout))
    return fail(KVQ_EUNSUPPORTED, "cache layout %d does not match this store (kvq_store takes any layout)",
                cache->layout);
  if (dtype < KVQ_F32 || dtype > KVQ_F16) return fail(KVQ_EINVAL, "unknown dtype %d", dtype);
  if (n_new < 0 || pos0 < 0) return fail(KVQ_EINVAL, "n_new and pos0 must be >= 0");
  if ((long long)pos0 + n_new > v.cap) return fail(KVQ_ECAPACITY, "pos0 + n_new = %lld > capacity %d",
                                                  (long long)pos0 + n_new, v.cap);
  if (n_new == 0) return KVQ_OK;
  if (!k_new || !v_new) return fail(KVQ_EINVAL, "k_new/v_new is NULL");
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(KVQ_EALIGN, "k_new/v_new not 16-byte aligned");
  return KVQ_OK;
}

kvq_status store_common(int want_layout, const kvq_cache *cache, const void *k_new, const void *v_new, int dtype,
                        int n_new, int pos0, kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::CacheView v;
  kvq_status st = check_store(want_layout, cache, k_new, v_new, dtype, n_new, pos0, v);
  if (st != KVQ_OK || n_new == 0) return st;
  cudaError_t e = kvq::launch_store(v, k_new, v_new, dtype, n_new, pos0, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "store launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

// Automatic split-K chunk, sized for the tensor-core kernel that will run. Decode (up to eight
// query rows per kv head), one wave: for the per-warp kernel four times the smallest multiple of
// 32 tokens (a warp's stage) that gives one slice to every resident warp (four warps per chunk);
// for the warp-specialised kernels (Q6_0, asymmetric) the smallest multiple of 64 that gives one
// chunk to every resident CTA. Many rows: about four waves of 64-row CTAs on the row-side kernel,
// the fewest waves x stages of 256-row CTAs on the tcgen05 kernel.
// `work` = body tokens summed over every (batch, kv head) (0: n_body for each of them); a ragged
// batch passes its true total so the chunk fits the work that exists.
// n_wchunks: window chunks per (batch, kv head) that the row-side kernel scores in the same grid.
int auto_chunk(const kvq::CacheView &c, int rows, int n_body, int n_heads, long long work = 0, int n_wchunks = 0) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool total_given = work > 0;
  if (!total_given) work = (long long)(n_body > 0 ? n_body : 1) * n_heads;
  long long chunk;
  if (c.layout == KVQ_Q6_0 && kvq::mma_q6_shape(c.D, rows) && !kvq::prefill_shape(c.layout, c.v_layout, c.D, rows)) {
    // one chunk per resident CTA; each group of four query rows has its own CTAs
    const long long ctas = (long long)sms * kvq::kMmaQ6CtasPerSm(c.D);
    const long long groups = (rows + 3) / 4;
    chunk = ((work * groups + ctas - 1) / ctas + 63) / 64 * 64;
  } else if (kvq::prefill_shape(c.layout, c.v_layout, c.D, rows) && rows <= 16 &&
             !kvq::decode_kernel(c.layout, c.v_layout)) {
    // row-side kernel in its decode form (one row block, the warps split the tokens): one chunk per
    // resident CTA, as many chunks per (batch, kv head) as fit one wave
    const long long ctas = (long long)sms * (kvq::is_hadamard(c.layout) ? kvq::kPrefillCtasPerSm : 2);
    long long per_head = ctas / (n_heads > 0 ? n_heads : 1);   // (the window is scored in phase 2)
    if (per_head < 1) per_head = 1;
    const long long body = total_given ? (work + n_heads - 1) / n_heads : (n_body > 0 ? n_body : 1);
    chunk = ((body + per_head - 1) / per_head + 63) / 64 * 64;
  } else if (kvq::tc_prefill_shape(c.layout, c.v_layout, c.D, rows)) {
    // tcgen05 kernel, one CTA of 256 rows per SM: the number of body chunks per row block (1..8)
    // whose grid takes the fewest waves x (stages per chunk + about two stages of fixed cost per CTA)
    const long long units = (long long)((rows + kvq::kTcRows - 1) / kvq::kTcRows) * n_heads;
    const long long body = total_given ? (work + n_heads - 1) / n_heads : (n_body > 0 ? n_body : 1);
    const long long stages = (body + 63) / 64;
    long long best = 1, best_cost = -1;
    for (long long n = 1; n <= 8; ++n) {
      const long long per = (stages + n - 1) / n;
      if (per * 64 > 8192) continue;
      const long long waves = (units * n + sms - 1) / sms;
      const long long cost = waves * (per + 2);
      if (best_cost < 0 || cost < best_cost) { best = n; best_cost = cost; }
    }
    chunk = ((stages + best - 1) / best) * 64;
  } else if (kvq::prefill_shape(c.layout, c.v_layout, c.D, rows)) {
    // row-side kernel: CTAs of 64 query rows; split the body into enough chunks for about four
    // waves of resident CTAs
    const long long row_ctas = (long long)((rows + kvq::kPrefillRows - 1) / kvq::kPrefillRows) * n_heads;
    const long long want = 4LL * sms * kvq::kPrefillCtasPerSm;
    long long n_chunks = (want + row_ctas - 1) / row_ctas;
    if (n_chunks < 1) n_chunks = 1;
    const long long body = total_given ? (work + n_heads - 1) / n_heads : (n_body > 0 ? n_body : 1);
    chunk = ((body + n_chunks - 1) / n_chunks + 63) / 64 * 64;
  } else if (kvq::uses_mma4(c.layout)) {
    // warp-specialised 4-bit kernel: one chunk per resident CTA, as many chunks per (batch, kv
    // head) as fit one wave
    const long long ctas = (long long)sms * kvq::kMma4CtasPerSm;
    long long per_head = ctas / (n_heads > 0 ? n_heads : 1);
    if (per_head < 1) per_head = 1;
    const long long body = total_given ? (work + n_heads - 1) / n_heads : (n_body > 0 ? n_body : 1);
    chunk = ((body + per_head - 1) / per_head + 63) / 64 * 64;
  } else {
    const long long warps = (long long)sms * kvq::kMmaWarpsPerSm;
    chunk = 4 * (((work + warps - 1) / warps + 31) / 32 * 32);   // a warp's slice: whole 32-token stages
  }
  if (chunk > 8192) chunk = 8192;
  return (int)chunk;
}

// Resolve the attention arguments and the workspace layout for a checked cache view `a.cache`
// (kv_len: the call's length, or the largest per-sequence length of a paged call). When `ws` is
// NULL only sizes are computed (returned through `need`).
kvq_status resolve_core(int n_q_heads, int n_q, int kv_len, int causal, int q_pos0, bool paged, int chunk,
                        kvq::AttendArgs &a, size_t &need, void *ws, long long work = 0) {
  const kvq::CacheView &c = a.cache;
  if (n_q_heads < 1 || n_q < 1) return fail(KVQ_EINVAL, "n_q_heads and n_q must be >= 1");
  if (n_q_heads % c.H) return fail(KVQ_ESHAPE, "n_q_heads %d not a multiple of n_kv_heads %d", n_q_heads, c.H);
  if (kv_len < 1) return fail(KVQ_EINVAL, "kv_len must be >= 1");
  if (kv_len > c.cap) return fail(KVQ_ECAPACITY, "kv_len %d > capacity %d", kv_len, c.cap);
  if (!paged && causal && (q_pos0 < 0 || (long long)q_pos0 + n_q > kv_len))
    return fail(KVQ_EINVAL, "causal call needs 0 <= q_pos0 and q_pos0 + n_q <= kv_len");
  if (chunk == 0)
  {
    const int n_win = kvq::is_hadamard(c.layout) ? (c.n_recent < kv_len ? c.n_recent : kv_len) : 0;
    chunk = auto_chunk(c, (n_q_heads / c.H) * n_q, kv_len - n_win, c.B * c.H, work,
                       (n_win + kvq::kWinChunk - 1) / kvq::kWinChunk);
  }
  if (chunk < 64 || chunk > 8192 || chunk % 64) return fail(KVQ_ESHAPE, "chunk %d not a multiple of 64 in [64, 8192]", chunk);
  a.Hq = n_q_heads; a.gqa = n_q_heads / c.H; a.n_q = n_q;
  a.kv_len = kv_len;
  a.n_win = kvq::is_hadamard(c.layout) ? (c.n_recent < kv_len ? c.n_recent : kv_len) : 0;
  a.n_body = kv_len - a.n_win;
  a.causal = causal ? 1 : 0;
  a.q_pos0 = causal ? q_pos0 : 0;
  a.chunk = chunk;
  a.n_chunks = (a.n_body + chunk - 1) / chunk;
  a.n_wchunks = (a.n_win + kvq::kWinChunk - 1) / kvq::kWinChunk;
  a.C = a.n_chunks + a.n_wchunks;
  a.win_in_reduce = 0;
  a.y_base = 0;
  a.q_prepped = 0;
  a.fresh_lo = 0;
  a.fresh_hi = INT_MAX;
  a.seq_lens = nullptr;
  a.fresh_tail = 0;
  a.cap_scores = nullptr;
  a.cap_sq = nullptr;
  const size_t rows = (size_t)c.B * n_q_heads * n_q;
  size_t off = 0;
  const size_t o_m = off; off = round_up(off + rows * a.C * sizeof(float), 256);
  const size_t o_l = off; off = round_up(off + rows * a.C * sizeof(float), 256);
  const size_t o_o = off; off = round_up(off + rows * a.C * (size_t)c.D * sizeof(float), 256);
  size_t o_q8 = 0, o_sq = 0, o_qr = 0;
  if (kvq::is_hadamard(c.layout)) {
    o_q8 = off; off = round_up(off + rows * (size_t)c.D, 256);
    o_sq = off; off = round_up(off + rows * sizeof(float), 256);
    o_qr = off; off = round_up(off + rows * (size_t)c.D * sizeof(float), 256);
  }
  need = off;
  if (ws) {
    char *w = static_cast<char *>(ws);
    a.part_m = reinterpret_cast<float *>(w + o_m);
    a.part_l = reinterpret_cast<float *>(w + o_l);
    a.part_o = reinterpret_cast<float *>(w + o_o);
    a.q8 = kvq::is_hadamard(c.layout) ? reinterpret_cast<int8_t *>(w + o_q8) : nullptr;
    a.s_q = kvq::is_hadamard(c.layout) ? reinterpret_cast<float *>(w + o_sq) : nullptr;
    a.q_rot = kvq::is_hadamard(c.layout) ? reinterpret_cast<float *>(w + o_qr) : nullptr;
  }
  return KVQ_OK;
}

kvq_status resolve_attend(const kvq_cache *cache, int n_q_heads, int n_q, int kv_len, int causal, int q_pos0,
                          int chunk, kvq::AttendArgs &a, size_t &need, void *ws) {
  kvq_status st = check_cache(cache, a.cache);
  if (st != KVQ_OK) return st;
  return resolve_core(n_q_heads, n_q, kv_len, causal, q_pos0, false, chunk, a, need, ws);
}

// Paged call: the grid is sized for max_kv_len; per-sequence lengths are read on the device.
kvq_status resolve_paged(const kvq_paged_cache *cache, int n_q_heads, int n_q, int max_kv_len, int causal, int chunk,
                         kvq::AttendArgs &a, size_t &need, void *ws, long long total_kv_len = 0) {
  kvq_status st = check_paged_cache(cache, a.cache);
  if (st != KVQ_OK) return st;
  long long work = 0;                                    // body tokens over all sequences and kv heads
  if (total_kv_len > 0) {
    const long long win = kvq::is_hadamard(cache->layout & 0xFF) ? (long long)cache->n_recent * cache->batch : 0;
    work = (total_kv_len > win ? total_kv_len - win : 1) * cache->n_kv_heads;
  }
  return resolve_core(n_q_heads, n_q, max_kv_len, causal, 0, true, chunk, a, need, ws, work);
}

}  // namespace

extern "C" {

size_t kvq_row_bytes(int32_t layout, int32_t head_dim) { return row_bytes_of(layout, head_dim); }

kvq_status kvq_cache_bytes(int32_t layout, int32_t batch, int32_t n_kv_heads, int32_t head_dim, int32_t capacity,
                           int32_t n_recent, size_t out_sizes[4]) {
  g_last_error[0] = 0;
  if (!out_sizes) return fail(KVQ_EINVAL, "out_sizes is NULL");
  const size_t rb = row_bytes_of(layout, head_dim);
  if (layout < KVQ_Q4_0 || layout > kvq::kLastLayout) return fail(KVQ_EINVAL, "unknown layout %d", layout);
  if (!rb) return fail(KVQ_ESHAPE, "head_dim %d not 128/256", head_dim);
  if (batch < 1 || n_kv_heads < 1 || capacity < 1 || n_recent < 0) return fail(KVQ_EINVAL, "bad sizes");
  const size_t rows = (size_t)batch * n_kv_heads * capacity;
  const size_t nb = (size_t)head_dim / kvq::kBlock;
  out_sizes[0] = rows * rb;
  out_sizes[1] = kvq::is_hadamard(layout) ? rows * sizeof(float) : rows * nb * 2;
  out_sizes[2] = layout == KVQ_ASYM4_G32 ? rows * nb * 2 : 0;
  out_sizes[3] = kvq::is_hadamard(layout) ? (size_t)batch * n_kv_heads * n_recent * head_dim * sizeof(float) : 0;
  return KVQ_OK;
}

kvq_status kvq_store_q4_0(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t dtype, int32_t n_new,
                          int32_t pos0, kvq_stream_t stream) {
  return store_common(KVQ_Q4_0, cache, k_new, v_new, dtype, n_new, pos0, stream);
}
kvq_status kvq_store_q6_0(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t dtype, int32_t n_new,
                          int32_t pos0, kvq_stream_t stream) {
  return store_common(KVQ_Q6_0, cache, k_new, v_new, dtype, n_new, pos0, stream);
}
kvq_status kvq_store_hadamard_int4(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t dtype,
                                   int32_t n_new, int32_t pos0, kvq_stream_t stream) {
  return store_common(KVQ_HAD_INT4, cache, k_new, v_new, dtype, n_new, pos0, stream);
}
kvq_status kvq_store_asym4_g32(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t dtype,
                               int32_t n_new, int32_t pos0, kvq_stream_t stream) {
  return store_common(KVQ_ASYM4_G32, cache, k_new, v_new, dtype, n_new, pos0, stream);
}
kvq_status kvq_store_q8_0(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t dtype, int32_t n_new,
                          int32_t pos0, kvq_stream_t stream) {
  return store_common(KVQ_Q8_0, cache, k_new, v_new, dtype, n_new, pos0, stream);
}
kvq_status kvq_store_hadamard_int2(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t dtype,
                                   int32_t n_new, int32_t pos0, kvq_stream_t stream) {
  return store_common(KVQ_HAD_INT2, cache, k_new, v_new, dtype, n_new, pos0, stream);
}
kvq_status kvq_store(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t dtype, int32_t n_new,
                     int32_t pos0, kvq_stream_t stream) {
  return store_common(-1, cache, k_new, v_new, dtype, n_new, pos0, stream);
}

size_t kvq_attend_workspace_bytes(const kvq_cache *cache, int32_t n_q_heads, int32_t n_q, int32_t kv_len,
                                  int32_t chunk) {
  kvq::AttendArgs a;
  size_t need = 0;
  if (resolve_attend(cache, n_q_heads, n_q, kv_len, 0, 0, chunk, a, need, nullptr) != KVQ_OK) return 0;
  return need;
}

int32_t kvq_attend_chunk(const kvq_cache *cache, int32_t n_q_heads, int32_t n_q, int32_t kv_len, int32_t chunk) {
  kvq::AttendArgs a;
  size_t need = 0;
  if (resolve_attend(cache, n_q_heads, n_q, kv_len, 0, 0, chunk, a, need, nullptr) != KVQ_OK) return 0;
  return a.chunk;
}

namespace {

// The query, output, workspace and scale arguments of an attention call.
kvq_status check_call(size_t need, const void *q, int32_t q_dtype, float attn_scale, const float *out,
                      const void *workspace, size_t workspace_bytes) {
  if (q_dtype < KVQ_F32 || q_dtype > KVQ_F16) return fail(KVQ_EINVAL, "unknown q dtype %d", q_dtype);
  if (!q || !out || !workspace) return fail(KVQ_EINVAL, "q/out/workspace is NULL");
  if (!aligned(q, 16) || !aligned(out, 16)) return fail(KVQ_EALIGN, "q/out not 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(KVQ_EALIGN, "workspace not 256-byte aligned");
  if (workspace_bytes < need) return fail(KVQ_EWORKSPACE, "workspace %zu < required %zu", workspace_bytes, need);
  if (!(attn_scale == attn_scale) || attn_scale > 3.0e38f || attn_scale < -3.0e38f)
    return fail(KVQ_EINVAL, "attn_scale must be finite");
  return KVQ_OK;
}

// Validation of an attention call and its workspace; on success `a` is fully resolved.
kvq_status prepare_attend(const kvq_cache *cache, const void *q, int32_t q_dtype, int32_t n_q_heads, int32_t n_q,
                          int32_t kv_len, int32_t causal, int32_t q_pos0, float attn_scale, int32_t chunk,
                          float *out, void *workspace, size_t workspace_bytes, kvq::AttendArgs &a) {
  size_t need = 0;
  kvq_status st = resolve_attend(cache, n_q_heads, n_q, kv_len, causal, q_pos0, chunk, a, need, nullptr);
  if (st != KVQ_OK) return st;
  st = check_call(need, q, q_dtype, attn_scale, out, workspace, workspace_bytes);
  if (st != KVQ_OK) return st;
  resolve_attend(cache, n_q_heads, n_q, kv_len, causal, q_pos0, chunk, a, need, workspace);
  a.q = q;
  a.q_dtype = q_dtype;
  a.scale = attn_scale;
  a.out = out;
  return KVQ_OK;
}

// Phase 1 (tensor-core or CUDA-core kernel) and phase 2 on `s`, with the optional phase-1 events.
cudaError_t launch_attend_sequence(kvq::AttendArgs &a, cudaStream_t s, bool events) {
  cudaError_t e = cudaSuccess;
  const bool mma = kvq::mma_supported(a);
  // the decode tensor-core kernels (and the row-side kernel's decode form) cover the body chunks only
  a.win_in_reduce = mma && a.n_win > 0 &&
                    (!kvq::prefill_supported(a) ||
                     kvq::dec_shape(a.cache.layout, a.cache.v_layout, a.cache.D, a.gqa * a.n_q));
  // the tensor-core kernels prepare the Hadamard query themselves; the CUDA-core one reads it
  if (kvq::is_hadamard(a.cache.layout) && !mma) {
    a.fresh_lo = 0;                                      // its predecessor is then the prep kernel
    a.fresh_hi = INT_MAX;
    a.fresh_tail = 0;
    e = kvq::launch_had_prep(a, s);
  }
  const bool prof = events && g_ev_begin && g_ev_end;
  // Under stream capture an event record must be external to become a graph node.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (e == cudaSuccess && prof) e = cudaStreamIsCapturing(s, &cap);
  const unsigned rec_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  if (e == cudaSuccess && prof) e = cudaEventRecordWithFlags(g_ev_begin, s, rec_flags);
  if (e == cudaSuccess) e = mma ? kvq::launch_attend_mma(a, s) : kvq::launch_attend_generic(a, s);
  if (e == cudaSuccess && prof) e = cudaEventRecordWithFlags(g_ev_end, s, rec_flags);
  if (e == cudaSuccess) e = kvq::launch_attend_reduce(a, s, true);
  return e;
}

// The append (when n_new > 0) and the attention of a validated append + attend call.
cudaError_t launch_append_attend(const kvq::CacheView &v, kvq::AttendArgs &a, const void *k_new, const void *v_new,
                                 int kv_dtype, int n_new, int pos0, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (n_new > 0) {
    e = kvq::launch_store(v, k_new, v_new, kv_dtype, n_new, pos0, s);
    a.fresh_lo = pos0;                                   // the rows (and window slots) it writes
    a.fresh_hi = pos0 + n_new;
  }
  if (e == cudaSuccess) e = launch_attend_sequence(a, s, true);
  return e;
}

size_t dtype_bytes(int32_t dt) { return dt == KVQ_F32 ? 4 : 2; }

// Device staging of a host-buffer call, in the caller's workspace after the attention partials:
// k_new, v_new, q, out and (paged) seq_lens, each from a 256-byte boundary.
struct HostStaging {
  size_t k = 0, v = 0, q = 0, out = 0, lens = 0, total = 0;
  size_t kv_bytes = 0, q_bytes = 0, out_bytes = 0, lens_bytes = 0;
};

HostStaging host_staging(size_t attend_need, int batch, int n_kv_heads, int head_dim, int kv_dtype, int n_new,
                         int q_dtype, int n_q_heads, int n_q, bool paged) {
  HostStaging h;
  h.kv_bytes = n_new > 0 ? (size_t)batch * n_kv_heads * n_new * head_dim * dtype_bytes(kv_dtype) : 0;
  h.q_bytes = (size_t)batch * n_q_heads * n_q * head_dim * dtype_bytes(q_dtype);
  h.out_bytes = (size_t)batch * n_q_heads * n_q * head_dim * sizeof(float);
  h.lens_bytes = paged ? (size_t)batch * sizeof(int32_t) : 0;
  // k_new, v_new and q back to back (each size is a multiple of 256 bytes: head_dim 128 or 256), so
  // host inputs that are back to back too arrive with one copy
  h.k = round_up(attend_need, 256);
  h.v = h.k + h.kv_bytes;
  h.q = h.v + h.kv_bytes;
  h.out = h.q + round_up(h.q_bytes, 256);
  h.lens = h.out + round_up(h.out_bytes, 256);
  h.total = h.lens + round_up(h.lens_bytes, 256);
  return h;
}

// The element types and row count that size a host-buffer call's staging.
kvq_status check_host_sizes(int kv_dtype, int n_new, int q_dtype) {
  if (q_dtype < KVQ_F32 || q_dtype > KVQ_F16) return fail(KVQ_EINVAL, "unknown q dtype %d", q_dtype);
  if (kv_dtype < KVQ_F32 || kv_dtype > KVQ_F16) return fail(KVQ_EINVAL, "unknown dtype %d", kv_dtype);
  if (n_new < 0) return fail(KVQ_EINVAL, "n_new must be >= 0");
  return KVQ_OK;
}

// The host-side arguments of a host-buffer call that the device entry points cannot see.
kvq_status check_host_args(int kv_dtype, int n_new, int q_dtype, const void *k_new, const void *v_new, const void *q,
                           const float *out, const void *workspace) {
  const kvq_status st = check_host_sizes(kv_dtype, n_new, q_dtype);
  if (st != KVQ_OK) return st;
  if (n_new > 0 && (!k_new || !v_new)) return fail(KVQ_EINVAL, "k_new/v_new is NULL");
  if (!q || !out || !workspace) return fail(KVQ_EINVAL, "q/out/workspace is NULL");
  return KVQ_OK;
}

// The device address of a host buffer that the GPU reads and writes in place: pinned memory
// (cudaHostAlloc / cudaMallocHost, or registered), which unified addressing maps into every
// device's address space, and 16-byte aligned like the device-buffer calls require; nullptr for
// anything else (pageable memory goes through the staging copies).
void *device_view(const void *p) {
  if (!p || !aligned(p, 16)) return nullptr;
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
    cudaGetLastError();                                  // not a CUDA-known pointer: clear the error
    return nullptr;
  }
  return pa.type == cudaMemoryTypeHost ? pa.devicePointer : nullptr;
}

// Where a host-buffer call's kernels find their inputs and put their output. Pinned caller
// buffers are used in place where that saves a copy operation: the store kernel reads k_new /
// v_new over the host link (each element once) and the reduce writes the result there. q is
// always staged in device memory, since every phase-1 CTA of a kv head reads it (reading it over
// the link measured slower than one small copy). Pageable buffers go through the staging area of
// the workspace with a copy each way.
struct HostIo {
  const void *k, *v, *q;
  float *out;
  bool copy_in, copy_out;                                // copy_in: k_new and v_new staged with q
};
HostIo host_io(const HostStaging &h, char *ws, int n_new, const void *k_new, const void *v_new, float *out) {
  HostIo io;
  const void *kd = n_new > 0 ? device_view(k_new) : nullptr, *vd = n_new > 0 ? device_view(v_new) : nullptr;
  io.copy_in = !(n_new == 0 || (kd && vd));
  io.k = io.copy_in ? ws + h.k : kd;
  io.v = io.copy_in ? ws + h.v : vd;
  io.q = ws + h.q;
  float *od = static_cast<float *>(device_view(out));
  io.copy_out = od == nullptr;
  io.out = io.copy_out ? reinterpret_cast<float *>(ws + h.out) : od;
  return io;
}

// Host -> staging copies of the inputs (cudaMemcpyDefault: pinned or pageable host memory).
cudaError_t copy_in(const HostStaging &h, char *ws, const void *k_new, const void *v_new, const void *q,
                    const void *seq_lens, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  const char *kb = static_cast<const char *>(k_new), *vb = static_cast<const char *>(v_new);
  if (h.kv_bytes && vb == kb + h.kv_bytes && static_cast<const char *>(q) == vb + h.kv_bytes) {
    e = cudaMemcpyAsync(ws + h.k, k_new, 2 * h.kv_bytes + h.q_bytes, cudaMemcpyDefault, s);   // one copy
  } else if (h.kv_bytes) {
    e = cudaMemcpyAsync(ws + h.k, k_new, h.kv_bytes, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ws + h.v, v_new, h.kv_bytes, cudaMemcpyDefault, s);
  }
  if (e == cudaSuccess && !(h.kv_bytes && vb == kb + h.kv_bytes && static_cast<const char *>(q) == vb + h.kv_bytes))
    e = cudaMemcpyAsync(ws + h.q, q, h.q_bytes, cudaMemcpyDefault, s);
  if (e == cudaSuccess && h.lens_bytes) e = cudaMemcpyAsync(ws + h.lens, seq_lens, h.lens_bytes, cudaMemcpyDefault, s);
  return e;
}

// Staging -> host copy of the output, then wait for the stream.
cudaError_t copy_out_and_wait(const HostStaging &h, const char *ws, float *out, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(out, ws + h.out, h.out_bytes, cudaMemcpyDefault, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e;
}

}  // namespace

kvq_status kvq_decode_attend(const kvq_cache *cache, const void *q, int32_t q_dtype, int32_t n_q_heads, int32_t n_q,
                             int32_t kv_len, int32_t causal, int32_t q_pos0, float attn_scale, int32_t chunk,
                             float *out, void *workspace, size_t workspace_bytes, kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::AttendArgs a;
  kvq_status st = prepare_attend(cache, q, q_dtype, n_q_heads, n_q, kv_len, causal, q_pos0, attn_scale, chunk, out,
                                 workspace, workspace_bytes, a);
  if (st != KVQ_OK) return st;
  cudaError_t e = launch_attend_sequence(a, reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "attend launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

kvq_status kvq_append_decode_attend(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t kv_dtype,
                                    int32_t n_new, int32_t pos0, const void *q, int32_t q_dtype, int32_t n_q_heads,
                                    int32_t n_q, int32_t kv_len, int32_t causal, int32_t q_pos0, float attn_scale,
                                    int32_t chunk, float *out, void *workspace, size_t workspace_bytes,
                                    kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::CacheView v;
  kvq_status st = check_store(-1, cache, k_new, v_new, kv_dtype, n_new, pos0, v);
  if (st != KVQ_OK) return st;
  kvq::AttendArgs a;
  st = prepare_attend(cache, q, q_dtype, n_q_heads, n_q, kv_len, causal, q_pos0, attn_scale, chunk, out, workspace,
                      workspace_bytes, a);
  if (st != KVQ_OK) return st;
  const cudaError_t e = launch_append_attend(v, a, k_new, v_new, kv_dtype, n_new, pos0,
                                             reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "append/attend launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

// ------------------------------------------------------------------ paged pool
kvq_status kvq_paged_cache_bytes(int32_t layout, int32_t n_pages, int32_t n_kv_heads, int32_t head_dim,
                                 int32_t page_size, int32_t batch, int32_t n_recent, size_t out_sizes[4]) {
  g_last_error[0] = 0;
  if (!out_sizes) return fail(KVQ_EINVAL, "out_sizes is NULL");
  if (layout < KVQ_Q4_0 || layout > kvq::kLastLayout) return fail(KVQ_EINVAL, "unknown layout %d", layout);
  const size_t rb = row_bytes_of(layout, head_dim);
  if (!rb) return fail(KVQ_ESHAPE, "head_dim %d not 128/256", head_dim);
  if (n_pages < 1 || n_kv_heads < 1 || page_size < 1 || batch < 1 || n_recent < 0) return fail(KVQ_EINVAL, "bad sizes");
  const size_t rows = (size_t)n_pages * n_kv_heads * page_size;
  const size_t nb = (size_t)head_dim / kvq::kBlock;
  out_sizes[0] = rows * rb;
  out_sizes[1] = kvq::is_hadamard(layout) ? rows * sizeof(float) : rows * nb * 2;
  out_sizes[2] = layout == KVQ_ASYM4_G32 ? rows * nb * 2 : 0;
  out_sizes[3] = kvq::is_hadamard(layout) ? (size_t)batch * n_kv_heads * n_recent * head_dim * sizeof(float) : 0;
  return KVQ_OK;
}

namespace {

kvq_status check_paged_store(const kvq_paged_cache *cache, const void *k_new, const void *v_new, int dtype, int n_new,
                             const void *positions, kvq::CacheView &v) {
  kvq_status st = check_paged_cache(cache, v);
  if (st != KVQ_OK) return st;
  if (dtype < KVQ_F32 || dtype > KVQ_F16) return fail(KVQ_EINVAL, "unknown dtype %d", dtype);
  if (n_new < 0) return fail(KVQ_EINVAL, "n_new must be >= 0");
  if (n_new > v.cap) return fail(KVQ_ECAPACITY, "n_new %d > sequence capacity %d", n_new, v.cap);
  if (n_new == 0) return KVQ_OK;
  if (!k_new || !v_new || !positions) return fail(KVQ_EINVAL, "k_new/v_new/positions is NULL");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(positions, 16))
    return fail(KVQ_EALIGN, "k_new/v_new/positions not 16-byte aligned");
  return KVQ_OK;
}

kvq_status prepare_paged(const kvq_paged_cache *cache, const void *q, int32_t q_dtype, int32_t n_q_heads, int32_t n_q,
                         const int32_t *seq_lens, int32_t max_kv_len, int32_t causal, float attn_scale, int32_t chunk,
                         float *out, void *workspace, size_t workspace_bytes, kvq::AttendArgs &a) {
  size_t need = 0;
  kvq_status st = resolve_paged(cache, n_q_heads, n_q, max_kv_len, causal, chunk, a, need, nullptr);
  if (st != KVQ_OK) return st;
  if (!seq_lens) return fail(KVQ_EINVAL, "seq_lens is NULL");
  if (!aligned(seq_lens, 16)) return fail(KVQ_EALIGN, "seq_lens not 16-byte aligned");
  st = check_call(need, q, q_dtype, attn_scale, out, workspace, workspace_bytes);
  if (st != KVQ_OK) return st;
  resolve_paged(cache, n_q_heads, n_q, max_kv_len, causal, chunk, a, need, workspace);
  a.seq_lens = seq_lens;
  a.q = q;
  a.q_dtype = q_dtype;
  a.scale = attn_scale;
  a.out = out;
  return KVQ_OK;
}

cudaError_t launch_paged_append_attend(const kvq::CacheView &v, kvq::AttendArgs &a, const void *k_new,
                                       const void *v_new, int kv_dtype, int n_new, const int32_t *seq_lens,
                                       cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (n_new > 0) {
    // the new tokens end each sequence: positions seq_lens[b] - n_new + j
    e = kvq::launch_store(v, k_new, v_new, kv_dtype, n_new, 0, s, seq_lens, -n_new);
    a.fresh_tail = n_new;                                 // the rows (and window slots) it writes
  }
  if (e == cudaSuccess) e = launch_attend_sequence(a, s, true);
  return e;
}

}  // namespace

kvq_status kvq_paged_store(const kvq_paged_cache *cache, const void *k_new, const void *v_new, int32_t dtype,
                           int32_t n_new, const int32_t *positions, kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::CacheView v;
  kvq_status st = check_paged_store(cache, k_new, v_new, dtype, n_new, positions, v);
  if (st != KVQ_OK || n_new == 0) return st;
  cudaError_t e = kvq::launch_store(v, k_new, v_new, dtype, n_new, 0, reinterpret_cast<cudaStream_t>(stream),
                                    positions, 0);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "store launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

namespace {

// Resident CTAs per SM of the phase-1 kernel a call with these shapes runs, and how many of its
// CTAs one (batch, kv head, chunk) unit takes (the row-side kernel: one per 64-query-row block).
void phase1_capacity(const kvq::CacheView &c, int rows, int q_dtype, int &ctas_per_sm, int &ctas_per_unit,
                     bool &window_ctas) {
  ctas_per_unit = 1;
  window_ctas = false;                                   // the decode kernels leave the window to phase 2
  if (c.layout == KVQ_Q6_0 && c.v_layout == KVQ_Q6_0 && kvq::mma_q6_shape(c.D, rows) &&
      !(kvq::prefill_shape(c.layout, c.v_layout, c.D, rows) && q_dtype != KVQ_F32)) {
    ctas_per_sm = kvq::kMmaQ6CtasPerSm(c.D);
    ctas_per_unit = (rows + 3) / 4;
  } else if (kvq::tc_prefill_shape(c.layout, c.v_layout, c.D, rows)) {
    ctas_per_sm = 1;                                     // the tcgen05 kernel: one CTA of 256 rows per SM
    ctas_per_unit = (rows + kvq::kTcRows - 1) / kvq::kTcRows;
  } else if (kvq::prefill_shape(c.layout, c.v_layout, c.D, rows) &&
             (kvq::is_hadamard(c.layout) || q_dtype != KVQ_F32)) {
    ctas_per_sm = kvq::is_hadamard(c.layout) ? kvq::kPrefillCtasPerSm : 2;
    const bool dec = rows <= 16 && !kvq::decode_kernel(c.layout, c.v_layout);
    ctas_per_unit = dec ? 1 : (rows + kvq::kPrefillRows - 1) / kvq::kPrefillRows;
    window_ctas = kvq::is_hadamard(c.layout) && !dec;    // the row-side kernel scores the window chunks
  } else if (c.layout == c.v_layout && kvq::uses_mma4(c.layout)) {
    ctas_per_sm = kvq::kMma4CtasPerSm;
  } else {
    ctas_per_sm = kvq::kMmaWarpsPerSm / 4;
  }
}

}  // namespace

int32_t kvq_paged_attend_plan_chunk(const kvq_paged_cache *cache, int32_t n_q_heads, int32_t n_q, int32_t q_dtype,
                                    const int32_t *host_seq_lens) {
  g_last_error[0] = 0;
  kvq::CacheView v;
  if (check_paged_cache(cache, v) != KVQ_OK) return 0;
  if (!host_seq_lens || n_q_heads < 1 || n_q < 1 || n_q_heads % v.H) {
    fail(KVQ_EINVAL, "host_seq_lens is NULL or bad head counts");
    return 0;
  }
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int per_sm = 1, per_unit = 1;
  bool window_ctas = false;
  phase1_capacity(v, (n_q_heads / v.H) * n_q, q_dtype, per_sm, per_unit, window_ctas);
  const long long capacity = (long long)sms * per_sm / per_unit;       // (head, chunk) units in one wave
  const int cap_len = v.cap;
  auto units = [&](int ch) {
    long long u = 0;
    for (int b = 0; b < v.B; ++b) {
      const int L = host_seq_lens[b] < 0 ? 0 : (host_seq_lens[b] > cap_len ? cap_len : host_seq_lens[b]);
      const int nw = kvq::is_hadamard(v.layout) ? (v.n_recent < L ? v.n_recent : L) : 0;
      const int nb = L - nw;
      u += nb > 0 ? (nb + ch - 1) / ch : 0;
      if (window_ctas) u += (nw + kvq::kWinChunk - 1) / kvq::kWinChunk;
    }
    return u * v.H;
  };
  // the shortest chunk whose units fit one wave: every CTA then has at most that many tokens
  for (int ch = 64; ch <= 8192; ch += 64)
    if (units(ch) <= capacity) return ch;
  // more work than one wave at the longest chunk: the least (waves x chunk)
  long long best = -1;
  int best_ch = 8192;
  for (int ch = 64; ch <= 8192; ch += 64) {
    const long long cost = (units(ch) + capacity - 1) / capacity * ch;
    if (best < 0 || cost < best) {
      best = cost;
      best_ch = ch;
    }
  }
  return best_ch;
}

size_t kvq_paged_attend_workspace_bytes(const kvq_paged_cache *cache, int32_t n_q_heads, int32_t n_q,
                                        int32_t max_kv_len, int32_t chunk) {
  kvq::AttendArgs a;
  size_t need = 0;
  if (resolve_paged(cache, n_q_heads, n_q, max_kv_len, 0, chunk, a, need, nullptr) != KVQ_OK) return 0;
  return need;
}

int32_t kvq_paged_attend_chunk(const kvq_paged_cache *cache, int32_t n_q_heads, int32_t n_q, int32_t max_kv_len,
                               int64_t total_kv_len, int32_t chunk) {
  kvq::AttendArgs a;
  size_t need = 0;
  if (total_kv_len < 0) return 0;
  if (resolve_paged(cache, n_q_heads, n_q, max_kv_len, 0, chunk, a, need, nullptr, total_kv_len) != KVQ_OK) return 0;
  return a.chunk;
}

kvq_status kvq_paged_decode_attend(const kvq_paged_cache *cache, const void *q, int32_t q_dtype, int32_t n_q_heads,
                                   int32_t n_q, const int32_t *seq_lens, int32_t max_kv_len, int32_t causal,
                                   float attn_scale, int32_t chunk, float *out, void *workspace,
                                   size_t workspace_bytes, kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::AttendArgs a;
  kvq_status st = prepare_paged(cache, q, q_dtype, n_q_heads, n_q, seq_lens, max_kv_len, causal, attn_scale, chunk,
                                out, workspace, workspace_bytes, a);
  if (st != KVQ_OK) return st;
  cudaError_t e = launch_attend_sequence(a, reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "attend launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

kvq_status kvq_paged_append_decode_attend(const kvq_paged_cache *cache, const void *k_new, const void *v_new,
                                          int32_t kv_dtype, int32_t n_new, const void *q, int32_t q_dtype,
                                          int32_t n_q_heads, int32_t n_q, const int32_t *seq_lens,
                                          int32_t max_kv_len, int32_t causal, float attn_scale, int32_t chunk,
                                          float *out, void *workspace, size_t workspace_bytes,
                                          kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::CacheView v;
  kvq_status st = check_paged_store(cache, k_new, v_new, kv_dtype, n_new, seq_lens, v);
  if (st != KVQ_OK) return st;
  kvq::AttendArgs a;
  st = prepare_paged(cache, q, q_dtype, n_q_heads, n_q, seq_lens, max_kv_len, causal, attn_scale, chunk, out,
                     workspace, workspace_bytes, a);
  if (st != KVQ_OK) return st;
  const cudaError_t e = launch_paged_append_attend(v, a, k_new, v_new, kv_dtype, n_new, seq_lens,
                                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "append/attend launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

// ------------------------------------------------------------------ host-buffer calls
size_t kvq_append_decode_attend_host_workspace_bytes(const kvq_cache *cache, int32_t kv_dtype, int32_t n_new,
                                                     int32_t q_dtype, int32_t n_q_heads, int32_t n_q,
                                                     int32_t kv_len, int32_t chunk) {
  kvq::AttendArgs a;
  size_t need = 0;
  if (resolve_attend(cache, n_q_heads, n_q, kv_len, 0, 0, chunk, a, need, nullptr) != KVQ_OK) return 0;
  if (check_host_sizes(kv_dtype, n_new, q_dtype) != KVQ_OK) return 0;
  return host_staging(need, cache->batch, cache->n_kv_heads, cache->head_dim, kv_dtype, n_new, q_dtype, n_q_heads,
                      n_q, false).total;
}

kvq_status kvq_append_decode_attend_host(const kvq_cache *cache, const void *k_new, const void *v_new,
                                         int32_t kv_dtype, int32_t n_new, int32_t pos0, const void *q,
                                         int32_t q_dtype, int32_t n_q_heads, int32_t n_q, int32_t kv_len,
                                         int32_t causal, int32_t q_pos0, float attn_scale, int32_t chunk,
                                         float *out, void *workspace, size_t workspace_bytes,
                                         kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::AttendArgs a;
  size_t need = 0;
  kvq_status st = resolve_attend(cache, n_q_heads, n_q, kv_len, causal, q_pos0, chunk, a, need, nullptr);
  if (st != KVQ_OK) return st;
  st = check_host_args(kv_dtype, n_new, q_dtype, k_new, v_new, q, out, workspace);
  if (st != KVQ_OK) return st;
  const HostStaging h = host_staging(need, cache->batch, cache->n_kv_heads, cache->head_dim, kv_dtype, n_new,
                                     q_dtype, n_q_heads, n_q, false);
  if (workspace_bytes < h.total)
    return fail(KVQ_EWORKSPACE, "workspace %zu < required %zu", workspace_bytes, h.total);
  char *ws = static_cast<char *>(workspace);
  const HostIo io = host_io(h, ws, n_new, k_new, v_new, out);
  // both parts validated against the addresses the kernels will use before anything is enqueued
  kvq::CacheView v;
  st = check_store(-1, cache, io.k, io.v, kv_dtype, n_new, pos0, v);
  if (st != KVQ_OK) return st;
  st = prepare_attend(cache, io.q, q_dtype, n_q_heads, n_q, kv_len, causal, q_pos0, attn_scale, chunk, io.out,
                      workspace, need, a);
  if (st != KVQ_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = io.copy_in ? copy_in(h, ws, k_new, v_new, q, nullptr, s)
                             : cudaMemcpyAsync(ws + h.q, q, h.q_bytes, cudaMemcpyDefault, s);   // q only
  if (e == cudaSuccess) e = launch_append_attend(v, a, io.k, io.v, kv_dtype, n_new, pos0, s);
  if (e == cudaSuccess) e = io.copy_out ? copy_out_and_wait(h, ws, out, s) : cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "host-buffer append/attend: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

size_t kvq_paged_append_decode_attend_host_workspace_bytes(const kvq_paged_cache *cache, int32_t kv_dtype,
                                                           int32_t n_new, int32_t q_dtype, int32_t n_q_heads,
                                                           int32_t n_q, int32_t max_kv_len, int32_t chunk) {
  kvq::AttendArgs a;
  size_t need = 0;
  if (resolve_paged(cache, n_q_heads, n_q, max_kv_len, 0, chunk, a, need, nullptr) != KVQ_OK) return 0;
  if (check_host_sizes(kv_dtype, n_new, q_dtype) != KVQ_OK) return 0;
  return host_staging(need, cache->batch, cache->n_kv_heads, cache->head_dim, kv_dtype, n_new, q_dtype, n_q_heads,
                      n_q, true).total;
}

kvq_status kvq_paged_append_decode_attend_host(const kvq_paged_cache *cache, const void *k_new, const void *v_new,
                                               int32_t kv_dtype, int32_t n_new, const void *q, int32_t q_dtype,
                                               int32_t n_q_heads, int32_t n_q, const int32_t *seq_lens,
                                               int32_t max_kv_len, int32_t causal, float attn_scale, int32_t chunk,
                                               float *out, void *workspace, size_t workspace_bytes,
                                               kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::AttendArgs a;
  size_t need = 0;
  kvq_status st = resolve_paged(cache, n_q_heads, n_q, max_kv_len, causal, chunk, a, need, nullptr);
  if (st != KVQ_OK) return st;
  st = check_host_args(kv_dtype, n_new, q_dtype, k_new, v_new, q, out, workspace);
  if (st != KVQ_OK) return st;
  if (!seq_lens) return fail(KVQ_EINVAL, "seq_lens is NULL");
  const HostStaging h = host_staging(need, cache->batch, cache->n_kv_heads, cache->head_dim, kv_dtype, n_new,
                                     q_dtype, n_q_heads, n_q, true);
  if (workspace_bytes < h.total)
    return fail(KVQ_EWORKSPACE, "workspace %zu < required %zu", workspace_bytes, h.total);
  char *ws = static_cast<char *>(workspace);
  const HostIo io = host_io(h, ws, n_new, k_new, v_new, out);
  // the sequence lengths are read by every CTA: always staged in device memory
  const int32_t *lens = reinterpret_cast<const int32_t *>(ws + h.lens);
  kvq::CacheView v;
  st = check_paged_store(cache, io.k, io.v, kv_dtype, n_new, lens, v);
  if (st != KVQ_OK) return st;
  st = prepare_paged(cache, io.q, q_dtype, n_q_heads, n_q, lens, max_kv_len, causal, attn_scale, chunk, io.out,
                     workspace, need, a);
  if (st != KVQ_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (io.copy_in) {
    e = copy_in(h, ws, k_new, v_new, q, seq_lens, s);
  } else {                                               // q and the lengths only
    e = cudaMemcpyAsync(ws + h.q, q, h.q_bytes, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ws + h.lens, seq_lens, h.lens_bytes, cudaMemcpyDefault, s);
  }
  if (e == cudaSuccess) e = launch_paged_append_attend(v, a, io.k, io.v, kv_dtype, n_new, lens, s);
  if (e == cudaSuccess) e = io.copy_out ? copy_out_and_wait(h, ws, out, s) : cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "host-buffer paged append/attend: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

kvq_status kvq_debug_scores_i32(const kvq_cache *cache, const void *q, int32_t q_dtype, int32_t n_q_heads,
                                int32_t n_q, int32_t kv_len, int32_t *scores_out, float *s_q_out,
                                kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::AttendArgs a;
  size_t need = 0;
  kvq_status st = resolve_attend(cache, n_q_heads, n_q, kv_len, 0, 0, 0, a, need, nullptr);
  if (st != KVQ_OK) return st;
  if (!kvq::is_hadamard(a.cache.layout)) return fail(KVQ_EUNSUPPORTED, "integer scores exist for the Hadamard layouts only");
  if (q_dtype < KVQ_F32 || q_dtype > KVQ_F16) return fail(KVQ_EINVAL, "unknown q dtype %d", q_dtype);
  if (!q || !scores_out || !s_q_out) return fail(KVQ_EINVAL, "q/scores_out/s_q_out is NULL");
  if (!aligned(q, 16) || !aligned(scores_out, 16) || !aligned(s_q_out, 16))
    return fail(KVQ_EALIGN, "q/scores_out/s_q_out not 16-byte aligned");
  cudaError_t e = kvq::launch_debug_scores(a.cache, q, q_dtype, n_q_heads, n_q, kv_len, a.n_body, scores_out, s_q_out,
                                           reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "debug scores launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

kvq_status kvq_debug_attend_scores_i32(const kvq_cache *cache, const void *q, int32_t q_dtype, int32_t n_q_heads,
                                       int32_t n_q, int32_t kv_len, int32_t causal, int32_t q_pos0, float attn_scale,
                                       int32_t chunk, float *out, void *workspace, size_t workspace_bytes,
                                       int32_t *scores_out, float *s_q_out, kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::AttendArgs a;
  kvq_status st = prepare_attend(cache, q, q_dtype, n_q_heads, n_q, kv_len, causal, q_pos0, attn_scale, chunk, out,
                                 workspace, workspace_bytes, a);
  if (st != KVQ_OK) return st;
  if (!scores_out || !s_q_out) return fail(KVQ_EINVAL, "scores_out/s_q_out is NULL");
  if (!aligned(scores_out, 16) || !aligned(s_q_out, 16)) return fail(KVQ_EALIGN, "scores_out/s_q_out not 16-byte aligned");
  if (!kvq::capture_supported(a))
    return fail(KVQ_EUNSUPPORTED, "score capture needs a contiguous Hadamard cache (one layout in both planes) "
                                  "whose body is scored by a tensor-core kernel");
  a.cap_scores = scores_out;
  a.cap_sq = s_q_out;
  cudaError_t e = launch_attend_sequence(a, reinterpret_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "attend launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

const char *kvq_status_string(int32_t status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_EINVAL: return "invalid argument";
    case KVQ_ESHAPE: return "unsupported shape";
    case KVQ_ECAPACITY: return "beyond cache capacity";
    case KVQ_EUNSUPPORTED: return "unsupported layout or option";
    case KVQ_EALIGN: return "misaligned pointer";
    case KVQ_ECUDA: return "CUDA launch error";
    case KVQ_EWORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

const char *kvq_last_error(void) { return g_last_error; }

kvq_status kvq_profile_phase1_events(void *phase1_begin, void *phase1_end) {
  g_ev_begin = static_cast<cudaEvent_t>(phase1_begin);
  g_ev_end = static_cast<cudaEvent_t>(phase1_end);
  return KVQ_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ allocation-free attention
// kvq_decode_attend_static: the same two-phase attention as kvq_decode_attend, for callers that
// cannot hand the library a workspace of their own. Its scratch is one file-scope device array
// of KVQ_STATIC_SCRATCH_BYTES, present on every device that loads the library for the life of
// the process. Host code resolves the array's device address with cudaGetSymbolAddress (the
// array's name is only a host-side stand-in) once per device, on the first call made with that
// device current, and keeps it.
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[KVQ_STATIC_SCRATCH_BYTES];
std::mutex g_static_mu;
void *g_static_ptr[kvq::kMaxDevices] = {};

cudaError_t static_scratch_of_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kvq::kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_decode_attend_static(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                               int32_t n_q_heads, int32_t n_q, int32_t kv_len, int32_t causal,
                                               int32_t q_pos0, float attn_scale, int32_t chunk, float *out,
                                               kvq_stream_t stream) {
  g_last_error[0] = 0;
  kvq::AttendArgs a;
  size_t need = 0;
  kvq_status st = resolve_attend(cache, n_q_heads, n_q, kv_len, causal, q_pos0, chunk, a, need, nullptr);
  if (st != KVQ_OK) return st;
  if (q_dtype < KVQ_F32 || q_dtype > KVQ_F16) return fail(KVQ_EINVAL, "unknown q dtype %d", q_dtype);
  if (!q || !out) return fail(KVQ_EINVAL, "q/out is NULL");
  if (!aligned(q, 16) || !aligned(out, 16)) return fail(KVQ_EALIGN, "q/out not 16-byte aligned");
  if (!(attn_scale == attn_scale) || attn_scale > 3.0e38f || attn_scale < -3.0e38f)
    return fail(KVQ_EINVAL, "attn_scale must be finite");
  if (need > (size_t)KVQ_STATIC_SCRATCH_BYTES)
    return fail(KVQ_EWORKSPACE, "call needs %zu bytes of scratch; the built-in scratch holds %zu", need,
                (size_t)KVQ_STATIC_SCRATCH_BYTES);
  void *ws = nullptr;
  cudaError_t e = static_scratch_of_current_device(&ws);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "built-in scratch address: %s", cudaGetErrorString(e));
  resolve_attend(cache, n_q_heads, n_q, kv_len, causal, q_pos0, chunk, a, need, ws);
  a.q = q;
  a.q_dtype = q_dtype;
  a.scale = attn_scale;
  a.out = out;
  e = launch_attend_sequence(a, reinterpret_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "attend launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}
