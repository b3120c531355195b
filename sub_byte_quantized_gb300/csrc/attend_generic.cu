// Split-K decode attention, CUDA-core form for every layout and shape, plus the phase-2
// LSE reduce and the Hadamard query preparation.
//
// Phase 1 (attend_generic_kernel): one CTA per (chunk, batch x kv head, group of 8 query
// rows). The chunk is walked in sub-tiles of T tokens; each sub-tile of K and V is unpacked
// from the packed cache into shared memory (nibbles / bit planes sign-extended in registers,
// times their scales), then each warp scores its query row against the sub-tile (one token
// per lane), keeps an online softmax (running max m, running sum l) and accumulates the
// unnormalised output o. The dequantised rows live only in shared memory for one sub-tile;
// nothing the size of the cache is ever written. Each (row, chunk) writes (m, l, o) to the
// workspace.
//
// Hadamard int4: body tokens hold their signed int4 codes in shared memory and are scored as
// the exact integer dot with the row's int8 query codes (sums of products of integers below
// 2^24 are exact in float32), times alpha * s_q * s_k. The exact-f32 ring forms one extra
// chunk scored with the float32 rotated query.
//
// Phase 2 (the LSE reduce) lives in reduce.cu.
#include <cfloat>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kRowsPerCta = 8;       // one warp per query row
constexpr int kThreads = kRowsPerCta * 32;

// Absolute token range of chunk c of a sequence: body chunks [c*chunk, min(n_body, (c+1)*chunk)),
// window chunk w = c - n_chunks: [n_body + w*kWinChunk, min(kv_len, n_body + (w+1)*kWinChunk)).
__device__ __forceinline__ void chunk_range(const AttendArgs &a, const SeqLen &sl, int c, int &t0, int &t1) {
  if (c < a.n_chunks) {
    t0 = c * sl.chunk;
    t1 = min(sl.n_body, t0 + sl.chunk);
  } else {
    t0 = sl.n_body + (c - a.n_chunks) * kWinChunk;
    t1 = min(sl.kv_len, t0 + kWinChunk);
  }
}

// Unpack 8 values (group gi of a token row) of a packed row into f32 (value = code * scale [+ zero]).
// For the Hadamard layouts the raw signed codes are produced (the per-token scale is applied by
// the caller).
__device__ __forceinline__ void unpack8(const CacheView &c, int kv, size_t row, int gi, float out[8]) {
  const int layout = kv ? c.v_layout : c.layout;          // each plane's own layout (mixed K/V)
  const uint8_t *p = (kv ? c.payload[1] : c.payload[0]) + row * (size_t)(kv ? c.v_row_bytes : c.row_bytes);
  const int blk = gi >> 2, sub = gi & 3;
  if (layout == KVQ_HAD_INT4) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(p + gi * 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = (float)((int)((w >> (4 * i)) & 0xFu ^ 0x8u) - 8);
    return;
  }
  if (layout == KVQ_HAD_INT2) {                       // four 2-bit fields per byte, (v ^ 2) - 2
    const uint32_t w = *reinterpret_cast<const uint16_t *>(p + gi * 2);
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = (float)((int)((w >> (2 * i)) & 0x3u ^ 0x2u) - 2);
    return;
  }
  const float s = __half2float(static_cast<const __half *>((kv ? c.scale[1] : c.scale[0]))[row * (c.D / kBlock) + blk]);
  if (layout == KVQ_Q4_0) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(p + blk * 16 + sub * 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = (float)((int)((w >> (4 * i)) & 0xFu ^ 0x8u) - 8) * s;
  } else if (layout == KVQ_Q6_0) {
    const uint32_t lo = *reinterpret_cast<const uint32_t *>(p + blk * 24 + sub * 4);
    const uint32_t hi = *reinterpret_cast<const uint16_t *>(p + blk * 24 + 16 + sub * 2);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t v = ((lo >> (4 * i)) & 0xFu) | (((hi >> (2 * i)) & 0x3u) << 4);
      out[i] = (float)((int)(v ^ 0x20u) - 0x20) * s;
    }
  } else if (layout == KVQ_Q8_0) {                    // byte i = value i, (v ^ 0x80) - 0x80
    const uint2 w = *reinterpret_cast<const uint2 *>(p + blk * 32 + sub * 8);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b = ((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFFu;
      out[i] = (float)((int)(b ^ 0x80u) - 0x80) * s;
    }
  } else {  // ASYM4_G32
    const float z = __half2float((kv ? c.zero[1] : c.zero[0])[row * (c.D / kBlock) + blk]);
    const uint32_t w = *reinterpret_cast<const uint32_t *>(p + blk * 16 + sub * 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = fmaf((float)((w >> (4 * i)) & 0xFu), s, z);
  }
}

// D: head dim; T: tokens per shared-memory sub-tile.
template <int D, int T>
__global__ void __launch_bounds__(kThreads) attend_generic_kernel(AttendArgs a) {
  extern __shared__ __align__(16) float smem[];
  float *Ks = smem;                          // [T][D + 1]
  float *Vs = Ks + T * (D + 1);              // [T][D]
  float *Qs = Vs + T * D;                    // [8][D]
  float *ks = Qs + kRowsPerCta * D;          // [T] HAD body: per-token K scale
  float *vs = ks + T;                        // [T] HAD body: per-token V scale

  const CacheView &c = a.cache;
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  // Let the phase-2 grid be scheduled early; it still waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");   // upstream store / query prep complete
#endif
  const int chunk_id = blockIdx.x;
  const int bh = blockIdx.y;                 // b * H_kv + kv head
  const int b = bh / c.H, kvh = bh - b * c.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = a.gqa * a.n_q;
  const int r = blockIdx.z * kRowsPerCta + warp;       // row within the GQA group
  const bool row_ok = r < R;
  const int hq = kvh * a.gqa + (row_ok ? r / a.n_q : 0);
  const int qi = row_ok ? r % a.n_q : 0;
  const size_t grow = ((size_t)b * a.Hq + hq) * a.n_q + qi;   // global query row

  const SeqLen sl = seq_of(a, b);
  int t0, t1;
  chunk_range(a, sl, chunk_id, t0, t1);
  const bool is_win = chunk_id >= a.n_chunks;
  const bool had = is_hadamard(c.layout);
  const int lim = row_ok ? row_limit(a, sl, qi) : -1;
  // Highest token any row of this CTA may see.
  int cta_lim = -1;
  for (int w = 0; w < kRowsPerCta; ++w) {
    const int rr = blockIdx.z * kRowsPerCta + w;
    if (rr < R) cta_lim = max(cta_lim, row_limit(a, sl, rr % a.n_q));
  }
  if (t0 > cta_lim || t0 >= t1) return;      // no row sees this chunk: phase 2 skips it too
  const int t_end = min(t1, cta_lim + 1);

  // Query row into shared memory: HAD body -> int8 codes; HAD window -> rotated f32; else q.
  constexpr int VPL = D / 32;
  if (row_ok) {
    for (int d = lane; d < D; d += 32) {
      float qv;
      if (had) {
        qv = is_win ? a.q_rot[grow * D + d] : (float)a.q8[grow * D + d];
      } else if (a.q_dtype == KVQ_F32) {
        qv = static_cast<const float *>(a.q)[grow * D + d];
      } else if (a.q_dtype == KVQ_BF16) {
        qv = bf16_bits_to_f32(static_cast<const uint16_t *>(a.q)[grow * D + d]);
      } else {
        qv = __half2float(static_cast<const __half *>(a.q)[grow * D + d]);
      }
      Qs[warp * D + d] = qv;
    }
  }
  const float sq = (had && !is_win && row_ok) ? a.s_q[grow] : 1.0f;

  float m = -INFINITY, l = 0.0f;
  float o[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) o[i] = 0.0f;

  for (int tb = t0; tb < t_end; tb += T) {
    const int nt = min(T, t_end - tb);
    __syncthreads();                                     // previous sub-tile fully consumed
    // Unpack K and V rows [tb, tb + nt) into shared memory.
    for (int idx = threadIdx.x; idx < 2 * T * (D / 8); idx += kThreads) {
      const int kv = idx >= T * (D / 8);
      const int rem = idx - kv * T * (D / 8);
      const int t = rem / (D / 8), gi = rem - t * (D / 8);
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (t >= nt && gi == 0) (kv ? vs : ks)[t] = 0.0f;   // tail tokens weigh exactly zero
      if (t < nt) {
        const int tok = tb + t;
        if (is_win) {
          const float *src = (kv ? c.ring[1] : c.ring[0]) + ((size_t)bh * c.n_recent + (size_t)(tok % c.n_recent)) * D + gi * 8;
          const float4 x0 = *reinterpret_cast<const float4 *>(src), x1 = *reinterpret_cast<const float4 *>(src + 4);
          v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w; v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
        } else {
          const size_t crow = cache_row(c, b, kvh, tok);
          unpack8(c, kv, crow, gi, v);
          if (had && gi == 0) {
            const float s = static_cast<const float *>((kv ? c.scale[1] : c.scale[0]))[crow];
            (kv ? vs : ks)[t] = s;
          }
        }
      }
      if (kv == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) Ks[t * (D + 1) + gi * 8 + i] = v[i];
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) Vs[t * D + gi * 8 + i] = v[i];
      }
    }
    __syncthreads();
    if (!row_ok) continue;

    // Scores: lane handles tokens lane, lane + 32, ...
    constexpr int TPL = T / 32;
    float s[TPL];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < TPL; ++j) {
      const int t = lane + 32 * j;
      const int tok = tb + t;
      float acc = 0.0f;
      const float *kr = Ks + t * (D + 1);
      const float *qr = Qs + warp * D;
#pragma unroll 8
      for (int d = 0; d < D; ++d) acc = fmaf(qr[d], kr[d], acc);
      float sc;
      if (had && !is_win) {
        sc = a.scale * sq * ks[t] * acc;       // acc is the exact integer dot
      } else {
        sc = a.scale * acc;
      }
      const bool vis = t < nt && tok <= lim;
      s[j] = vis ? sc : -INFINITY;
      tmax = fmaxf(tmax, s[j]);
    }
#pragma unroll
    for (int mk = 16; mk; mk >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, mk));
    if (tmax == -INFINITY) continue;             // nothing visible for this row in the sub-tile
    const float m_new = fmaxf(m, tmax);
    const float corr = __expf(m - m_new);        // m = -inf -> 0
    l *= corr;
#pragma unroll
    for (int i = 0; i < VPL; ++i) o[i] *= corr;
    m = m_new;
    float p[TPL];
    float psum = 0.0f;
#pragma unroll
    for (int j = 0; j < TPL; ++j) {
      p[j] = s[j] == -INFINITY ? 0.0f : __expf(s[j] - m);
      psum += p[j];
      if (had && !is_win) p[j] *= vs[lane + 32 * j];    // fold the V token scale into p
    }
#pragma unroll
    for (int mk = 16; mk; mk >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, mk);
    l += psum;
    // o[d] += sum_t p_t V[t][d]; lane owns dims lane + 32 i.
#pragma unroll
    for (int j = 0; j < TPL; ++j) {
      for (int src = 0; src < 32; ++src) {
        const float pt = __shfl_sync(0xffffffffu, p[j], src);
        const float *vr = Vs + (src + 32 * j) * D;
#pragma unroll
        for (int i = 0; i < VPL; ++i) o[i] = fmaf(pt, vr[lane + 32 * i], o[i]);
      }
    }
  }
  if (!row_ok || t0 > lim) return;               // this row does not see the chunk
  const size_t pi = grow * a.C + chunk_id;
  if (lane == 0) {
    a.part_m[pi] = m;
    a.part_l[pi] = l;
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) a.part_o[pi * D + lane + 32 * i] = o[i];
}

// Hadamard query preparation: one warp per query row.
template <int V>
__global__ void __launch_bounds__(256) had_prep_kernel(AttendArgs a, int rows, bool write_rot) {
  // It reads only the query: it may run alongside the preceding kernel (this call's append), except
  // its first CTA, which waits for it, so that the grid completes after it and a kernel waiting on
  // this grid also sees the append. Its consumers wait for it in every CTA.
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  pdl_wait_if(false);
  const int lane = threadIdx.x & 31;
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (r >= rows) return;
  constexpr int D = V * 32;
  float x[V];
  int q8[V];
  if (V == 4) load4_f32(a.q, a.q_dtype, (size_t)r * D + lane * 4, x);
  else load8_f32(a.q, a.q_dtype, (size_t)r * D + lane * 8, x);
  const float s = had_query_row<V>(x, q8, lane);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    a.q8[(size_t)r * D + lane * V + i] = (int8_t)q8[i];
    if (write_rot) a.q_rot[(size_t)r * D + lane * V + i] = x[i];
  }
  if (lane == 0) a.s_q[r] = s;
}

// Debug hook: exact int32 body scores. One CTA of 128 threads per (query row, 128 tokens);
// warp 0 first prepares the row (FWHT, int8 codes) into shared memory.
template <int V>
__global__ void __launch_bounds__(128) debug_scores_kernel(CacheView c, const void *q, int q_dtype, int Hq,
                                                           int n_q, int n_body, int32_t *scores,
                                                           float *s_q_out) {
  constexpr int D = V * 32;
  __shared__ int q8s[D];
  const int row = blockIdx.y;                    // (b * Hq + h) * n_q + i
  const int gqa = Hq / c.H;
  const int b = row / (Hq * n_q);
  const int h = (row / n_q) % Hq;
  const int kvh = h / gqa;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float x[V];
    int qq[V];
    if (V == 4) load4_f32(q, q_dtype, (size_t)row * D + lane * 4, x);
    else load8_f32(q, q_dtype, (size_t)row * D + lane * 8, x);
    const float s = had_query_row<V>(x, qq, lane);
#pragma unroll
    for (int i = 0; i < V; ++i) q8s[lane * V + i] = qq[i];
    if (lane == 0 && blockIdx.x == 0) s_q_out[row] = s;
  }
  __syncthreads();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n_body) return;
  const uint8_t *p = c.payload[0] + ((size_t)(b * c.H + kvh) * c.cap + t) * (size_t)c.row_bytes;
  int acc = 0;
  if (c.layout == KVQ_HAD_INT2) {
    for (int g = 0; g < D / 8; ++g) {
      const uint32_t w = *reinterpret_cast<const uint16_t *>(p + g * 2);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc += q8s[g * 8 + i] * ((int)((w >> (2 * i)) & 0x3u ^ 0x2u) - 2);
    }
  } else {
    for (int g = 0; g < D / 8; ++g) {
      const uint32_t w = *reinterpret_cast<const uint32_t *>(p + g * 4);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc += q8s[g * 8 + i] * ((int)((w >> (4 * i)) & 0xFu ^ 0x8u) - 8);
    }
  }
  scores[(size_t)row * n_body + t] = acc;
}

template <int D, int T>
cudaError_t launch_generic_dt(const AttendArgs &a, cudaStream_t st) {
  const size_t smem = sizeof(float) * ((size_t)T * (D + 1) + (size_t)T * D + kRowsPerCta * D + 2 * T);
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = set_smem_once(configured, attend_generic_kernel<D, T>, (int)smem);
  if (e != cudaSuccess) return e;
  const int R = a.gqa * a.n_q;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.C, a.cache.B * a.cache.H, (R + kRowsPerCta - 1) / kRowsPerCta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_generic_kernel<D, T>, a);
}

}  // namespace

cudaError_t launch_attend_generic(const AttendArgs &a, cudaStream_t st) {
  return a.cache.D == 128 ? launch_generic_dt<128, 64>(a, st) : launch_generic_dt<256, 32>(a, st);
}

cudaError_t launch_had_prep(const AttendArgs &a, cudaStream_t st, bool write_rot) {
  const int rows = a.cache.B * a.Hq * a.n_q;
  const unsigned blocks = (unsigned)(((size_t)rows * 32 + 255) / 256);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.cache.D == 128 ? cudaLaunchKernelEx(&cfg, had_prep_kernel<4>, a, rows, write_rot)
                          : cudaLaunchKernelEx(&cfg, had_prep_kernel<8>, a, rows, write_rot);
}

cudaError_t launch_debug_scores(const CacheView &c, const void *q, int q_dtype, int Hq, int n_q, int kv_len,
                                int n_body, int32_t *scores, float *s_q, cudaStream_t st) {
  (void)kv_len;
  const int rows = c.B * Hq * n_q;
  dim3 grid((unsigned)max(1, (n_body + 127) / 128), (unsigned)rows);
  if (c.D == 128) debug_scores_kernel<4><<<grid, 128, 0, st>>>(c, q, q_dtype, Hq, n_q, n_body, scores, s_q);
  else debug_scores_kernel<8><<<grid, 128, 0, st>>>(c, q, q_dtype, Hq, n_q, n_body, scores, s_q);
  return cudaGetLastError();
}

}  // namespace kvq
