// Phase 2 of the split-K decode attention: combine the per-chunk partials (m_c, l_c, o_c) of
// every query row with the online-softmax correction
//   M = max_c m_c,  L = sum_c l_c e^(m_c - M),  out = sum_c o_c e^(m_c - M) / L,
// over the chunks the row can see (a chunk beyond a row's causal limit has no partial). For the
// Hadamard layout the combined output is still in the rotated basis and is un-rotated here
// (in-warp FWHT times 1/sqrt(D)).
//
// Two shapes. Few rows (decode): one CTA per (query row, 32-dim slice) -- one CTA per row for the
// Hadamard layout, whose un-rotation needs the whole row. Eight warps split the chunks; each lane
// owns one (or D/32) output dims and keeps a running (M, L, O) over batches of eight chunks whose
// loads are all in flight together. The warps are combined in shared memory. Many rows (prefill
// chunks, large batches): one warp per row, eight rows per CTA, the lane owning D/32 consecutive
// dims, no shared memory.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kWarps = 8;
constexpr int kBatch = 8;

template <int D, bool HAD>
__global__ void __launch_bounds__(kWarps * 32) attend_reduce_kernel(AttendArgs a) {
  constexpr int DS = HAD ? D : 32;         // dims per CTA
  constexpr int VPL = DS / 32;             // dims per lane
  __shared__ float sm_m[kWarps], sm_l[kWarps];
  __shared__ __align__(16) float sm_o[kWarps][DS];
  __shared__ __align__(16) float sm_qw[HAD ? kWarps : 1][HAD ? D : 4];   // per-warp rotated query (window)
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.wait;" ::: "memory");     // phase-1 partials are complete
#endif
  const size_t row = blockIdx.x;                          // (b * H_q + h) * n_q + i
  const int qi = (int)(row % a.n_q);
  const int d0 = HAD ? 0 : blockIdx.y * 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqLen sl = seq_of(a, a.seq_lens ? (int)(row / ((size_t)a.Hq * a.n_q)) : 0);
  const int lim = row_limit(a, sl, qi);                  // negative: the row sees nothing
  const int n_vis_body = lim < 0 ? 0 : min(sl.n_chunks, lim / sl.chunk + 1);
  const bool win_vis = sl.kv_len > sl.n_body && sl.n_body <= lim;
  const float *pm = a.part_m + row * a.C;
  const float *pl = a.part_l + row * a.C;
  const float *po = a.part_o + row * a.C * (size_t)D;

  float M = -INFINITY, L = 0.0f, O[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) O[i] = 0.0f;
  if constexpr (HAD) {
  if (a.win_in_reduce && win_vis) {
    // The exact-f32 recent window (tokens n_body .. kv_len-1, ring slot t mod n_recent), scored
    // with the float32 rotated query. Warp w takes window tokens 8w .. 8w+7 of each group of 64,
    // two groups per pass: lane l scores token l / 4 of each group over dims (l % 4) * D/4 .. +D/4
    // (reduced over the token's four lanes) and accumulates its output dims lane * VPL .. +VPL for
    // the sixteen tokens; every K and V load of a pass is in flight before the first score. The
    // warp's state then joins the chunk partials below.
    const CacheView &cv = a.cache;
    const size_t bh = (row / a.n_q) / a.Hq * cv.H + ((row / a.n_q) % a.Hq) / a.gqa;
    // rotated query row (the tensor-core phase 1 prepares its int8 codes itself, so rotate here)
    float qv[VPL];
    int q8v[VPL];
    if (VPL == 4) load4_f32(a.q, a.q_dtype, row * D + lane * 4, qv);
    else load8_f32(a.q, a.q_dtype, row * D + lane * 8, qv);
    had_query_row<VPL>(qv, q8v, lane);
    constexpr int QS = D / 4;                             // dims per lane in the score
    float *sm_q = sm_qw[HAD ? warp : 0];
#pragma unroll
    for (int i = 0; i < VPL; ++i) sm_q[lane * VPL + i] = qv[i];
    __syncwarp();
    float qs[QS];
#pragma unroll
    for (int i = 0; i < QS; ++i) qs[i] = sm_q[(lane & 3) * QS + i];
    const int tl = lane >> 2;                             // this lane's token within the warp's eight
    const int n_w = sl.kv_len - sl.n_body;
    // two groups of 64 tokens per pass: both groups' K and V loads are issued before any score
    // is formed, so a pass costs one memory round trip
    constexpr int NG = 2;
    for (int g0 = 0; g0 < n_w; g0 += 64 * NG) {
      float4 kq[NG][QS / 4];
      float4 vv[NG][8][VPL / 4];
      bool tv[NG];
#pragma unroll
      for (int k = 0; k < NG; ++k) {
        const int t = sl.n_body + g0 + 64 * k + 8 * warp + tl;   // this lane's token of group k
        tv[k] = t < sl.kv_len && t <= lim;
        const size_t slot = (bh * cv.n_recent + (size_t)((tv[k] ? t : sl.n_body) % cv.n_recent)) * D;
        const float *kr = cv.ring[0] + slot + (lane & 3) * QS;
#pragma unroll
        for (int i = 0; i < QS / 4; ++i)
          kq[k][i] = tv[k] ? *reinterpret_cast<const float4 *>(kr + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
        // the eight V rows' slices (invalid tokens read a valid slot and get weight 0)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int tu = sl.n_body + g0 + 64 * k + 8 * warp + u;
          const int ts = tu < sl.kv_len ? tu : sl.n_body;
          const float *vr = cv.ring[1] + (bh * cv.n_recent + (size_t)(ts % cv.n_recent)) * D + lane * VPL;
#pragma unroll
          for (int i = 0; i < VPL / 4; ++i) vv[k][u][i] = *reinterpret_cast<const float4 *>(vr + 4 * i);
        }
      }
      float sc[NG];
      float gm = -INFINITY;
#pragma unroll
      for (int k = 0; k < NG; ++k) {
        float dot = 0.0f;
#pragma unroll
        for (int i = 0; i < QS / 4; ++i) {
          dot = fmaf(qs[4 * i], kq[k][i].x, dot);
          dot = fmaf(qs[4 * i + 1], kq[k][i].y, dot);
          dot = fmaf(qs[4 * i + 2], kq[k][i].z, dot);
          dot = fmaf(qs[4 * i + 3], kq[k][i].w, dot);
        }
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
        sc[k] = tv[k] ? a.scale * dot : -INFINITY;
        gm = fmaxf(gm, sc[k]);
      }
#pragma unroll
      for (int k = 4; k < 32; k <<= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, k));
      if (gm == -INFINITY) continue;                      // no visible token in this warp's sixteen
      const float mn = fmaxf(M, gm);
      const float corr = __expf(M - mn);                  // M = -inf -> 0
      float p[NG], ps = 0.0f;
#pragma unroll
      for (int k = 0; k < NG; ++k) {
        p[k] = tv[k] ? __expf(sc[k] - mn) : 0.0f;
        ps += (lane & 3) == 0 ? p[k] : 0.0f;              // each token counted once
      }
#pragma unroll
      for (int k = 4; k < 32; k <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, k);
      L = fmaf(L, corr, ps);
#pragma unroll
      for (int i = 0; i < VPL; ++i) O[i] *= corr;
#pragma unroll
      for (int k = 0; k < NG; ++k) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float pu = __shfl_sync(0xffffffffu, p[k], 4 * u);
#pragma unroll
          for (int i = 0; i < VPL / 4; ++i) {
            O[4 * i] = fmaf(pu, vv[k][u][i].x, O[4 * i]);
            O[4 * i + 1] = fmaf(pu, vv[k][u][i].y, O[4 * i + 1]);
            O[4 * i + 2] = fmaf(pu, vv[k][u][i].z, O[4 * i + 2]);
            O[4 * i + 3] = fmaf(pu, vv[k][u][i].w, O[4 * i + 3]);
          }
        }
      }
      M = mn;
    }
  }
  }
  for (int base = warp; base < a.C; base += kWarps * kBatch) {
    float mc[kBatch], lc[kBatch], oc[kBatch][VPL];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = base + u * kWarps;
      const int wt0 = sl.n_body + (c - a.n_chunks) * kWinChunk;      // window chunk's first token
      const bool vis = c < a.C && (c < a.n_chunks ? c < n_vis_body
                                                  : !a.win_in_reduce && wt0 < sl.kv_len && wt0 <= lim);
      mc[u] = vis ? pm[c] : -INFINITY;
      lc[u] = vis ? pl[c] : 0.0f;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int d = HAD ? lane * VPL + i : d0 + lane;
        oc[u][i] = vis ? po[(size_t)c * D + d] : 0.0f;
      }
    }
    float bm = M;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) bm = fmaxf(bm, mc[u]);
    if (bm == -INFINITY) continue;
    const float corr = __expf(M - bm);                    // M = -inf -> 0
    L *= corr;
#pragma unroll
    for (int i = 0; i < VPL; ++i) O[i] *= corr;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const float w = __expf(mc[u] - bm);                 // invisible chunks: exp(-inf) = 0
      L = fmaf(lc[u], w, L);
#pragma unroll
      for (int i = 0; i < VPL; ++i) O[i] = fmaf(oc[u][i], w, O[i]);
    }
    M = bm;
  }
  if (lane == 0) {
    sm_m[warp] = M;
    sm_l[warp] = L;
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) sm_o[warp][HAD ? lane * VPL + i : lane] = O[i];
  __syncthreads();
  if (warp != 0) return;
  float Mt = sm_m[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) Mt = fmaxf(Mt, sm_m[w]);
  float Lt = 0.0f, x[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) x[i] = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float wt = sm_m[w] == -INFINITY ? 0.0f : __expf(sm_m[w] - Mt);
    Lt = fmaf(sm_l[w], wt, Lt);
#pragma unroll
    for (int i = 0; i < VPL; ++i) x[i] = fmaf(sm_o[w][HAD ? lane * VPL + i : lane], wt, x[i]);
  }
  const float inv = Lt > 0.0f ? 1.0f / Lt : 0.0f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) x[i] *= inv;
  if (HAD) {
    warp_fwht<VPL>(x, lane);
    const float cD = inv_sqrt_dim(D);
#pragma unroll
    for (int i = 0; i < VPL; ++i) a.out[row * D + lane * VPL + i] = x[i] * cD;
  } else {
    a.out[row * D + d0 + lane] = x[0];
  }
}

// One warp per row (many rows; the window, if any, is a partial of its own). KB = partials loaded
// per batch: as many as the rows have (up to eight), since the registers they take bound the rows in
// flight per SM (a causal prefill chunk with one body chunk and one window chunk: two).
template <int D, bool HAD, int KB>
__global__ void __launch_bounds__(kWarps * 32, KB >= 8 ? 1 : (D == 128 ? 8 - KB : 6 - KB)) attend_reduce_rows_kernel(AttendArgs a, unsigned rows) {
  constexpr int VPL = D / 32;
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.wait;" ::: "memory");     // phase-1 partials are complete
#endif
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * kWarps + warp;
  if (row >= rows) return;
  const int qi = (int)(row % a.n_q);
  const SeqLen sl = seq_of(a, a.seq_lens ? (int)(row / ((size_t)a.Hq * a.n_q)) : 0);
  const int lim = row_limit(a, sl, qi);                  // negative: the row sees nothing
  const int n_vis_body = lim < 0 ? 0 : min(sl.n_chunks, lim / sl.chunk + 1);
  const float *pm = a.part_m + row * a.C;
  const float *pl = a.part_l + row * a.C;
  const float *po = a.part_o + row * a.C * (size_t)D + lane * VPL;
  float M = -INFINITY, L = 0.0f, O[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) O[i] = 0.0f;
  for (int base = 0; base < a.C; base += KB) {
    float mc[KB], lc[KB], oc[KB][VPL];
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const int c = base + u;
      const int wt0 = sl.n_body + (c - a.n_chunks) * kWinChunk;      // window chunk's first token
      const bool vis = c < a.C && (c < a.n_chunks ? c < n_vis_body : wt0 < sl.kv_len && wt0 <= lim);
      mc[u] = vis ? pm[c] : -INFINITY;
      lc[u] = vis ? pl[c] : 0.0f;
      if constexpr (VPL == 4) {
        const float4 v = vis ? *reinterpret_cast<const float4 *>(po + (size_t)c * D) : make_float4(0.f, 0.f, 0.f, 0.f);
        oc[u][0] = v.x; oc[u][1] = v.y; oc[u][2] = v.z; oc[u][3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < VPL; ++i) oc[u][i] = vis ? po[(size_t)c * D + i] : 0.0f;
      }
    }
    float bm = M;
#pragma unroll
    for (int u = 0; u < KB; ++u) bm = fmaxf(bm, mc[u]);
    if (bm == -INFINITY) continue;
    const float corr = __expf(M - bm);
    L *= corr;
#pragma unroll
    for (int i = 0; i < VPL; ++i) O[i] *= corr;
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const float w = __expf(mc[u] - bm);
      L = fmaf(lc[u], w, L);
#pragma unroll
      for (int i = 0; i < VPL; ++i) O[i] = fmaf(oc[u][i], w, O[i]);
    }
    M = bm;
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) O[i] *= inv;
  if (HAD) {
    warp_fwht<VPL>(O, lane);
    const float cD = inv_sqrt_dim(D);
#pragma unroll
    for (int i = 0; i < VPL; ++i) O[i] *= cD;
  }
  float *out = a.out + row * D + lane * VPL;
  if constexpr (VPL == 4) {
    *reinterpret_cast<float4 *>(out) = make_float4(O[0], O[1], O[2], O[3]);
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i) out[i] = O[i];
  }
}

template <int KB>
cudaError_t launch_rows(cudaLaunchConfig_t &cfg, const AttendArgs &a, unsigned rows, bool had) {
  if (a.cache.D == 128)
    return had ? cudaLaunchKernelEx(&cfg, attend_reduce_rows_kernel<128, true, KB>, a, rows)
               : cudaLaunchKernelEx(&cfg, attend_reduce_rows_kernel<128, false, KB>, a, rows);
  return had ? cudaLaunchKernelEx(&cfg, attend_reduce_rows_kernel<256, true, KB>, a, rows)
             : cudaLaunchKernelEx(&cfg, attend_reduce_rows_kernel<256, false, KB>, a, rows);
}

}  // namespace

cudaError_t launch_attend_reduce(const AttendArgs &a, cudaStream_t st, bool pdl) {
  const unsigned rows = (unsigned)((size_t)a.cache.B * a.Hq * a.n_q);
  const bool had = is_hadamard(a.cache.layout);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // many rows and no window work here: one warp per row
  const bool per_warp = !a.win_in_reduce && rows >= 4u * (unsigned)sms * kWarps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = per_warp ? dim3((rows + kWarps - 1) / kWarps) : dim3(rows, had ? 1 : a.cache.D / 32);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (per_warp) {
    if (a.C <= 2) return launch_rows<2>(cfg, a, rows, had);
    if (a.C <= 4) return launch_rows<4>(cfg, a, rows, had);
    return launch_rows<kBatch>(cfg, a, rows, had);
  }
  if (a.cache.D == 128)
    return had ? cudaLaunchKernelEx(&cfg, attend_reduce_kernel<128, true>, a)
               : cudaLaunchKernelEx(&cfg, attend_reduce_kernel<128, false>, a);
  return had ? cudaLaunchKernelEx(&cfg, attend_reduce_kernel<256, true>, a)
             : cudaLaunchKernelEx(&cfg, attend_reduce_kernel<256, false>, a);
}

}  // namespace kvq
