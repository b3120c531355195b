// Tensor-core phase 1 for many query rows per kv head: causal prefill chunks (and any call whose
// GQA group times query rows exceeds eight), Hadamard int4 layout, head_dim 128 (tract
// discussion #2402, "Architecture: State" and the prefill remarks: the query rows of a chunk
// attend the cached body with causal limits; the body scores are exact integer dot products of
// the int8 rotated query and the int4 rotated keys).
//
// Here the rows are the M side of the contraction (FlashAttention-2 orientation), with
// mma.sync.m16n8k16 (f16 in, f32 accumulate):
//   QK:  S[16 rows][8 tokens] += Q8[16 rows][16 dims] . K^T[16 dims][8 tokens]
//   PV:  O[16 rows][8 dims]   += P'[16 rows][16 tokens] . V[16 tokens][8 dims]
// Q8 holds the int8 query codes (exact in f16; the ones facing high nibbles divided by 16); K
// enters as exact f16 subnormals u * 2^-24 of u = code + 8, with -8 * sum(q8) * 2^-24 as the
// accumulator's initial value, so every score is the exact integer dot times 2^-24 (|dot| <
// 2^18). score = alpha * s_q[row] * s_k[t] * dot. V enters as its exact signed codes; the
// per-token V scale is folded into the probabilities, P' = p * s_v, kept as f16 hi + lo parts
// (two mma per step). The probabilities stay in registers between the two products: the S
// accumulator of two 8-token tiles is the A fragment of one 16-token PV step.
//
// A CTA of four warps takes 64 consecutive query rows of one (batch, kv head) and one chunk of
// body tokens; the warps share a three-stage cp.async ring of 64-token stages (K and V payload
// rows with the 64-byte XOR swizzle, per-token f32 scales), and each warp keeps the online
// softmax of its 16 rows. The exact-f32 recent window is one more chunk (blockIdx.y ==
// n_chunks): its CTAs stream the f32 rotated K/V rows of the ring and score them with the f32
// rotated query on the CUDA cores.
#include <cfloat>
#include <climits>

#include "kvq_internal.cuh"
#include "mma_util.cuh"

namespace kvq {
namespace {
using namespace mma;

constexpr int kWarps = 4;
constexpr int kRows = kPrefillRows;     // query rows per CTA (16 per warp)
constexpr int kStage = 64;              // tokens per stage
constexpr int kRing = 3;
constexpr int kD = 128;
constexpr int kRowBytes = 64;
constexpr int kOffV = kStage * kRowBytes;
constexpr int kOffSK = 2 * kStage * kRowBytes;
constexpr int kOffSV = kOffSK + kStage * 4;
constexpr int kStageBytes = kOffSV + kStage * 4;
constexpr int kOffQ = kRing * kStageBytes;      // int8 query codes [64 rows][128]
constexpr int kOffSQ = kOffQ + kRows * kD;      // their scales [64]
constexpr int kQrPitch = kD * 4 + 16;            // f32 rotated query rows, padded (window chunk)
constexpr int kOffQR = kOffSQ + kRows * 4;
constexpr int kSmem = kOffQR + kRows * kQrPitch;
constexpr int kWinStage = 8;                     // window tokens per stage (f32 K and V rows)
constexpr int kWinPitch = kD * 4 + 16;
static_assert(2 * kWinStage * kWinPitch <= kStageBytes, "window stage fits a ring slot");
constexpr int kCtasPerSm = kPrefillCtasPerSm;
static_assert(kRows == 16 * kWarps, "16 query rows per warp");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Byte offset of (row, 16-byte column j) inside a swizzled 64-byte-row slab.
__device__ __forceinline__ uint32_t swz(int row, int j) {
  return (uint32_t)(row * kRowBytes + ((j ^ ((row >> 1) & 3)) << 4));
}

__device__ __forceinline__ int row_limit_of(const AttendArgs &a, int r) {
  const int qi = r % a.n_q;
  return a.causal ? min(a.kv_len - 1, a.q_pos0 + qi) : a.kv_len - 1;
}

__global__ void __launch_bounds__(kWarps * 32, kCtasPerSm) attend_prefill_had_kernel(AttendArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");   // upstream store complete before any read
#endif
  const CacheView &cv = a.cache;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int row0 = blockIdx.x * kRows;
  const int chunk_id = blockIdx.y;
  const int bh = blockIdx.z;
  const int bb = bh / cv.H, kvh = bh - bb * cv.H;
  const int R = a.gqa * a.n_q;

  const bool win = chunk_id == a.n_chunks;            // the recent-window chunk
  const int t0 = win ? a.n_body : chunk_id * a.chunk;
  const int t1 = win ? a.kv_len : min(a.n_body, t0 + a.chunk);
  int w_lim = -1;
  for (int r = row0; r < min(row0 + kRows, R); ++r) w_lim = max(w_lim, row_limit_of(a, r));
  if (t0 > w_lim) return;                              // no row of this CTA sees the chunk
  const int t_end = min(t1, w_lim + 1);
  const int stage_len = win ? kWinStage : kStage;
  const int n_stages = (t_end - t0 + stage_len - 1) / stage_len;

  const size_t head_row0 = (size_t)bh * cv.cap;
  const uint8_t *kp = cv.payload[0] + head_row0 * kRowBytes;
  const uint8_t *vp = cv.payload[1] + head_row0 * kRowBytes;
  const float *ksc = static_cast<const float *>(cv.scale[0]) + head_row0;
  const float *vsc = static_cast<const float *>(cv.scale[1]) + head_row0;

  // ---- CTA-wide stage copy: 256 16-byte pieces per payload plane (two per thread), one 4-byte
  // scale per thread; rows past t_end are zero-filled
  auto issue = [&](int s) {
    if (win) {                                         // window: 8 f32 K and V rows, ring slot t mod n_recent
      if (s < n_stages) {
        const int ts = t0 + s * kWinStage;
        uint8_t *sb = smem + (s % kRing) * kStageBytes;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int q = threadIdx.x + 128 * k;          // piece: row q / 32, 16-byte column q % 32
          const int row = q >> 5, pc = q & 31;
          const int t = ts + row;
          const bool ok = t < t_end;
          const size_t off = ((size_t)bh * cv.n_recent + (size_t)((ok ? t : t0) % cv.n_recent)) * kD + 4 * pc;
          cp_async16(smem_addr(sb + row * kWinPitch + 16 * pc), cv.ring[0] + off, ok ? 16 : 0);
          cp_async16(smem_addr(sb + (kWinStage + row) * kWinPitch + 16 * pc), cv.ring[1] + off, ok ? 16 : 0);
        }
      }
      cp_async_commit();
      return;
    }
    if (s < n_stages) {
      const int ts = t0 + s * kStage;
      uint8_t *sb = smem + (s % kRing) * kStageBytes;
      const uint32_t sK = smem_addr(sb), sV = smem_addr(sb + kOffV);
      const bool full = ts + kStage <= t_end;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int q = threadIdx.x + 128 * k;            // piece: row q / 4, column q % 4
        const int row = q >> 2, j = q & 3;
        const bool ok = full || ts + row < t_end;
        const size_t off = (size_t)(ok ? ts + row : t0) * kRowBytes + 16 * j;
        cp_async16(sK + swz(row, j), kp + off, ok ? 16 : 0);
        cp_async16(sV + swz(row, j), vp + off, ok ? 16 : 0);
      }
      {
        const int kv = threadIdx.x >> 6, row = threadIdx.x & 63;   // one token's f32 scale per thread
        const bool ok = ts + row < t_end;
        cp_async4(smem_addr(sb + (kv ? kOffSV : kOffSK) + 4 * row), (kv ? vsc : ksc) + (ok ? ts + row : t0), ok ? 4 : 0);
      }
    }
    cp_async_commit();
  };
  issue(0);
  issue(1);

  // ---- query prologue: each warp rotates and quantises its 16 rows (warp FWHT, int8 codes,
  // one f32 scale per row) into shared memory, then reads back its A fragments
  uint8_t *q8s = smem + kOffQ;
  float *sqs = reinterpret_cast<float *>(smem + kOffSQ);
  for (int i = 0; i < 16; ++i) {
    const int lr = 16 * warp + i, r = row0 + lr;
    uint32_t packed = 0u;
    float sq = 0.0f;
    if (r < R) {
      const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
      const size_t grow = ((size_t)bb * a.Hq + hq) * a.n_q + qi;
      float x[4];
      int q8v[4];
      load4_f32(a.q, a.q_dtype, grow * kD + lane * 4, x);
      sq = had_query_row<4>(x, q8v, lane);
      *reinterpret_cast<float4 *>(smem + kOffQR + lr * kQrPitch + lane * 16) = make_float4(x[0], x[1], x[2], x[3]);
      packed = (uint32_t)(q8v[0] & 0xFF) | ((uint32_t)(q8v[1] & 0xFF) << 8) | ((uint32_t)(q8v[2] & 0xFF) << 16) |
               ((uint32_t)(q8v[3] & 0xFF) << 24);
    }
    else *reinterpret_cast<float4 *>(smem + kOffQR + lr * kQrPitch + lane * 16) = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<uint32_t *>(q8s + lr * kD + lane * 4) = packed;
    if (lane == 0) sqs[lr] = sq;
  }
  __syncwarp();
  const int rg = row0 + 16 * warp + g, rg8 = rg + 8;
  const int lim_g = rg < R ? row_limit_of(a, rg) : -1;
  const int lim_g8 = rg8 < R ? row_limit_of(a, rg8) : -1;
  const float alpha_g = (rg < R ? a.scale * sqs[16 * warp + g] : 0.0f) * 16777216.0f * kLog2e;
  const float alpha_g8 = (rg8 < R ? a.scale * sqs[16 * warp + g + 8] : 0.0f) * 16777216.0f * kLog2e;
  const float walpha = a.scale * kLog2e;               // window scores: alpha * q_rot . k_y (base 2)
  int warp_lim = max(lim_g, lim_g8), warp_min = INT_MAX;
  if (lim_g >= 0) warp_min = lim_g;
  if (lim_g8 >= 0) warp_min = min(warp_min, lim_g8);
#pragma unroll
  for (int k = 4; k < 32; k <<= 1) {
    warp_lim = max(warp_lim, __shfl_xor_sync(0xffffffffu, warp_lim, k));
    warp_min = min(warp_min, __shfl_xor_sync(0xffffffffu, warp_min, k));
  }

  float m_g = -INFINITY, m_g8 = -INFINITY, l_g = 0.0f, l_g8 = 0.0f;
  float O[4][4][4];                                      // [block][j'][c0..c3]: dims 32b + 4n + j'
#pragma unroll
  for (int b = 0; b < 4; ++b)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) O[b][j][k] = 0.0f;

  // ---------------- the recent window: exact f32 scores on the CUDA cores; lane (g, c) scores
  // rows g, g+8 against tokens 2c, 2c+1 of each 8-token stage and accumulates the O layout of
  // the body path (rows g, g+8; dims 32b + 8c + 0..7)
  for (int i = 0; win && i < n_stages; ++i) {
    cp_async_wait<kRing - 2>();
    __syncthreads();
    issue(i + kRing - 1);
    const int ts = t0 + i * kWinStage;
    if (ts > warp_lim) continue;
    const uint8_t *sb = smem + (i % kRing) * kStageBytes;
    const float *qa = reinterpret_cast<const float *>(smem + kOffQR + (16 * warp + g) * kQrPitch);
    const float *qb = reinterpret_cast<const float *>(smem + kOffQR + (16 * warp + g + 8) * kQrPitch);
    const float *ka = reinterpret_cast<const float *>(sb + (2 * c) * kWinPitch);
    const float *kb = reinterpret_cast<const float *>(sb + (2 * c + 1) * kWinPitch);
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;       // (g, 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1)
#pragma unroll 8
    for (int d = 0; d < kD; d += 4) {
      const float4 x = *reinterpret_cast<const float4 *>(qa + d), y = *reinterpret_cast<const float4 *>(qb + d);
      const float4 u = *reinterpret_cast<const float4 *>(ka + d), v = *reinterpret_cast<const float4 *>(kb + d);
      s0 = fmaf(x.x, u.x, s0); s0 = fmaf(x.y, u.y, s0); s0 = fmaf(x.z, u.z, s0); s0 = fmaf(x.w, u.w, s0);
      s1 = fmaf(x.x, v.x, s1); s1 = fmaf(x.y, v.y, s1); s1 = fmaf(x.z, v.z, s1); s1 = fmaf(x.w, v.w, s1);
      s2 = fmaf(y.x, u.x, s2); s2 = fmaf(y.y, u.y, s2); s2 = fmaf(y.z, u.z, s2); s2 = fmaf(y.w, u.w, s2);
      s3 = fmaf(y.x, v.x, s3); s3 = fmaf(y.y, v.y, s3); s3 = fmaf(y.z, v.z, s3); s3 = fmaf(y.w, v.w, s3);
    }
    const int ta = ts + 2 * c, tb = ta + 1;
    s0 = (ta < t1 && ta <= lim_g) ? s0 * walpha : -INFINITY;
    s1 = (tb < t1 && tb <= lim_g) ? s1 * walpha : -INFINITY;
    s2 = (ta < t1 && ta <= lim_g8) ? s2 * walpha : -INFINITY;
    s3 = (tb < t1 && tb <= lim_g8) ? s3 * walpha : -INFINITY;
    float mx_g = fmaxf(s0, s1), mx_g8 = fmaxf(s2, s3);
    mx_g = fmaxf(mx_g, __shfl_xor_sync(0xffffffffu, mx_g, 1));
    mx_g = fmaxf(mx_g, __shfl_xor_sync(0xffffffffu, mx_g, 2));
    mx_g8 = fmaxf(mx_g8, __shfl_xor_sync(0xffffffffu, mx_g8, 1));
    mx_g8 = fmaxf(mx_g8, __shfl_xor_sync(0xffffffffu, mx_g8, 2));
    const float mn_g = fmaxf(m_g, mx_g), mn_g8 = fmaxf(m_g8, mx_g8);
    const float mu_g = mn_g == -INFINITY ? 0.0f : mn_g, mu_g8 = mn_g8 == -INFINITY ? 0.0f : mn_g8;
    const float corr_g = ex2(m_g - mu_g), corr_g8 = ex2(m_g8 - mu_g8);
    m_g = mn_g;
    m_g8 = mn_g8;
    s0 = ex2(s0 - mu_g);
    s1 = ex2(s1 - mu_g);
    s2 = ex2(s2 - mu_g8);
    s3 = ex2(s3 - mu_g8);
    l_g = fmaf(l_g, corr_g, s0 + s1);
    l_g8 = fmaf(l_g8, corr_g8, s2 + s3);
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        O[b][j][0] *= corr_g;
        O[b][j][1] *= corr_g;
        O[b][j][2] *= corr_g8;
        O[b][j][3] *= corr_g8;
      }
#pragma unroll
    for (int t = 0; t < kWinStage; ++t) {
      const int src = (lane & ~3) | (t >> 1);            // lane (g, t / 2) holds token t's p
      const float pg = __shfl_sync(0xffffffffu, (t & 1) ? s1 : s0, src);
      const float pg8 = __shfl_sync(0xffffffffu, (t & 1) ? s3 : s2, src);
      const float *vr = reinterpret_cast<const float *>(sb + (kWinStage + t) * kWinPitch) + 8 * c;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float4 v0 = *reinterpret_cast<const float4 *>(vr + 32 * b);
        const float4 v1 = *reinterpret_cast<const float4 *>(vr + 32 * b + 4);
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          O[b][j][0] = fmaf(pg, v[j], O[b][j][0]);
          O[b][j][1] = fmaf(pg, v[4 + j], O[b][j][1]);
          O[b][j][2] = fmaf(pg8, v[j], O[b][j][2]);
          O[b][j][3] = fmaf(pg8, v[4 + j], O[b][j][3]);
        }
      }
    }
  }

  if (!win) {
    // A fragment of k-step 2b + st: rows g / g+8, k slots (2c, 2c+1) = dims (8c + 2st, 8c + 2st + 4)
    // of block b, slots (2c+8, 2c+9) = dims (8c + 2st + 1, 8c + 2st + 5) divided by 16
    uint32_t aq[8][4];
    float zq_g, zq_g8;
    {
      int qs_g = 0, qs_g8 = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint2 wg = *reinterpret_cast<const uint2 *>(q8s + (16 * warp + g) * kD + 32 * b + 8 * c);
        const uint2 wg8 = *reinterpret_cast<const uint2 *>(q8s + (16 * warp + g + 8) * kD + 32 * b + 8 * c);
        float h[8], h8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int v = (int)(int8_t)(((i < 4 ? wg.x : wg.y) >> (8 * (i & 3))) & 0xFFu);
          const int v8 = (int)(int8_t)(((i < 4 ? wg8.x : wg8.y) >> (8 * (i & 3))) & 0xFFu);
          qs_g += v;
          qs_g8 += v8;
          h[i] = (float)v;
          h8[i] = (float)v8;
        }
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          aq[2 * b + st][0] = pack_f16x2(h[2 * st], h[2 * st + 4]);
          aq[2 * b + st][1] = pack_f16x2(h8[2 * st], h8[2 * st + 4]);
          aq[2 * b + st][2] = pack_f16x2(h[2 * st + 1] * 0.0625f, h[2 * st + 5] * 0.0625f);
          aq[2 * b + st][3] = pack_f16x2(h8[2 * st + 1] * 0.0625f, h8[2 * st + 5] * 0.0625f);
        }
      }
      qs_g += __shfl_xor_sync(0xffffffffu, qs_g, 1);
      qs_g += __shfl_xor_sync(0xffffffffu, qs_g, 2);
      qs_g8 += __shfl_xor_sync(0xffffffffu, qs_g8, 1);
      qs_g8 += __shfl_xor_sync(0xffffffffu, qs_g8, 2);
      zq_g = -8.0f * (float)qs_g * 5.9604644775390625e-8f;     // exact: |8 qs| < 2^17
      zq_g8 = -8.0f * (float)qs_g8 * 5.9604644775390625e-8f;
    }
    for (int i = 0; i < n_stages; ++i) {
      cp_async_wait<kRing - 2>();
      __syncthreads();                                     // stage i landed; stage i-1 fully read
      issue(i + kRing - 1);
      const int ts = t0 + i * kStage;
      if (ts > warp_lim) continue;                         // none of this warp's rows sees the stage
      const uint8_t *sb = smem + (i % kRing) * kStageBytes;
      const uint32_t sK = smem_addr(sb), sV = smem_addr(sb + kOffV);
      const float *skf = reinterpret_cast<const float *>(sb + kOffSK);
      const float *svf = reinterpret_cast<const float *>(sb + kOffSV);

      // two 32-token halves: S = Q8 . K^T for four 8-token tiles, online softmax, O += P' . V
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int tsub = ts + 32 * hh;
        if (tsub > warp_lim) break;
        float s[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t kw[4];                                    // token 8j + g, blocks 0..3, word c
          ldsm_x4(sK + swz(32 * hh + 8 * j + (lane & 7), lane >> 3), kw);
          float d[4] = {zq_g, zq_g, zq_g8, zq_g8};
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t u[4];
            unpack8_sub<false>(kw[b], u);
            mma16816(d, aq[2 * b], u[0], u[1]);
            mma16816(d, aq[2 * b + 1], u[2], u[3]);
          }
          const float2 sk = *reinterpret_cast<const float2 *>(skf + 32 * hh + 8 * j + 2 * c);
          s[j][0] = d[0] * alpha_g * sk.x;
          s[j][1] = d[1] * alpha_g * sk.y;
          s[j][2] = d[2] * alpha_g8 * sk.x;
          s[j][3] = d[3] * alpha_g8 * sk.y;
        }
        if (tsub + 32 > t1 || tsub + 31 > warp_min) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int ta = tsub + 8 * j + 2 * c, tb = ta + 1;
            if (!(ta < t1 && ta <= lim_g)) s[j][0] = -INFINITY;
            if (!(tb < t1 && tb <= lim_g)) s[j][1] = -INFINITY;
            if (!(ta < t1 && ta <= lim_g8)) s[j][2] = -INFINITY;
            if (!(tb < t1 && tb <= lim_g8)) s[j][3] = -INFINITY;
          }
        }
        // ---------------- online softmax (base 2), rows g and g+8
        float mx_g = fmaxf(s[0][0], s[0][1]), mx_g8 = fmaxf(s[0][2], s[0][3]);
#pragma unroll
        for (int j = 1; j < 4; ++j) {
          mx_g = fmaxf(mx_g, fmaxf(s[j][0], s[j][1]));
          mx_g8 = fmaxf(mx_g8, fmaxf(s[j][2], s[j][3]));
        }
        mx_g = fmaxf(mx_g, __shfl_xor_sync(0xffffffffu, mx_g, 1));
        mx_g = fmaxf(mx_g, __shfl_xor_sync(0xffffffffu, mx_g, 2));
        mx_g8 = fmaxf(mx_g8, __shfl_xor_sync(0xffffffffu, mx_g8, 1));
        mx_g8 = fmaxf(mx_g8, __shfl_xor_sync(0xffffffffu, mx_g8, 2));
        const float mn_g = fmaxf(m_g, mx_g), mn_g8 = fmaxf(m_g8, mx_g8);
        const float mu_g = mn_g == -INFINITY ? 0.0f : mn_g, mu_g8 = mn_g8 == -INFINITY ? 0.0f : mn_g8;
        const float corr_g = ex2(m_g - mu_g), corr_g8 = ex2(m_g8 - mu_g8);
        m_g = mn_g;
        m_g8 = mn_g8;
        if (__any_sync(0xffffffffu, corr_g != 1.0f || corr_g8 != 1.0f)) {
#pragma unroll
          for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              O[b][j][0] *= corr_g;
              O[b][j][1] *= corr_g;
              O[b][j][2] *= corr_g8;
              O[b][j][3] *= corr_g8;
            }
        }
        float ls_g = 0.0f, ls_g8 = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s[j][0] = ex2(s[j][0] - mu_g);
          s[j][1] = ex2(s[j][1] - mu_g);
          s[j][2] = ex2(s[j][2] - mu_g8);
          s[j][3] = ex2(s[j][3] - mu_g8);
          ls_g += s[j][0] + s[j][1];
          ls_g8 += s[j][2] + s[j][3];
          const float2 sv = *reinterpret_cast<const float2 *>(svf + 32 * hh + 8 * j + 2 * c);
          s[j][0] *= sv.x;                                   // P' = p * s_v
          s[j][1] *= sv.y;
          s[j][2] *= sv.x;
          s[j][3] *= sv.y;
        }
        l_g = fmaf(l_g, corr_g, ls_g);
        l_g8 = fmaf(l_g8, corr_g8, ls_g8);

        // O += P' . V, two 16-token steps
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          uint32_t ah[4], al[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // e = 0: (row g, tile 2kk), 1: (row g+8, tile 2kk), 2: (row g, tile 2kk+1), 3: (row g+8, tile 2kk+1)
            const int j = 2 * kk + (e >> 1), xx = (e & 1) ? 2 : 0;
            ah[e] = pack_f16x2(s[j][xx], s[j][xx + 1]);
            const float2 f = __half22float2(u32_as_h2(ah[e]));
            al[e] = pack_f16x2(s[j][xx] - f.x, s[j][xx + 1] - f.y);
          }
          // A order: a0 = (row g, tokens 2c..), a1 = (row g+8, tokens 2c..), a2 = (row g, tokens 8+2c..),
          // a3 = (row g+8, tokens 8+2c..)
          const uint32_t Ah[4] = {ah[0], ah[1], ah[2], ah[3]};
          const uint32_t Al[4] = {al[0], al[1], al[2], al[3]};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t vw[4];                                  // (2c.., block 2h), (8+2c.., 2h), (2c.., 2h+1), (8+2c.., 2h+1)
            const int mi = lane >> 3;
            ldsm_x4_t(sV + swz(32 * hh + 16 * kk + (mi & 1) * 8 + (lane & 7), 2 * h + (mi >> 1)), vw);
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int b = 2 * h + e2;
              uint32_t ua[4], ub[4];
              unpack8_q4(vw[2 * e2], ua);
              unpack8_q4(vw[2 * e2 + 1], ub);
#pragma unroll
              for (int jp = 0; jp < 4; ++jp) {
                mma16816(O[b][jp], Ah, ua[jp], ub[jp]);
                mma16816(O[b][jp], Al, ua[jp], ub[jp]);
              }
            }
          }
        }
      }
    }

  }

  // ---------------- rows g and g+8: l over the four lanes of the row, then this chunk's partial
  l_g += __shfl_xor_sync(0xffffffffu, l_g, 1);
  l_g += __shfl_xor_sync(0xffffffffu, l_g, 2);
  l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 1);
  l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 2);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rg8 : rg;
    const int lim = half ? lim_g8 : lim_g;
    if (r >= R || t0 > lim) continue;                    // row does not see this chunk
    const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
    const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
    float *po = a.part_o + pi * kD;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      // c0 / c2 of tile (b, j') are dim 32b + 8c + j', c1 / c3 dim 32b + 8c + 4 + j'
      *reinterpret_cast<float4 *>(po + 32 * b + 8 * c) =
          make_float4(O[b][0][2 * half], O[b][1][2 * half], O[b][2][2 * half], O[b][3][2 * half]);
      *reinterpret_cast<float4 *>(po + 32 * b + 8 * c + 4) =
          make_float4(O[b][0][2 * half + 1], O[b][1][2 * half + 1], O[b][2][2 * half + 1], O[b][3][2 * half + 1]);
    }
    if (c == 0) {
      a.part_m[pi] = (half ? m_g8 : m_g) * kLn2;         // natural-log units, like the other kernels
      a.part_l[pi] = half ? l_g8 : l_g;
    }
  }
}

}  // namespace

bool prefill_supported(const AttendArgs &a) {
  return prefill_shape(a.cache.layout, a.cache.D, a.gqa * a.n_q) && a.n_body > 0 && a.chunk % kStage == 0;
}

cudaError_t launch_attend_prefill(const AttendArgs &a, cudaStream_t st) {
  static bool configured[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(attend_prefill_had_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int R = a.gqa * a.n_q;
  cudaLaunchConfig_t cfg = {};
  // one more chunk index for the recent window (when present)
  cfg.gridDim = dim3((R + kRows - 1) / kRows, a.n_chunks + (a.n_win > 0 ? 1 : 0), a.cache.B * a.cache.H);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_prefill_had_kernel, a);
}

}  // namespace kvq
