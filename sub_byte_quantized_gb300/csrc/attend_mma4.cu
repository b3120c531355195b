// Warp-specialised tensor-core phase 1 for the 4-bit layouts (Q4_0, the asymmetric g=32 layout and
// the per-token Hadamard int4 body), head_dim 128, up to 8 query rows per kv head; the library runs
// it for the asymmetric layout (where the per-warp kernel runs out of registers). The arithmetic
// is the one of the per-warp kernel (attend_mma.cu):
//   QK:  S^T[16 tokens][8 rows] += K[16 tokens][16 dims] . Q^T[16 dims][8 rows]
//   PV:  O^T[16 dims][8 rows]   += V^T[16 dims][16 tokens] . P'^T[16 tokens][8 rows]
// with the codes as exact f16 operands (K as subnormals u * 2^-24 with the offset in the
// accumulator's initial value; V by the exact f16 fix-up: asymmetric V as n - 8, the group's
// midpoint z + 8 s coming from one small mma per tile), exact query operands (power-of-two
// prescale, hi + lo parts for f32 queries; int8 codes for the Hadamard layout) and P' = p * s_v
// kept as f16 hi + lo parts.
//
// Work split: a CTA of eight warps streams one chunk in 128-token stages. Warps 0-3 ("K warps") each
// score two 16-token tiles of stage i and run the online softmax; warps 4-7 ("V warps") accumulate
// P'V for the same tiles one stage later, reading the probabilities (already transposed into the
// mma B layout, as f16 hi + lo parts) and the rescale factors that the K warps left in shared
// memory. The per-stage CTA barrier orders the hand-off. K and V stream through separate
// three-slot rings: 16-byte cp.async of the 64-byte payload rows (64-byte XOR swizzle for the
// ldmatrix reads) plus the per-token scales (and zero-points); the copy of stage i+2 of K and
// stage i+1 of V is issued while stage i is scored. For the Hadamard layout the per-token V scale
// travels with K, so that the K warps form p * s_v before the hi/lo split. At the end the four
// tile states are combined in shared memory and the CTA writes one (m, l, o) partial per row.
#include <cfloat>
#include <climits>

#include "kvq_internal.cuh"
#include "mma_util.cuh"

namespace kvq {
namespace {
using namespace mma;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
#ifndef KVQ_MMA4_TPW
#define KVQ_MMA4_TPW 2
#endif
constexpr int kTPW = KVQ_MMA4_TPW;      // 16-token tiles per warp per stage
constexpr int kTiles = 4 * kTPW;        // tiles per stage
constexpr int kStage = 16 * kTiles;     // tokens per stage
constexpr int kRing = 3;
constexpr int kD = 128;
constexpr int kRowBytes = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int L>
struct Geo4 {
  static constexpr bool HAD = L == KVQ_HAD_INT4, ASYM = L == KVQ_ASYM4_G32;
  static constexpr int SCB = HAD ? 4 : 8;                 // scale bytes per token
  static constexpr int OFF_SC = kStage * kRowBytes;       // scales after the payload rows
  static constexpr int OFF_X2 = OFF_SC + kStage * SCB;    // asym zero-points / Hadamard s_v (K slot)
  static constexpr int X2B = ASYM ? 8 : (HAD ? 4 : 0);
  static constexpr int SLOT = OFF_X2 + kStage * X2B;
  static constexpr int OFF_V = kRing * SLOT;              // K ring, then V ring
  static constexpr int OFF_X = 2 * kRing * SLOT;          // hand-off [tile][parity][lane] 32 bytes
  static constexpr int QSCR = 8 * 128 + 8 * 4;            // Hadamard: int8 query codes + scales per K warp
  static constexpr int OFF_Q = OFF_X + kTiles * 2 * 32 * 32;
  static constexpr int SMEM = OFF_Q + (HAD ? 4 * QSCR : 0);
  static_assert((64 + 32 * kD) * 4 <= OFF_X, "combine area (cm, cl, co) fits below the hand-off");
};

// Last token query row r (of the gqa * n_q rows of a kv head) may see; negative if none.
__device__ __forceinline__ int row_limit_of(const AttendArgs &a, const SeqLen &sl, int r) {
  return row_limit(a, sl, r % a.n_q);
}

// Byte offset of (row, 16-byte column j) inside a swizzled 64-byte-row slab.
__device__ __forceinline__ uint32_t swz(int row, int j) {
  return (uint32_t)(row * kRowBytes + ((j ^ ((row >> 1) & 3)) << 4));
}

template <int LAYOUT, bool QSPLIT, bool PAGED>
__global__ void __launch_bounds__(kThreads, kMma4CtasPerSm) attend_mma4_kernel(AttendArgs a) {
  using G = Geo4<LAYOUT>;
  constexpr bool ASYM = G::ASYM, HAD = G::HAD;
  constexpr int SCB = G::SCB;
  extern __shared__ __align__(1024) uint8_t smem[];
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  const CacheView &cv = a.cache;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int tw = warp & 3;
  const bool kwarp = warp < 4;
  const int chunk_id = blockIdx.x;
  const int bh = blockIdx.y;
  const int bb = bh / cv.H, kvh = bh - bb * cv.H;
  const SeqLen sl = seq_of_t<PAGED>(a, bb);             // this sequence's lengths
  const int R = a.gqa * a.n_q;

  const int t0 = chunk_id * sl.chunk;
  const int t1 = min(sl.n_body, t0 + sl.chunk);
  // the rows' limits, folded here so that nothing of the sequence's lengths stays live below:
  // the widest and narrowest limit, this thread's two accumulator rows, and a mask of the rows
  // that see this chunk
  int w_lim = -1, min_lim = INT_MAX, lim0 = -1, lim1 = -1;
  unsigned row_vis = 0u;
  for (int r = 0; r < R; ++r) {
    const int l = row_limit_of(a, sl, r);
    w_lim = max(w_lim, l);
    min_lim = min(min_lim, l);
    if (r == 2 * c) lim0 = l;
    if (r == 2 * c + 1) lim1 = l;
    if (t0 <= l) row_vis |= 1u << r;
  }
  // rows appended by the preceding kernel: only the CTAs that read them wait for it
  pdl_wait_if(t0 <= w_lim && t0 < sl.fresh_hi && sl.fresh_lo < min(t1, w_lim + 1));
  if (t0 > w_lim || t0 >= t1) return;                 // no row sees this chunk (phase 2 skips it)
  const int t_end = min(t1, w_lim + 1);
  const int n_stages = (t_end - t0 + kStage - 1) / kStage;

  // ---- CTA-wide copy of plane kvp's stage s into a ring slot: the payload in 16-byte pieces
  // (iteration k of each thread covers rows 64k .. 64k+63), one scale per token (threads 0-127)
  // and, in the same slot, the asymmetric zero-points or (K slot, Hadamard) the V scales (threads
  // 128-255). Rows past t_end read as zero. Each 64-token half of the stage is a run of
  // consecutive plane rows (a page holds at least 64 aligned tokens): one base row per half.
  static_assert(kStage == 128 && kThreads == 256, "two 64-row halves, one payload piece per thread each");
  const size_t head_row0 = (size_t)bh * cv.cap;           // contiguous cache: row of token 0
  auto copy_stage = [&](int kvp, uint8_t *slot, int s) {
    const int ts = t0 + s * kStage;
    const uint32_t sd = smem_addr(slot);
    const int row = threadIdx.x & (kStage - 1);          // scale / zero-point row of this thread
    const bool second = threadIdx.x >= kStage;
    const bool ok_row = ts + row < t_end;
    size_t tok;                                          // plane row of that token (or a valid row)
    if constexpr (!PAGED) {
      const uint8_t *pl = cv.payload[kvp] + head_row0 * kRowBytes;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int q = threadIdx.x + kThreads * k, r = q >> 2, j = q & 3;
        const bool ok = ts + r < t_end;
        const size_t off = ok ? (size_t)ts * kRowBytes + 16 * q : (size_t)t0 * kRowBytes;
        cp_async16(sd + swz(r, j), pl + off, ok ? 16 : 0);
      }
      tok = head_row0 + (size_t)(ok_row ? ts + row : t0);
    } else {
      const size_t rb0 = cache_row_paged(cv, bb, kvh, ts);
      const size_t rb1 = ts + 64 < t_end ? cache_row_paged(cv, bb, kvh, ts + 64) : rb0;
      const int rr = threadIdx.x >> 2, j = threadIdx.x & 3;   // row within a half, 16-byte column
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint8_t *src = cv.payload[kvp] + (k ? rb1 : rb0) * kRowBytes;
        const bool ok = ts + 64 * k + rr < t_end;
        cp_async16(sd + swz(64 * k + rr, j), src + (ok ? rr * kRowBytes + 16 * j : 0), ok ? 16 : 0);
      }
      tok = ok_row ? (row < 64 ? rb0 + row : rb1 + (row - 64)) : rb0;
    }
    if (!second) {
      cp_async_scale<SCB>(sd + G::OFF_SC + row * SCB, static_cast<const uint8_t *>(cv.scale[kvp]) + tok * SCB,
                          ok_row ? SCB : 0);
    } else if (ASYM) {
      cp_async8(sd + G::OFF_X2 + row * 8, reinterpret_cast<const uint8_t *>(cv.zero[kvp]) + tok * 8, ok_row ? 8 : 0);
    } else if (HAD && kvp == 0) {
      cp_async4(sd + G::OFF_X2 + row * 4, static_cast<const uint8_t *>(cv.scale[1]) + tok * 4, ok_row ? 4 : 0);
    }
  };
  // one commit group per call: K of stage s and V of stage s - 1
  auto issue = [&](int s) {
    if (s < n_stages) copy_stage(0, smem + (s % kRing) * G::SLOT, s);
    if (s >= 1 && s - 1 < n_stages)      // V slot: the asymmetric zero-points only (Hadamard s_v rides with K)
      copy_stage(1, smem + G::OFF_V + ((s - 1) % kRing) * G::SLOT, s - 1);
    cp_async_commit();
  };
  issue(0);
  issue(1);

  uint8_t *xch = smem + G::OFF_X;
  const int r0 = 2 * c, r1 = 2 * c + 1;                 // the thread's two accumulator columns (query rows)

  if (kwarp) {
    // =============================== K warps: scores and online softmax
    // query fragments (B operand of QK): row g of the group, dims 32b + 8c + 0..7
    uint32_t bq_hi[8][2], bq_lo[QSPLIT ? 8 : 1][2];
    float qsum[4];
    float row_alpha;
    if (HAD) {
      // int8 query codes of the R rows, rotated and quantised per K warp into its scratch
      uint8_t *qs8 = smem + G::OFF_Q + tw * G::QSCR;
      float *qsq = reinterpret_cast<float *>(qs8 + 8 * 128);
      for (int r = 0; r < R; ++r) {
        const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
        const size_t grow = ((size_t)bb * a.Hq + hq) * a.n_q + qi;
        float x[4];
        int q8v[4];
        load4_f32(a.q, a.q_dtype, grow * kD + lane * 4, x);
        const float sq = had_query_row<4>(x, q8v, lane);
        *reinterpret_cast<uint32_t *>(qs8 + r * 128 + lane * 4) =
            (uint32_t)(q8v[0] & 0xFF) | ((uint32_t)(q8v[1] & 0xFF) << 8) | ((uint32_t)(q8v[2] & 0xFF) << 16) |
            ((uint32_t)(q8v[3] & 0xFF) << 24);
        if (lane == 0) qsq[r] = sq;
      }
      __syncwarp();
      const bool live = g < R;
      row_alpha = (live ? a.scale * qsq[g] : 0.0f) * 16777216.0f * kLog2e;
      float qs = 0.0f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float h[8];
        const uint2 w8 = live ? *reinterpret_cast<const uint2 *>(qs8 + g * 128 + 32 * b + 8 * c) : make_uint2(0u, 0u);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t word = i < 4 ? w8.x : w8.y;
          h[i] = (float)(int8_t)((word >> (8 * (i & 3))) & 0xFFu);
          qs += h[i];
        }
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          bq_hi[2 * b + st][0] = pack_f16x2(h[2 * st], h[2 * st + 4]);
          bq_hi[2 * b + st][1] = pack_f16x2(h[2 * st + 1] * 0.0625f, h[2 * st + 5] * 0.0625f);
        }
        qsum[b] = 0.0f;
      }
      qs += __shfl_xor_sync(0xffffffffu, qs, 1);
      qs += __shfl_xor_sync(0xffffffffu, qs, 2);
      qsum[0] = qs;                                      // whole-row sum (one accumulator per token)
    } else {
      float x[4][8];
      const bool live = g < R;
      const int hq = kvh * a.gqa + (live ? g / a.n_q : 0);
      const int qi = live ? g % a.n_q : 0;
      const size_t grow = ((size_t)bb * a.Hq + hq) * a.n_q + qi;
      float mx = 0.0f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (live) {
          load8_f32(a.q, a.q_dtype, grow * kD + 32 * b + 8 * c, x[b]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) x[b][i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(x[b][i]));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      // power-of-two prescale: the row's largest |q| lands in [2^13, 2^14), exact and clear of
      // f16 overflow; the inverse goes into the row's alpha
      int e = 0;
      if (mx > 0.0f) e = min(max(((__float_as_int(mx) >> 23) & 0xFF) - 127 - 13, -100), 100);
      const float pre = ldexpf(1.0f, -e), post = ldexpf(1.0f, e);
      row_alpha = a.scale * post * 16777216.0f * kLog2e;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float s = 0.0f, h[8], l[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float v = x[b][i] * pre;
          s += v;
          h[i] = __half2float(__float2half_rn(v));
          l[i] = v - h[i];
        }
        qsum[b] = s;
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          // odd dims face the high 4-bit fields (16 u * 2^-24): their query entries are / 16
          bq_hi[2 * b + st][0] = pack_f16x2(h[2 * st], h[2 * st + 4]);
          bq_hi[2 * b + st][1] = pack_f16x2(h[2 * st + 1] * 0.0625f, h[2 * st + 5] * 0.0625f);
          if (QSPLIT) {
            bq_lo[2 * b + st][0] = pack_f16x2(l[2 * st], l[2 * st + 4]);
            bq_lo[2 * b + st][1] = pack_f16x2(l[2 * st + 1] * 0.0625f, l[2 * st + 5] * 0.0625f);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        qsum[b] += __shfl_xor_sync(0xffffffffu, qsum[b], 1);
        qsum[b] += __shfl_xor_sync(0xffffffffu, qsum[b], 2);
      }
    }
    const float alpha0 = __shfl_sync(0xffffffffu, row_alpha, r0 * 4);
    const float alpha1 = __shfl_sync(0xffffffffu, row_alpha, r1 * 4);
    // zq: per-block row sums of q in accumulator units (x 2^-24). ASYM: multiplied by each
    // token's zero-point; Q4_0 and Hadamard: -8 zq is the accumulator's initial value.
    float zq0[4], zq1[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      zq0[b] = __shfl_sync(0xffffffffu, qsum[b], r0 * 4) * 5.9604644775390625e-8f;
      zq1[b] = __shfl_sync(0xffffffffu, qsum[b], r1 * 4) * 5.9604644775390625e-8f;
      if (!ASYM) {
        zq0[b] *= -8.0f;
        zq1[b] *= -8.0f;
      }
    }
    const int mi = lane >> 3;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

    for (int i = 0; i <= n_stages; ++i) {
      cp_async_wait<1>();
      __syncthreads();                                   // K(i), V(i-1) landed; refilled slots are free
      issue(i + 2);
      if (i == n_stages) continue;
#pragma unroll
      for (int tt = 0; tt < kTPW; ++tt) {
      const int tile = kTPW * tw + tt;
      const int ts = t0 + i * kStage + 16 * tile;
      // (a tile past t_end is zero-filled and fully masked: it contributes nothing)
      const uint8_t *sb = smem + (i % kRing) * G::SLOT;
      const uint32_t sK = smem_addr(sb);
      const int trow = 16 * tile;
      uint32_t kw[2][4];
#pragma unroll
      for (int half = 0; half < 2; ++half)
        ldsm_x4(sK + swz(trow + (mi & 1) * 8 + (lane & 7), 2 * half + (mi >> 1)), kw[half]);
      float s[4];
      if (HAD) {
        // one per-token scale: the eight k-steps accumulate the exact integer dot (x 2^-24) in
        // two chains
        float dA[4] = {zq0[0], zq1[0], zq0[0], zq1[0]}, dB[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t ug[4], u8[4];
          unpack8_sub<false>(kw[b >> 1][(b & 1) * 2 + 0], ug);
          unpack8_sub<false>(kw[b >> 1][(b & 1) * 2 + 1], u8);
          const uint32_t A0[4] = {ug[0], u8[0], ug[1], u8[1]};
          const uint32_t A1[4] = {ug[2], u8[2], ug[3], u8[3]};
          float(&d)[4] = (b & 1) ? dB : dA;
          mma16816(d, A0, bq_hi[2 * b][0], bq_hi[2 * b][1]);
          mma16816(d, A1, bq_hi[2 * b + 1][0], bq_hi[2 * b + 1][1]);
        }
        const float skg = *reinterpret_cast<const float *>(sb + G::OFF_SC + (trow + g) * 4);
        const float skg8 = *reinterpret_cast<const float *>(sb + G::OFF_SC + (trow + g + 8) * 4);
        s[0] = (dA[0] + dB[0]) * skg * alpha0;
        s[1] = (dA[1] + dB[1]) * skg * alpha1;
        s[2] = (dA[2] + dB[2]) * skg8 * alpha0;
        s[3] = (dA[3] + dB[3]) * skg8 * alpha1;
      } else {
        const uint2 skg = *reinterpret_cast<const uint2 *>(sb + G::OFF_SC + (trow + g) * 8);
        const uint2 skg8 = *reinterpret_cast<const uint2 *>(sb + G::OFF_SC + (trow + g + 8) * 8);
        const float2 sg01 = __half22float2(u32_as_h2(skg.x)), sg23 = __half22float2(u32_as_h2(skg.y));
        const float2 s801 = __half22float2(u32_as_h2(skg8.x)), s823 = __half22float2(u32_as_h2(skg8.y));
        const float skg_f[4] = {sg01.x, sg01.y, sg23.x, sg23.y};
        const float skg8_f[4] = {s801.x, s801.y, s823.x, s823.y};
        float zg_f[4] = {0.f, 0.f, 0.f, 0.f}, zg8_f[4] = {0.f, 0.f, 0.f, 0.f};
        if (ASYM) {
          const uint2 zg = *reinterpret_cast<const uint2 *>(sb + G::OFF_X2 + (trow + g) * 8);
          const uint2 zg8 = *reinterpret_cast<const uint2 *>(sb + G::OFF_X2 + (trow + g + 8) * 8);
          const float2 a01 = __half22float2(u32_as_h2(zg.x)), a23 = __half22float2(u32_as_h2(zg.y));
          const float2 b01 = __half22float2(u32_as_h2(zg8.x)), b23 = __half22float2(u32_as_h2(zg8.y));
          zg_f[0] = a01.x; zg_f[1] = a01.y; zg_f[2] = a23.x; zg_f[3] = a23.y;
          zg8_f[0] = b01.x; zg8_f[1] = b01.y; zg8_f[2] = b23.x; zg8_f[3] = b23.y;
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t ug[4], u8[4];
          unpack8_sub<ASYM>(kw[b >> 1][(b & 1) * 2 + 0], ug);
          unpack8_sub<ASYM>(kw[b >> 1][(b & 1) * 2 + 1], u8);
          const uint32_t A0[4] = {ug[0], u8[0], ug[1], u8[1]};
          const uint32_t A1[4] = {ug[2], u8[2], ug[3], u8[3]};
          // the first mma takes the offset (ASYM: zero) as its separate C operand: no register copies
          float d[4];
          const float c0 = ASYM ? 0.0f : zq0[b], c1 = ASYM ? 0.0f : zq1[b];
          mma16816_c(d, A0, bq_hi[2 * b][0], bq_hi[2 * b][1], c0, c1, c0, c1);
          mma16816(d, A1, bq_hi[2 * b + 1][0], bq_hi[2 * b + 1][1]);
          if (QSPLIT) {
            mma16816(d, A0, bq_lo[2 * b][0], bq_lo[2 * b][1]);
            mma16816(d, A1, bq_lo[2 * b + 1][0], bq_lo[2 * b + 1][1]);
          }
          acc[0] = fmaf(skg_f[b], d[0], acc[0]);
          acc[1] = fmaf(skg_f[b], d[1], acc[1]);
          acc[2] = fmaf(skg8_f[b], d[2], acc[2]);
          acc[3] = fmaf(skg8_f[b], d[3], acc[3]);
          if (ASYM) {
            acc[0] = fmaf(zg_f[b], zq0[b], acc[0]);
            acc[1] = fmaf(zg_f[b], zq1[b], acc[1]);
            acc[2] = fmaf(zg8_f[b], zq0[b], acc[2]);
            acc[3] = fmaf(zg8_f[b], zq1[b], acc[3]);
          }
        }
        s[0] = acc[0] * alpha0;
        s[1] = acc[1] * alpha1;
        s[2] = acc[2] * alpha0;
        s[3] = acc[3] * alpha1;
      }
      if (ts + 16 > t1 || ts + 15 > min_lim) {
        const int ta = ts + g, tb = ta + 8;
        if (!(ta < t1 && ta <= lim0)) s[0] = -INFINITY;
        if (!(ta < t1 && ta <= lim1)) s[1] = -INFINITY;
        if (!(tb < t1 && tb <= lim0)) s[2] = -INFINITY;
        if (!(tb < t1 && tb <= lim1)) s[3] = -INFINITY;
      }
      // online softmax (base 2), rows r0 / r1
      float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
      for (int k = 4; k < 32; k <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, k));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, k));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = mn0 == -INFINITY ? 0.0f : mn0, mu1 = mn1 == -INFINITY ? 0.0f : mn1;
      const float corr0 = ex2(m0 - mu0), corr1 = ex2(m1 - mu1);
      m0 = mn0;
      m1 = mn1;
      float p0 = ex2(s[0] - mu0), p1 = ex2(s[1] - mu1), p2 = ex2(s[2] - mu0), p3 = ex2(s[3] - mu1);
      l0 = fmaf(l0, corr0, p0 + p2);
      l1 = fmaf(l1, corr1, p1 + p3);
      if (HAD) {                                         // per-token V scale: P' = p * s_v before the split
        const float svg = *reinterpret_cast<const float *>(sb + G::OFF_X2 + (trow + g) * 4);
        const float svg8 = *reinterpret_cast<const float *>(sb + G::OFF_X2 + (trow + g + 8) * 4);
        p0 *= svg;
        p1 *= svg;
        p2 *= svg8;
        p3 *= svg8;
      }
      // p -> exact hi + lo f16 parts, transposed once into the B layout: each f16 pair holds one
      // query row g and two consecutive tokens (2c, 2c+1) or (2c+8, 2c+9)
      const uint32_t h01 = pack_f16x2(p0, p1), h23 = pack_f16x2(p2, p3);
      const float2 f01 = __half22float2(u32_as_h2(h01)), f23 = __half22float2(u32_as_h2(h23));
      const uint32_t l01 = pack_f16x2(p0 - f01.x, p1 - f01.y), l23 = pack_f16x2(p2 - f23.x, p3 - f23.y);
      uint4 pb;
      pb.x = movm_t(h01);
      pb.y = movm_t(h23);
      pb.z = movm_t(l01);
      pb.w = movm_t(l23);
      uint8_t *xs = xch + ((tile * 2 + (i & 1)) * 32 + lane) * 32;
      *reinterpret_cast<uint4 *>(xs) = pb;
      *reinterpret_cast<float2 *>(xs + 16) = make_float2(corr0, corr1);
      }
    }
    // reduce l over the token lanes; publish (m, l) per row
#pragma unroll
    for (int k = 4; k < 32; k <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, k);
      l1 += __shfl_xor_sync(0xffffffffu, l1, k);
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();                                     // every warp is done with the rings
    float *cm = reinterpret_cast<float *>(smem);
    float *cl = cm + 32;
    if (g == 0) {
      cm[tw * 8 + r0] = m0;
      cm[tw * 8 + r1] = m1;
      cl[tw * 8 + r0] = l0;
      cl[tw * 8 + r1] = l1;
    }
  } else {
    // =============================== V warps: O^T += V^T . P'^T per 32-dim block
    float O[4][2][4];
    // ASYM: Dw[b][r] (+ Dw[b + 8][r]) = sum_t p_t x[t][b], x = z_v + 8 s_v the group midpoint
    // (hi part in rows b, lo part in rows b + 8), from one small mma per tile
    float Dw[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t wsel = (g & 1) ? 0x7632u : 0x5410u;
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k) O[b][h][k] = 0.0f;
    const int mi = lane >> 3;

    for (int i = 0; i <= n_stages; ++i) {
      cp_async_wait<1>();
      __syncthreads();
      issue(i + 2);
      const int j = i - 1;                               // the stage these warps consume
      if (j < 0) continue;
#pragma unroll
      for (int tt = 0; tt < kTPW; ++tt) {
      const int tile = kTPW * tw + tt;
      // (a tile past t_end is zero-filled and fully masked: it contributes nothing)
      const uint8_t *xs = xch + ((tile * 2 + (j & 1)) * 32 + lane) * 32;
      const uint4 pb = *reinterpret_cast<const uint4 *>(xs);
      const float2 cr = *reinterpret_cast<const float2 *>(xs + 16);
      if (__any_sync(0xffffffffu, cr.x != 1.0f || cr.y != 1.0f)) {
        Dw[0] *= cr.x;
        Dw[1] *= cr.y;
        Dw[2] *= cr.x;
        Dw[3] *= cr.y;
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            O[b][h][0] *= cr.x;
            O[b][h][1] *= cr.y;
            O[b][h][2] *= cr.x;
            O[b][h][3] *= cr.y;
          }
      }
      const uint8_t *sb = smem + G::OFF_V + (j % kRing) * G::SLOT;
      const uint32_t sV = smem_addr(sb);
      const int trow = 16 * tile;
      uint32_t vw[2][4];
#pragma unroll
      for (int half = 0; half < 2; ++half)
        ldsm_x4_t(sV + swz(trow + (mi & 1) * 8 + (lane & 7), 2 * half + (mi >> 1)), vw[half]);
      if (HAD) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t ua[4], ub[4];
          unpack8_q4(vw[b >> 1][(b & 1) * 2 + 0], ua);
          unpack8_q4(vw[b >> 1][(b & 1) * 2 + 1], ub);
          const uint32_t A0[4] = {ua[0], ua[1], ub[0], ub[1]};
          const uint32_t A1[4] = {ua[2], ua[3], ub[2], ub[3]};
          mma16816(O[b][0], A0, pb.x, pb.y);
          mma16816(O[b][0], A0, pb.z, pb.w);
          mma16816(O[b][1], A1, pb.x, pb.y);
          mma16816(O[b][1], A1, pb.z, pb.w);
        }
        continue;
      }
      // V block scales paired (s_v[2c][b], s_v[2c+1][b]), (s_v[2c+8][b], s_v[2c+9][b])
      const uint8_t *svb = sb + G::OFF_SC + trow * 8;
      const uint2 sa = *reinterpret_cast<const uint2 *>(svb + (2 * c) * 8);
      const uint2 sbv = *reinterpret_cast<const uint2 *>(svb + (2 * c + 1) * 8);
      const uint2 sc = *reinterpret_cast<const uint2 *>(svb + (2 * c + 8) * 8);
      const uint2 sd = *reinterpret_cast<const uint2 *>(svb + (2 * c + 9) * 8);
      const uint32_t sp0[4] = {__byte_perm(sa.x, sbv.x, 0x5410), __byte_perm(sa.x, sbv.x, 0x7632),
                               __byte_perm(sa.y, sbv.y, 0x5410), __byte_perm(sa.y, sbv.y, 0x7632)};
      const uint32_t sp1[4] = {__byte_perm(sc.x, sd.x, 0x5410), __byte_perm(sc.x, sd.x, 0x7632),
                               __byte_perm(sc.y, sd.y, 0x5410), __byte_perm(sc.y, sd.y, 0x7632)};
      if (ASYM) {
        // W operand (group midpoints): rows g < 4 hold the hi part of block g's x = z_v + 8 s_v for
        // tokens (2c, 2c+1), (2c+8, 2c+9), rows g + 8 its lo part. With the codes centred (n - 8)
        // neither the O accumulators nor this one carry an offset mass: an offset form (codes n,
        // zero-point z_v) adds two large sums that cancel, and the tensor core's truncated adds of
        // the small p lo products against them cost about 15x the error of this form.
        const uint8_t *zvb = sb + G::OFF_X2 + trow * 8;
        const uint2 wa = *reinterpret_cast<const uint2 *>(zvb + (2 * c) * 8);
        const uint2 wb = *reinterpret_cast<const uint2 *>(zvb + (2 * c + 1) * 8);
        const uint2 wc = *reinterpret_cast<const uint2 *>(zvb + (2 * c + 8) * 8);
        const uint2 wd = *reinterpret_cast<const uint2 *>(zvb + (2 * c + 9) * 8);
        const bool lo2 = g < 2;
        const uint32_t z0 = __byte_perm(lo2 ? wa.x : wa.y, lo2 ? wb.x : wb.y, wsel);
        const uint32_t z1 = __byte_perm(lo2 ? wc.x : wc.y, lo2 ? wd.x : wd.y, wsel);
        const uint32_t s0 = __byte_perm(lo2 ? sa.x : sa.y, lo2 ? sbv.x : sbv.y, wsel);
        const uint32_t s1 = __byte_perm(lo2 ? sc.x : sc.y, lo2 ? sd.x : sd.y, wsel);
        uint32_t h0, l0, h1, l1;
        midpoint_split(z0, s0, h0, l0);
        midpoint_split(z1, s1, h1, l1);
        if (g >= 4) h0 = l0 = h1 = l1 = 0u;
        const uint32_t Aw[4] = {h0, l0, h1, l1};
        mma16816(Dw, Aw, pb.x, pb.y);
        mma16816(Dw, Aw, pb.z, pb.w);
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // P' = (p_hi + p_lo) * s_v as hi + lo f16 (TwoProduct with the f16 fma):
        //   hi = rn(p_hi * s),  r = p_hi * s - hi (exact),  lo = rn(p_lo * s + r)
        const uint32_t hi0 = hmul2(pb.x, sp0[b]), hi1 = hmul2(pb.y, sp1[b]);
        const uint32_t e0 = hfma2_negc(pb.x, sp0[b], hi0), e1 = hfma2_negc(pb.y, sp1[b], hi1);
        const uint32_t lo0 = hfma2(pb.z, sp0[b], e0), lo1 = hfma2(pb.w, sp1[b], e1);
        uint32_t ua[4], ub[4];
        if (ASYM) {
          unpack8_u4m8(vw[b >> 1][(b & 1) * 2 + 0], ua);
          unpack8_u4m8(vw[b >> 1][(b & 1) * 2 + 1], ub);
        } else {
          unpack8_q4(vw[b >> 1][(b & 1) * 2 + 0], ua);
          unpack8_q4(vw[b >> 1][(b & 1) * 2 + 1], ub);
        }
        const uint32_t A0[4] = {ua[0], ua[1], ub[0], ub[1]};   // dims 4g+0 (row g), 4g+1 (row g+8)
        const uint32_t A1[4] = {ua[2], ua[3], ub[2], ub[3]};   // dims 4g+2, 4g+3
        mma16816(O[b][0], A0, hi0, hi1);
        mma16816(O[b][0], A0, lo0, lo1);
        mma16816(O[b][1], A1, hi0, hi1);
        mma16816(O[b][1], A1, lo0, lo1);
      }
      }
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();                                     // every warp is done with the rings
    // O holds s_v * code (asymmetric: s_v (n - 8)); asymmetric values add the midpoint term,
    // s_v n + z_v = s_v (n - 8) + (z_v + 8 s_v).
    float *co = reinterpret_cast<float *>(smem) + 64;    // [tile][8][128] after cm/cl
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float w0 = 0.0f, w1 = 0.0f;
      if (ASYM) {
        w0 = __shfl_sync(0xffffffffu, Dw[0] + Dw[2], 4 * b + c);
        w1 = __shfl_sync(0xffffffffu, Dw[1] + Dw[3], 4 * b + c);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int d = 32 * b + 4 * g + 2 * h;
        *reinterpret_cast<float2 *>(co + (tw * 8 + r0) * kD + d) = make_float2(O[b][h][0] + w0, O[b][h][2] + w0);
        *reinterpret_cast<float2 *>(co + (tw * 8 + r1) * kD + d) = make_float2(O[b][h][1] + w1, O[b][h][3] + w1);
      }
    }
  }
  __syncthreads();
  // ---------------- combine the four tiles: cm/cl [tile][8], co [tile][8][128]
  const float *cm = reinterpret_cast<const float *>(smem);
  const float *cl = cm + 32;
  const float *co = cm + 64;
  for (int r = 0; r < R; ++r) {
    if (!((row_vis >> r) & 1u)) continue;                // row does not see this chunk
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * 8 + r]);
    float wt[4], L = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      wt[w] = cm[w * 8 + r] == -INFINITY ? 0.0f : ex2(cm[w * 8 + r] - M);
      L = fmaf(cl[w * 8 + r], wt[w], L);
    }
    const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
    const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
    if (threadIdx.x < kD) {
      const int d = threadIdx.x;
      float acc = 0.0f;
#pragma unroll
      for (int w = 0; w < 4; ++w) acc = fmaf(co[(w * 8 + r) * kD + d], wt[w], acc);
      a.part_o[pi * kD + d] = acc;
    }
    if (threadIdx.x == 0) {
      a.part_m[pi] = M * kLn2;                           // natural-log units, like the other kernels
      a.part_l[pi] = L;
    }
  }
}

template <int LAYOUT, bool QSPLIT, bool PAGED>
cudaError_t launch_t(const AttendArgs &a, cudaStream_t st) {
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = set_smem_once(configured, attend_mma4_kernel<LAYOUT, QSPLIT, PAGED>, Geo4<LAYOUT>::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks, a.cache.B * a.cache.H);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Geo4<LAYOUT>::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_mma4_kernel<LAYOUT, QSPLIT, PAGED>, a);
}

}  // namespace

cudaError_t launch_attend_mma4(const AttendArgs &a, cudaStream_t st) {
  const bool split = a.q_dtype == KVQ_F32;
  const bool paged = a.cache.page_shift >= 0;
  if (a.cache.layout != KVQ_ASYM4_G32) return cudaErrorNotSupported;   // built for the layout that uses it
  if (split) return paged ? launch_t<KVQ_ASYM4_G32, true, true>(a, st) : launch_t<KVQ_ASYM4_G32, true, false>(a, st);
  return paged ? launch_t<KVQ_ASYM4_G32, false, true>(a, st) : launch_t<KVQ_ASYM4_G32, false, false>(a, st);
}

}  // namespace kvq
