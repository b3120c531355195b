// Tensor-core phase 1 of the split-K decode attention for the Q6_0 layout (per 32-value block:
// a 16-byte plane of low nibbles, an 8-byte plane of 2-bit high fields, one fp16 scale;
// "Storage layouts", q6_0, of the FreeToken cache-quantisation PR), head_dim 128 or 256, any number
// of query rows per kv head (the GQA group times the query rows of the call): a CTA takes a group of
// up to four of them (the grid's third dimension), so a call with more rows streams each chunk once
// per group of four.
//
// The contraction is the same as in the 4-bit kernel, with mma.sync.m16n8k16 (f16 in, f32
// accumulate):
//   QK:  S^T[16 tokens][8 cols] += K[16 tokens][16 dims] . Q^T[16 dims][8 cols]
//   PV:  O^T[16 dims][8 cols]   += V^T[16 dims][16 tokens] . P'^T[16 tokens][8 cols]
// With at most four query rows the eight mma columns hold each row twice: columns 0-3 the f16
// "hi" parts, columns 4-7 the "lo" parts (q = hi + lo for f32 queries, P' = hi + lo for the
// scaled probabilities), so one mma carries both halves; the two column groups are added at the
// end.
//
// Operands: a 6-bit code u = code + 32 in [0, 63] enters as the exact f16 subnormal u * 2^-24 (low-
// nibble positions) or 16 u * 2^-24 (high-nibble positions, whose query entries are divided by
// 16). The low-plane word of 8 nibbles is masked per pair as in the 4-bit kernel, and the
// matching 2-bit fields of the high plane (sign bit flipped: u = v ^ 0x20) are shifted into bits
// 4-5 or 8-9 of the same f16 lanes. The -32 offset of K goes into the accumulator's initial value
// (-32 * sum(q) * 2^-24 per block); for V it comes from one extra small mma per tile,
// W[block][row] = sum_t s_v[t][block] * p[t][row], subtracted as 32 W in the epilogue.
//
// Work split: a CTA of eight warps streams its chunk in 64-token stages. Warps 0-3 ("K warps")
// each score one 16-token tile of stage i (all blocks) and run the online softmax; warps 4-7
// ("V warps") accumulate P'V for the same tiles one stage later, reading the probabilities and
// the rescale factors that the K warps left in shared memory. The per-stage CTA barrier orders
// the hand-off, so the two roles overlap without further synchronisation. K and V stream through
// separate three-slot rings (16-byte cp.async of whole token rows, contiguous in the cache, into
// rows padded by 16 bytes so that the per-lane 32/64-bit fragment reads are free of bank
// conflicts); the copy of stage i+2 of K and stage i+1 of V is issued while stage i is scored.
// At the end the four tile states are combined in shared memory and the CTA writes one
// (m, l, o) partial per query row.
#include <cfloat>
#include <climits>

#include "kvq_internal.cuh"
#include "mma_util.cuh"

namespace kvq {
namespace {
using namespace mma;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStage = 64;   // tokens per stage: four 16-token tiles
constexpr int kRing = 3;     // slots per ring (K and V each)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Geom {
  static constexpr int NB = D / 32;            // blocks per token row
  static constexpr int RB = 24 * NB;           // packed payload bytes per token
  static constexpr int PITCH = RB + 16;        // shared-memory row pitch (conflict-free reads)
  static constexpr int SB = 2 * NB;            // scale bytes per token
  static constexpr int PIECES = kStage * RB / 16;   // 16-byte copies per plane per stage
  static constexpr int OFF_SC = kStage * PITCH;     // scales after the rows, in each slot
  static constexpr int SLOT = OFF_SC + kStage * SB;
  static constexpr int OFF_V = kRing * SLOT;        // K ring, then V ring
  static constexpr int OFF_X = 2 * kRing * SLOT;    // hand-off: [tile][slot][lane] 32 bytes
  static constexpr int SMEM = OFF_X + 4 * 2 * 32 * 32;
};

// Eight 6-bit values -> four f16 subnormal pairs. w: eight low nibbles n0..n7 (n0 = bits 0-3),
// h: the matching 2-bit high fields t0..t3 in byte 0 and t4..t7 in byte 2 (t_i at bits 2i of its
// byte; bytes 1 and 3 are ignored). Pairs (0,4), (1,5), (2,6), (3,7); the code plus 32 is
// u = n + 16 (t ^ 2), at weight 1 for the even pairs' positions and 16 for the odd ones.
__device__ __forceinline__ void unpack6(uint32_t w, uint32_t h, uint32_t (&o)[4]) {
  const uint32_t hx = h ^ 0x00AA00AAu;        // flip the sign bit of every field
  const uint32_t w8 = w >> 8;
  // (a & c) | b with b pre-masked: lop3 LUT 0xEC
  o[0] = lop3<0xEC>(w, (hx << 4) & 0x00300030u, 0x000F000Fu);
  o[1] = lop3<0xEC>(w, (hx << 6) & 0x03000300u, 0x00F000F0u);
  o[2] = lop3<0xEC>(w8, hx & 0x00300030u, 0x000F000Fu);
  o[3] = lop3<0xEC>(w8, (hx << 2) & 0x03000300u, 0x00F000F0u);
}

// Last token query row r (of the gqa * n_q rows of a kv head) may see; negative if none.
__device__ __forceinline__ int row_limit_of(const AttendArgs &a, const SeqLen &sl, int r) {
  return row_limit(a, sl, r % a.n_q);
}

__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

template <int D, bool PAGED>
__global__ void __launch_bounds__(kThreads, kMmaQ6CtasPerSm(D)) attend_mma_q6_kernel(AttendArgs a) {
  using G = Geom<D>;
  constexpr int NB = G::NB;
  extern __shared__ __align__(1024) uint8_t smem[];
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  const CacheView &cv = a.cache;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int tw = warp & 3;                             // tile of the stage
  const bool kwarp = warp < 4;                         // role: K (scores) or V (P'V)
  const int chunk_id = blockIdx.x;
  const int bh = blockIdx.y;
  const int bb = bh / cv.H, kvh = bh - bb * cv.H;
  const SeqLen sl = seq_of_t<PAGED>(a, bb);             // this sequence's lengths
  // rows of this CTA: group blockIdx.z of four of the kv head's gqa * n_q rows (local row r is row
  // rbase + r of the kv head)
  const int rbase = 4 * blockIdx.z;
  const int R = min(4, a.gqa * a.n_q - rbase);

  const int t0 = chunk_id * sl.chunk;
  const int t1 = min(sl.n_body, t0 + sl.chunk);
  // the rows' limits, folded here so that nothing of the sequence's lengths stays live below:
  // the widest and narrowest limit, this thread's two accumulator rows, and a mask of the rows
  // that see this chunk
  int w_lim = -1, min_lim = INT_MAX, lim0 = -1, lim1 = -1;
  unsigned row_vis = 0u;
  for (int r = 0; r < R; ++r) {
    const int l = row_limit_of(a, sl, rbase + r);
    w_lim = max(w_lim, l);
    min_lim = min(min_lim, l);
    if (r == 2 * (c & 1)) lim0 = l;
    if (r == 2 * (c & 1) + 1) lim1 = l;
    if (t0 <= l) row_vis |= 1u << r;
  }
  // rows appended by the preceding kernel: only the CTAs that read them wait for it
  pdl_wait_if(t0 <= w_lim && t0 < sl.fresh_hi && sl.fresh_lo < min(t1, w_lim + 1));
  if (t0 > w_lim || t0 >= t1) return;                 // no row sees this chunk (phase 2 skips it)
  const int t_end = min(t1, w_lim + 1);
  const int n_stages = (t_end - t0 + kStage - 1) / kStage;

  // ---- copy of plane kvp's stage s into a ring slot: the stage's rows are consecutive plane
  // rows (a page holds at least 64 aligned tokens); 16-byte piece q goes to row q / (RB/16) of the
  // padded slot. Rows past t_end are zero-filled.
  const size_t head_row0 = (size_t)bh * cv.cap;           // contiguous cache: row of token 0
  auto copy_stage = [&](int kvp, uint8_t *slot, int s) {
    const int ts = t0 + s * kStage;
    const size_t r0 = cache_row_t<PAGED>(cv, bb, kvh, head_row0, ts);
    const uint8_t *pl = cv.payload[kvp] + r0 * G::RB;
    const uint8_t *sc = static_cast<const uint8_t *>(cv.scale[kvp]) + r0 * G::SB;
    const uint32_t sd = smem_addr(slot);
    if (ts + kStage <= t_end) {                          // full stage: no per-row bounds
      const uint8_t *src = pl;
#pragma unroll
      for (int j = 0; j < (G::PIECES + kThreads - 1) / kThreads; ++j) {
        const int q = threadIdx.x + kThreads * j;
        if (q < G::PIECES) {
          const int row = q / (G::RB / 16);
          cp_async16(sd + row * G::PITCH + 16 * (q - row * (G::RB / 16)), src + 16 * q, 16);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < (G::PIECES + kThreads - 1) / kThreads; ++j) {
        const int q = threadIdx.x + kThreads * j;
        if (q < G::PIECES) {
          const int row = q / (G::RB / 16), pc = q - row * (G::RB / 16);
          const bool ok = ts + row < t_end;
          const size_t off = ok ? (size_t)16 * q : 0;
          cp_async16(sd + row * G::PITCH + 16 * pc, pl + off, ok ? 16 : 0);
        }
      }
    }
    if (threadIdx.x < kStage) {
      const int row = threadIdx.x;
      const bool ok = ts + row < t_end;
      const uint8_t *src = sc + (size_t)(ok ? row : 0) * G::SB;
      const uint32_t dst = sd + G::OFF_SC + row * G::SB;
      if (G::SB == 16) cp_async16(dst, src, ok ? 16 : 0);
      else cp_async8(dst, src, ok ? 8 : 0);
    }
  };
  // one commit group per call: K of stage s and V of stage s - 1
  auto issue = [&](int s) {
    if (s < n_stages) copy_stage(0, smem + (s % kRing) * G::SLOT, s);
    if (s >= 1 && s - 1 < n_stages) copy_stage(1, smem + G::OFF_V + ((s - 1) % kRing) * G::SLOT, s - 1);
    cp_async_commit();
  };
  issue(0);
  issue(1);

  // hand-off slot of (tile, stage parity): per lane {bm0, bm1, ba0, ba1} and {corr0, corr1}
  uint8_t *xch = smem + G::OFF_X;
  const int r0 = 2 * (c & 1), r1 = r0 + 1;             // the thread's rows (accumulator columns 2c, 2c+1)

  if (kwarp) {
    // =============================== K warps: scores and online softmax
    // query fragments: lane (g, c) holds column g = row (g & 3), its f16 hi part (g < 4) or lo
    // part (g >= 4), dims 32b + 8c + 0..7 of every block b
    uint32_t bq[2 * NB][2];
    float qsum[NB];
    float row_alpha;
    {
      const int rq = g & 3;
      const bool live = rq < R;
      const int hq = kvh * a.gqa + (live ? (rbase + rq) / a.n_q : 0);
      const int qi = live ? (rbase + rq) % a.n_q : 0;
      const size_t grow = ((size_t)bb * a.Hq + hq) * a.n_q + qi;
      float x[NB][8];
      float mx = 0.0f;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (live) {
          load8_f32(a.q, a.q_dtype, grow * D + 32 * b + 8 * c, x[b]);
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
      row_alpha = live ? a.scale * post * 16777216.0f * kLog2e : 0.0f;
      const bool hi_col = g < 4;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float sm = 0.0f, u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float v = x[b][i] * pre;
          sm += v;
          const float h = __half2float(__float2half_rn(v));
          u[i] = hi_col ? h : v - h;
        }
        qsum[b] = sm;
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          bq[2 * b + st][0] = pack_f16x2(u[2 * st], u[2 * st + 4]);
          bq[2 * b + st][1] = pack_f16x2(u[2 * st + 1] * 0.0625f, u[2 * st + 5] * 0.0625f);
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        qsum[b] += __shfl_xor_sync(0xffffffffu, qsum[b], 1);
        qsum[b] += __shfl_xor_sync(0xffffffffu, qsum[b], 2);
      }
    }
    const float alpha0 = __shfl_sync(0xffffffffu, row_alpha, r0 * 4);
    const float alpha1 = __shfl_sync(0xffffffffu, row_alpha, r1 * 4);
    // K offset: -32 * sum(q) of the block in accumulator units (x 2^-24), in the hi columns only
    float zq0[NB], zq1[NB];
    {
      const float zf = c < 2 ? -32.0f * 5.9604644775390625e-8f : 0.0f;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        zq0[b] = __shfl_sync(0xffffffffu, qsum[b], r0 * 4) * zf;
        zq1[b] = __shfl_sync(0xffffffffu, qsum[b], r1 * 4) * zf;
      }
    }
    // bytes 2c, 2c+1 of a block's eight high bytes -> bytes 0 and 2
    const uint32_t sel_k = (uint32_t)(2 * c) | ((uint32_t)(2 * c + 1) << 8);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

    for (int i = 0; i <= n_stages; ++i) {
      cp_async_wait<1>();
      __syncthreads();                                   // K(i), V(i-1) landed; the slots refilled below are free
      issue(i + 2);
      const int tr = 16 * tw;
      const int ts = t0 + i * kStage + tr;
      if (i == n_stages || ts >= t_end) continue;
      const uint8_t *sb = smem + (i % kRing) * G::SLOT;
      const uint8_t *kg = sb + (tr + g) * G::PITCH, *kg8 = kg + 8 * G::PITCH;
      const uint8_t *kss = sb + G::OFF_SC;
      uint32_t skg[NB / 2], skg8[NB / 2];                // K scales of tokens g, g+8 (f16 pairs)
      if constexpr (NB == 8) {
        const uint4 x0 = *reinterpret_cast<const uint4 *>(kss + (tr + g) * G::SB);
        const uint4 x1 = *reinterpret_cast<const uint4 *>(kss + (tr + g + 8) * G::SB);
        skg[0] = x0.x; skg[1] = x0.y; skg[2] = x0.z; skg[3] = x0.w;
        skg8[0] = x1.x; skg8[1] = x1.y; skg8[2] = x1.z; skg8[3] = x1.w;
      } else {
        const uint2 x0 = *reinterpret_cast<const uint2 *>(kss + (tr + g) * G::SB);
        const uint2 x1 = *reinterpret_cast<const uint2 *>(kss + (tr + g + 8) * G::SB);
        skg[0] = x0.x; skg[1] = x0.y;
        skg8[0] = x1.x; skg8[1] = x1.y;
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint32_t wg = lds32(kg + 24 * b + 4 * c), wg8 = lds32(kg8 + 24 * b + 4 * c);
        const uint2 hg = *reinterpret_cast<const uint2 *>(kg + 24 * b + 16);
        const uint2 hg8 = *reinterpret_cast<const uint2 *>(kg8 + 24 * b + 16);
        uint32_t ug[4], u8[4];
        unpack6(wg, prmt(hg.x, hg.y, sel_k), ug);
        unpack6(wg8, prmt(hg8.x, hg8.y, sel_k), u8);
        const uint32_t A0[4] = {ug[0], u8[0], ug[1], u8[1]};
        const uint32_t A1[4] = {ug[2], u8[2], ug[3], u8[3]};
        float d[4];
        mma16816_c(d, A0, bq[2 * b][0], bq[2 * b][1], zq0[b], zq1[b], zq0[b], zq1[b]);
        mma16816(d, A1, bq[2 * b + 1][0], bq[2 * b + 1][1]);
        const float2 sg = __half22float2(u32_as_h2(skg[b >> 1])), sg8 = __half22float2(u32_as_h2(skg8[b >> 1]));
        const float kgs = (b & 1) ? sg.y : sg.x, kgs8 = (b & 1) ? sg8.y : sg8.x;
        acc[0] = fmaf(kgs, d[0], acc[0]);
        acc[1] = fmaf(kgs, d[1], acc[1]);
        acc[2] = fmaf(kgs8, d[2], acc[2]);
        acc[3] = fmaf(kgs8, d[3], acc[3]);
      }
      // hi + lo columns -> whole scores of rows r0, r1 (lanes c and c ^ 2 then agree)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], 2);
      float s[4] = {acc[0] * alpha0, acc[1] * alpha1, acc[2] * alpha0, acc[3] * alpha1};
      if (ts + 16 > t1 || ts + 15 > min_lim) {
        const int ta = ts + g, tb = ta + 8;
        if (!(ta < t1 && ta <= lim0)) s[0] = -INFINITY;
        if (!(ta < t1 && ta <= lim1)) s[1] = -INFINITY;
        if (!(tb < t1 && tb <= lim0)) s[2] = -INFINITY;
        if (!(tb < t1 && tb <= lim1)) s[3] = -INFINITY;
      }
      // online softmax (base 2)
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
      const float p0 = ex2(s[0] - mu0), p1 = ex2(s[1] - mu1), p2 = ex2(s[2] - mu0), p3 = ex2(s[3] - mu1);
      l0 = fmaf(l0, corr0, p0 + p2);
      l1 = fmaf(l1, corr1, p1 + p3);
      // P into the B layout: columns 0-3 hi parts, 4-7 lo parts of rows 0-3; for the lo columns
      // also the hi part of the same row (the scale product's error term)
      const uint32_t h01 = pack_f16x2(p0, p1), h23 = pack_f16x2(p2, p3);
      const float2 f01 = __half22float2(u32_as_h2(h01)), f23 = __half22float2(u32_as_h2(h23));
      const uint32_t l01 = pack_f16x2(p0 - f01.x, p1 - f01.y), l23 = pack_f16x2(p2 - f23.x, p3 - f23.y);
      uint4 pb;
      pb.x = movm_t(c >= 2 ? l01 : h01);                 // main part of column g
      pb.y = movm_t(c >= 2 ? l23 : h23);
      pb.z = movm_t(h01);
      pb.w = movm_t(h23);
      if (g < 4) pb.z = pb.w = 0u;
      uint8_t *xs = xch + ((tw * 2 + (i & 1)) * 32 + lane) * 32;
      *reinterpret_cast<uint4 *>(xs) = pb;
      *reinterpret_cast<float2 *>(xs + 16) = make_float2(corr0, corr1);
    }
    // reduce l over the token lanes; one lane per row pair publishes (m, l)
#pragma unroll
    for (int k = 4; k < 32; k <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, k);
      l1 += __shfl_xor_sync(0xffffffffu, l1, k);
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();                                     // every warp is done with the rings
    float *cm = reinterpret_cast<float *>(smem);
    float *cl = cm + 16;
    if (g == 0 && c < 2) {
      cm[tw * 4 + r0] = m0;
      cm[tw * 4 + r1] = m1;
      cl[tw * 4 + r0] = l0;
      cl[tw * 4 + r1] = l1;
    }
  } else {
    // =============================== V warps: O^T += V^T . P'^T per block, P' = p * s_v
    float O[NB][2][4];
    float Dw[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k) O[b][h][k] = 0.0f;
    // byte (g & 3) of two tokens' high words into bytes 0 and 2; halfword (g & 1) of two
    // tokens' low-plane words into one word
    const uint32_t sel_v = (uint32_t)(g & 3) | ((uint32_t)(4 + (g & 3)) << 8);
    const uint32_t sel_h = (g & 1) ? 0x7632u : 0x5410u;
    const int gb = min(g, NB - 1);

    for (int i = 0; i <= n_stages; ++i) {
      cp_async_wait<1>();
      __syncthreads();
      issue(i + 2);
      const int j = i - 1;                               // the stage these warps consume
      const int tr = 16 * tw;
      const int ts = t0 + j * kStage + tr;
      if (j < 0 || ts >= t_end) continue;
      const uint8_t *xs = xch + ((tw * 2 + (j & 1)) * 32 + lane) * 32;
      const uint4 pb = *reinterpret_cast<const uint4 *>(xs);
      const float2 cr = *reinterpret_cast<const float2 *>(xs + 16);
      if (__any_sync(0xffffffffu, cr.x != 1.0f || cr.y != 1.0f)) {
        Dw[0] *= cr.x;
        Dw[1] *= cr.y;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            O[b][h][0] *= cr.x;
            O[b][h][1] *= cr.y;
            O[b][h][2] *= cr.x;
            O[b][h][3] *= cr.y;
          }
      }
      const uint8_t *sb = smem + G::OFF_V + (j % kRing) * G::SLOT;
      // V rows of tokens 2c, 2c+1, 2c+8, 2c+9 and their scale rows
      const uint8_t *va = sb + (tr + 2 * c) * G::PITCH, *vb = va + G::PITCH;
      const uint8_t *vc = va + 8 * G::PITCH, *vd = va + 9 * G::PITCH;
      const uint8_t *sa = sb + G::OFF_SC + (tr + 2 * c) * G::SB;
      uint32_t s2c[NB / 2], s2c1[NB / 2], s2c8[NB / 2], s2c9[NB / 2];
      if constexpr (NB == 8) {
        const uint4 x0 = *reinterpret_cast<const uint4 *>(sa), x1 = *reinterpret_cast<const uint4 *>(sa + G::SB);
        const uint4 x8 = *reinterpret_cast<const uint4 *>(sa + 8 * G::SB), x9 = *reinterpret_cast<const uint4 *>(sa + 9 * G::SB);
        s2c[0] = x0.x; s2c[1] = x0.y; s2c[2] = x0.z; s2c[3] = x0.w;
        s2c1[0] = x1.x; s2c1[1] = x1.y; s2c1[2] = x1.z; s2c1[3] = x1.w;
        s2c8[0] = x8.x; s2c8[1] = x8.y; s2c8[2] = x8.z; s2c8[3] = x8.w;
        s2c9[0] = x9.x; s2c9[1] = x9.y; s2c9[2] = x9.z; s2c9[3] = x9.w;
      } else {
        const uint2 x0 = *reinterpret_cast<const uint2 *>(sa), x1 = *reinterpret_cast<const uint2 *>(sa + G::SB);
        const uint2 x8 = *reinterpret_cast<const uint2 *>(sa + 8 * G::SB), x9 = *reinterpret_cast<const uint2 *>(sa + 9 * G::SB);
        s2c[0] = x0.x; s2c[1] = x0.y; s2c1[0] = x1.x; s2c1[1] = x1.y;
        s2c8[0] = x8.x; s2c8[1] = x8.y; s2c9[0] = x9.x; s2c9[1] = x9.y;
      }
      // W term: rows g < NB of its A operand hold block g's V scales
      {
        const uint32_t wa = *reinterpret_cast<const uint16_t *>(sa + 2 * gb);
        const uint32_t wb = *reinterpret_cast<const uint16_t *>(sa + G::SB + 2 * gb);
        const uint32_t wc = *reinterpret_cast<const uint16_t *>(sa + 8 * G::SB + 2 * gb);
        const uint32_t wd = *reinterpret_cast<const uint16_t *>(sa + 9 * G::SB + 2 * gb);
        const uint32_t Aw[4] = {g < NB ? (wa | (wb << 16)) : 0u, 0u, g < NB ? (wc | (wd << 16)) : 0u, 0u};
        mma16816(Dw, Aw, pb.x, pb.y);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int lo = 24 * b + 4 * (g >> 1), hi = 24 * b + 16 + 4 * (g >> 2);
        const uint32_t wa = prmt(lds32(va + lo), lds32(vb + lo), sel_h);
        const uint32_t wb = prmt(lds32(vc + lo), lds32(vd + lo), sel_h);
        const uint32_t Ha = prmt(lds32(va + hi), lds32(vb + hi), sel_v);
        const uint32_t Hb = prmt(lds32(vc + hi), lds32(vd + hi), sel_v);
        uint32_t ua[4], ub[4];
        unpack6(wa, Ha, ua);
        unpack6(wb, Hb, ub);
        const uint32_t sel = (b & 1) ? 0x7632u : 0x5410u;
        const uint32_t sp0 = prmt(s2c[b >> 1], s2c1[b >> 1], sel), sp1 = prmt(s2c8[b >> 1], s2c9[b >> 1], sel);
        // hi columns: rn(p_hi s); lo columns: rn(p_lo s + (p_hi s - rn(p_hi s))), the error term
        // exact by the f16 fma
        const uint32_t th0 = hmul2(pb.z, sp0), th1 = hmul2(pb.w, sp1);
        const uint32_t x0 = hfma2(pb.z, sp0, th0 ^ 0x80008000u), x1 = hfma2(pb.w, sp1, th1 ^ 0x80008000u);
        const uint32_t B0 = hfma2(pb.x, sp0, x0), B1 = hfma2(pb.y, sp1, x1);
        const uint32_t A0[4] = {ua[0], ua[1], ub[0], ub[1]};   // dims 4g (row g), 4g+1 (row g+8)
        const uint32_t A1[4] = {ua[2], ua[3], ub[2], ub[3]};   // dims 4g+2, 4g+3
        mma16816(O[b][0], A0, B0, B1);
        mma16816(O[b][1], A1, B0, B1);
      }
    }
    // hi + lo columns of O and W
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k) O[b][h][k] += __shfl_xor_sync(0xffffffffu, O[b][h][k], 2);
    Dw[0] += __shfl_xor_sync(0xffffffffu, Dw[0], 2);
    Dw[1] += __shfl_xor_sync(0xffffffffu, Dw[1], 2);
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();                                     // every warp is done with the rings
    float *co = reinterpret_cast<float *>(smem) + 32;     // [tile][4][D] after cm/cl
    // value = u * s_v - 32 s_v: even dims entered as u * 2^-24, odd dims as 16 u * 2^-24
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float w0 = 32.0f * __shfl_sync(0xffffffffu, Dw[0], 4 * b + c);
      const float w1 = 32.0f * __shfl_sync(0xffffffffu, Dw[1], 4 * b + c);
      if (c < 2) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int d = 32 * b + 4 * g + 2 * h;
          *reinterpret_cast<float2 *>(co + (tw * 4 + r0) * D + d) =
              make_float2(fmaf(O[b][h][0], 16777216.0f, -w0), fmaf(O[b][h][2], 1048576.0f, -w0));
          *reinterpret_cast<float2 *>(co + (tw * 4 + r1) * D + d) =
              make_float2(fmaf(O[b][h][1], 16777216.0f, -w1), fmaf(O[b][h][3], 1048576.0f, -w1));
        }
      }
    }
  }
  __syncthreads();
  // ---------------- combine the four tiles: cm/cl [tile][4], co [tile][4][D]
  const float *cm = reinterpret_cast<const float *>(smem);
  const float *cl = cm + 16;
  const float *co = cm + 32;
  for (int r = 0; r < R; ++r) {
    if (!((row_vis >> r) & 1u)) continue;                // row does not see this chunk
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * 4 + r]);
    float wt[4], L = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      wt[w] = cm[w * 4 + r] == -INFINITY ? 0.0f : ex2(cm[w * 4 + r] - M);
      L = fmaf(cl[w * 4 + r], wt[w], L);
    }
    const int hq = kvh * a.gqa + (rbase + r) / a.n_q, qi = (rbase + r) % a.n_q;
    const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
    for (int d = threadIdx.x; d < D; d += kThreads) {
      float acc = 0.0f;
#pragma unroll
      for (int w = 0; w < 4; ++w) acc = fmaf(co[(w * 4 + r) * D + d], wt[w], acc);
      a.part_o[pi * D + d] = acc;
    }
    if (threadIdx.x == 0) {
      a.part_m[pi] = M * kLn2;                           // natural-log units, like the other kernels
      a.part_l[pi] = L;
    }
  }
}

template <int D, bool PAGED>
cudaError_t launch_t(const AttendArgs &a, cudaStream_t st) {
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = set_smem_once(configured, attend_mma_q6_kernel<D, PAGED>, Geom<D>::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks, a.cache.B * a.cache.H, (a.gqa * a.n_q + 3) / 4);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Geom<D>::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_mma_q6_kernel<D, PAGED>, a);
}

}  // namespace

bool mma_q6_supported(const AttendArgs &a) {
  return a.cache.layout == KVQ_Q6_0 && mma_q6_shape(a.cache.D, a.gqa * a.n_q) && a.n_body > 0 &&
         a.chunk % kStage == 0;
}

cudaError_t launch_attend_mma_q6(const AttendArgs &a, cudaStream_t st) {
  if (a.cache.page_shift >= 0) return a.cache.D == 256 ? launch_t<256, true>(a, st) : launch_t<128, true>(a, st);
  return a.cache.D == 256 ? launch_t<256, false>(a, st) : launch_t<128, false>(a, st);
}

}  // namespace kvq
