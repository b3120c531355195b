// Tensor-core phase 1 of the split-K decode attention for the block layouts with 4- and 8-bit
// codes (Q4_0, Q8_0, Q4_0 keys with Q8_0 values) and the per-token Hadamard int4 and int2
// bodies, head_dim 128, up to 8 query rows per kv head (the GQA group times the query rows of the
// call). For the Hadamard layouts the exact-f32 recent window is scored in phase 2.
//
// Why tensor cores: every kv head is shared by gqa query heads, so per packed K/V element the
// step does 4*gqa flops (QK and PV); at gqa 8 that is ~57 flops per packed byte, beyond what
// the CUDA cores sustain at HBM rate. The group is a dense contraction, done with
// mma.sync.m16n8k16 (f16 in, f32 accumulate):
//   QK:  S^T[16 tokens][8 rows] += K[16 tokens][16 dims] . Q^T[16 dims][8 rows]
//   PV:  O^T[16 dims][8 rows]   += V^T[16 dims][16 tokens] . P'^T[16 tokens][8 rows]
// Exactness: 4- and 8-bit codes are exact in f16; queries given in bf16/f16 are exact in f16
// after a per-row power-of-two prescale (f32 queries are split into hi + lo f16 parts); the block
// scale of K (per token and 32-dim block) multiplies each block's f32 partial sum; the block
// scale of V is folded into the probabilities, P' = p * s_v, kept as hi + lo f16 parts (p is
// split once per tile, and each block's scale is applied with an exact f16 TwoProduct).
//
// Data movement: each warp pulls its chunk HBM -> shared memory in 32-token stages with
// 16-byte cp.async (two stages in flight per warp; measured on GB300, 64-token stages or deeper
// rings, i.e. more bytes in flight, were slower at the same occupancy). Payload rows (64 bytes
// for 4-bit codes, 128 for 8-bit) are placed with an XOR swizzle of their 16-byte columns so that
// the ldmatrix reads (8 rows x 16 bytes per phase) are bank-conflict free. ldmatrix gives each
// lane the code words of its fragment: plain for K (one token, 8 consecutive dims of 4-bit codes
// or 4 of 8-bit codes), transposed for V (two tokens, 4 consecutive dims of 4-bit codes or 2 of
// 8-bit codes). K codes become exact subnormal f16 values u * 2^-24 of the offset code u (one
// lop3 per nibble pair; one byte permute per 8-bit pair), the offset going into the
// accumulator's initial value; V codes become exact signed f16 values (the code under the
// exponent of 1024, one f16 add), so that the long PV accumulation carries no offset mass.
//
// Hadamard int2 (32-byte rows, value f of a byte at bits 2f): one ldmatrix gives a lane 16
// consecutive dims of a token per word; two byte permutes split a word into two f16 lanes and one
// lop3 per pair keeps the fields k of both lanes in place with their sign bit flipped, i.e. the
// subnormal u * 4^k * 2^-24 of u = code + 2 (K: the query entries facing field k are divided by
// 4^k and -2 * sum(q) is the accumulator's initial value). V codes become exact signed f16 values
// (a shift, the lop3 under the exponent of 1024, one f16 add per pair).
//
// Each CTA handles one chunk of one (batch, kv head); each of its four warps streams a contiguous
// quarter of the chunk through a private two-stage shared-memory ring and keeps its online
// softmax state in registers. At the end the warps combine their states in shared memory and
// the CTA writes one (m, l, o) partial per query row.
#include <cfloat>
#include <climits>

#include "kvq_internal.cuh"
#include "mma_util.cuh"

namespace kvq {
namespace {
using namespace mma;

constexpr int kWarps = 4;
#ifndef KVQ_MMA_STAGE
#define KVQ_MMA_STAGE 32
#endif
constexpr int kStage = KVQ_MMA_STAGE;   // tokens per pipeline stage (16-token tiles)
#ifndef KVQ_MMA_RING
#define KVQ_MMA_RING 2
#endif
constexpr int kRing = KVQ_MMA_RING;     // stages per warp in flight
static_assert(kStage % 16 == 0 && 64 % kStage == 0, "a stage is whole tiles and never straddles a 64-token page");
static_assert(kRing >= 2, "at least one stage loads while another is read");
constexpr int kTiles = kStage / 16;
constexpr int kMinBlocks = KVQ_MMA_MIN_BLOCKS; // resident CTAs per SM
constexpr int kD = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Stage buffer: K payload, V payload (swizzled rows of 64 bytes for 4-bit codes, 128 bytes for
// Q8_0, 32 bytes for Hadamard int2), K and V scales (4 f16 per token, or one f32 per token for the
// Hadamard layouts).
template <int L>
__host__ __device__ constexpr int plane_row_bytes() { return L == KVQ_Q8_0 ? 128 : (L == KVQ_HAD_INT2 ? 32 : 64); }
template <int L>
__host__ __device__ constexpr int scale_bytes() { return is_hadamard(L) ? 4 : 8; }
template <int L, int VL>
__host__ __device__ constexpr int off_v() { return kStage * plane_row_bytes<L>(); }
template <int L, int VL>
__host__ __device__ constexpr int off_sk() { return off_v<L, VL>() + kStage * plane_row_bytes<VL>(); }
template <int L, int VL>
__host__ __device__ constexpr int off_sv() { return off_sk<L, VL>() + kStage * scale_bytes<L>(); }
template <int L, int VL>
__host__ __device__ constexpr int stage_bytes() { return off_sv<L, VL>() + kStage * scale_bytes<VL>(); }
// Hadamard: per-warp scratch for the int8 query codes of up to 8 rows and their scales
constexpr int kQScratch = 8 * 128 + 8 * 4;
template <int L, int VL>
__host__ __device__ constexpr int smem_bytes() {
  return kWarps * kRing * stage_bytes<L, VL>() + (is_hadamard(L) ? kWarps * kQScratch : 0);
}
// the warps' final (m, l, o) states reuse the stage buffers
static_assert(kWarps * 8 * (2 + kD) * 4 <= kWarps * kRing * stage_bytes<KVQ_HAD_INT2, KVQ_HAD_INT2>(),
              "combine buffer fits");
static_assert(smem_bytes<KVQ_Q8_0, KVQ_Q8_0>() * kMinBlocks <= 227 * 1024, "Q8_0 stages fit the resident CTAs");

// Last token query row r (of the gqa * n_q rows of a kv head) may see; negative if none.
__device__ __forceinline__ int row_limit_of(const AttendArgs &a, const SeqLen &sl, int r) {
  return row_limit(a, sl, r % a.n_q);
}

// Byte offset of (row, 16-byte column j) inside a swizzled slab of RB-byte rows: the column is
// XORed with bits of the row so that the 8 rows an ldmatrix phase reads at one column fall in
// different banks (32-byte rows: (row / 4) % 2; 64-byte rows: (row / 2) % 4; 128-byte rows: row % 8).
template <int RB>
__device__ __forceinline__ uint32_t swz(int row, int j) {
  return (uint32_t)(row * RB + ((j ^ (RB == 32 ? (row >> 2) & 1 : RB == 64 ? (row >> 1) & 3 : row & 7)) << 4));
}

// 8-bit K word (dims 4c..4c+3 of one token, two's complement codes) -> two f16 pairs holding the
// exact subnormals u * 2^-24 of u = code + 128: dims (4c, 4c+1) and (4c+2, 4c+3).
__device__ __forceinline__ void unpack4_s8_sub(uint32_t w, uint32_t &p01, uint32_t &p23) {
  const uint32_t x = w ^ 0x80808080u;
  p01 = __byte_perm(x, 0u, 0x4140);
  p23 = __byte_perm(x, 0u, 0x4342);
}
// Transposed 8-bit V word (bytes: token 2c dims d, d+1, then token 2c+1 dims d, d+1) -> exact
// signed f16 pairs (dim d of both tokens) and (dim d+1 of both tokens): the byte u = code + 128
// goes under the exponent of 1024 and one f16 add removes 1152.
__device__ __forceinline__ void unpack4_s8_t(uint32_t w, uint32_t &d0, uint32_t &d1) {
  const uint32_t x = w ^ 0x80808080u;
  d0 = hadd2(__byte_perm(x, 0x64646464u, 0x4240), 0xE480E480u);
  d1 = hadd2(__byte_perm(x, 0x64646464u, 0x4341), 0xE480E480u);
}

// CAP: score capture (Hadamard layout, contiguous cache): the exact integer score of every
// (row, body token) this CTA computes and each row's int8 query scale go to a.cap_scores / a.cap_sq.
template <int LAYOUT, int VLAYOUT, bool QSPLIT, bool PAGED, bool CAP = false>
__global__ void __launch_bounds__(kWarps * 32, kMinBlocks) attend_mma_kernel(AttendArgs a) {
  constexpr bool HAD = is_hadamard(LAYOUT), HAD2 = LAYOUT == KVQ_HAD_INT2;
  static_assert(LAYOUT != KVQ_ASYM4_G32 && VLAYOUT != KVQ_ASYM4_G32, "the asymmetric layout has its own kernel");
  constexpr bool K8 = LAYOUT == KVQ_Q8_0, V8 = VLAYOUT == KVQ_Q8_0;   // 8-bit code planes
  constexpr int KRB = plane_row_bytes<LAYOUT>(), VRB = plane_row_bytes<VLAYOUT>();
  constexpr int SCB = scale_bytes<LAYOUT>(), OFF_V = off_v<LAYOUT, VLAYOUT>(), OFF_SK = off_sk<LAYOUT, VLAYOUT>();
  constexpr int OFF_SV = off_sv<LAYOUT, VLAYOUT>(), STAGE_BYTES = stage_bytes<LAYOUT, VLAYOUT>();
  static_assert(VLAYOUT == LAYOUT || (LAYOUT == KVQ_Q4_0 && VLAYOUT == KVQ_Q8_0), "supported plane pairs");
  static_assert(!CAP || (HAD && !PAGED), "score capture: Hadamard layout, contiguous cache");
  extern __shared__ __align__(1024) uint8_t smem[];
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  const CacheView &cv = a.cache;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  // One chunk per CTA; warp w takes a contiguous quarter of the chunk's stages.
  const int chunk_id = blockIdx.x;
  const int bh = blockIdx.y;
  const int bb = bh / cv.H, kvh = bh - bb * cv.H;
  const SeqLen sl = seq_of_t<PAGED>(a, bb);             // this sequence's lengths
  const int R = a.gqa * a.n_q;

  const int t0 = chunk_id * sl.chunk;
  const int t1 = min(sl.n_body, t0 + sl.chunk);
  int w_lim = -1, min_lim = INT_MAX;
  for (int r = 0; r < R; ++r) {
    const int l = row_limit_of(a, sl, r);
    w_lim = max(w_lim, l);
    min_lim = min(min_lim, l);
  }
  // rows appended by the preceding kernel: only the CTAs that read them wait for it
  pdl_wait_if(t0 <= w_lim && t0 < sl.fresh_hi && sl.fresh_lo < min(t1, w_lim + 1));
  if (t0 > w_lim || t0 >= t1) return;                 // no row sees this chunk (phase 2 skips it)
  const int t_end = min(t1, w_lim + 1);
  const int n_stages = (t_end - t0 + kStage - 1) / kStage;
  const int spw = (n_stages + kWarps - 1) / kWarps;      // stages per warp
  const int s_first = min(n_stages, warp * spw);
  const int n_mine = min(n_stages, s_first + spw) - s_first;
  const int tw0 = t0 + s_first * kStage;                 // this warp's first token

  // ---- per-warp stage pipeline
  uint8_t *wbuf = smem + warp * kRing * STAGE_BYTES;
  // contiguous cache: the planes' rows of token 0 of this (batch, kv head)
  const size_t head_row0 = (size_t)bh * cv.cap;
  const uint8_t *kp0 = cv.payload[0] + head_row0 * KRB, *vp0 = cv.payload[1] + head_row0 * VRB;
  const uint8_t *ksc0 = static_cast<const uint8_t *>(cv.scale[0]) + head_row0 * SCB;
  const uint8_t *vsc0 = static_cast<const uint8_t *>(cv.scale[1]) + head_row0 * SCB;

  auto issue = [&](int i) {
    if (i < n_mine) {
      const int ts = tw0 + i * kStage;
      // the stage's rows are consecutive plane rows (a page holds at least 64 aligned tokens)
      size_t r0 = (size_t)ts;                             // row offset from the base pointers
      const uint8_t *kb = kp0, *vb = vp0, *ksb = ksc0, *vsb = vsc0;
      if constexpr (PAGED) {
        r0 = cache_row_paged(cv, bb, kvh, ts);
        kb = cv.payload[0]; vb = cv.payload[1];
        ksb = static_cast<const uint8_t *>(cv.scale[0]); vsb = static_cast<const uint8_t *>(cv.scale[1]);
      }
      const uint8_t *kp = kb + r0 * KRB, *vp = vb + r0 * VRB;
      const uint8_t *ksc = ksb + r0 * SCB, *vsc = vsb + r0 * SCB;
      uint8_t *sb = wbuf + (i % kRing) * STAGE_BYTES;
      const uint32_t sK = smem_addr(sb), sV = smem_addr(sb + OFF_V);
      if (ts + kStage <= t_end) {                        // full stage: no per-row bounds
        if constexpr (KRB == VRB) {
          constexpr int CPR = KRB / 16;                  // 16-byte pieces per row
#pragma unroll
          for (int k = 0; k < kStage * CPR / 32; ++k) {
            const int q = lane + 32 * k;                 // 16-byte piece: row q / CPR, column q % CPR
            const int row = q / CPR, j = q % CPR;
            cp_async16(sK + swz<KRB>(row, j), kp + 16 * q, 16);
            cp_async16(sV + swz<VRB>(row, j), vp + 16 * q, 16);
          }
        } else {
#pragma unroll
          for (int k = 0; k < kStage * (KRB / 16) / 32; ++k) {
            const int q = lane + 32 * k;
            cp_async16(sK + swz<KRB>(q / (KRB / 16), q % (KRB / 16)), kp + 16 * q, 16);
          }
#pragma unroll
          for (int k = 0; k < kStage * (VRB / 16) / 32; ++k) {
            const int q = lane + 32 * k;
            cp_async16(sV + swz<VRB>(q / (VRB / 16), q % (VRB / 16)), vp + 16 * q, 16);
          }
        }
#pragma unroll
        for (int k = 0; k < (kStage + 31) / 32; ++k) {
          const int row = lane + 32 * k;
          if (kStage % 32 && row >= kStage) break;
          const size_t tok = (size_t)row;
          cp_async_scale<SCB>(smem_addr(sb + OFF_SK + row * SCB), ksc + tok * SCB, SCB);
          cp_async_scale<SCB>(smem_addr(sb + OFF_SV + row * SCB), vsc + tok * SCB, SCB);
        }
      } else {                                           // tail stage: rows past t_end are zero-filled
        if constexpr (KRB == VRB) {
          constexpr int CPR = KRB / 16;
#pragma unroll
          for (int k = 0; k < kStage * CPR / 32; ++k) {
            const int q = lane + 32 * k;
            const int row = q / CPR, j = q % CPR;
            const bool ok = ts + row < t_end;
            const size_t off = (size_t)(ok ? row : 0) * KRB + 16 * j;
            cp_async16(sK + swz<KRB>(row, j), kp + off, ok ? 16 : 0);
            cp_async16(sV + swz<VRB>(row, j), vp + off, ok ? 16 : 0);
          }
        } else {
#pragma unroll
          for (int k = 0; k < kStage * (KRB / 16) / 32; ++k) {
            const int q = lane + 32 * k;
            const int row = q / (KRB / 16), j = q % (KRB / 16);
            const bool ok = ts + row < t_end;
            cp_async16(sK + swz<KRB>(row, j), kp + (size_t)(ok ? row : 0) * KRB + 16 * j, ok ? 16 : 0);
          }
#pragma unroll
          for (int k = 0; k < kStage * (VRB / 16) / 32; ++k) {
            const int q = lane + 32 * k;
            const int row = q / (VRB / 16), j = q % (VRB / 16);
            const bool ok = ts + row < t_end;
            cp_async16(sV + swz<VRB>(row, j), vp + (size_t)(ok ? row : 0) * VRB + 16 * j, ok ? 16 : 0);
          }
        }
#pragma unroll
        for (int k = 0; k < (kStage + 31) / 32; ++k) {
          const int row = lane + 32 * k;
          if (kStage % 32 && row >= kStage) break;
          const bool ok = ts + row < t_end;
          const size_t tok = (size_t)(ok ? row : 0);
          cp_async_scale<SCB>(smem_addr(sb + OFF_SK + row * SCB), ksc + tok * SCB, ok ? SCB : 0);
          cp_async_scale<SCB>(smem_addr(sb + OFF_SV + row * SCB), vsc + tok * SCB, ok ? SCB : 0);
        }
      }
    }
    cp_async_commit();                                   // always one group per call
  };
  // start streaming the first stages before the query prologue so their latency overlaps it
#pragma unroll
  for (int i = 0; i < kRing; ++i) issue(i);

  // ---- query fragments (B operand of QK): row g of the group, dims 32b + 8c + 0..7
  uint32_t bq_hi[8][2], bq_lo[QSPLIT ? 8 : 1][2];
  float qsum[4];                                        // per-block sum of the prescaled q (row g)
  float row_alpha;                                      // alpha * 2^e * 2^24 * log2(e) for row g
  if (HAD) {
    // Query preparation in the prologue: each warp rotates and quantises the R <= 8 query rows of
    // the group (warp FWHT, int8 codes, one f32 scale per row), parks the codes in its shared
    // scratch and reads them back in fragment order. The int8 codes are exact in f16; the row's
    // s_q goes into its alpha and -8 * sum(q8) into the accumulator start value.
    uint8_t *qs8 = smem + kWarps * kRing * STAGE_BYTES + warp * kQScratch;
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
      if (CAP && lane == 0 && warp == 0 && chunk_id == 0) a.cap_sq[grow] = sq;
    }
    __syncwarp();
    const bool live = g < R;
    row_alpha = (live ? a.scale * qsq[g] : 0.0f) * 16777216.0f * kLog2e;
    float qs = 0.0f;
    if constexpr (HAD2) {
      // 2-bit key codes: k-step 4 ch + k pairs dims (16c + k, 16c + 8 + k) and (16c + 4 + k,
      // 16c + 12 + k) of the column block ch (dims 64 ch ..), whose fields sit at bits 2k of their
      // bytes: the code operands are u * 4^k * 2^-24, so these query entries are divided by 4^k
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        float h[16];
        const uint4 w16 = live ? *reinterpret_cast<const uint4 *>(qs8 + g * 128 + 64 * ch + 16 * c) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t wv[4] = {w16.x, w16.y, w16.z, w16.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          h[i] = (float)(int8_t)((wv[i >> 2] >> (8 * (i & 3))) & 0xFFu);
          qs += h[i];
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float f = 1.0f / (float)(1 << (2 * k));
          bq_hi[4 * ch + k][0] = pack_f16x2(h[k] * f, h[8 + k] * f);
          bq_hi[4 * ch + k][1] = pack_f16x2(h[4 + k] * f, h[12 + k] * f);
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) qsum[b] = 0.0f;
    } else {
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
    }
    qs += __shfl_xor_sync(0xffffffffu, qs, 1);
    qs += __shfl_xor_sync(0xffffffffu, qs, 2);
    qsum[0] = qs;                                        // whole-row sum (one accumulator per token)
  } else {
    float x[4][8];
    const bool live = g < R;
    const int hq = kvh * a.gqa + (live ? g / a.n_q : 0);
    const int qi = live ? g % a.n_q : 0;
    const size_t grow = ((size_t)bb * a.Hq + hq) * a.n_q + qi;
    float mx = 0.0f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      if (live && K8) {                                  // dims 32b + 4c + 0..3 and 32b + 16 + 4c + 0..3
        load4_f32(a.q, a.q_dtype, grow * kD + 32 * b + 4 * c, x[b]);
        load4_f32(a.q, a.q_dtype, grow * kD + 32 * b + 16 + 4 * c, x[b] + 4);
      } else if (live) {                                 // dims 32b + 8c + 0..7
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
    // power-of-two prescale so that the row's largest |q| lands in [2^13, 2^14): exact, and
    // safe from f16 overflow; the inverse scale goes into the row's alpha.
    int e = 0;
    if (mx > 0.0f) e = min(max(((__float_as_int(mx) >> 23) & 0xFF) - 127 - 13, -100), 100);
    const float pre = ldexpf(1.0f, -e), post = ldexpf(1.0f, e);
    row_alpha = a.scale * post * 16777216.0f * kLog2e;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float s = 0.0f;
      float h[8], l[8];
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
        if (K8) {
          // 8-bit codes: k-step st covers dims 32b + 16 st + 4c + 0..3, in pairs (0, 1) and (2, 3)
          bq_hi[2 * b + st][0] = pack_f16x2(h[4 * st], h[4 * st + 1]);
          bq_hi[2 * b + st][1] = pack_f16x2(h[4 * st + 2], h[4 * st + 3]);
          if (QSPLIT) {
            bq_lo[2 * b + st][0] = pack_f16x2(l[4 * st], l[4 * st + 1]);
            bq_lo[2 * b + st][1] = pack_f16x2(l[4 * st + 2], l[4 * st + 3]);
          }
          continue;
        }
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
  // the thread's two S^T columns are query rows 2c and 2c+1
  const int r0 = 2 * c, r1 = 2 * c + 1;
  const float alpha0 = __shfl_sync(0xffffffffu, row_alpha, r0 * 4);
  const float alpha1 = __shfl_sync(0xffffffffu, row_alpha, r1 * 4);
  // zq: per-block row sums of q in accumulator units (x 2^-24) times minus the code offset
  // (Q4_0 / Hadamard int4: 8, Q8_0: 128, Hadamard int2: 2), the accumulator's initial value (the
  // K codes enter as code + offset).
  float zq0[4], zq1[4];
  {
    constexpr float kOff = K8 ? -128.0f : (HAD2 ? -2.0f : -8.0f);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      zq0[b] = __shfl_sync(0xffffffffu, qsum[b], r0 * 4) * (5.9604644775390625e-8f * kOff);
      zq1[b] = __shfl_sync(0xffffffffu, qsum[b], r1 * 4) * (5.9604644775390625e-8f * kOff);
    }
  }
  const int lim0 = r0 < R ? row_limit_of(a, sl, r0) : -1;
  const int lim1 = r1 < R ? row_limit_of(a, sl, r1) : -1;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  float O[4][2][4];                                      // [block][half][c0..c3]
#pragma unroll
  for (int b = 0; b < 4; ++b) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int k = 0; k < 4; ++k) O[b][h][k] = 0.0f;
  }

  for (int i = 0; i < n_mine; ++i) {
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint8_t *sb = wbuf + (i % kRing) * STAGE_BYTES;
    const uint32_t sK = smem_addr(sb), sV = smem_addr(sb + OFF_V);
    const int ts = tw0 + i * kStage;

    // ---------------- scores S^T for the 4 tiles of the stage
    float s[kTiles][4];
#pragma unroll
    for (int tile = 0; tile < kTiles; ++tile) {
      uint32_t kw[2][4];
      if constexpr (!K8) {
#pragma unroll
        for (int half = 0; half < (HAD2 ? 1 : 2); ++half) {
          const int mi = lane >> 3;
          const int row = tile * 16 + (mi & 1) * 8 + (lane & 7);
          ldsm_x4(sK + swz<KRB>(row, 2 * half + (mi >> 1)), kw[half]);
        }
      }
      if (HAD) {
        // one per-token scale: all 8 k-steps accumulate the exact integer dot (x 2^-24) in two
        // chains; score = alpha * s_q * s_k * dot
        float dA[4], dB[4];                              // the first mma of each chain takes its C operand
        if constexpr (HAD2) {
          // kw[0][2 ch] = token g, dims 64 ch + 16c .. +15 (field f at bits 2f); [2 ch + 1] = token
          // g + 8. Bytes (0, 2) and (1, 3) go to the two f16 lanes; per k one lop3 keeps fields
          // (k, 8 + k) or (4 + k, 12 + k) at bits 2k and flips their sign bit: u = code + 2 as the
          // subnormal u * 4^k * 2^-24 (the query entries carry the 4^-k)
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const uint32_t wg = kw[0][2 * ch], w8 = kw[0][2 * ch + 1];
            const uint32_t gA = prmt(wg, 0u, 0x4240u), gB = prmt(wg, 0u, 0x4341u);
            const uint32_t eA = prmt(w8, 0u, 0x4240u), eB = prmt(w8, 0u, 0x4341u);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t m = 0x00030003u << (2 * k), x = 0x00020002u << (2 * k);
              const uint32_t A[4] = {lop3<0x6a>(gA, m, x), lop3<0x6a>(eA, m, x), lop3<0x6a>(gB, m, x),
                                     lop3<0x6a>(eB, m, x)};
              const int ks = 4 * ch + k;
              float(&d)[4] = (ks & 1) ? dB : dA;
              if (ks == 0)
                mma16816_c(d, A, bq_hi[0][0], bq_hi[0][1], zq0[0], zq1[0], zq0[0], zq1[0]);
              else if (ks == 1)
                mma16816_c(d, A, bq_hi[1][0], bq_hi[1][1], 0.0f, 0.0f, 0.0f, 0.0f);
              else
                mma16816(d, A, bq_hi[ks][0], bq_hi[ks][1]);
            }
          }
        } else {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t ug[4], u8[4];
          unpack8_sub<false>(kw[b >> 1][(b & 1) * 2 + 0], ug);
          unpack8_sub<false>(kw[b >> 1][(b & 1) * 2 + 1], u8);
          const uint32_t A0[4] = {ug[0], u8[0], ug[1], u8[1]};
          const uint32_t A1[4] = {ug[2], u8[2], ug[3], u8[3]};
          float(&d)[4] = (b & 1) ? dB : dA;
          if (b == 0)
            mma16816_c(d, A0, bq_hi[0][0], bq_hi[0][1], zq0[0], zq1[0], zq0[0], zq1[0]);
          else if (b == 1)
            mma16816_c(d, A0, bq_hi[2][0], bq_hi[2][1], 0.0f, 0.0f, 0.0f, 0.0f);
          else
            mma16816(d, A0, bq_hi[2 * b][0], bq_hi[2 * b][1]);
          mma16816(d, A1, bq_hi[2 * b + 1][0], bq_hi[2 * b + 1][1]);
        }
        }
        if constexpr (CAP) {
          // the two chains hold the exact dot x 2^-24 (|dot| < 2^18): (dA + dB) x 2^24 is the integer
          const int ta = ts + tile * 16 + g, tb = ta + 8;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int r = (k & 1) ? r1 : r0, t = (k & 2) ? tb : ta;
            if (r < R && t < t_end) capture_score(a, bb, kvh, r, t, __float2int_rn((dA[k] + dB[k]) * 16777216.0f));
          }
        }
        const float skg = *reinterpret_cast<const float *>(sb + OFF_SK + (tile * 16 + g) * 4);
        const float skg8 = *reinterpret_cast<const float *>(sb + OFF_SK + (tile * 16 + g + 8) * 4);
        s[tile][0] = (dA[0] + dB[0]) * skg * alpha0;
        s[tile][1] = (dA[1] + dB[1]) * skg * alpha1;
        s[tile][2] = (dA[2] + dB[2]) * skg8 * alpha0;
        s[tile][3] = (dA[3] + dB[3]) * skg8 * alpha1;
        continue;
      }
      const uint2 skg = *reinterpret_cast<const uint2 *>(sb + OFF_SK + (tile * 16 + g) * 8);
      const uint2 skg8 = *reinterpret_cast<const uint2 *>(sb + OFF_SK + (tile * 16 + g + 8) * 8);
      const float2 sg01 = __half22float2(u32_as_h2(skg.x)), sg23 = __half22float2(u32_as_h2(skg.y));
      const float2 s801 = __half22float2(u32_as_h2(skg8.x)), s823 = __half22float2(u32_as_h2(skg8.y));
      const float skg_f[4] = {sg01.x, sg01.y, sg23.x, sg23.y};
      const float skg8_f[4] = {s801.x, s801.y, s823.x, s823.y};
      float acc_s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint32_t A0[4], A1[4];
        if constexpr (K8) {
          // block b = 16-byte columns 2b, 2b+1: kb[0] / kb[1] = tokens g / g+8, dims 32b + 4c..;
          // kb[2] / kb[3] the same tokens, dims 32b + 16 + 4c..
          uint32_t kb[4];
          const int mi = lane >> 3;
          ldsm_x4(sK + swz<KRB>(tile * 16 + (mi & 1) * 8 + (lane & 7), 2 * b + (mi >> 1)), kb);
          unpack4_s8_sub(kb[0], A0[0], A0[2]);
          unpack4_s8_sub(kb[1], A0[1], A0[3]);
          unpack4_s8_sub(kb[2], A1[0], A1[2]);
          unpack4_s8_sub(kb[3], A1[1], A1[3]);
        } else {
          // kw[b/2][(b%2)*2 + 0] = (token g, block b); [.. + 1] = (token g+8, block b)
          uint32_t ug[4], u8[4];
          unpack8_sub<false>(kw[b >> 1][(b & 1) * 2 + 0], ug);
          unpack8_sub<false>(kw[b >> 1][(b & 1) * 2 + 1], u8);
          A0[0] = ug[0]; A0[1] = u8[0]; A0[2] = ug[1]; A0[3] = u8[1];
          A1[0] = ug[2]; A1[1] = u8[2]; A1[2] = ug[3]; A1[3] = u8[3];
        }
        // the first mma takes the offset as its separate C operand: no register copies
        float d[4];
        mma16816_c(d, A0, bq_hi[2 * b][0], bq_hi[2 * b][1], zq0[b], zq1[b], zq0[b], zq1[b]);
        mma16816(d, A1, bq_hi[2 * b + 1][0], bq_hi[2 * b + 1][1]);
        if (QSPLIT) {
          mma16816(d, A0, bq_lo[2 * b][0], bq_lo[2 * b][1]);
          mma16816(d, A1, bq_lo[2 * b + 1][0], bq_lo[2 * b + 1][1]);
        }
        acc_s[0] = fmaf(skg_f[b], d[0], acc_s[0]);
        acc_s[1] = fmaf(skg_f[b], d[1], acc_s[1]);
        acc_s[2] = fmaf(skg8_f[b], d[2], acc_s[2]);
        acc_s[3] = fmaf(skg8_f[b], d[3], acc_s[3]);
      }
      s[tile][0] = acc_s[0] * alpha0;
      s[tile][1] = acc_s[1] * alpha1;
      s[tile][2] = acc_s[2] * alpha0;
      s[tile][3] = acc_s[3] * alpha1;
    }
    // ---------------- mask (only at the chunk tail or a causal boundary)
    if (ts + kStage > t1 || ts + kStage - 1 > min_lim) {
#pragma unroll
      for (int tile = 0; tile < kTiles; ++tile) {
        const int ta = ts + tile * 16 + g, tb = ta + 8;
        if (!(ta < t1 && ta <= lim0)) s[tile][0] = -INFINITY;
        if (!(ta < t1 && ta <= lim1)) s[tile][1] = -INFINITY;
        if (!(tb < t1 && tb <= lim0)) s[tile][2] = -INFINITY;
        if (!(tb < t1 && tb <= lim1)) s[tile][3] = -INFINITY;
      }
    }
    // ---------------- online softmax (base 2), rows r0 / r1
    float mx0 = fmaxf(s[0][0], s[0][2]), mx1 = fmaxf(s[0][1], s[0][3]);
#pragma unroll
    for (int tile = 1; tile < kTiles; ++tile) {
      mx0 = fmaxf(mx0, fmaxf(s[tile][0], s[tile][2]));
      mx1 = fmaxf(mx1, fmaxf(s[tile][1], s[tile][3]));
    }
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
    l0 *= corr0;
    l1 *= corr1;
    // once the running maxima settle, corr is exactly 1 for every row: skip the rescale
    if (__any_sync(0xffffffffu, corr0 != 1.0f || corr1 != 1.0f)) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          O[b][h][0] *= corr0;
          O[b][h][1] *= corr1;
          O[b][h][2] *= corr0;
          O[b][h][3] *= corr1;
        }
      }
    }
#pragma unroll
    for (int tile = 0; tile < kTiles; ++tile) {
      s[tile][0] = ex2(s[tile][0] - mu0);
      s[tile][1] = ex2(s[tile][1] - mu1);
      s[tile][2] = ex2(s[tile][2] - mu0);
      s[tile][3] = ex2(s[tile][3] - mu1);
      l0 += s[tile][0] + s[tile][2];
      l1 += s[tile][1] + s[tile][3];
    }

    // ---------------- O^T += V^T . (P * s_v)^T per 32-dim block
#pragma unroll
    for (int tile = 0; tile < kTiles; ++tile) {
      uint32_t vw[2][4];
      if constexpr (!V8) {
#pragma unroll
        for (int half = 0; half < (HAD2 ? 1 : 2); ++half) {
          const int mi = lane >> 3;
          const int row = tile * 16 + (mi & 1) * 8 + (lane & 7);
          ldsm_x4_t(sV + swz<VRB>(row, 2 * half + (mi >> 1)), vw[half]);
        }
      }
      // p -> exact hi + lo f16 parts, transposed once into the B layout: each f16 pair holds one
      // query row g and two consecutive tokens (2c, 2c+1) or (2c+8, 2c+9)
      uint32_t bh0, bh1, bl0, bl1;
      {
        float p0 = s[tile][0], p1 = s[tile][1], p2 = s[tile][2], p3 = s[tile][3];
        if (HAD) {                                       // per-token V scale: P' = p * s_v before the split
          const float svg = *reinterpret_cast<const float *>(sb + OFF_SV + (tile * 16 + g) * 4);
          const float svg8 = *reinterpret_cast<const float *>(sb + OFF_SV + (tile * 16 + g + 8) * 4);
          p0 *= svg;
          p1 *= svg;
          p2 *= svg8;
          p3 *= svg8;
        }
        const uint32_t h01 = pack_f16x2(p0, p1), h23 = pack_f16x2(p2, p3);
        const float2 f01 = __half22float2(u32_as_h2(h01)), f23 = __half22float2(u32_as_h2(h23));
        const uint32_t l01 = pack_f16x2(p0 - f01.x, p1 - f01.y);
        const uint32_t l23 = pack_f16x2(p2 - f23.x, p3 - f23.y);
        bh0 = movm_t(h01);
        bh1 = movm_t(h23);
        bl0 = movm_t(l01);
        bl1 = movm_t(l23);
      }
      // Hadamard V codes (s_v already in P') enter as exact signed f16 values (lop3 + one f16
      // fix-up per pair), like the Q4_0 and Q8_0 codes. An offset form (u = code + 8 as a
      // subnormal, with -8 sum_t P'_t added at the end) is a little cheaper, but its accumulator
      // holds about 8 sum_t P'_t, and the tensor core's truncated adds of the small P' lo
      // products against it cost about 20x the error of the signed form.
      if (HAD) {
        if constexpr (HAD2) {
          // vw[0][2 ch] = tokens (2c, 2c+1) of 16-bit unit g of column block ch (dims 64 ch + 8g ..
          // +7, field f at bits 2f of each token's half), vw[0][2 ch + 1] = tokens (2c+8, 2c+9).
          // One mma per field pair (f, f + 4): rows g and g + 8 of its A operand are dims
          // 64 ch + 8g + f and + 4 as exact signed f16 codes (the field under the exponent of 1024
          // with its sign bit flipped, then 1026 removed). No offset term: with u = code + 2 as a
          // subnormal, the accumulator would hold about 2 sum(P') and the true sum only after
          // subtracting 2 W, where the tensor core's truncated adds of the small P' lo products
          // would show.
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const uint32_t v0 = vw[0][2 * ch], v1 = vw[0][2 * ch + 1];
#pragma unroll
            for (int f = 0; f < 4; ++f) {
              const uint32_t A[4] = {
                  hadd2(lop3<0x6a>(v0 >> (2 * f), 0x00030003u, 0x64026402u), 0xE402E402u),
                  hadd2(lop3<0x6a>(v0 >> (8 + 2 * f), 0x00030003u, 0x64026402u), 0xE402E402u),
                  hadd2(lop3<0x6a>(v1 >> (2 * f), 0x00030003u, 0x64026402u), 0xE402E402u),
                  hadd2(lop3<0x6a>(v1 >> (8 + 2 * f), 0x00030003u, 0x64026402u), 0xE402E402u)};
              float(&o)[4] = O[(4 * ch + f) >> 1][(4 * ch + f) & 1];
              mma16816(o, A, bh0, bh1);
              mma16816(o, A, bl0, bl1);
            }
          }
        } else {
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t ua[4], ub[4];
            unpack8_q4(vw[b >> 1][(b & 1) * 2 + 0], ua);
            unpack8_q4(vw[b >> 1][(b & 1) * 2 + 1], ub);
            const uint32_t A0[4] = {ua[0], ua[1], ub[0], ub[1]};
            const uint32_t A1[4] = {ua[2], ua[3], ub[2], ub[3]};
            mma16816(O[b][0], A0, bh0, bh1);
            mma16816(O[b][0], A0, bl0, bl1);
            mma16816(O[b][1], A1, bh0, bh1);
            mma16816(O[b][1], A1, bl0, bl1);
          }
        }
        continue;
      }
      // V block scales paired the same way: (s_v[2c][b], s_v[2c+1][b]), (s_v[2c+8][b], s_v[2c+9][b])
      const uint8_t *svb = sb + OFF_SV + tile * 16 * 8;
      const uint2 sa = *reinterpret_cast<const uint2 *>(svb + (2 * c) * 8);
      const uint2 sbv = *reinterpret_cast<const uint2 *>(svb + (2 * c + 1) * 8);
      const uint2 sc = *reinterpret_cast<const uint2 *>(svb + (2 * c + 8) * 8);
      const uint2 sd = *reinterpret_cast<const uint2 *>(svb + (2 * c + 9) * 8);
      const uint32_t sp0[4] = {__byte_perm(sa.x, sbv.x, 0x5410), __byte_perm(sa.x, sbv.x, 0x7632),
                               __byte_perm(sa.y, sbv.y, 0x5410), __byte_perm(sa.y, sbv.y, 0x7632)};
      const uint32_t sp1[4] = {__byte_perm(sc.x, sd.x, 0x5410), __byte_perm(sc.x, sd.x, 0x7632),
                               __byte_perm(sc.y, sd.y, 0x5410), __byte_perm(sc.y, sd.y, 0x7632)};
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // P' = (p_hi + p_lo) * s_v split into hi + lo f16 exactly enough (TwoProduct with f16 fma):
        //   hi = rn(p_hi * s),  r = p_hi * s - hi (exact),  lo = rn(p_lo * s + r)
        const uint32_t hi0 = hmul2(bh0, sp0[b]), hi1 = hmul2(bh1, sp1[b]);
        const uint32_t r0 = hfma2_negc(bh0, sp0[b], hi0), r1 = hfma2_negc(bh1, sp1[b], hi1);
        const uint32_t lo0 = hfma2(bl0, sp0[b], r0), lo1 = hfma2(bl1, sp1[b], r1);
        uint32_t A0[4], A1[4];
        if constexpr (V8) {
          // block b = 16-byte columns 2b, 2b+1, transposed: vb[0] / vb[1] = tokens (2c, 2c+1) /
          // (2c+8, 2c+9) at dims 32b + 2g, 2g+1; vb[2] / vb[3] the same at dims 32b + 16 + 2g, 2g+1.
          // A0: dims 32b + 2g (row g), 2g+1 (row g+8); A1: dims 32b + 16 + 2g, 2g+1
          uint32_t vb[4];
          const int mi = lane >> 3;
          ldsm_x4_t(sV + swz<VRB>(tile * 16 + (mi & 1) * 8 + (lane & 7), 2 * b + (mi >> 1)), vb);
          unpack4_s8_t(vb[0], A0[0], A0[1]);
          unpack4_s8_t(vb[1], A0[2], A0[3]);
          unpack4_s8_t(vb[2], A1[0], A1[1]);
          unpack4_s8_t(vb[3], A1[2], A1[3]);
        } else {
          // vw[b/2][(b%2)*2 + 0] = tokens (2c, 2c+1) of block b; [.. + 1] = tokens (2c+8, 2c+9)
          uint32_t ua[4], ub[4];
          unpack8_q4(vw[b >> 1][(b & 1) * 2 + 0], ua);
          unpack8_q4(vw[b >> 1][(b & 1) * 2 + 1], ub);
          A0[0] = ua[0]; A0[1] = ua[1]; A0[2] = ub[0]; A0[3] = ub[1];   // dims 4g+0 (row g), 4g+1 (row g+8)
          A1[0] = ua[2]; A1[1] = ua[3]; A1[2] = ub[2]; A1[3] = ub[3];   // dims 4g+2, 4g+3
        }
        mma16816(O[b][0], A0, hi0, hi1);
        mma16816(O[b][0], A0, lo0, lo1);
        mma16816(O[b][1], A1, hi0, hi1);
        mma16816(O[b][1], A1, lo0, lo1);
      }
    }
    __syncwarp();                                        // buffer fully read before reuse
    issue(i + kRing);
  }

  // ---------------- warp state: reduce l (and the zero-point sums) over the token lanes
#pragma unroll
  for (int k = 4; k < 32; k <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, k);
    l1 += __shfl_xor_sync(0xffffffffu, l1, k);
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();                                       // every warp is done with its stages

  // ---------------- combine the four warps in shared memory: cm/cl [warp][8], co [warp][8][128]
  float *cm = reinterpret_cast<float *>(smem);
  float *cl = cm + kWarps * 8;
  float *co = cl + kWarps * 8;
  if (g == 0) {
    cm[warp * 8 + r0] = m0;
    cm[warp * 8 + r1] = m1;
    cl[warp * 8 + r0] = l0;
    cl[warp * 8 + r1] = l1;
  }
  // O holds the values directly (the V codes entered as exact signed values)
  if constexpr (HAD2) {
    // accumulator j = 4 ch + f: dims 64 ch + 8g + f (values 0, 1: rows r0, r1) and + 4 (2, 3), the
    // codes entered as exact signed values
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int da = 64 * (j >> 2) + 8 * g + (j & 3), db = da + 4;
      const float(&o)[4] = O[j >> 1][j & 1];
      co[(warp * 8 + r0) * kD + da] = o[0];
      co[(warp * 8 + r1) * kD + da] = o[1];
      co[(warp * 8 + r0) * kD + db] = o[2];
      co[(warp * 8 + r1) * kD + db] = o[3];
    }
  }
#pragma unroll
  for (int b = 0; b < (HAD2 ? 0 : 4); ++b) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int d = V8 ? 32 * b + 16 * h + 2 * g : 32 * b + 4 * g + 2 * h;
      *reinterpret_cast<float2 *>(co + (warp * 8 + r0) * kD + d) = make_float2(O[b][h][0], O[b][h][2]);
      *reinterpret_cast<float2 *>(co + (warp * 8 + r1) * kD + d) = make_float2(O[b][h][1], O[b][h][3]);
    }
  }
  __syncthreads();
  const int d = threadIdx.x;                             // 128 threads <-> 128 dims
  for (int r = 0; r < R; ++r) {
    if (t0 > row_limit_of(a, sl, r)) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cm[w * 8 + r]);
    float L = 0.0f, acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = cm[w * 8 + r] == -INFINITY ? 0.0f : ex2(cm[w * 8 + r] - M);
      L = fmaf(cl[w * 8 + r], wt, L);
      acc = fmaf(co[(w * 8 + r) * kD + d], wt, acc);
    }
    const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
    const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
    a.part_o[pi * kD + d] = acc;
    if (d == 0) {
      a.part_m[pi] = M * kLn2;                           // natural-log units, like the other kernels
      a.part_l[pi] = L;
    }
  }
}

template <int LAYOUT, int VLAYOUT, bool QSPLIT, bool PAGED, bool CAP = false>
cudaError_t launch_t(const AttendArgs &a, cudaStream_t st) {
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = set_smem_once(configured, attend_mma_kernel<LAYOUT, VLAYOUT, QSPLIT, PAGED, CAP>, smem_bytes<LAYOUT, VLAYOUT>());
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks, a.cache.B * a.cache.H);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem_bytes<LAYOUT, VLAYOUT>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_mma_kernel<LAYOUT, VLAYOUT, QSPLIT, PAGED, CAP>, a);
}

template <int LAYOUT, int VLAYOUT>
cudaError_t launch_pair_t(const AttendArgs &a, cudaStream_t st) {
  const bool paged = a.cache.page_shift >= 0;
  if (a.q_dtype == KVQ_F32)
    return paged ? launch_t<LAYOUT, VLAYOUT, true, true>(a, st) : launch_t<LAYOUT, VLAYOUT, true, false>(a, st);
  return paged ? launch_t<LAYOUT, VLAYOUT, false, true>(a, st) : launch_t<LAYOUT, VLAYOUT, false, false>(a, st);
}

}  // namespace

bool capture_supported(const AttendArgs &a) {
  const int L = a.cache.layout;
  return is_hadamard(L) && a.cache.v_layout == L && a.cache.page_shift < 0 && mma_supported(a);
}

bool mma_supported(const AttendArgs &a) {
  const int L = a.cache.layout, VL = a.cache.v_layout;
  if (prefill_supported(a)) return true;                 // includes the mixed K/V pairs it is built for
  if (L == KVQ_Q6_0 && VL == L) return mma_q6_supported(a);
  return decode_kernel(L, VL) && a.cache.D == kD && a.gqa * a.n_q <= 8 && a.n_body > 0 && a.chunk % kStage == 0;
}

cudaError_t launch_attend_mma(const AttendArgs &a, cudaStream_t st) {
  if (prefill_supported(a)) return launch_attend_prefill(a, st);
  if (a.cap_scores && !is_hadamard(a.cache.layout)) return cudaErrorNotSupported;
  if (uses_mma4(a.cache.layout)) return launch_attend_mma4(a, st);
  const bool paged = a.cache.page_shift >= 0;
  const int L = a.cache.layout, VL = a.cache.v_layout;
  if (L == KVQ_Q6_0) return launch_attend_mma_q6(a, st);
  if (L == KVQ_HAD_INT4) {                               // int8 query codes are exact
    if (a.cap_scores) return paged ? cudaErrorNotSupported : launch_t<KVQ_HAD_INT4, KVQ_HAD_INT4, false, false, true>(a, st);
    return paged ? launch_t<KVQ_HAD_INT4, KVQ_HAD_INT4, false, true>(a, st)
                 : launch_t<KVQ_HAD_INT4, KVQ_HAD_INT4, false, false>(a, st);
  }
  if (L == KVQ_HAD_INT2) {
    if (a.cap_scores) return paged ? cudaErrorNotSupported : launch_t<KVQ_HAD_INT2, KVQ_HAD_INT2, false, false, true>(a, st);
    return paged ? launch_t<KVQ_HAD_INT2, KVQ_HAD_INT2, false, true>(a, st)
                 : launch_t<KVQ_HAD_INT2, KVQ_HAD_INT2, false, false>(a, st);
  }
  if (L == KVQ_Q4_0 && VL == KVQ_Q4_0) return launch_pair_t<KVQ_Q4_0, KVQ_Q4_0>(a, st);
  if (L == KVQ_Q8_0 && VL == KVQ_Q8_0) return launch_pair_t<KVQ_Q8_0, KVQ_Q8_0>(a, st);
  if (L == KVQ_Q4_0 && VL == KVQ_Q8_0) return launch_pair_t<KVQ_Q4_0, KVQ_Q8_0>(a, st);
  return cudaErrorNotSupported;                          // the asymmetric layout runs attend_mma4.cu
}

}  // namespace kvq
