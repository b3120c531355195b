// Tensor-core phase 1 for many query rows per kv head: causal prefill chunks (and any call whose
// GQA group times query rows exceeds eight), head_dim 128, for the Hadamard int4 layout (tract
// discussion #2402, "Architecture: State" and the prefill remarks: the query rows of a chunk
// attend the cached body with causal limits; the body scores are exact integer dot products of
// the int8 rotated query and the int4 rotated keys) and for the per-block Q4_0 and asymmetric g=32
// layouts (bf16/f16 queries).
//
// Here the rows are the M side of the contraction (FlashAttention-2 orientation), with
// mma.sync.m16n8k16 (f16 in, f32 accumulate):
//   QK:  S[16 rows][8 tokens] += Q8[16 rows][16 dims] . K^T[16 dims][8 tokens]
//   PV:  O[16 rows][8 dims]   += P'[16 rows][16 tokens] . V[16 tokens][8 dims]
// Hadamard: Q8 holds the int8 query codes and K, V their signed int4 codes, all exact in f16, so
// every score is the exact integer dot (|dot| < 2^17, exact in the f32 accumulator);
// score = alpha * s_q[row] * s_k[t] * dot. The per-token V scale is folded into the
// probabilities, P' = p * s_v, kept as f16 hi + lo parts (two mma per step).
// Q4_0 / asymmetric: the per-block scale varies along the contracted dims, so the stage is
// unpacked into code * scale itself, split exactly into f16 hi + lo tiles (at most 15 significant
// bits): S = Q . (K_hi + K_lo)^T with the query exact in f16 after a per-row power-of-two
// prescale, and O += P_hi . V_hi + P_hi . V_lo + P_lo . V_hi. Asymmetric: the tiles hold the
// values v = s n + z themselves, formed in f32 and split into f16 hi + lo parts (|error| below
// 2^-23 |v|, not exact like code * scale). Keeping z out of the tiles in extra mma terms would
// be exact per element, but in a block with an outlier dim (z far from the other dims' values)
// the code and zero-point sums are large and cancel, and the tensor core's truncated
// accumulation over the chunk shows in the difference.
// The probabilities stay in registers between the two products: the S accumulator of two
// 8-token tiles is the A fragment of one 16-token PV step.
//
// A CTA of four warps takes 64 consecutive query rows of one (batch, kv head) and one chunk of
// body tokens. The packed rows stream through a three-stage cp.async ring of 64-token stages;
// each stage is unpacked once by the whole CTA into f16 code tiles (K and V, [token][128] with a
// 16-byte XOR swizzle), which the warps read with ldmatrix. Within each 8-dim group the tiles
// keep the unpacker's order (0,4,1,5,2,6,3,7); the query fragments and the output columns follow
// it. Each warp keeps the online softmax of its 16 rows.
//
// Hadamard: the exact-f32 recent window is more chunks of kWinChunk tokens (blockIdx.y >=
// n_chunks; a wide window is spread over several CTAs): their CTAs
// stream the f32 rotated K/V rows of the ring and score them with the f32 rotated query on the
// CUDA cores.
#pragma once
#include <cfloat>
#include <climits>

#include "kvq_internal.cuh"
#include "mma_util.cuh"

namespace kvq {
namespace {
using namespace mma;

constexpr int kWarps = 4;
constexpr int kRows = kPrefillRows;     // query rows per CTA (16 per warp)
static_assert(kRows == 16 * kWarps, "16 query rows per warp");
constexpr int kStage = 64;              // tokens per stage
constexpr int kD = 128;
constexpr int kTileRow = kD * 2;                       // f16 code/value tile [64 tokens][128], 256-byte rows
constexpr int kTile = kStage * kTileRow;
constexpr int kQrPitch = kD * 4 + 16;                  // window chunk: f32 rotated query rows (padded)
constexpr int kWinStage = 8;                           // window tokens per stage
constexpr int kWinPitch = kD * 4 + 16;

// One plane's layout in this kernel: code width, payload row bytes, per-token scale / zero bytes,
// and how the CTA's 128 threads split a 64-token stage of it into 16-byte pieces (every row has
// 16 eight-value chunks; a piece holds 16 / PPR of them).
template <int PL>
struct PlaneL {
  static constexpr bool HAD = is_hadamard(PL), ASYM = PL == KVQ_ASYM4_G32;
  static constexpr int BITS = PL == KVQ_Q8_0 ? 8 : (PL == KVQ_HAD_INT2 ? 2 : (PL == KVQ_Q6_0 ? 6 : 4));
  static constexpr int RB = kD * BITS / 8;               // payload bytes per token row
  static constexpr int SCB = HAD ? 4 : 8;                // scale bytes per token (f32 / 4 x f16)
  static constexpr int ZB = ASYM ? 8 : 0;                // zero-point bytes per token (4 x f16)
  static constexpr int PPR = RB / 16;                    // 16-byte pieces per row
  static constexpr int CPP = 16 / PPR;                   // 8-value chunks per piece (not used for 6-bit rows)
  static constexpr int PPT = kStage * PPR / (kWarps * 32);   // pieces per thread per stage
  static_assert(PPT >= 1 && PPT * kWarps * 32 == kStage * PPR, "whole pieces per thread");
};

// Shared memory of a (K layout, V layout) pair: a ring of raw stage slots (payload rows, scales,
// zero-points), then one region that first holds the query rows (prologue) and then the f16
// tiles of the unpacked stage (K, V; for block layouts also the K and V lo parts), then the
// per-row alpha factors. Three ring slots when they fit
// the CTAs-per-SM budget, else two.
template <int KL, int VL>
struct PGeo {
  using K = PlaneL<KL>;
  using V = PlaneL<VL>;
  static_assert(K::HAD == V::HAD, "one basis for both planes");
  static constexpr bool HAD = K::HAD;
  static constexpr int OFF_V = kStage * K::RB;
  static constexpr int OFF_SK = OFF_V + kStage * V::RB;
  static constexpr int OFF_SV = OFF_SK + kStage * K::SCB;
  static constexpr int OFF_ZK = OFF_SV + kStage * V::SCB;
  static constexpr int OFF_ZV = OFF_ZK + kStage * K::ZB;
  static constexpr int RAW = OFF_ZV + kStage * V::ZB;
  static constexpr int WIN = 2 * kWinStage * kWinPitch;  // window stage (Hadamard) in a slot
  static constexpr int SLOT = ((HAD && WIN > RAW ? WIN : RAW) + 127) / 128 * 128;
  static constexpr int NT = HAD ? 2 : 4;                 // f16 tiles
  static constexpr int QB = HAD ? kD : 2 * kD;           // query bytes per row: int8 codes / prescaled f16
  static constexpr int REG_T = NT * kTile, REG_Q = kRows * QB, REG_W = HAD ? kRows * kQrPitch : 0;
  static constexpr int REGION = REG_T > REG_Q ? (REG_T > REG_W ? REG_T : REG_W) : (REG_Q > REG_W ? REG_Q : REG_W);
  static constexpr int TAIL = kRows * 4;
  static constexpr int CTAS = HAD ? kPrefillCtasPerSm : 2;
  static constexpr int BUDGET = (233472 - 1024 * CTAS) / CTAS;   // 228 KB per SM, 1 KB reserved per CTA
  static constexpr int RING = 3 * SLOT + REGION + TAIL <= BUDGET ? 3 : 2;
  static constexpr int OFF_T = RING * SLOT;
  static constexpr int OFF_Q = OFF_T;                    // the query rows, then the tiles
  static constexpr int OFF_QR = OFF_T;                   // window chunk: rotated f32 query rows
  static constexpr int OFF_SQ = OFF_T + REGION;          // per row: s_q (Hadamard) / alpha factor
  static constexpr int SMEM = OFF_SQ + TAIL;
  static_assert(SMEM <= BUDGET, "shared memory fits the CTAs per SM");
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Byte offset of (token row, 16-byte chunk) in an f16 code tile. Within each 128-byte half of the
// row the chunk is XORed with (row & 7), and with 2 in the upper half: ldmatrix phases (8 rows,
// one chunk) and the unpacker's 16-byte store phases (2 rows x chunks e, 4+e, 8+e, 12+e) both hit
// 8 distinct bank groups.
__device__ __forceinline__ uint32_t toff(int row, int chunk) {
  return (uint32_t)(row * kTileRow + (((chunk & 8) | ((chunk ^ (row & 7) ^ ((chunk >> 3) << 1)) & 7)) << 4));
}

// Last token query row r (of the gqa * n_q rows of a kv head) may see; negative if none.
// Unpack one plane of a raw stage slot (`pay`: 64 rows of PL's payload, `sc`: its per-token
// scales, `zr`: its per-token zero-points, asymmetric layout only) into the f16 tile at shared
// address `tile` (block layouts: hi parts; lo parts at tile + 2 * kTile).
template <int PL>
__device__ __forceinline__ void unpack_plane(const uint8_t *pay, const uint8_t *sc, const uint8_t *zr, uint32_t tile) {
  using P = PlaneL<PL>;
  if constexpr (P::BITS == 6) {
    // Q6_0: each thread takes two (row, 32-value block) units; a block is 16 low-plane bytes then
    // 8 high-plane bytes (24-byte blocks: 8-byte reads). Chunk k of the block (values 8k .. 8k+7)
    // is low-plane word k plus high-plane bytes 2k, 2k+1. In one store instruction a warp covers 8
    // rows x chunks (k, 4+k, 8+k, 12+k): the tile swizzle keeps each 8-lane phase conflict-free.
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int u = threadIdx.x + kWarps * 32 * k2;
      const int row = u >> 2, blk = u & 3;
      const uint8_t *bp = pay + row * P::RB + 24 * blk;
      const uint2 l0 = *reinterpret_cast<const uint2 *>(bp), l1 = *reinterpret_cast<const uint2 *>(bp + 8);
      const uint2 hh = *reinterpret_cast<const uint2 *>(bp + 16);
      const uint32_t lw[4] = {l0.x, l0.y, l1.x, l1.y};
      const uint32_t s2 = 0x00010001u * *reinterpret_cast<const uint16_t *>(sc + row * 8 + 2 * blk);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t o[4];
        unpack8_s6(lw[k], ((k < 2) ? hh.x : hh.y) >> (16 * (k & 1)), o);
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          hi[x] = hmul2(o[x], s2);                                         // rn(c s)
          lo[x] = hfma2(o[x], s2, hi[x] ^ 0x80008000u);                    // c s - rn(c s), exact
        }
        const uint32_t off = toff(row, 4 * blk + k);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(tile + off),
                     "r"(hi[0]), "r"(hi[1]), "r"(hi[2]), "r"(hi[3]) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(tile + 2 * kTile + off),
                     "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3]) : "memory");
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < P::PPT; ++k) {
    const int u = threadIdx.x + kWarps * 32 * k;          // piece: row u / PPR, 16-byte column u % PPR
    const int row = u / P::PPR, q = u % P::PPR;
    const uint4 w = *reinterpret_cast<const uint4 *>(pay + 16 * u);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < P::CPP; ++e) {
      // 8- and 2-bit rows: half of the lanes of each 8-lane store phase take their chunks in a
      // rotated order, so that the phase's eight 16-byte stores land in eight distinct bank groups
      // of the swizzled tile (in plain order they would pair up: a 2-way conflict)
      int ee = e;
      if constexpr (P::BITS == 8) ee = e ^ ((q >> 2) & 1);
      if constexpr (P::BITS == 2) ee = e ^ (q << 2);
      const int ch = q * P::CPP + ee;                     // chunk: dims 8 ch .. 8 ch + 7
      uint32_t o[4];
      if constexpr (P::BITS == 8) {
        unpack8_s8(ee ? ws[2] : ws[0], ee ? ws[3] : ws[1], o);
      } else if constexpr (P::BITS == 2) {
        const uint32_t wd = q ? ws[(e >> 1) ^ 2] : ws[e >> 1];
        unpack8_s2(wd >> (16 * (e & 1)), o);
      } else if constexpr (P::ASYM) {
        unpack8_u4(ws[e], o);
      } else {
        unpack8_q4(ws[e], o);
      }
      const uint32_t off = toff(row, ch);
      if constexpr (P::HAD) {
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(tile + off),
                     "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]) : "memory");
      } else {
        uint32_t hi[4], lo[4];
        if constexpr (P::ASYM) {
          // v = s n + z in f32 (s n is exact), then hi = rn(v), lo = rn(v - hi)
          const float sf = __half2float(*reinterpret_cast<const __half *>(sc + row * 8 + 2 * (ch >> 2)));
          const float zf = __half2float(*reinterpret_cast<const __half *>(zr + row * 8 + 2 * (ch >> 2)));
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const float2 nf = __half22float2(u32_as_h2(o[x]));
            const float v0 = fmaf(sf, nf.x, zf), v1 = fmaf(sf, nf.y, zf);
            hi[x] = pack_f16x2(v0, v1);
            const float2 hf = __half22float2(u32_as_h2(hi[x]));
            lo[x] = pack_f16x2(v0 - hf.x, v1 - hf.y);
          }
        } else {
          const uint32_t s2 = 0x00010001u * *reinterpret_cast<const uint16_t *>(sc + row * 8 + 2 * (ch >> 2));
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            hi[x] = hmul2(o[x], s2);                                       // rn(c s)
            lo[x] = hfma2(o[x], s2, hi[x] ^ 0x80008000u);                  // c s - rn(c s), exact
          }
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(tile + off),
                     "r"(hi[0]), "r"(hi[1]), "r"(hi[2]), "r"(hi[3]) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(tile + 2 * kTile + off),
                     "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3]) : "memory");
      }
    }
  }
}

__device__ __forceinline__ int row_limit_of(const AttendArgs &a, const SeqLen &sl, int r) {
  return row_limit(a, sl, r % a.n_q);
}

// DEC (at most 16 query rows per kv head, one row block): the four warps split each stage's
// tokens (16 each) over the same 16 rows and merge their softmax states at the end, instead of
// one warp scoring every token while the other three only unpack.
// CAP: score capture (Hadamard layouts, contiguous cache): every exact integer body score the CTA
// computes and each row's int8 query scale also go to a.cap_scores / a.cap_sq.
template <int KL, int VL, bool PAGED, bool DEC, bool CAP = false>
__global__ void __launch_bounds__(kWarps * 32, PGeo<KL, VL>::CTAS) attend_prefill_kernel(AttendArgs a) {
  using G = PGeo<KL, VL>;
  constexpr int NTJ = DEC ? 2 : 4;                       // 8-token score tiles per pass
  constexpr int NKK = DEC ? 1 : 2;                       // 16-token PV steps per pass
  constexpr int NPASS = DEC ? 1 : 2;                     // passes per 64-token stage
  constexpr int TPP = 8 * NTJ;                           // tokens per pass
  using PK = typename G::K;
  using PV = typename G::V;
  constexpr bool HAD = G::HAD, ASYMK = PK::ASYM, ASYMV = PV::ASYM;
  constexpr int kRing = G::RING;
  static_assert(!CAP || (HAD && !PAGED), "score capture: Hadamard layouts, contiguous cache");
  extern __shared__ __align__(1024) uint8_t smem[];
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  const CacheView &cv = a.cache;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int row0 = blockIdx.x * kRows;
  const int chunk_id = blockIdx.y + a.y_base;
  const int bh = blockIdx.z;
  const int bb = bh / cv.H, kvh = bh - bb * cv.H;
  const SeqLen sl = seq_of_t<PAGED>(a, bb);             // this sequence's lengths
  const int R = a.gqa * a.n_q;

  const bool win = HAD && chunk_id >= a.n_chunks;     // a chunk of the recent window
  const int t0 = win ? sl.n_body + (chunk_id - a.n_chunks) * kWinChunk : chunk_id * sl.chunk;
  const int t1 = win ? min(sl.kv_len, t0 + kWinChunk) : min(sl.n_body, t0 + sl.chunk);
  int w_lim = -1;
  for (int r = row0; r < min(row0 + kRows, R); ++r) w_lim = max(w_lim, row_limit_of(a, sl, r));
  // rows appended by the preceding kernel (cache rows or window ring): only the CTAs that read
  // them wait for it; a window chunk whose rotated query rows were prepared by an earlier launch
  // always waits (the preceding grid's CTAs may have let it start before they waited for that
  // preparation themselves)
  pdl_wait_if((HAD && win && a.q_prepped) || (t0 <= w_lim && t0 < sl.fresh_hi && sl.fresh_lo < min(t1, w_lim + 1)));
  if (t0 > w_lim || t0 >= t1) return;                 // no row of this CTA sees the chunk
  const int t_end = min(t1, w_lim + 1);
  const int stage_len = win ? kWinStage : kStage;
  const int n_stages = (t_end - t0 + stage_len - 1) / stage_len;


  const size_t head_row0 = (size_t)bh * cv.cap;           // contiguous cache: row of token 0
  // ---- CTA-wide copy of stage s into ring slot s % 3; rows past t_end are zero-filled.
  // Body: 256 16-byte pieces per packed plane (two per thread), one token's scales per thread (and
  // zero-points). Window: 8 f32 K and V rows from ring slot t mod n_recent.
  auto issue = [&](int s) {
    if (s < n_stages) {
      uint8_t *sb = smem + (s % kRing) * G::SLOT;
      if (win) {
        const int ts = t0 + s * kWinStage;
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
      } else {
        const int ts = t0 + s * kStage;
        // the stage's 64 rows are consecutive plane rows (a page holds at least 64 aligned tokens)
        const size_t r0 = cache_row_t<PAGED>(cv, bb, kvh, head_row0, ts);
        const uint8_t *kp = cv.payload[0] + r0 * PK::RB, *vp = cv.payload[1] + r0 * PV::RB;
        const bool full = ts + kStage <= t_end;
#pragma unroll
        for (int k = 0; k < PK::PPT; ++k) {             // K pieces: row q / PPR, 16-byte column q % PPR
          const int q = threadIdx.x + 128 * k;
          const bool ok = full || ts + q / PK::PPR < t_end;
          cp_async16(smem_addr(sb + 16 * q), kp + (ok ? (size_t)16 * q : 0), ok ? 16 : 0);
        }
#pragma unroll
        for (int k = 0; k < PV::PPT; ++k) {             // V pieces
          const int q = threadIdx.x + 128 * k;
          const bool ok = full || ts + q / PV::PPR < t_end;
          cp_async16(smem_addr(sb + G::OFF_V + 16 * q), vp + (ok ? (size_t)16 * q : 0), ok ? 16 : 0);
        }
        const int kv = threadIdx.x >> 6, row = threadIdx.x & 63;   // one token's scales per thread
        const bool ok = ts + row < t_end;
        const size_t tok = r0 + (size_t)(ok ? row : 0);
        if (kv == 0) {
          cp_async_scale<PK::SCB>(smem_addr(sb + G::OFF_SK + PK::SCB * row),
                                  static_cast<const uint8_t *>(cv.scale[0]) + tok * PK::SCB, ok ? PK::SCB : 0);
          if (ASYMK) cp_async8(smem_addr(sb + G::OFF_ZK + 8 * row), reinterpret_cast<const uint8_t *>(cv.zero[0]) + tok * 8,
                               ok ? 8 : 0);
        } else {
          cp_async_scale<PV::SCB>(smem_addr(sb + G::OFF_SV + PV::SCB * row),
                                  static_cast<const uint8_t *>(cv.scale[1]) + tok * PV::SCB, ok ? PV::SCB : 0);
          if (ASYMV) cp_async8(smem_addr(sb + G::OFF_ZV + 8 * row), reinterpret_cast<const uint8_t *>(cv.zero[1]) + tok * 8,
                               ok ? 8 : 0);
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < kRing - 1; ++s) issue(s);

  // ---- query prologue, each warp for its 16 rows. Hadamard: rotate and quantise (warp FWHT, int8
  // codes and one f32 scale per row; the window chunk keeps the f32 rotated rows instead).
  // Others: a per-row power-of-two prescale (largest |q| in [2^13, 2^14), asymmetric [2^8, 2^9) so
  // that a block sum stays below the f16 range; bf16 / f16 rows stay exact) and the prescaled f16
  // row; the row's alpha * 2^e * log2(e) goes with it (asymmetric: and its four block sums).
  uint8_t *qsm = smem + G::OFF_Q;
  float *sqs = reinterpret_cast<float *>(smem + G::OFF_SQ);
  for (int i = 0; i < 16; ++i) {
    const int lr = 16 * warp + i, r = row0 + lr;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    size_t grow = 0;
    if (r < R) {
      const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
      grow = ((size_t)bb * a.Hq + hq) * a.n_q + qi;
      if (!(HAD && win && a.q_prepped)) load4_f32(a.q, a.q_dtype, grow * kD + lane * 4, x);
    }
    if (HAD && win && a.q_prepped) {                   // the rotated rows are already prepared
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < R) v = *reinterpret_cast<const float4 *>(a.q_rot + grow * kD + lane * 4);
      *reinterpret_cast<float4 *>(smem + G::OFF_QR + lr * kQrPitch + lane * 16) = v;
      continue;
    }
    if constexpr (HAD) {
      int q8v[4] = {0, 0, 0, 0};
      float sq = 0.0f;
      if (r < R) sq = had_query_row<4>(x, q8v, lane);
      if (win) {
        *reinterpret_cast<float4 *>(smem + G::OFF_QR + lr * kQrPitch + lane * 16) = make_float4(x[0], x[1], x[2], x[3]);
      } else {
        *reinterpret_cast<uint32_t *>(qsm + lr * kD + lane * 4) =
            (uint32_t)(q8v[0] & 0xFF) | ((uint32_t)(q8v[1] & 0xFF) << 8) | ((uint32_t)(q8v[2] & 0xFF) << 16) |
            ((uint32_t)(q8v[3] & 0xFF) << 24);
        if (lane == 0) sqs[lr] = sq;
        if (CAP && lane == 0 && chunk_id == 0 && r < R) a.cap_sq[grow] = sq;
      }
    } else {
      float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
      int e = 0;
      if (mx > 0.0f) e = min(max(((__float_as_int(mx) >> 23) & 0xFF) - 127 - 13, -100), 100);
      const float pre = ldexpf(1.0f, -e);
      const uint2 qp = make_uint2(pack_f16x2(x[0] * pre, x[1] * pre), pack_f16x2(x[2] * pre, x[3] * pre));
      *reinterpret_cast<uint2 *>(qsm + lr * 2 * kD + lane * 8) = qp;
      if (lane == 0) sqs[lr] = r < R ? a.scale * ldexpf(1.0f, e) * kLog2e : 0.0f;
    }
  }
  // DEC: every warp reads block 0's query rows and factors, which warp 0 wrote
  if constexpr (DEC) __syncthreads();
  else __syncwarp();
  // the warp's 16 rows: its own block, except in the body chunks of DEC where all warps share block 0
  const int rw = (DEC && !win) ? 0 : warp;
  const int rg = row0 + 16 * rw + g, rg8 = rg + 8;
  const int lim_g = rg < R ? row_limit_of(a, sl, rg) : -1;
  const int lim_g8 = rg8 < R ? row_limit_of(a, sl, rg8) : -1;
  int warp_lim = max(lim_g, lim_g8), warp_min = INT_MAX;
  if (lim_g >= 0) warp_min = lim_g;
  if (lim_g8 >= 0) warp_min = min(warp_min, lim_g8);
#pragma unroll
  for (int k = 4; k < 32; k <<= 1) {
    warp_lim = max(warp_lim, __shfl_xor_sync(0xffffffffu, warp_lim, k));
    warp_min = min(warp_min, __shfl_xor_sync(0xffffffffu, warp_min, k));
  }
  float m_g = -INFINITY, m_g8 = -INFINITY, l_g = 0.0f, l_g8 = 0.0f;

  if constexpr (HAD) {
  if (win) {
    // =============== the recent window on the tensor cores, accurate to f32: every f32 operand is
    // split into tf32 hi + lo parts and each product takes three m16n8k8 MMAs (lo * hi, hi * lo,
    // hi * hi; the dropped lo * lo term is below 2^-21 of the product). Per 8-token stage, warp w
    // scores its rows 16 w + g and 16 w + g + 8 (g = lane / 4) against tokens 2c and 2c + 1
    // (c = lane % 4), the layout of an m16n8 accumulator, and keeps O[16 rows][128 dims] in 16 of
    // them: Ow[n] holds dims 8n + 2c, 8n + 2c + 1 of rows g (0, 1) and g + 8 (2, 3).
    const float walpha = a.scale * kLog2e;
    float Ow[kD / 8][4];
#pragma unroll
    for (int n = 0; n < kD / 8; ++n)
#pragma unroll
      for (int k = 0; k < 4; ++k) Ow[n][k] = 0.0f;
    for (int i = 0; i < n_stages; ++i) {
      cp_async_wait<kRing - 2>();
      __syncthreads();
      issue(i + kRing - 1);
      const int ts = t0 + i * kWinStage;
      if (ts > warp_lim) continue;
      const uint8_t *sb = smem + (i % kRing) * G::SLOT;
      const float *qa = reinterpret_cast<const float *>(smem + G::OFF_QR + (16 * warp + g) * kQrPitch);
      const float *qb = reinterpret_cast<const float *>(smem + G::OFF_QR + (16 * warp + g + 8) * kQrPitch);
      const float *kr = reinterpret_cast<const float *>(sb + g * kWinPitch);   // token g: column g of K^T
      // S = Q . K^T over the 16 8-dim k-steps; the three product terms in separate accumulators
      float slh[4] = {0.f, 0.f, 0.f, 0.f}, shl[4] = {0.f, 0.f, 0.f, 0.f}, shh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < kD / 8; ++ks) {
        const int d0 = 8 * ks + c;
        uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
        split_tf32(qa[d0], ah[0], al[0]);
        split_tf32(qb[d0], ah[1], al[1]);
        split_tf32(qa[d0 + 4], ah[2], al[2]);
        split_tf32(qb[d0 + 4], ah[3], al[3]);
        split_tf32(kr[d0], bh0, bl0);
        split_tf32(kr[d0 + 4], bh1, bl1);
        mma1688_tf32(slh, al, bh0, bh1);
        mma1688_tf32(shl, ah, bl0, bl1);
        mma1688_tf32(shh, ah, bh0, bh1);
      }
      // (g, 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1)
      float s0 = (slh[0] + shl[0]) + shh[0], s1 = (slh[1] + shl[1]) + shh[1];
      float s2 = (slh[2] + shl[2]) + shh[2], s3 = (slh[3] + shl[3]) + shh[3];
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
      // O += P . V: the probabilities are the A operand as they stand (k = c <-> token 2c,
      // k = c + 4 <-> token 2c + 1), V's rows 2c and 2c + 1 the matching B entries
      uint32_t ph[4], pl[4];
      split_tf32(s0, ph[0], pl[0]);
      split_tf32(s2, ph[1], pl[1]);
      split_tf32(s1, ph[2], pl[2]);
      split_tf32(s3, ph[3], pl[3]);
      const float *va = reinterpret_cast<const float *>(sb + (kWinStage + 2 * c) * kWinPitch);
      const float *vb = reinterpret_cast<const float *>(sb + (kWinStage + 2 * c + 1) * kWinPitch);
#pragma unroll
      for (int n = 0; n < kD / 8; ++n) {
        Ow[n][0] *= corr_g;
        Ow[n][1] *= corr_g;
        Ow[n][2] *= corr_g8;
        Ow[n][3] *= corr_g8;
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(va[8 * n + g], bh0, bl0);
        split_tf32(vb[8 * n + g], bh1, bl1);
        mma1688_tf32(Ow[n], pl, bh0, bh1);
        mma1688_tf32(Ow[n], ph, bl0, bl1);
        mma1688_tf32(Ow[n], ph, bh0, bh1);
      }
    }
    l_g += __shfl_xor_sync(0xffffffffu, l_g, 1);
    l_g += __shfl_xor_sync(0xffffffffu, l_g, 2);
    l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 1);
    l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 2);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? rg8 : rg;
      const int lim = half ? lim_g8 : lim_g;
      if (r >= R || t0 > lim) continue;                  // row does not see the window
      const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
      const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
      float *po = a.part_o + pi * kD;
#pragma unroll
      for (int n = 0; n < kD / 8; ++n)
        *reinterpret_cast<float2 *>(po + 8 * n + 2 * c) = make_float2(Ow[n][2 * half], Ow[n][2 * half + 1]);
      if (c == 0) {
        a.part_m[pi] = (half ? m_g8 : m_g) * kLn2;
        a.part_l[pi] = half ? l_g8 : l_g;
      }
    }
    return;
  }
  }

  // =============== body chunk on the tensor cores
  // A fragment of k-step ks (tile columns 16ks .. 16ks+15): rows g / g+8; tile column 8m + 2i
  // holds dim 8m + i and column 8m + 2i + 1 holds dim 8m + 4 + i (the unpacker's pair order)
  uint32_t aq[8][4];
  float alpha_g, alpha_g8;
  if constexpr (HAD) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int8_t *qg = reinterpret_cast<const int8_t *>(qsm + (16 * rw + g) * kD + 16 * ks);
      const int8_t *qg8 = qg + 8 * kD;
      aq[ks][0] = pack_f16x2((float)qg[c], (float)qg[4 + c]);
      aq[ks][1] = pack_f16x2((float)qg8[c], (float)qg8[4 + c]);
      aq[ks][2] = pack_f16x2((float)qg[8 + c], (float)qg[12 + c]);
      aq[ks][3] = pack_f16x2((float)qg8[8 + c], (float)qg8[12 + c]);
    }
    alpha_g = (rg < R ? a.scale * sqs[16 * rw + g] : 0.0f) * kLog2e;
    alpha_g8 = (rg8 < R ? a.scale * sqs[16 * rw + g + 8] : 0.0f) * kLog2e;
  } else {
    const uint16_t *qh = reinterpret_cast<const uint16_t *>(qsm);
    auto pk = [](uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); };
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint16_t *qg = qh + (16 * rw + g) * kD + 16 * ks, *qg8 = qg + 8 * kD;
      aq[ks][0] = pk(qg[c], qg[4 + c]);
      aq[ks][1] = pk(qg8[c], qg8[4 + c]);
      aq[ks][2] = pk(qg[8 + c], qg[12 + c]);
      aq[ks][3] = pk(qg8[8 + c], qg8[12 + c]);
    }
    alpha_g = sqs[16 * rw + g];                        // alpha * 2^e * log2(e), 0 for rows past R
    alpha_g8 = sqs[16 * rw + g + 8];
  }
  float O[16][4];                                        // tile j: dims 8j + c (c0/c2), 8j + 4 + c (c1/c3)
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) O[j][k] = 0.0f;
  const uint32_t sKT = smem_addr(smem + G::OFF_T), sVT = sKT + kTile;
  const int mi = lane >> 3;
  // ldmatrix addresses: every row this lane points at has (row & 7) == (lane & 7), so the tile
  // swizzle reduces to a per-lane constant XOR a compile-time constant per chunk.
  // K: rows 8j + (lane & 7), chunk 4m + mi.  V: rows 16kk + 8 (mi & 1) + (lane & 7), chunk 2p + (mi >> 1).
  const uint32_t kbase = sKT + (uint32_t)(lane & 7) * kTileRow;
  const uint32_t vbase = sVT + (uint32_t)((mi & 1) * 8 + (lane & 7)) * kTileRow;
  const int kx = mi ^ (lane & 7), vx = (mi >> 1) ^ (lane & 7);
  auto kofs = [&](int m) -> uint32_t {                   // chunk 4m + mi
    return (uint32_t)((((kx ^ (((m & 1) << 2) | ((m >> 1) << 1))) & 7) | ((m >> 1) << 3)) << 4);
  };
  auto vofs = [&](int p) -> uint32_t {                   // chunk 2p + (mi >> 1)
    return (uint32_t)((((vx ^ ((2 * p) ^ ((p >> 2) << 1))) & 7) | ((p >> 2) << 3)) << 4);
  };

  for (int i = 0; i < n_stages; ++i) {
    cp_async_wait<kRing - 2>();
    __syncthreads();                                     // stage i landed; the tiles are free
    issue(i + kRing - 1);
    const uint8_t *sb = smem + (i % kRing) * G::SLOT;
    // ---- unpack the stage into the f16 tiles, plane by plane (each thread: PPT 16-byte pieces of
    // CPP eight-value chunks per plane). Hadamard: the signed codes. Block layouts: the values
    // code * scale of each chunk's 32-dim block as f16 hi + lo parts (exact TwoProduct: code * scale
    // has at most 19 significant bits); asymmetric zero-points enter by their own mma terms.
    unpack_plane<KL>(sb, sb + G::OFF_SK, sb + G::OFF_ZK, sKT);
    unpack_plane<VL>(sb + G::OFF_V, sb + G::OFF_SV, sb + G::OFF_ZV, sVT);
    __syncthreads();                                     // tiles complete
    const int ts = t0 + i * kStage;
    if (ts > warp_lim) continue;                         // none of this warp's rows sees the stage
    const float *skf = reinterpret_cast<const float *>(sb + G::OFF_SK);   // Hadamard per-token scales
    const float *svf = reinterpret_cast<const float *>(sb + G::OFF_SV);

    // passes over the stage (two 32-token halves; DEC: this warp's 16 tokens): S = Q . K^T for
    // NTJ 8-token tiles, online softmax, O += P' . V
    // the first token (within the stage) of pass hh: the halves of the stage, or (DEC) this warp's 16
    const auto pass_tok = [warp](int hh) { return DEC ? 16 * warp : 32 * hh; };
#pragma unroll 1
    for (int hh = 0; hh < NPASS; ++hh) {
      const int tsub = ts + pass_tok(hh);
      if (tsub > warp_lim) break;
      float s[NTJ][4];
      {
        // k-step pairs outermost: consecutive mma on one tile's accumulator are four apart
        float d[NTJ][4] = {};
#pragma unroll
        for (int m = 0; m < 4; ++m) {                    // k-steps 2m, 2m+1
          uint32_t kw[NTJ][4];
#pragma unroll
          for (int j = 0; j < NTJ; ++j) ldsm_x4(kbase + (pass_tok(hh) + 8 * j) * kTileRow + kofs(m), kw[j]);
#pragma unroll
          for (int j = 0; j < NTJ; ++j) mma16816(d[j], aq[2 * m], kw[j][0], kw[j][1]);
#pragma unroll
          for (int j = 0; j < NTJ; ++j) mma16816(d[j], aq[2 * m + 1], kw[j][2], kw[j][3]);
          if constexpr (!HAD) {                          // + the lo parts of the K values
#pragma unroll
            for (int j = 0; j < NTJ; ++j) ldsm_x4(kbase + 2 * kTile + (pass_tok(hh) + 8 * j) * kTileRow + kofs(m), kw[j]);
#pragma unroll
            for (int j = 0; j < NTJ; ++j) mma16816(d[j], aq[2 * m], kw[j][0], kw[j][1]);
#pragma unroll
            for (int j = 0; j < NTJ; ++j) mma16816(d[j], aq[2 * m + 1], kw[j][2], kw[j][3]);
          }
        }
        if constexpr (CAP) {                             // d holds the exact integer dots
#pragma unroll
          for (int j = 0; j < NTJ; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int r = (k & 2) ? rg8 : rg, t = tsub + 8 * j + 2 * c + (k & 1);
              if (r < R && t < t_end) capture_score(a, bb, kvh, r, t, __float2int_rn(d[j][k]));
            }
        }
#pragma unroll
        for (int j = 0; j < NTJ; ++j) {
          float2 sk = make_float2(1.0f, 1.0f);
          if constexpr (HAD) sk = *reinterpret_cast<const float2 *>(skf + pass_tok(hh) + 8 * j + 2 * c);
          s[j][0] = d[j][0] * alpha_g * sk.x;
          s[j][1] = d[j][1] * alpha_g * sk.y;
          s[j][2] = d[j][2] * alpha_g8 * sk.x;
          s[j][3] = d[j][3] * alpha_g8 * sk.y;
        }
      }
      if (tsub + TPP > t1 || tsub + TPP - 1 > warp_min) {
#pragma unroll
        for (int j = 0; j < NTJ; ++j) {
          const int ta = tsub + 8 * j + 2 * c, tb = ta + 1;
          if (!(ta < t1 && ta <= lim_g)) s[j][0] = -INFINITY;
          if (!(tb < t1 && tb <= lim_g)) s[j][1] = -INFINITY;
          if (!(ta < t1 && ta <= lim_g8)) s[j][2] = -INFINITY;
          if (!(tb < t1 && tb <= lim_g8)) s[j][3] = -INFINITY;
        }
      }
      // online softmax (base 2), rows g and g+8
      float mx_g = fmaxf(s[0][0], s[0][1]), mx_g8 = fmaxf(s[0][2], s[0][3]);
#pragma unroll
      for (int j = 1; j < NTJ; ++j) {
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
        for (int j = 0; j < 16; ++j) {
          O[j][0] *= corr_g;
          O[j][1] *= corr_g;
          O[j][2] *= corr_g8;
          O[j][3] *= corr_g8;
        }
      }
      float ls_g = 0.0f, ls_g8 = 0.0f;
#pragma unroll
      for (int j = 0; j < NTJ; ++j) {
        s[j][0] = ex2(s[j][0] - mu_g);
        s[j][1] = ex2(s[j][1] - mu_g);
        s[j][2] = ex2(s[j][2] - mu_g8);
        s[j][3] = ex2(s[j][3] - mu_g8);
        ls_g += s[j][0] + s[j][1];
        ls_g8 += s[j][2] + s[j][3];
        if constexpr (HAD) {                             // P' = p * s_v
          const float2 sv = *reinterpret_cast<const float2 *>(svf + pass_tok(hh) + 8 * j + 2 * c);
          s[j][0] *= sv.x;
          s[j][1] *= sv.y;
          s[j][2] *= sv.x;
          s[j][3] *= sv.y;
        }
      }
      l_g = fmaf(l_g, corr_g, ls_g);
      l_g8 = fmaf(l_g8, corr_g8, ls_g8);

      // O += P' . V, two 16-token steps
#pragma unroll
      for (int kk = 0; kk < NKK; ++kk) {
        // A: a0 = (row g, tokens 2c..), a1 = (row g+8, tokens 2c..), a2 = (row g, tokens 8+2c..),
        // a3 = (row g+8, tokens 8+2c..), as f16 hi + lo parts
        uint32_t ah[4], al[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 2 * kk + (e >> 1), xx = (e & 1) ? 2 : 0;
          ah[e] = pack_f16x2(s[j][xx], s[j][xx + 1]);
          const float2 f = __half22float2(u32_as_h2(ah[e]));
          al[e] = pack_f16x2(s[j][xx] - f.x, s[j][xx + 1] - f.y);
        }
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {                 // output tiles 8pg .. 8pg+7
          uint32_t vw[4][4];                             // per p: b0/b1 of tile 2p, b0/b1 of tile 2p+1
#pragma unroll
          for (int p4 = 0; p4 < 4; ++p4)
            ldsm_x4_t(vbase + (pass_tok(hh) + 16 * kk) * kTileRow + vofs(4 * pg + p4), vw[p4]);
          // hi parts of the eight tiles, then the lo parts: eight mma between two on one tile
#pragma unroll
          for (int p4 = 0; p4 < 4; ++p4) {
            mma16816(O[2 * (4 * pg + p4)], ah, vw[p4][0], vw[p4][1]);
            mma16816(O[2 * (4 * pg + p4) + 1], ah, vw[p4][2], vw[p4][3]);
          }
#pragma unroll
          for (int p4 = 0; p4 < 4; ++p4) {
            mma16816(O[2 * (4 * pg + p4)], al, vw[p4][0], vw[p4][1]);
            mma16816(O[2 * (4 * pg + p4) + 1], al, vw[p4][2], vw[p4][3]);
          }
          if constexpr (!HAD) {                          // + P_hi . V_lo
#pragma unroll
            for (int p4 = 0; p4 < 4; ++p4)
              ldsm_x4_t(vbase + 2 * kTile + (pass_tok(hh) + 16 * kk) * kTileRow + vofs(4 * pg + p4), vw[p4]);
#pragma unroll
            for (int p4 = 0; p4 < 4; ++p4) {
              mma16816(O[2 * (4 * pg + p4)], ah, vw[p4][0], vw[p4][1]);
              mma16816(O[2 * (4 * pg + p4) + 1], ah, vw[p4][2], vw[p4][3]);
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
  if constexpr (DEC) {
    // the four warps scored different tokens of the same 16 rows: merge their (m, l, O) through
    // shared memory (the tile region, free once every warp is past its last stage), one thread
    // per output dim
    __syncthreads();
    float *xm = reinterpret_cast<float *>(smem + G::OFF_T);   // [warp][row] m (log2 units)
    float *xl = xm + kWarps * 16;                             // [warp][row] l
    float *xo = xl + kWarps * 16;                             // [warp][row][dim] O
    static_assert((2 * kWarps * 16 + kWarps * 16 * kD) * 4 <= G::REGION, "merge area fits the tile region");
    if (c == 0) {
      xm[warp * 16 + g] = m_g;
      xm[warp * 16 + g + 8] = m_g8;
      xl[warp * 16 + g] = l_g;
      xl[warp * 16 + g + 8] = l_g8;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float *o0 = xo + (warp * 16 + g) * kD + 8 * j, *o8 = o0 + 8 * kD;
      o0[c] = O[j][0];
      o0[4 + c] = O[j][1];
      o8[c] = O[j][2];
      o8[4 + c] = O[j][3];
    }
    __syncthreads();
    const int d = threadIdx.x;                               // 128 threads <-> 128 dims
    for (int r = 0; r < 16; ++r) {
      const int rr = row0 + r;
      if (rr >= R || t0 > row_limit_of(a, sl, rr)) continue;   // row does not see this chunk
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, xm[w * 16 + r]);
      float L = 0.0f, acc = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float wt = xm[w * 16 + r] == -INFINITY ? 0.0f : ex2(xm[w * 16 + r] - M);
        L = fmaf(xl[w * 16 + r], wt, L);
        acc = fmaf(xo[(w * 16 + r) * kD + d], wt, acc);
      }
      const int hq = kvh * a.gqa + rr / a.n_q, qi = rr % a.n_q;
      const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
      a.part_o[pi * kD + d] = acc;
      if (d == 0) {
        a.part_m[pi] = M * kLn2;
        a.part_l[pi] = L;
      }
    }
    return;
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rg8 : rg;
    const int lim = half ? lim_g8 : lim_g;
    if (r >= R || t0 > lim) continue;                    // row does not see this chunk
    const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
    const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
    float *po = a.part_o + pi * kD;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      po[8 * j + c] = O[j][2 * half];
      po[8 * j + 4 + c] = O[j][2 * half + 1];
    }
    if (c == 0) {
      a.part_m[pi] = (half ? m_g8 : m_g) * kLn2;         // natural-log units, like the other kernels
      a.part_l[pi] = half ? l_g8 : l_g;
    }
  }
}

template <int KL, int VL, bool PAGED, bool DEC, bool CAP = false>
cudaError_t launch_t(const AttendArgs &a, cudaStream_t st) {
  using G = PGeo<KL, VL>;
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = set_smem_once(configured, attend_prefill_kernel<KL, VL, PAGED, DEC, CAP>, G::SMEM);
  if (e != cudaSuccess) return e;
  const int R = a.gqa * a.n_q;
  cudaLaunchConfig_t cfg = {};
  // Hadamard: more chunk indices for the recent window (unless phase 2 scores it)
  cfg.gridDim = dim3((R + kRows - 1) / kRows, a.n_chunks + (G::HAD && !a.win_in_reduce ? a.n_wchunks : 0) - a.y_base,
                     a.cache.B * a.cache.H);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = G::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_prefill_kernel<KL, VL, PAGED, DEC, CAP>, a);
}

// The launch for a layout pair: contiguous or paged; DEC for one row block when the pair has no
// decode kernel of its own (the only shapes such pairs send here with few rows).
template <int KL, int VL>
cudaError_t launch_pair(const AttendArgs &a, cudaStream_t st) {
  const bool paged = a.cache.page_shift >= 0;
  if (a.cap_scores) {                                    // score capture: one layout of the Hadamard pair
    if constexpr (is_hadamard(KL) && KL == VL) {
      if (paged) return cudaErrorNotSupported;
      if (!decode_kernel(KL, VL) && a.gqa * a.n_q <= 16) return launch_t<KL, VL, false, true, true>(a, st);
      return launch_t<KL, VL, false, false, true>(a, st);
    } else {
      return cudaErrorNotSupported;
    }
  }
  if constexpr (!decode_kernel(KL, VL)) {
    if (a.gqa * a.n_q <= 16)
      return paged ? launch_t<KL, VL, true, true>(a, st) : launch_t<KL, VL, false, true>(a, st);
  }
  return paged ? launch_t<KL, VL, true, false>(a, st) : launch_t<KL, VL, false, false>(a, st);
}

}  // namespace
}  // namespace kvq
