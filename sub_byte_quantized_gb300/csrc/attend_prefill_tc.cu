// Phase 1 of the causal prefill chunk on the fifth-generation tensor cores (tcgen05): the body of a
// Hadamard int4 / int2 cache (one layout in both planes) scored and weighted for many query rows per
// kv head at once (tract discussion #2402, "Architecture: Data flow (decode)": the query rows of an
// appended chunk attend the cached body with their causal limits; "What's done": the body score is
// the exact integer dot int8(q_rot) . int4(k_rot)).
//
// A body CTA = 256 query rows of one (batch, kv head), as two blocks of 128, x one split-K chunk of
// body tokens. The rows are the M side of both products, and the accumulators live in tensor memory
// (TMEM, all 512 columns; per block b):
//   S  = Q8 . K^T       M 128 x N 64 tokens x K 128 dims   -> TMEM columns 64 b .. +63
//   O += P' . V         M 128 x N 128 dims x K 64 tokens   -> TMEM columns 128 + 128 b .. +127, with
//                                                            P' (A) read from columns 384 + 64 b .. +63
// Q8 holds the int8 query codes and K, V the signed 2- or 4-bit codes, all exact in f16 (kind::f16,
// f32 accumulate), so S is the exact integer dot (|dot| < 2^17). score = alpha * s_q * s_k * dot;
// the per-token V scale is folded into the probabilities, P' = p * s_v, which go to the PV product
// as exact f16 hi + lo parts (two MMAs per k-step). The two blocks share every K/V tile and take
// turns on the tensor core: per stage the MMA lane issues, for block 0 and then block 1, the P'V of
// the previous stage (once the block's softmax has stored its P') and then the block's S of this
// stage, so one block's softmax overlaps the other's MMAs.
//
// Warp roles (12 warps), connected by mbarriers; every wait is bounded in time and a CTA whose wait
// gives up writes NaN partials for its rows, so a failure shows in the output instead of hanging:
//   warps 0-7   softmax: warp w serves block w / 4, TMEM lanes (query rows) 32 (w % 4) .. +31; each
//               thread owns a whole row (64 scores per stage); online softmax in base 2 with a lazily
//               moved reference maximum (below), the row's score factor folded into the exponent's
//               fma; P' hi/lo into tensor memory, the A operand of the PV product
//   warp  8     copy: packed K/V rows and per-token scales of each 64-token stage -> a three-slot raw
//               ring (16-byte cp.async, completion counted on the slot's mbarrier)
//   warp  9     one lane issues the MMAs and commits them to mbarriers; the warp owns the TMEM
//               allocation
//   warps 10-11 unpack: raw codes -> f16 code tiles (three tile buffers, 128-byte swizzle), scales ->
//               per-stage arrays
// (Twelve warps put at most three on a scheduler, so a thread may hold 168 registers: the whole-row
// softmax needs them.)
// Operand layouts (shared-memory descriptors, 128-byte swizzle): Q [128 rows][128 dims] per block
// and K [64 tokens][128 dims] K-major in two 64-dim column blocks; V [64 tokens][128 dims] read as
// the MN-major B operand of the PV product; P' in TMEM, lane = row, two tokens per 32-bit column (16
// tokens = 8 columns per MMA k-step; the hi parts of a stage, then its lo parts). Within each 8-dim
// group the tiles keep the unpacker's order (dims 0,4,1,5,2,6,3,7); the output columns follow it.
//
// Lazy rescaling: O and l are kept relative to a reference maximum m per row, which moves only when
// a stage's maximum exceeds it by more than tau (log2 units); then O is rescaled in TMEM (after the
// previous P'V completes). Otherwise p = 2^(s - m) <= 2^tau, and tau is chosen per stage from the
// stage's largest V scale so that p * s_v < 2^15 stays well inside the f16 range (tau <= 8). The
// partial (m, l, O) is exact softmax algebra for any reference, so the result does not depend on
// when m moves; what tau saves is the wait for the tensor core on almost every stage.
//
// The int8 query codes and scales, and the rotated f32 query rows, come from the query-preparation
// kernel launched just before (one pass over the rows instead of one per chunk). The exact-f32
// recent window is scored by more CTAs of the same grid, after the body CTAs in launch order
// (window_chunk below).
#include <cfloat>
#include <climits>

#include "kvq_internal.cuh"
#include "mma_util.cuh"

namespace kvq {
namespace {
using namespace mma;

constexpr int kRows = 128;              // query rows per block = TMEM lanes
constexpr int kBlk = 2;                 // row blocks per CTA, taking turns on the tensor core
constexpr int kCtaRows = kBlk * kRows;
static_assert(kCtaRows == kTcRows, "the chunk planner's rows per CTA");
constexpr int kStage = 64;              // tokens per stage
constexpr int kD = 128;
constexpr int kRing = 3;                // raw stage slots
constexpr int kTB = 3;                  // code tile buffers (the unpackers run up to two stages ahead)
constexpr int kWCopy = 8, kWMma = 9, kWUnp = 10, kUnpThreads = 64;
// Tensor memory (columns of 32 bits, lane = query row of the block): per block b, S at 64 b, O at
// 128 + 128 b, and P' at 384 + 64 b (the f16 hi parts of the stage's 64 tokens in 32 columns, then
// the lo parts), read by the PV product as its A operand.
constexpr int kTmemCols = 512;
__host__ __device__ constexpr uint32_t tm_s(int b) { return 64u * b; }
__host__ __device__ constexpr uint32_t tm_o(int b) { return 128u + 128u * b; }
__host__ __device__ constexpr uint32_t tm_p(int b) { return 384u + 64u * b; }
constexpr int kThreads = kWUnp * 32 + kUnpThreads;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Shared memory (bytes). Swizzled operand tiles start on 1 KB boundaries.
constexpr int kSQ = 0;                          // Q codes f16 per block: two 64-dim column blocks of [128][64]
constexpr int kQBlk = 32768;
constexpr int kST = kSQ + kBlk * kQBlk;         // kTB tile buffers of K (16 KB) + V (16 KB)
constexpr int kTileBuf = 32768;
constexpr int kSTsc = kST + kTB * kTileBuf;     // kTB x (s_k[64], s_v[64]) f32
constexpr int kSRaw = kSTsc + kTB * 512;       // raw ring
template <int L>
struct RawGeo {
  static constexpr int RB = L == KVQ_HAD_INT2 ? 32 : 64;     // payload bytes per token row
  static constexpr int OFF_V = kStage * RB, OFF_SK = 2 * kStage * RB, OFF_SV = OFF_SK + 4 * kStage;
  static constexpr int SLOT = OFF_SV + 4 * kStage;
  static constexpr int SVMAX = kSRaw + kRing * SLOT;          // per tile buffer: the stage's largest s_v, two halves
  static constexpr int BAR = SVMAX + 8 * kTB;                 // mbarriers
  static constexpr int SMEM = BAR + 256;
  static_assert(SMEM <= 227 * 1024, "fits one CTA per SM");
};
static_assert(kST % 1024 == 0, "swizzled tiles on 1 KB boundaries");
// mbarriers (SF, PF, PVD: one per row block)
enum { B_RAWF = 0, B_RAWE = kRing, B_TF = 2 * kRing, B_TE = B_TF + kTB, B_SF = B_TE + kTB, B_PF = B_SF + kBlk,
       B_PVD = B_PF + kBlk, B_DR = B_PVD + kBlk, N_BAR = B_DR + 1 };
static_assert(N_BAR * 8 <= 256, "mbarriers fit");
// Shared-memory matrix descriptor, 128-byte swizzle: start, leading and stride byte offsets.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16: f16 A and B, f32 accumulator, M x N, B K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t id, uint32_t accumulate) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
               ::"r"(d_tmem), "l"(da), "l"(db), "r"(id), "r"(accumulate));
}
// The same with the A operand in tensor memory (lane = row, two f16 values per 32-bit column along K).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t db, uint32_t id, uint32_t accumulate) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
               ::"r"(d_tmem), "r"(a_tmem), "l"(db), "r"(id), "r"(accumulate));
}
// The mbarrier gets one arrival once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(b)));
}
// Byte offset of (row, byte) in a [rows][128 bytes] operand block with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(int row, int byte) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15));
}
// 32 consecutive TMEM columns of this warp's 32 lanes (one f32 per column per thread).
__device__ __forceinline__ void tm_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 64 consecutive TMEM columns of this warp's 32 lanes in one load and one wait; the wait names the
// destination registers, so that no use of them is scheduled above it.
__device__ __forceinline__ void tm_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]),
        "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
        "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]),
        "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
        "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
        "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]),
        "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]),
        "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]),
        "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]),
        "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]),
        "+r"(r[63])
      :
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tm_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
// 16 consecutive TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tm_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// The tiles keep each 8-dim group in the unpacker's pair order: position p of the group holds dim
// perm8(p) = (p >> 1) + 4 (p & 1).

// One chunk of the exact-f32 recent window (kWinChunk tokens of the rotated f32 K/V ring) for the
// CTA's 256 query rows, scored with the prepared rotated f32 query rows on the tensor cores and
// accurate to f32. Every f32 operand is split into f16 hi + lo parts (hi = x rounded to f16, lo =
// the remainder rounded to f16: 22 significant bits), and each product takes three m16n8k16 MMAs
// (lo * hi, hi * lo, hi * hi; the dropped lo * lo term is below 2^-21 of the product). To keep the
// parts inside the f16 range every operand is first scaled by an exact power of two that lands its
// largest magnitude in [2^13, 2^14): each query row and each key token for S = Q K^T (their factors
// multiply each score back), each value dim for O = P V (its factor multiplies the dim's output;
// the probabilities need none, p <= 1). K and V are split once per CTA into f16 planes (V
// transposed, so that a B fragment's two tokens are adjacent); the rows are taken 128 at a time
// (eight warps of 16 rows), each warp scoring its rows against all 64 tokens (eight m16n8
// accumulators: rows g and g + 8 against tokens 8t + 2c and 8t + 2c + 1, g = lane / 4,
// c = lane % 4), taking the softmax over them in one pass and accumulating O[16 rows][128 dims] in
// sixteen more, with the probabilities reused as A fragments in place. These CTAs come last in the
// grid, so they run on the SMs that the body CTAs leave free.
constexpr int kWp = kD + 4;                     // floats per staged f32 row (16 bytes of padding)
constexpr int kKPitch = kD + 8;                 // halves per K plane row (token): 68 words
constexpr int kVPitch = kWinChunk + 8;          // halves per transposed V plane row (dim): 36 words
constexpr int kWinRows = 128 * kWp * 4;                            // 128 staged f32 rows
static_assert(kWinRows == 2 * kWinChunk * kWp * 4, "the chunk's K and V rows fill one staging area");
constexpr int kWinA = 0;                                          // f32 K, V rows, later the second half's query rows
constexpr int kWinB = kWinA + kWinRows;                           // the first half's f32 query rows
constexpr int kWinKh = kWinB + kWinRows;                          // K hi, K lo [token][dim] f16
constexpr int kWinKl = kWinKh + kWinChunk * kKPitch * 2;
constexpr int kWinVh = kWinKl + kWinChunk * kKPitch * 2;          // V hi, V lo [dim][token] f16
constexpr int kWinVl = kWinVh + kD * kVPitch * 2;
constexpr int kWinSc = kWinVl + kD * kVPitch * 2;                 // f32: key factors [64], value-dim factors [128], row factors [2][128]
constexpr int kWinVmax = kWinSc + (kWinChunk + kD + 256) * 4;     // per value dim: largest magnitude (bit pattern)
constexpr int kWinEnd = kWinVmax + kD * 4;
static_assert(kWinEnd <= 227 * 1024, "window chunk fits one CTA");
template <int L>
constexpr int tc_smem() { return RawGeo<L>::SMEM > kWinEnd ? RawGeo<L>::SMEM : kWinEnd; }
// 2^e with e chosen so that m * 2^e lies in [2^13, 2^14) (m > 0; 1 for m = 0), and its inverse
__device__ __forceinline__ void pow2_scale(float m, float &up, float &down) {
  int e = 0;
  if (m > 0.0f) e = min(max(13 - (((__float_as_int(m) >> 23) & 0xFF) - 127), -100), 100);
  up = __int_as_float((e + 127) << 23);
  down = __int_as_float((127 - e) << 23);
}
// (x0, x1) -> f16 pairs hi = rn(x), lo = rn(x - hi)
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  hi = pack_f16x2(x0, x1);
  const float2 h = __half22float2(u32_as_h2(hi));
  lo = pack_f16x2(x0 - h.x, x1 - h.y);
}
template <bool PAGED>
__device__ __forceinline__ void window_chunk(const AttendArgs &a, uint8_t *sm, int row0, int bh, int wc) {
  const CacheView &cv = a.cache;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  constexpr int kWarpsAll = kThreads / 32;
  const int bb = bh / cv.H, kvh = bh - bb * cv.H;
  const SeqLen sl = seq_of_t<PAGED>(a, bb);
  const int R = a.gqa * a.n_q;
  const int t0 = sl.n_body + wc * kWinChunk, t1 = min(sl.kv_len, t0 + kWinChunk);
  const int w_lim = max_row_limit(a, sl, row0, min(row0 + kCtaRows, R));
  if (t0 > w_lim || t0 >= t1) return;                   // no row of this CTA sees the chunk
  const int t_end = min(t1, w_lim + 1);
  float *wa = reinterpret_cast<float *>(sm + kWinA), *wb = reinterpret_cast<float *>(sm + kWinB);
  uint16_t *kh = reinterpret_cast<uint16_t *>(sm + kWinKh), *kl = reinterpret_cast<uint16_t *>(sm + kWinKl);
  uint16_t *vh = reinterpret_cast<uint16_t *>(sm + kWinVh), *vl = reinterpret_cast<uint16_t *>(sm + kWinVl);
  float *kdown = reinterpret_cast<float *>(sm + kWinSc), *vdown = kdown + kWinChunk, *qdown = vdown + kD;
  uint32_t *vmax = reinterpret_cast<uint32_t *>(sm + kWinVmax);
  // the rotated f32 query rows of rows hr0 .. hr0 + 127 into a staging area (zeros past the last row)
  auto stage_rows = [&](float *dst, int hr0) {
    for (int u = tid; u < 128 * 32; u += kThreads) {
      const int lr = u >> 5, pc = u & 31, r = hr0 + lr;
      const bool in = r < R;
      const float *src = a.q_rot + query_row_index(a, bb, kvh, in ? r : hr0) * kD + 4 * pc;
      cp_async16(smem_addr(dst + lr * kWp + 4 * pc), src, in ? 16 : 0);
    }
  };
  // each staged row scaled in place by its power of two (one warp per row)
  auto scale_rows = [&](float *rows, float *down) {
#pragma unroll 4
    for (int lr = warp; lr < 128; lr += kWarpsAll) {
      const float4 x = *reinterpret_cast<const float4 *>(rows + lr * kWp + 4 * lane);
      float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
      for (int k = 16; k >= 1; k >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, k));
      float up, dn;
      pow2_scale(m, up, dn);
      *reinterpret_cast<float4 *>(rows + lr * kWp + 4 * lane) = make_float4(x.x * up, x.y * up, x.z * up, x.w * up);
      if (lane == 0) down[lr] = dn;
    }
  };
  // ---- all copies in flight at once: the chunk's f32 K and V rows from the ring (slot t mod
  // n_recent; zeros past t_end) and the first half's query rows
  for (int u = tid; u < 2 * kWinChunk * 32; u += kThreads) {
    const int pl = u / (kWinChunk * 32), row = (u >> 5) % kWinChunk, pc = u & 31;
    const int t = t0 + row;
    const bool in = t < t_end;
    const float *src = cv.ring[pl] + ((size_t)bh * cv.n_recent + (size_t)((in ? t : t0) % cv.n_recent)) * kD + 4 * pc;
    cp_async16(smem_addr(wa + (pl * kWinChunk + row) * kWp + 4 * pc), src, in ? 16 : 0);
  }
  stage_rows(wb, row0);
  for (int d = tid; d < kD; d += kThreads) vmax[d] = 0u;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  // ---- K: one warp per token, scaled by its power of two and split into the hi / lo planes; V:
  // the largest magnitude of each dim (every warp over its tokens, merged with an atomic max on
  // the bit patterns, which order like non-negative floats)
  for (int t = warp; t < kWinChunk; t += kWarpsAll) {
    const float4 x = *reinterpret_cast<const float4 *>(wa + t * kWp + 4 * lane);
    float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, k));
    float up, down;
    pow2_scale(m, up, down);
    uint32_t h0, l0, h1, l1;
    split_f16x2(x.x * up, x.y * up, h0, l0);
    split_f16x2(x.z * up, x.w * up, h1, l1);
    *reinterpret_cast<uint2 *>(kh + t * kKPitch + 4 * lane) = make_uint2(h0, h1);
    *reinterpret_cast<uint2 *>(kl + t * kKPitch + 4 * lane) = make_uint2(l0, l1);
    if (lane == 0) kdown[t] = down;
  }
  {
    float4 m4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t = warp; t < kWinChunk; t += kWarpsAll) {
      const float4 x = *reinterpret_cast<const float4 *>(wa + (kWinChunk + t) * kWp + 4 * lane);
      m4 = make_float4(fmaxf(m4.x, fabsf(x.x)), fmaxf(m4.y, fabsf(x.y)), fmaxf(m4.z, fabsf(x.z)), fmaxf(m4.w, fabsf(x.w)));
    }
    atomicMax(vmax + 4 * lane, __float_as_uint(m4.x));
    atomicMax(vmax + 4 * lane + 1, __float_as_uint(m4.y));
    atomicMax(vmax + 4 * lane + 2, __float_as_uint(m4.z));
    atomicMax(vmax + 4 * lane + 3, __float_as_uint(m4.w));
  }
  scale_rows(wb, qdown);
  __syncthreads();
  // ---- V: scaled by each dim's power of two, split and transposed (one (dim, token pair) per item)
  for (int u = tid; u < kD * (kWinChunk / 2); u += kThreads) {
    const int d = u & (kD - 1), tp = u / kD;
    float up, down;
    pow2_scale(__uint_as_float(vmax[d]), up, down);
    const float *col = wa + (kWinChunk + 2 * tp) * kWp + d;
    uint32_t h, l;
    split_f16x2(col[0] * up, col[kWp] * up, h, l);
    *reinterpret_cast<uint32_t *>(vh + d * kVPitch + 2 * tp) = h;
    *reinterpret_cast<uint32_t *>(vl + d * kVPitch + 2 * tp) = l;
    if (tp == 0) vdown[d] = down;
  }
  __syncthreads();                                      // the K/V staging area is free
  const bool two = row0 + 128 < R;
  if (two) stage_rows(wa, row0 + 128);                  // the second half's rows, while the first is scored
  const float walpha = a.scale * kLog2e;
  for (int half = 0; half < 2 && row0 + 128 * half < R; ++half) {
    const int hr0 = row0 + 128 * half;
    const float *wf = half ? wa : wb;
    const float *qd = qdown + 128 * half;
    if (half == 1) {
      asm volatile("cp.async.wait_all;" ::: "memory");
      __syncthreads();
      scale_rows(wa, qdown + 128);
      __syncthreads();
    }
    if (warp >= 8) continue;
    const int rg = hr0 + 16 * warp + g, rg8 = rg + 8;
    const int lim_g = rg < R ? row_limit(a, sl, rg % a.n_q) : -1;
    const int lim_g8 = rg8 < R ? row_limit(a, sl, rg8 % a.n_q) : -1;
    if (!__any_sync(0xffffffffu, t0 <= max(lim_g, lim_g8))) continue;
    // ---- S = Q . K^T over eight 16-dim k-steps
    const float *qa = wf + (16 * warp + g) * kWp, *qb = qa + 8 * kWp;
    float sc[kWinChunk / 8][4];
#pragma unroll
    for (int t = 0; t < kWinChunk / 8; ++t)
#pragma unroll
      for (int k = 0; k < 4; ++k) sc[t][k] = 0.0f;
#pragma unroll 2
    for (int ks = 0; ks < kD / 16; ++ks) {
      const int d0 = 16 * ks + 2 * c;
      uint32_t ah[4], al[4];
      const float2 x0 = *reinterpret_cast<const float2 *>(qa + d0), x1 = *reinterpret_cast<const float2 *>(qb + d0);
      const float2 x2 = *reinterpret_cast<const float2 *>(qa + d0 + 8), x3 = *reinterpret_cast<const float2 *>(qb + d0 + 8);
      split_f16x2(x0.x, x0.y, ah[0], al[0]);
      split_f16x2(x1.x, x1.y, ah[1], al[1]);
      split_f16x2(x2.x, x2.y, ah[2], al[2]);
      split_f16x2(x3.x, x3.y, ah[3], al[3]);
#pragma unroll
      for (int t = 0; t < kWinChunk / 8; ++t) {
        const int kr = (8 * t + g) * kKPitch + d0;      // token 8t + g: column g of K^T
        const uint32_t bh0 = *reinterpret_cast<const uint32_t *>(kh + kr), bh1 = *reinterpret_cast<const uint32_t *>(kh + kr + 8);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t *>(kl + kr), bl1 = *reinterpret_cast<const uint32_t *>(kl + kr + 8);
        mma16816(sc[t], al, bh0, bh1);
        mma16816(sc[t], ah, bl0, bl1);
        mma16816(sc[t], ah, bh0, bh1);
      }
    }
    // ---- softmax over the chunk (base 2): sc[t] = (g, 8t+2c), (g, 8t+2c+1), (g+8, 8t+2c), (g+8, 8t+2c+1)
    const float fg = walpha * qd[16 * warp + g], fg8 = walpha * qd[16 * warp + g + 8];
    float m_g = -INFINITY, m_g8 = -INFINITY;
#pragma unroll
    for (int t = 0; t < kWinChunk / 8; ++t) {
      const int ta = t0 + 8 * t + 2 * c, tb = ta + 1;
      const float ka = kdown[8 * t + 2 * c], kb = kdown[8 * t + 2 * c + 1];
      sc[t][0] = (ta < t1 && ta <= lim_g) ? sc[t][0] * ka * fg : -INFINITY;
      sc[t][1] = (tb < t1 && tb <= lim_g) ? sc[t][1] * kb * fg : -INFINITY;
      sc[t][2] = (ta < t1 && ta <= lim_g8) ? sc[t][2] * ka * fg8 : -INFINITY;
      sc[t][3] = (tb < t1 && tb <= lim_g8) ? sc[t][3] * kb * fg8 : -INFINITY;
      m_g = fmaxf(m_g, fmaxf(sc[t][0], sc[t][1]));
      m_g8 = fmaxf(m_g8, fmaxf(sc[t][2], sc[t][3]));
    }
    m_g = fmaxf(m_g, __shfl_xor_sync(0xffffffffu, m_g, 1));
    m_g = fmaxf(m_g, __shfl_xor_sync(0xffffffffu, m_g, 2));
    m_g8 = fmaxf(m_g8, __shfl_xor_sync(0xffffffffu, m_g8, 1));
    m_g8 = fmaxf(m_g8, __shfl_xor_sync(0xffffffffu, m_g8, 2));
    const float mu_g = m_g == -INFINITY ? 0.0f : m_g, mu_g8 = m_g8 == -INFINITY ? 0.0f : m_g8;
    float l_g = 0.0f, l_g8 = 0.0f;
#pragma unroll
    for (int t = 0; t < kWinChunk / 8; ++t) {
      sc[t][0] = ex2(sc[t][0] - mu_g);
      sc[t][1] = ex2(sc[t][1] - mu_g);
      sc[t][2] = ex2(sc[t][2] - mu_g8);
      sc[t][3] = ex2(sc[t][3] - mu_g8);
      l_g += sc[t][0] + sc[t][1];
      l_g8 += sc[t][2] + sc[t][3];
    }
    l_g += __shfl_xor_sync(0xffffffffu, l_g, 1);
    l_g += __shfl_xor_sync(0xffffffffu, l_g, 2);
    l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 1);
    l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 2);
    // ---- O = P . V over four 16-token k-steps: the probabilities of tiles 2kk and 2kk + 1 are the
    // A fragment as they stand (k = 2c, 2c + 1 <-> tile 2kk's tokens, k = 2c + 8, 2c + 9 <-> tile
    // 2kk + 1's); B fragments from the transposed V planes
    float o[kD / 8][4];
#pragma unroll
    for (int n = 0; n < kD / 8; ++n)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[n][k] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < kWinChunk / 16; ++kk) {
      uint32_t ph[4], pl[4];
      split_f16x2(sc[2 * kk][0], sc[2 * kk][1], ph[0], pl[0]);
      split_f16x2(sc[2 * kk][2], sc[2 * kk][3], ph[1], pl[1]);
      split_f16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[2], pl[2]);
      split_f16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
      for (int n = 0; n < kD / 8; ++n) {
        const int vr = (8 * n + g) * kVPitch + 16 * kk + 2 * c;   // dim 8n + g, tokens 16kk + 2c, +1
        const uint32_t bh0 = *reinterpret_cast<const uint32_t *>(vh + vr), bh1 = *reinterpret_cast<const uint32_t *>(vh + vr + 8);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t *>(vl + vr), bl1 = *reinterpret_cast<const uint32_t *>(vl + vr + 8);
        mma16816(o[n], pl, bh0, bh1);
        mma16816(o[n], ph, bl0, bl1);
        mma16816(o[n], ph, bh0, bh1);
      }
    }
    // ---- partials of the rows that see the chunk (partial index n_chunks + wc)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = hh ? rg8 : rg, lim = hh ? lim_g8 : lim_g;
      if (r >= R || t0 > lim) continue;
      const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
      const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + a.n_chunks + wc;
      float *po = a.part_o + pi * kD;
#pragma unroll
      for (int n = 0; n < kD / 8; ++n)
        *reinterpret_cast<float2 *>(po + 8 * n + 2 * c) =
            make_float2(o[n][2 * hh] * vdown[8 * n + 2 * c], o[n][2 * hh + 1] * vdown[8 * n + 2 * c + 1]);
      if (c == 0) {
        a.part_m[pi] = (hh ? m_g8 : m_g) * kLn2;        // natural-log units, like the other kernels
        a.part_l[pi] = hh ? l_g8 : l_g;
      }
    }
  }
}

template <int L, bool PAGED, bool CAP>
__global__ void __launch_bounds__(kThreads, 1) attend_prefill_tc_kernel(AttendArgs a) {
  using RG = RawGeo<L>;
  static_assert(!CAP || !PAGED, "score capture: contiguous cache");
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint32_t tmem_base;
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the query codes come from the preceding kernel
#endif
  const CacheView &cv = a.cache;
  const int heads = cv.B * cv.H;
  if ((int)blockIdx.z >= heads) {
    // window chunks: the CTAs after the body's, (z - heads, y) numbering (head, window chunk) pairs
    const int wl = ((int)blockIdx.z - heads) * (int)gridDim.y + (int)blockIdx.y;
    if (!CAP && wl < heads * a.n_wchunks)
      window_chunk<PAGED>(a, sm, blockIdx.x * kCtaRows, wl / a.n_wchunks, wl % a.n_wchunks);
    return;
  }
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + RG::BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = blockIdx.x * kCtaRows, chunk_id = blockIdx.y, bh = blockIdx.z;
  const int bb = bh / cv.H, kvh = bh - bb * cv.H;
  const SeqLen sl = seq_of_t<PAGED>(a, bb);
  const int R = a.gqa * a.n_q;
  const int t0 = chunk_id * sl.chunk, t1 = min(sl.n_body, t0 + sl.chunk);
  const int w_lim = max_row_limit(a, sl, row0, min(row0 + kCtaRows, R));
  if (t0 > w_lim || t0 >= t1) return;                   // no row of this CTA sees the chunk
  const int t_end = min(t1, w_lim + 1);
  const int n_st = (t_end - t0 + kStage - 1) / kStage;
  const int nblk = R - row0 > kRows ? 2 : 1;            // row blocks with live rows
  const size_t head_row0 = (size_t)bh * cv.cap;

  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      bar_init(bar + B_RAWF + i, 32);                   // the copy lanes' cp.async completions
      bar_init(bar + B_RAWE + i, kUnpThreads);
    }
    for (int i = 0; i < kTB; ++i) {
      bar_init(bar + B_TF + i, kUnpThreads);
      bar_init(bar + B_TE + i, 1);
    }
    for (int i = 0; i < kBlk; ++i) {
      bar_init(bar + B_SF + i, 1);
      bar_init(bar + B_PF + i, 128);                    // the block's softmax threads
      bar_init(bar + B_PVD + i, 1);
    }
    bar_init(bar + B_DR, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // ---- query codes of the CTA's rows as exact f16 in the tiles' dim order: each unit is one
  // 8-dim group of one row (16 int8 -> one 16-byte store of four (dim i, dim i + 4) pairs)
  for (int u = tid; u < kCtaRows * 16; u += kThreads) {
    const int cr = u >> 4, gi = u & 15, r = row0 + cr;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (r < R) {
      const uint2 c8 = *reinterpret_cast<const uint2 *>(a.q8 + query_row_index(a, bb, kvh, r) * kD + 8 * gi);
      const int8_t *cb = reinterpret_cast<const int8_t *>(&c8);
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = pack_f16x2((float)cb[k], (float)cb[k + 4]);
    }
    *reinterpret_cast<uint4 *>(sm + kSQ + (cr >> 7) * kQBlk + (gi >> 3) * 16384 + sw128(cr & 127, 16 * (gi & 7))) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (warp == kWMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor-core reads
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = tmem_base;
  bool ok = true;

  if (warp == kWCopy) {
    // ---------------- copy: stage j -> raw slot j % kRing; rows past t_end are zero-filled
    for (int j = 0; j < n_st && ok; ++j) {
      const int slot = j % kRing;
      if (j >= kRing) ok = bar_wait_relaxed(bar + B_RAWE + slot, ((j / kRing) - 1) & 1);
      if (!ok) break;
      const int ts = t0 + j * kStage;
      const size_t r0 = cache_row_t<PAGED>(cv, bb, kvh, head_row0, ts);   // 64 consecutive plane rows
      uint8_t *raw = sm + kSRaw + slot * RG::SLOT;
      const uint8_t *kp = cv.payload[0] + r0 * RG::RB, *vp = cv.payload[1] + r0 * RG::RB;
#pragma unroll
      for (int k = 0; k < kStage * RG::RB / 16 / 32; ++k) {
        const int q = lane + 32 * k;                     // 16-byte piece q of the stage's rows
        const bool in = ts + q / (RG::RB / 16) < t_end;
        cp_async16(smem_addr(raw + 16 * q), kp + (in ? 16 * q : 0), in ? 16 : 0);
        cp_async16(smem_addr(raw + RG::OFF_V + 16 * q), vp + (in ? 16 * q : 0), in ? 16 : 0);
      }
      const float *skp = static_cast<const float *>(cv.scale[0]) + r0;
      const float *svp = static_cast<const float *>(cv.scale[1]) + r0;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int t = lane + 32 * k;
        const bool in = ts + t < t_end;
        cp_async4(smem_addr(raw + RG::OFF_SK + 4 * t), skp + (in ? t : 0), in ? 4 : 0);
        cp_async4(smem_addr(raw + RG::OFF_SV + 4 * t), svp + (in ? t : 0), in ? 4 : 0);
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar + B_RAWF + slot)) : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp >= kWUnp) {
    // ---------------- unpack: raw slot -> tile buffer j % kTB (each thread 16 (row, 8-dim group) units per plane)
    const int ut = tid - kWUnp * 32;
    for (int j = 0; j < n_st && ok; ++j) {
      const int slot = j % kRing, tb = j % kTB;
      ok = bar_wait_relaxed(bar + B_RAWF + slot, (j / kRing) & 1);
      if (ok && j >= kTB) ok = bar_wait_relaxed(bar + B_TE + tb, ((j - kTB) / kTB) & 1);   // P'V of stage j - kTB done
      if (!ok) break;
      const uint8_t *raw = sm + kSRaw + slot * RG::SLOT;
      uint8_t *tk = sm + kST + tb * kTileBuf, *tv = tk + 16384;
#pragma unroll
      for (int k = 0; k < kStage * 16 / kUnpThreads; ++k) {
        const int u = ut + kUnpThreads * k;
        const int row = u >> 4, gi = u & 15;
        const uint32_t off = (uint32_t)(gi >> 3) * 8192 + sw128(row, 16 * (gi & 7));
        uint32_t o[4];
        if constexpr (L == KVQ_HAD_INT2) {
          unpack8_s2(*reinterpret_cast<const uint16_t *>(raw + row * RG::RB + 2 * gi), o);
          *reinterpret_cast<uint4 *>(tk + off) = make_uint4(o[0], o[1], o[2], o[3]);
          unpack8_s2(*reinterpret_cast<const uint16_t *>(raw + RG::OFF_V + row * RG::RB + 2 * gi), o);
          *reinterpret_cast<uint4 *>(tv + off) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          unpack8_q4(*reinterpret_cast<const uint32_t *>(raw + row * RG::RB + 4 * gi), o);
          *reinterpret_cast<uint4 *>(tk + off) = make_uint4(o[0], o[1], o[2], o[3]);
          unpack8_q4(*reinterpret_cast<const uint32_t *>(raw + RG::OFF_V + row * RG::RB + 4 * gi), o);
          *reinterpret_cast<uint4 *>(tv + off) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      // per-stage scales: s_k[0..63], s_v[0..63]; each unpack warp also records the largest s_v of
      // its 32 tokens (non-negative floats order like their bit patterns)
      static_assert(kUnpThreads == kStage, "one key and one value scale per unpack thread");
      const float sck = *reinterpret_cast<const float *>(raw + RG::OFF_SK + 4 * ut);
      const float scv = *reinterpret_cast<const float *>(raw + RG::OFF_SV + 4 * ut);
      reinterpret_cast<float *>(sm + kSTsc + tb * 512)[ut] = sck;
      reinterpret_cast<float *>(sm + kSTsc + tb * 512)[64 + ut] = scv;
      const uint32_t mxv = __reduce_max_sync(0xffffffffu, __float_as_uint(fmaxf(scv, 0.0f)));
      if (lane == 0) reinterpret_cast<uint32_t *>(sm + RG::SVMAX)[2 * tb + (ut >> 5)] = mxv;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      bar_arrive(bar + B_RAWE + slot);
      bar_arrive(bar + B_TF + tb);
    }
  } else if (warp == kWMma) {
    // ---------------- MMA issue (one thread). Per stage j and block b: P'V of stage j - 1 (once the
    // block's softmax has stored its P'), then S of stage j into the same block's S columns, which
    // that softmax has finished reading. The blocks take turns, so while one block's softmax works
    // the tensor core serves the other.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc(kRows, kStage, false), id_o = idesc(kRows, kD, true);
      auto pv = [&](int b, int i) {
        ok = ok && bar_wait(bar + B_PF + b, i & 1);
        if (!ok) return;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t vt = smem_addr(sm + kST + (i % kTB) * kTileBuf + 16384);
#pragma unroll
        for (int ks = 0; ks < kStage / 16; ++ks) {
          const uint64_t db = sdesc(vt + 2048 * ks, 8192, 1024);
          const uint32_t pa = tmem + tm_p(b) + 8 * ks;    // 16 tokens = 8 columns
          mma_f16_ta(tmem + tm_o(b), pa, db, id_o, (i > 0 || ks > 0) ? 1u : 0u);
          mma_f16_ta(tmem + tm_o(b), pa + 32, db, id_o, 1u);
        }
        mma_commit(bar + B_PVD + b);                    // O holds stage i; P' free
        if (b == nblk - 1) mma_commit(bar + B_TE + (i % kTB));   // tile buffer free
      };
      for (int j = 0; j < n_st && ok; ++j) {
        const int tb = j % kTB;
        ok = bar_wait(bar + B_TF + tb, (j / kTB) & 1);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t kt = smem_addr(sm + kST + tb * kTileBuf);
        for (int b = 0; b < nblk && ok; ++b) {
          if (j >= 1) pv(b, j - 1);
          if (!ok) break;
          const uint32_t qt = smem_addr(sm + kSQ + b * kQBlk);
#pragma unroll
          for (int kb = 0; kb < kD / 16; ++kb) {
            const uint64_t da = sdesc(qt + (kb >> 2) * 16384 + 32 * (kb & 3), 16, 1024);
            const uint64_t db = sdesc(kt + (kb >> 2) * 8192 + 32 * (kb & 3), 16, 1024);
            mma_f16(tmem + tm_s(b), da, db, id_s, kb > 0 ? 1u : 0u);
          }
          mma_commit(bar + B_SF + b);
        }
      }
      for (int b = 0; b < nblk && ok; ++b) pv(b, n_st - 1);
      mma_commit(bar + B_DR);                           // drain: every MMA issued above completes
      if (!bar_wait(bar + B_DR, 0)) ok = false;
    }
  } else if ((warp >> 2) < nblk) {
    // ---------------- softmax: block b = warp / 4, row lr = TMEM lane, whole rows (64 scores per stage)
    const int b = warp >> 2, q4 = warp & 3;
    const int lr = 32 * q4 + lane, r = row0 + kRows * b + lr;
    const bool live = r < R;
    const int lim = live ? row_limit(a, sl, r % a.n_q) : -1;
    const size_t qrow = live ? query_row_index(a, bb, kvh, r) : 0;
    // the row's score factor alpha * s_q * log2(e) (never 0, so that a masked -inf stays -inf in
    // the exponent's fma; a zero factor only arises with all-zero query codes, whose dots are 0)
    float arow = live ? a.scale * a.s_q[qrow] * kLog2e : 1.0f;
    if (arow == 0.0f) arow = 1e-30f;
    const bool fneg = arow < 0.0f;                      // the maximum of z * arow is then at the minimum z
    const float fabs_row = fabsf(arow);
    if (CAP && live && chunk_id == 0) a.cap_sq[qrow] = a.s_q[qrow];
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    float m = -INFINITY, l = 0.0f;
    for (int j = 0; j < n_st && ok; ++j) {
      const int tb = j % kTB, ts = t0 + j * kStage;
      ok = __all_sync(0xffffffffu, bar_wait(bar + B_TF + tb, (j / kTB) & 1) && bar_wait(bar + B_SF + b, j & 1));
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;");
      const float *tsc = reinterpret_cast<const float *>(sm + kSTsc + tb * 512);
      float s[64];
      tm_ld64(tmem + lane_base + tm_s(b), s);
      if constexpr (CAP) {
        if (live) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (ts + i < t_end) a.cap_scores[qrow * a.n_body + ts + i] = __float2int_rn(s[i]);
        }
      }
      // z = dot * s_k (key scales as broadcast 16-byte loads); the score in log2 units is z * arow,
      // which enters the exponent as one fma
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const float4 k4 = *reinterpret_cast<const float4 *>(tsc + i);
        s[i] *= k4.x;
        s[i + 1] *= k4.y;
        s[i + 2] *= k4.z;
        s[i + 3] *= k4.w;
      }
      if (ts + 63 > lim || ts + 64 > t_end) {           // a masked token's score must be -inf
        const float zmask = fneg ? INFINITY : -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (!(ts + i <= lim && ts + i < t_end)) s[i] = zmask;
      }
      float mx16[16];                                   // max of sign(arow) * z as a tree
      if (!fneg) {
#pragma unroll
        for (int i = 0; i < 16; ++i) mx16[i] = fmaxf(fmaxf(s[i], s[i + 16]), fmaxf(s[i + 32], s[i + 48]));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) mx16[i] = fmaxf(fmaxf(-s[i], -s[i + 16]), fmaxf(-s[i + 32], -s[i + 48]));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) mx16[i] = fmaxf(fmaxf(mx16[i], mx16[i + 4]), fmaxf(mx16[i + 8], mx16[i + 12]));
      const float ztop = fmaxf(fmaxf(mx16[0], mx16[1]), fmaxf(mx16[2], mx16[3]));
      const float mx = ztop == -INFINITY ? -INFINITY : fabs_row * ztop;   // the stage's row maximum
      // tau: p * s_v < 2^15 for p <= 2^tau (svmax < 2^(e + 1))
      const float *svm = reinterpret_cast<const float *>(sm + RG::SVMAX) + 2 * tb;
      const float svmax = fmaxf(svm[0], svm[1]);
      const int e = (int)((__float_as_uint(svmax) >> 23) & 0xFF) - 127;
      const float tau = (float)min(8, max(0, 14 - e));
      const bool bump = mx > m + tau;                   // m = -inf: the first visible stage
      const float m_new = bump ? mx : m;
      const float mu = m_new == -INFINITY ? 0.0f : m_new;
      const float corr = bump ? ex2(m - mu) : 1.0f;     // m = -inf -> 0
      if (j >= 1) {
        // P'V of stage j - 1 has read P' and updated O (it precedes S of stage j on the tensor core)
        ok = __all_sync(0xffffffffu, bar_wait(bar + B_PVD + b, (j - 1) & 1));
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        if (__any_sync(0xffffffffu, bump && m != -INFINITY)) {   // rescale the block's O rows
#pragma unroll
          for (int c = 0; c < kD; c += 32) {
            float o[32];
            tm_ld32(tmem + lane_base + tm_o(b) + c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= corr;
            tm_st32(tmem + lane_base + tm_o(b) + c, o);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
      }
      // P' = p * s_v as exact f16 hi + lo, tokens 32 hh + 8 k .. +7, in two halves of 32 tokens
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};              // four independent partial sums
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t hiv[16], lov[16];                      // P' of this half's 32 tokens (TMEM form)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 va = *reinterpret_cast<const float4 *>(tsc + 64 + 32 * hh + 8 * k);   // value scales
          const float4 vb = *reinterpret_cast<const float4 *>(tsc + 64 + 32 * hh + 8 * k + 4);
          const float svv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int i = 32 * hh + 8 * k + 2 * e2;
            const float p0 = ex2(fmaf(s[i], arow, -mu)), p1 = ex2(fmaf(s[i + 1], arow, -mu));
            sum4[e2] += p0 + p1;
            const float q0 = p0 * svv[2 * e2], q1 = p1 * svv[2 * e2 + 1];
            const uint32_t hi = pack_f16x2(q0, q1);
            const float2 hf = __half22float2(u32_as_h2(hi));
            hiv[4 * k + e2] = hi;
            lov[4 * k + e2] = pack_f16x2(q0 - hf.x, q1 - hf.y);
          }
        }
        // tokens 32 hh .. +31 are TMEM columns 16 hh .. +15 of the hi half and of the lo half
        tm_st16(tmem + lane_base + tm_p(b) + 16 * hh, hiv);
        tm_st16(tmem + lane_base + tm_p(b) + 32 + 16 * hh, lov);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      l = l * corr + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
      m = m_new;
      asm volatile("tcgen05.fence::before_thread_sync;");   // the TMEM stores above precede the MMAs
      bar_arrive(bar + B_PF + b);
    }
    if (ok) ok = __all_sync(0xffffffffu, bar_wait(bar + B_PVD + b, (n_st - 1) & 1));
    if (ok) {                                           // warp-uniform: the TMEM loads need the whole warp
      asm volatile("tcgen05.fence::after_thread_sync;");
      const bool write = live && t0 <= lim;
      const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
      const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
      float *po = a.part_o + pi * kD;
#pragma unroll
      for (int c = 0; c < kD; c += 32) {
        float o[32];
        tm_ld32(tmem + lane_base + tm_o(b) + c, o);
        if (write) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {              // position 8 g8 + p holds dim 8 g8 + perm8(p)
            const float *x = o + 8 * g8;
            *reinterpret_cast<float4 *>(po + c + 8 * g8) = make_float4(x[0], x[2], x[4], x[6]);
            *reinterpret_cast<float4 *>(po + c + 8 * g8 + 4) = make_float4(x[1], x[3], x[5], x[7]);
          }
        }
      }
      if (write) {
        a.part_m[pi] = m * kLn2;                        // natural-log units, like the other kernels
        a.part_l[pi] = l;
      }
    }
  }
  // a wait that gave up anywhere in the CTA: its rows' partials become NaN (m = 0, l = NaN), which
  // the reduce turns into NaN outputs
  const bool failed = __syncthreads_or(!ok);
  if (failed && warp < 8) {
    const int r = row0 + kRows * (warp >> 2) + 32 * (warp & 3) + lane;
    if (r < R && t0 <= row_limit(a, sl, r % a.n_q)) {
      const int hq = kvh * a.gqa + r / a.n_q, qi = r % a.n_q;
      const size_t pi = (((size_t)bb * a.Hq + hq) * a.n_q + qi) * a.C + chunk_id;
      for (int d = 0; d < kD; ++d) a.part_o[pi * kD + d] = __int_as_float(0x7fc00000);
      a.part_m[pi] = 0.0f;
      a.part_l[pi] = __int_as_float(0x7fc00000);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  if (warp == kWMma) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
}

template <int L, bool PAGED, bool CAP>
cudaError_t launch_tc(const AttendArgs &a, cudaStream_t st) {
  static std::atomic<bool> configured[kMaxDevices];
  cudaError_t e = set_smem_once(configured, attend_prefill_tc_kernel<L, PAGED, CAP>, tc_smem<L>());
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  // body CTAs (row block, chunk, head), then the window CTAs in extra z slices
  const int heads = a.cache.B * a.cache.H;
  const int wz = CAP ? 0 : (heads * a.n_wchunks + a.n_chunks - 1) / a.n_chunks;
  cfg.gridDim = dim3((a.gqa * a.n_q + kCtaRows - 1) / kCtaRows, a.n_chunks, heads + wz);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = tc_smem<L>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_prefill_tc_kernel<L, PAGED, CAP>, a);
}

template <int L>
cudaError_t launch_layout(const AttendArgs &a, cudaStream_t st) {
  const bool paged = a.cache.page_shift >= 0;
  if (a.cap_scores) return paged ? cudaErrorNotSupported : launch_tc<L, false, true>(a, st);
  return paged ? launch_tc<L, true, false>(a, st) : launch_tc<L, false, false>(a, st);
}

}  // namespace

cudaError_t launch_attend_prefill_tc_body(const AttendArgs &a, cudaStream_t st) {
  if (a.cache.layout == KVQ_HAD_INT2) return launch_layout<KVQ_HAD_INT2>(a, st);
  return launch_layout<KVQ_HAD_INT4>(a, st);
}

}  // namespace kvq
