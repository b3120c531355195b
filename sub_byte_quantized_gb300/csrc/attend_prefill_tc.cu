// Phase 1 of the causal prefill chunk on the fifth-generation tensor cores (tcgen05): the body of a
// Hadamard int4 / int2 cache (one layout in both planes) scored and weighted for many query rows per
// kv head at once (tract discussion #2402, "Architecture: Data flow (decode)": the query rows of an
// appended chunk attend the cached body with their causal limits; "What's done": the body score is
// the exact integer dot int8(q_rot) . int4(k_rot)).
//
// One CTA = 128 query rows of one (batch, kv head) x one split-K chunk of body tokens. The rows are
// the M side of both products, and the accumulators live in tensor memory (TMEM, 256 columns):
//   S  = Q8 . K^T       M 128 x N 64 tokens x K 128 dims   -> TMEM columns 0-63 / 64-127 (two stages)
//   O += P' . V         M 128 x N 128 dims x K 64 tokens   -> TMEM columns 128-255, with P' (A) read
//                                                            from TMEM columns 256-383 (two stages)
// Q8 holds the int8 query codes and K, V the signed 2- or 4-bit codes, all exact in f16 (kind::f16,
// f32 accumulate), so S is the exact integer dot (|dot| < 2^17). score = alpha * s_q * s_k * dot;
// the per-token V scale is folded into the probabilities, P' = p * s_v, which go to the PV product
// as exact f16 hi + lo parts (two MMAs per k-step).
//
// Warp roles (14 warps), connected by mbarriers; every wait is bounded in time and a CTA whose wait
// gives up writes NaN partials for its rows, so a failure shows in the output instead of hanging:
//   warps 0-7   softmax: warp w serves TMEM lanes (query rows) 32 (w % 4) .. +31 and the column half
//               w / 4 (S columns 32 h .. +31, O columns 64 h .. +63); the two halves of a row exchange
//               their maxima through shared memory; online softmax in base 2 with a lazily moved
//               reference maximum (below), the row's score factor folded into the exponent's fma;
//               P' hi/lo into tensor memory (two stage buffers), the A operand of the PV product
//   warp  8     copy: packed K/V rows and per-token scales of each 64-token stage -> a three-slot raw
//               ring (16-byte cp.async, completion counted on the slot's mbarrier)
//   warp  9     one lane issues the MMAs (S of stage j, then P'V of stage j - 1) and commits them to
//               mbarriers; the warp owns the TMEM allocation
//   warps 10-13 unpack: raw codes -> f16 code tiles (two tile buffers, 128-byte swizzle), scales ->
//               per-stage arrays
// Operand layouts (shared-memory descriptors, 128-byte swizzle): Q [128 rows][128 dims] and K
// [64 tokens][128 dims] K-major in two 64-dim column blocks; V [64 tokens][128 dims] read as the
// MN-major B operand of the PV product; P' in TMEM, lane = row, two tokens per 32-bit column (16
// tokens = 8 columns per MMA k-step; the hi parts of a stage, then its lo parts). Within each 8-dim group
// the tiles keep the unpacker's order (dims 0,4,1,5,2,6,3,7); the output columns follow it.
//
// Lazy rescaling: O and l are kept relative to a reference maximum m per row, which moves only when
// a stage's maximum exceeds it by more than tau (log2 units); then O is rescaled in TMEM (after the
// previous P'V completes). Otherwise p = 2^(s - m) <= 2^tau, and tau is chosen per stage from the
// stage's largest V scale so that p * s_v < 2^15 stays well inside the f16 range (tau <= 8). The
// partial (m, l, O) is exact softmax algebra for any reference, so the result does not depend on
// when m moves; what tau saves is the wait for the tensor core on almost every stage.
//
// The int8 query codes and scales come from the query-preparation kernel launched just before (one
// pass over the rows instead of one per chunk); the exact-f32 recent window is scored by the
// row-side kernel's window chunks, launched after this one.
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
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + RG::BAR);
  const CacheView &cv = a.cache;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = blockIdx.x * kCtaRows, chunk_id = blockIdx.y, bh = blockIdx.z;
  const int bb = bh / cv.H, kvh = bh - bb * cv.H;
  const SeqLen sl = seq_of_t<PAGED>(a, bb);
  const int R = a.gqa * a.n_q;
  const int t0 = chunk_id * sl.chunk, t1 = min(sl.n_body, t0 + sl.chunk);
  int w_lim = -1;
  for (int r = row0; r < min(row0 + kCtaRows, R); ++r) w_lim = max(w_lim, row_limit(a, sl, r % a.n_q));
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
      {
        float h0[32], h1[32];
        tm_ld32(tmem + lane_base + tm_s(b), h0);
        tm_ld32(tmem + lane_base + tm_s(b) + 32, h1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = h0[i];
          s[32 + i] = h1[i];
        }
      }
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
  cudaError_t e = set_smem_once(configured, attend_prefill_tc_kernel<L, PAGED, CAP>, RawGeo<L>::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.gqa * a.n_q + kCtaRows - 1) / kCtaRows, a.n_chunks, a.cache.B * a.cache.H);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = RawGeo<L>::SMEM;
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
