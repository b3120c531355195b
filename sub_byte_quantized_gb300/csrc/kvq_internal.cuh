// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <atomic>
#include <climits>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq.h"

namespace kvq {

constexpr int kBlock = 32;          // values per Q4_0 / Q6_0 / Q8_0 / asymmetric block
constexpr int kLastLayout = KVQ_HAD_INT2;
// Tokens per chunk of the exact-f32 window (a wide window is split over several chunks).
constexpr int kWinChunk = 64;
// Layouts in the fixed Hadamard basis: one f32 scale per token, rotated query, optional f32 window.
__host__ __device__ constexpr bool is_hadamard(int layout) {
  return layout == KVQ_HAD_INT4 || layout == KVQ_HAD_INT2;
}
constexpr int kMaxDevices = 64;     // per-device one-time kernel attribute set-up

// Tensor-core phase 1: resident CTAs (of four warps) per SM the kernel is built for; the
// automatic split-K chunk sizes one wave of that many warps.
#ifndef KVQ_MMA_MIN_BLOCKS
#define KVQ_MMA_MIN_BLOCKS 3
#endif
constexpr int kMmaWarpsPerSm = 4 * KVQ_MMA_MIN_BLOCKS;
// Warp-specialised tensor-core phase 1 (CTAs of eight warps, two per SM; the automatic chunk gives
// every resident CTA one chunk): used for the asymmetric layout, whose per-warp kernel runs out of
// registers; Q4_0 and the Hadamard body keep the per-warp kernel (faster there on this part).
constexpr int kMma4CtasPerSm = 2;
__host__ __device__ constexpr bool uses_mma4(int layout) { return layout == KVQ_ASYM4_G32; }
// Tensor-core phase 1 for Q6_0: resident CTAs (of eight warps) per SM (shared-memory ring of three
// 64-token stages plus the score exchange: 92 KB at D = 256, 53 KB at D = 128).
__host__ __device__ constexpr int kMmaQ6CtasPerSm(int D) { return D == 256 ? 2 : 2; }
// Shapes the Q6_0 tensor-core kernel covers: head_dim 128 or 256, any rows per kv head (gqa * n_q)
// in groups of four.
__host__ __device__ constexpr bool mma_q6_shape(int D, int rows) { return (D == 128 || D == 256) && rows >= 1; }
// tcgen05 kernel for the body of many-row Hadamard calls (causal prefill chunks): 256 query rows per
// CTA (two blocks of 128), one CTA per SM; one Hadamard layout in both planes, head_dim 128, more than
// 64 rows per kv head.
constexpr int kTcRows = 256;
__host__ __device__ constexpr bool tc_prefill_shape(int kl, int vl, int D, int rows) {
  return kl == vl && is_hadamard(kl) && D == 128 && rows > 64;
}
// Row-side tensor-core kernel: 64 query rows per CTA; three resident CTAs per SM for the Hadamard
// layout, two for Q4_0 / asymmetric (their value tiles are hi + lo pairs).
constexpr int kPrefillRows = 64;
constexpr int kPrefillCtasPerSm = 3;
#ifndef KVQ_PREFILL_BLOCK_LAYOUTS
#define KVQ_PREFILL_BLOCK_LAYOUTS 1
#endif
// (K layout, V layout) pairs the row-side kernel is built for: one layout of Q4_0, asym, Q6_0, Q8_0,
// Hadamard int4 / int2 in both planes, or the mixed pairs 4-bit keys + Q8_0 values and int2 key
// body + int4 value body.
__host__ __device__ constexpr bool prefill_pair(int kl, int vl) {
  return (kl == vl && (kl == KVQ_HAD_INT4 || kl == KVQ_HAD_INT2 || kl == KVQ_Q8_0 ||
                       (KVQ_PREFILL_BLOCK_LAYOUTS && (kl == KVQ_Q4_0 || kl == KVQ_ASYM4_G32 || kl == KVQ_Q6_0)))) ||
         (vl == KVQ_Q8_0 && (kl == KVQ_Q4_0 || kl == KVQ_ASYM4_G32)) || (kl == KVQ_HAD_INT2 && vl == KVQ_HAD_INT4);
}
// Pairs with a decode kernel of their own (at most eight query rows per kv head; Q6_0: its kernel
// takes groups of four rows).
__host__ __device__ constexpr bool decode_kernel(int kl, int vl) {
  return (kl == vl && (kl == KVQ_Q4_0 || kl == KVQ_ASYM4_G32 || kl == KVQ_HAD_INT4 || kl == KVQ_HAD_INT2 ||
                       kl == KVQ_Q8_0 || kl == KVQ_Q6_0)) ||
         (kl == KVQ_Q4_0 && vl == KVQ_Q8_0);
}
// The row-side kernel takes many query rows per kv head, and every row count of the pairs that
// have no decode kernel.
__host__ __device__ constexpr bool prefill_shape(int kl, int vl, int D, int rows) {
  return D == 128 && prefill_pair(kl, vl) && (rows > 8 || !decode_kernel(kl, vl));
}
// The row-side kernel's decode form (DEC: one block of at most 16 rows, the warps split the tokens).
// Its Hadamard window is scored in phase 2, one CTA per query row, like the decode kernels'.
__host__ __device__ constexpr bool dec_shape(int kl, int vl, int D, int rows) {
  return prefill_shape(kl, vl, D, rows) && rows <= 16 && !decode_kernel(kl, vl);
}

// The opt-in dynamic shared-memory size of `kernel` is a per-device function attribute: set it
// the first time the kernel is launched on each device. `done` is the caller's flag array (one
// per kernel); threads that race on a first launch may both set the attribute, which is harmless.
template <class K>
inline cudaError_t set_smem_once(std::atomic<bool> (&done)[kMaxDevices], K *kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

// Device-side view of a cache; index 0 = K, 1 = V. Rows of the payload / scale / zero planes:
// contiguous [B][H][cap] (page_shift < 0), or a paged pool [n_pages][H][page] addressed through
// the block table [B][table_stride] (page = 1 << page_shift tokens, at least 64; cap is then the
// logical capacity of one sequence, table_stride pages). The ring is per sequence either way.
struct CacheView {
  int layout, B, H, D, cap, n_recent;      // layout: the K plane's (and, unless mixed, V's)
  int row_bytes;
  int v_layout, v_row_bytes;               // the V plane's layout and row bytes
  uint8_t *payload[2];
  void *scale[2];
  __half *zero[2];
  float *ring[2];
  int page_shift, table_stride, n_pages;
  const int32_t *table;
};
constexpr int kMinPageShift = 6;    // pages of at least 64 tokens: a 64-token stage never straddles two

// Plane row of token t of (batch bb, kv head kvh). A table entry outside the pool is clamped into
// it (the caller guarantees valid entries; the clamp only keeps every access inside the pool).
__device__ __forceinline__ size_t cache_row_paged(const CacheView &c, int bb, int kvh, int t) {
  int pg = __ldg(c.table + (size_t)bb * c.table_stride + (t >> c.page_shift));
  pg = min(max(pg, 0), c.n_pages - 1);
  return (((size_t)pg * c.H + kvh) << c.page_shift) + (t & ((1 << c.page_shift) - 1));
}
__device__ __forceinline__ size_t cache_row(const CacheView &c, int bb, int kvh, int t) {
  if (c.page_shift < 0) return ((size_t)bb * c.H + kvh) * c.cap + t;
  return cache_row_paged(c, bb, kvh, t);
}
// The same with the layout fixed at compile time (the streaming kernels are built for both):
// contiguous rows are head_row0 + t with head_row0 = (bb * H + kvh) * cap.
template <bool PAGED>
__device__ __forceinline__ size_t cache_row_t(const CacheView &c, int bb, int kvh, size_t head_row0, int t) {
  if constexpr (PAGED) return cache_row_paged(c, bb, kvh, t);
  else return head_row0 + t;
}

// Arguments of one decode-attention call, resolved on the host.
struct AttendArgs {
  CacheView cache;
  const void *q;
  int q_dtype;
  int Hq, gqa, n_q;         // query heads, H_q / H_kv, query rows per head
  int kv_len, n_win, n_body; // n_win = HAD ring tokens in use, n_body = kv_len - n_win
  int causal, q_pos0;
  float scale;              // attention scale alpha
  int chunk, n_chunks;      // body chunks = ceil(n_body / chunk)
  int n_wchunks;            // window chunks of kWinChunk tokens (0 without a window)
  int C;                    // total partials per row: n_chunks + n_wchunks
  int win_in_reduce;        // HAD: phase 2 computes the window chunk's partial itself
  int y_base;               // row-side kernel: chunk index of its grid's first y (window-only launches)
  int q_prepped;            // row-side window chunks: the f32 rotated query rows are in q_rot
  // Token rows [fresh_lo, fresh_hi) were written by the kernel launched just before phase 1 (an
  // append in the same call): only phase-1 CTAs that read them, and the first CTA, wait for it.
  // [0, INT_MAX) when the preceding kernel is unknown (every CTA waits).
  int fresh_lo, fresh_hi;
  // Per-sequence lengths (paged calls): seq_lens [B] on the device, each clamped into
  // [0, kv_len]; kv_len, n_win, n_body and the chunk counts are then the maxima the grid is sized
  // for, causal rows are the sequence's newest n_q tokens (q_pos0 = length - n_q), and
  // fresh_tail > 0 marks the newest fresh_tail tokens of every sequence as just appended.
  // seq_lens == nullptr: every sequence has kv_len tokens.
  const int32_t *seq_lens;
  int fresh_tail;
  float *out;
  // workspace regions
  float *part_m, *part_l, *part_o;   // [rows][C], [rows][C], [rows][C][D]
  int8_t *q8;                         // HAD: [rows][D]
  float *s_q, *q_rot;                 // HAD: [rows], [rows][D]
  // Score capture (Hadamard layouts, contiguous cache; nullptr in every ordinary call): the
  // tensor-core kernel that scores the body also writes each exact integer score it computes to
  // cap_scores [B][Hq][n_q][n_body] and each row's int8 query scale to cap_sq [B][Hq][n_q].
  int32_t *cap_scores;
  float *cap_sq;
};
// Row index (b, hq, qi) of query row r (of the gqa * n_q rows of kv head kvh).
__device__ __forceinline__ size_t query_row_index(const AttendArgs &a, int bb, int kvh, int r) {
  return ((size_t)bb * a.Hq + kvh * a.gqa + r / a.n_q) * a.n_q + r % a.n_q;
}
// Score capture: the integer score of query row r against body token t.
__device__ __forceinline__ void capture_score(const AttendArgs &a, int bb, int kvh, int r, int t, int v) {
  a.cap_scores[query_row_index(a, bb, kvh, r) * a.n_body + t] = v;
}

// Launchers (return cudaGetLastError() after enqueueing).
// Append n_new rows per (batch, kv head) at positions pos0 + j, or (seq_pos != nullptr) at the
// per-sequence positions seq_pos[b] + pos_offset + j; rows outside [0, cap) are not written.
cudaError_t launch_store(const CacheView &c, const void *k_new, const void *v_new, int dtype,
                         int n_new, int pos0, cudaStream_t st, const int32_t *seq_pos = nullptr,
                         int pos_offset = 0);
// Hadamard query preparation into the workspace: int8 codes and scales, and (write_rot) the f32
// rotated rows.
cudaError_t launch_had_prep(const AttendArgs &a, cudaStream_t st, bool write_rot = true);
cudaError_t launch_attend_generic(const AttendArgs &a, cudaStream_t st);
cudaError_t launch_attend_reduce(const AttendArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_debug_scores(const CacheView &c, const void *q, int q_dtype, int Hq, int n_q,
                                int kv_len, int n_body, int32_t *scores, float *s_q,
                                cudaStream_t st);
// Tensor-core phase 1 for the shapes it covers; returns cudaErrorNotSupported when it does not
// cover the call (the caller then uses the generic kernel).
bool mma_supported(const AttendArgs &a);
// Whether the call's body is scored by a tensor-core kernel that is also built with score capture.
bool capture_supported(const AttendArgs &a);
cudaError_t launch_attend_mma(const AttendArgs &a, cudaStream_t st);
cudaError_t launch_attend_mma4(const AttendArgs &a, cudaStream_t st);
bool mma_q6_supported(const AttendArgs &a);
cudaError_t launch_attend_mma_q6(const AttendArgs &a, cudaStream_t st);
// Tensor-core phase 1 with the query rows on the M side (more than eight rows per kv head, e.g.
// causal prefill chunks), Hadamard int4 layout.
bool prefill_supported(const AttendArgs &a);
cudaError_t launch_attend_prefill(const AttendArgs &a, cudaStream_t st);
// The body chunks of a tc_prefill_shape call on the tcgen05 kernel (the query codes and scales must
// already be in the workspace: launch_had_prep with write_rot = false).
cudaError_t launch_attend_prefill_tc_body(const AttendArgs &a, cudaStream_t st);
cudaError_t launch_attend_prefill_mixed(const AttendArgs &a, cudaStream_t st);

// ----------------------------------------------------------------- device helpers
// Programmatic dependent launch: wait for the preceding kernel (and its memory) when this CTA
// reads rows it wrote, or when it is the grid's first CTA -- so that the grid never completes
// before its predecessor, and later kernels that wait on this grid also see the predecessor's
// writes.
__device__ __forceinline__ void pdl_wait_if(bool reads_fresh) {
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  const bool first = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  if (first || reads_fresh) asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// The lengths of sequence bb that a kernel works with.
struct SeqLen {
  int kv_len, n_body, q_pos0, fresh_lo, fresh_hi;
  int chunk, n_chunks;     // this sequence's split of its body (paged calls: equal chunks)
};
__device__ __forceinline__ SeqLen seq_of(const AttendArgs &a, int bb) {
  SeqLen s;
  if (a.seq_lens == nullptr) {
    s.kv_len = a.kv_len;
    s.n_body = a.n_body;
    s.q_pos0 = a.q_pos0;
    s.fresh_lo = a.fresh_lo;
    s.fresh_hi = a.fresh_hi;
    s.chunk = a.chunk;
    s.n_chunks = a.n_chunks;
    return s;
  }
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  // unless the preceding kernel is this call's own append (which does not write the lengths),
  // the lengths may come from it: wait for it before reading them
  if (a.fresh_tail == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
  const int L = min(max(__ldg(a.seq_lens + bb), 0), a.kv_len);
  s.kv_len = L;
  s.n_body = L - min(a.cache.n_recent, L);
  s.q_pos0 = L - a.n_q;
  s.fresh_lo = a.fresh_tail > 0 ? L - a.fresh_tail : 0;
  s.fresh_hi = a.fresh_tail > 0 ? L : INT_MAX;
  // the body in ceil(n_body / chunk) equal chunks (multiples of 64 tokens, none longer than
  // a.chunk), so that a short sequence's last chunk is not a sliver while its others are full
  s.n_chunks = s.n_body > 0 ? (s.n_body + a.chunk - 1) / a.chunk : 0;
  s.chunk = s.n_chunks > 0 ? ((s.n_body + s.n_chunks - 1) / s.n_chunks + 63) / 64 * 64 : a.chunk;
  return s;
}
// The same for a kernel built for one cache kind: paged calls always pass per-sequence lengths,
// contiguous calls never do, so a contiguous instantiation reads the call's values directly.
template <bool PAGED>
__device__ __forceinline__ SeqLen seq_of_t(const AttendArgs &a, int bb) {
  if constexpr (PAGED) {
    return seq_of(a, bb);
  } else {
    SeqLen s;
    s.kv_len = a.kv_len;
    s.n_body = a.n_body;
    s.q_pos0 = a.q_pos0;
    s.fresh_lo = a.fresh_lo;
    s.fresh_hi = a.fresh_hi;
    s.chunk = a.chunk;
    s.n_chunks = a.n_chunks;
    return s;
  }
}
// Last token query row i (of n_q) of the sequence may see; negative when it sees none.
__device__ __forceinline__ int row_limit(const AttendArgs &a, const SeqLen &s, int qi) {
  return a.causal ? min(s.kv_len - 1, s.q_pos0 + qi) : s.kv_len - 1;
}

// The largest row limit among query rows [r_lo, r_hi) of a kv head (negative if the range is empty):
// row_limit grows with the query index qi = r % n_q, so only the largest qi in the range matters.
__device__ __forceinline__ int max_row_limit(const AttendArgs &a, const SeqLen &s, int r_lo, int r_hi) {
  if (r_hi <= r_lo) return -1;
  const int lo = r_lo % a.n_q, hi = (r_hi - 1) % a.n_q;
  const int qmax = (r_hi - r_lo >= a.n_q || lo > hi) ? a.n_q - 1 : hi;
  return row_limit(a, s, qmax);
}

// Load 8 consecutive input elements starting at element index `e` (8-aligned) as f32.
__device__ __forceinline__ void load8_f32(const void *base, int dtype, size_t e, float v[8]) {
  if (dtype == KVQ_F32) {
    const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e);
    float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + e));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (dtype == KVQ_BF16) {
        v[2 * k] = bf16_bits_to_f32(u[k] & 0xFFFFu);
        v[2 * k + 1] = bf16_bits_to_f32(u[k] >> 16);
      } else {
        v[2 * k] = __half2float(__ushort_as_half((unsigned short)(u[k] & 0xFFFFu)));
        v[2 * k + 1] = __half2float(__ushort_as_half((unsigned short)(u[k] >> 16)));
      }
    }
  }
}

// Load 4 consecutive elements (4-aligned) as f32.
__device__ __forceinline__ void load4_f32(const void *base, int dtype, size_t e, float v[4]) {
  if (dtype == KVQ_F32) {
    float4 a = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  } else {
    const uint2 w = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(base) + e));
    const uint32_t u[2] = {w.x, w.y};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (dtype == KVQ_BF16) {
        v[2 * k] = bf16_bits_to_f32(u[k] & 0xFFFFu);
        v[2 * k + 1] = bf16_bits_to_f32(u[k] >> 16);
      } else {
        v[2 * k] = __half2float(__ushort_as_half((unsigned short)(u[k] & 0xFFFFu)));
        v[2 * k + 1] = __half2float(__ushort_as_half((unsigned short)(u[k] >> 16)));
      }
    }
  }
}

// fp32 nearest to 1/sqrt(D) for the orthonormal Hadamard rotation (D = 128 or 256).
__device__ __forceinline__ float inv_sqrt_dim(int D) {
  return D == 128 ? 0x1.6a09e6p-4f : 0x1.0p-4f;
}

// In-warp unnormalised FWHT of a D-vector held as V = D/32 consecutive values per lane
// (element lane*V + i). Butterflies (a, b) -> (a + b, a - b) with half-span 1, 2, ..., D/2 in
// ascending order; every add/subtract rounded once.
template <int V>
__device__ __forceinline__ void warp_fwht(float (&x)[V], int lane) {
#pragma unroll
  for (int h = 1; h < V; h <<= 1) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = __fadd_rn(a, b);
        x[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = (lane & m) ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
    }
  }
}

// Hadamard query preparation of one row, in one warp: x (V = D/32 consecutive values per lane,
// already loaded) -> rotated row q_rot = FWHT(x) * fp32(1/sqrt(D)), its int8 codes
// clamp(rint(q_rot / s_q), -127, 127) and s_q = amax(|q_rot|) / 127, all in correctly rounded
// float32 steps. Every kernel that needs the int8 query codes uses this one routine.
template <int V>
__device__ __forceinline__ float had_query_row(float (&x)[V], int (&q8)[V], int lane) {
  warp_fwht<V>(x, lane);
  const float cD = inv_sqrt_dim(V * 32);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    x[i] = __fmul_rn(x[i], cD);
    amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int m = 16; m; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    q8[i] = 0;
    if (s > 0.0f) q8[i] = (int)fminf(fmaxf(rintf(__fdiv_rn(x[i], s)), -127.0f), 127.0f);
  }
  return s;
}

}  // namespace kvq
