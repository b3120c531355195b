// Store (append) kernels: quantise new K/V rows and write them into the packed cache.
//
// Bit-exactness: every value is produced by one IEEE float32 operation at a time
// (__fdiv_rn / __fsub_rn / __fmul_rn, rintf = round half to even, __float2half_rn), and this
// file is compiled with -fmad=false so no multiply-add is ever contracted.
//
// Q4_0 / Q6_0 / Q8_0 / asymmetric: 4 threads per 32-value block, 8 values per thread; the
// block's amax (or min/max) is reduced over those 4 lanes with shuffles. Loads are 16-byte
// vectors, stores are the thread's 4 payload bytes (+ 2 high-plane bytes for Q6_0; 8 bytes for
// Q8_0).
// Hadamard int4 / int2: one warp per token row; the FWHT runs in registers and shuffles.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr float kF16Max = 65504.0f;

struct StoreGeom {
  int B, H, D, cap, n_new, pos0, row_bytes, nb;
  long long rows_per_tensor;   // B * H * n_new
  long long n_rows;            // rows of this launch: both planes (2 * rows_per_tensor) or one
  int kv_only;                 // -1: K and V in one launch; 0 / 1: this launch covers that plane only
  // per-sequence first position seq_pos[b] + pos_offset (device), or nullptr: pos0 for every one
  const int32_t *seq_pos;
  int pos_offset;
};

// Decompose a global row id into (tensor, input row, plane row, row j of the append, position,
// batch * H + head). False when the position is outside [0, cap): a per-sequence position the
// host could not check; such a row is computed but not written.
__device__ __forceinline__ bool row_coords(const CacheView &c, const StoreGeom &g, long long r, int &kv,
                                           long long &in_row, long long &crow, int &j, int &pos, long long &bh) {
  kv = g.kv_only >= 0 ? g.kv_only : (r >= g.rows_per_tensor ? 1 : 0);
  const long long rr = g.kv_only >= 0 ? r : r - (long long)kv * g.rows_per_tensor;
  in_row = rr;
  int bb, kvh;
  if (g.rows_per_tensor <= 0x7FFFFFFFLL) {                // 32-bit index arithmetic (every realistic call)
    const unsigned ur = (unsigned)rr, nn = (unsigned)g.n_new, hh = (unsigned)g.H;
    const unsigned ubh = ur / nn, ubb = ubh / hh;
    j = (int)(ur - ubh * nn);
    bh = ubh;
    bb = (int)ubb;
    kvh = (int)(ubh - ubb * hh);
  } else {
    bh = rr / g.n_new;
    j = (int)(rr - bh * g.n_new);
    bb = (int)(bh / g.H);
    kvh = (int)(bh - (long long)bb * g.H);
  }
  pos = (g.seq_pos ? __ldg(g.seq_pos + bb) + g.pos_offset : g.pos0) + j;
  const bool ok = pos >= 0 && pos < g.cap;
  crow = ok ? (long long)cache_row(c, bb, kvh, pos) : 0;
  return ok;
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_min(float v) {
  v = fminf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fminf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

__device__ __forceinline__ __half f16_sat(float x) {
  return __float2half_rn(fminf(fmaxf(x, -kF16Max), kF16Max));
}

// q = clamp(rint(x / s), lo, hi), or 0 when s == 0.
__device__ __forceinline__ int sym_code(float x, float s, int lo, int hi) {
  if (!(s > 0.0f)) return 0;
  const float r = rintf(__fdiv_rn(x, s));
  return (int)fminf(fmaxf(r, (float)lo), (float)hi);
}

// LAYOUT: KVQ_Q4_0, KVQ_Q6_0, KVQ_Q8_0 or KVQ_ASYM4_G32.
template <int LAYOUT>
__global__ void __launch_bounds__(256) store_block_kernel(CacheView c, const void *__restrict__ k_new,
                                                          const void *__restrict__ v_new, int dtype,
                                                          StoreGeom g) {
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");   // attention may launch and wait on us
#endif
  const int tpr_shift = g.D == 128 ? 4 : 5;                // D / 8 threads per row
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long r = gt >> tpr_shift;
  const int tr = (int)(gt & ((1 << tpr_shift) - 1));      // thread within row
  // Threads past the last row still take part in the quad shuffles (full-warp masks) but load
  // and store nothing.
  bool valid = r < g.n_rows;
  int kv = 0, j = 0, pos = 0;
  long long in_row = 0, crow = 0, bh = 0;
  if (valid) valid = row_coords(c, g, r, kv, in_row, crow, j, pos, bh);
  const int blk = tr >> 2, lb = tr & 3;

  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (valid) load8_f32(kv ? v_new : k_new, dtype, (size_t)in_row * g.D + (size_t)tr * 8, v);
  uint8_t *prow = (kv ? c.payload[1] : c.payload[0]) + (size_t)crow * g.row_bytes;
  __half *srow = static_cast<__half *>((kv ? c.scale[1] : c.scale[0])) + (size_t)crow * g.nb;

  if (LAYOUT == KVQ_ASYM4_G32) {
    float mn = v[0], mx = v[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) { mn = fminf(mn, v[i]); mx = fmaxf(mx, v[i]); }
    mn = quad_min(mn);
    mx = quad_max(mx);
    const __half sh = f16_sat(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
    const __half zh = f16_sat(mn);
    const float s = __half2float(sh), z = __half2float(zh);
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int q = 0;
      if (s > 0.0f) {
        const float rr = rintf(__fdiv_rn(__fsub_rn(v[i], z), s));
        q = (int)fminf(fmaxf(rr, 0.0f), 15.0f);
      }
      w |= (uint32_t)q << (4 * i);
    }
    if (!valid) return;
    *reinterpret_cast<uint32_t *>(prow + blk * 16 + lb * 4) = w;
    if (lb == 0) {
      srow[blk] = sh;
      (kv ? c.zero[1] : c.zero[0])[(size_t)crow * g.nb + blk] = zh;
    }
    return;
  }

  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = quad_max(amax);
  if (LAYOUT == KVQ_Q4_0) {
    const __half sh = f16_sat(__fdiv_rn(amax, 8.0f));
    const float s = __half2float(sh);
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) w |= ((uint32_t)sym_code(v[i], s, -8, 7) & 0xFu) << (4 * i);
    if (!valid) return;
    *reinterpret_cast<uint32_t *>(prow + blk * 16 + lb * 4) = w;
    if (lb == 0) srow[blk] = sh;
  } else if (LAYOUT == KVQ_Q8_0) {
    const __half sh = f16_sat(__fdiv_rn(amax, 128.0f));
    const float s = __half2float(sh);
    uint32_t w0 = 0, w1 = 0;                   // byte i = value i (two's complement)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w0 |= ((uint32_t)sym_code(v[i], s, -128, 127) & 0xFFu) << (8 * i);
      w1 |= ((uint32_t)sym_code(v[4 + i], s, -128, 127) & 0xFFu) << (8 * i);
    }
    if (!valid) return;
    *reinterpret_cast<uint2 *>(prow + blk * 32 + lb * 8) = make_uint2(w0, w1);
    if (lb == 0) srow[blk] = sh;
  } else {  // Q6_0
    const __half sh = f16_sat(__fdiv_rn(amax, 32.0f));
    const float s = __half2float(sh);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t u = (uint32_t)sym_code(v[i], s, -32, 31) & 0x3Fu;
      lo |= (u & 0xFu) << (4 * i);
      hi |= ((u >> 4) & 0x3u) << (2 * i);      // values 4k..4k+3 -> byte k, bits 0,2,4,6
    }
    if (!valid) return;
    uint8_t *bp = prow + blk * 24;
    *reinterpret_cast<uint32_t *>(bp + lb * 4) = lo;
    *reinterpret_cast<uint16_t *>(bp + 16 + lb * 2) = (uint16_t)hi;
    if (lb == 0) srow[blk] = sh;
  }
}

// Hadamard int4 (BITS 4: scale amax / 7, codes [-7, 7], two per byte) or int2 (BITS 2: scale
// amax, codes [-1, 1], four per byte): one warp per token row, V = D/32 values per lane.
template <int V, int BITS>
__global__ void __launch_bounds__(256) store_had_kernel(CacheView c, const void *__restrict__ k_new,
                                                        const void *__restrict__ v_new, int dtype,
                                                        StoreGeom g) {
#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 900
  asm volatile("griddepcontrol.launch_dependents;");   // attention may launch and wait on us
#endif
  const int lane = threadIdx.x & 31;
  const long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (r >= g.n_rows) return;                               // whole warp exits together
  int kv, j, pos;
  long long in_row, crow, bh;
  if (!row_coords(c, g, r, kv, in_row, crow, j, pos, bh)) return;   // whole warp (one row)
  float x[V];
  const void *src = kv ? v_new : k_new;
  if (V == 4) {
    load4_f32(src, dtype, (size_t)in_row * g.D + lane * 4, x);
  } else {
    load8_f32(src, dtype, (size_t)in_row * g.D + lane * 8, x);
  }
  warp_fwht<V>(x, lane);
  const float cD = inv_sqrt_dim(g.D);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    x[i] = __fmul_rn(x[i], cD);
    amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int m = 16; m; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  constexpr int QMAX = BITS == 4 ? 7 : 1;
  const float s = __fdiv_rn(amax, (float)QMAX);
  uint32_t w = 0;                                           // field i of the lane at bits BITS*i
#pragma unroll
  for (int i = 0; i < V; ++i)
    w |= ((uint32_t)sym_code(x[i], s, -QMAX, QMAX) & ((1u << BITS) - 1u)) << (BITS * i);
  uint8_t *prow = (kv ? c.payload[1] : c.payload[0]) + (size_t)crow * g.row_bytes;
  if (V * BITS == 8) {
    prow[lane] = (uint8_t)w;
  } else if (V * BITS == 16) {
    *reinterpret_cast<uint16_t *>(prow + lane * 2) = (uint16_t)w;
  } else {
    *reinterpret_cast<uint32_t *>(prow + lane * 4) = w;
  }
  if (lane == 0) static_cast<float *>((kv ? c.scale[1] : c.scale[0]))[crow] = s;
  // Exact-f32 ring of the newest tokens: only the last min(n_new, n_recent) rows of this call,
  // so no two rows of one call write the same slot.
  if (c.n_recent > 0 && j >= g.n_new - c.n_recent) {
    float *dst = (kv ? c.ring[1] : c.ring[0]) + ((size_t)bh * c.n_recent + (size_t)(pos % c.n_recent)) * g.D + lane * V;
#pragma unroll
    for (int i = 0; i < V; i += 4)
      *reinterpret_cast<float4 *>(dst + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
  }
}

}  // namespace

namespace {

// One launch of the store kernel for `layout` over both planes (kv_only < 0) or one plane.
cudaError_t launch_store_plane(const CacheView &c, int layout, const void *k_new, const void *v_new, int dtype,
                               StoreGeom g, cudaStream_t st) {
  const long long rows = g.n_rows;
  if (is_hadamard(layout)) {
    const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
    const bool two = layout == KVQ_HAD_INT2;
    if (c.D == 128) {
      if (two) store_had_kernel<4, 2><<<blocks, 256, 0, st>>>(c, k_new, v_new, dtype, g);
      else store_had_kernel<4, 4><<<blocks, 256, 0, st>>>(c, k_new, v_new, dtype, g);
    } else {
      if (two) store_had_kernel<8, 2><<<blocks, 256, 0, st>>>(c, k_new, v_new, dtype, g);
      else store_had_kernel<8, 4><<<blocks, 256, 0, st>>>(c, k_new, v_new, dtype, g);
    }
  } else {
    const long long threads = rows * (c.D / 8);
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    switch (layout) {
      case KVQ_Q4_0: store_block_kernel<KVQ_Q4_0><<<blocks, 256, 0, st>>>(c, k_new, v_new, dtype, g); break;
      case KVQ_Q6_0: store_block_kernel<KVQ_Q6_0><<<blocks, 256, 0, st>>>(c, k_new, v_new, dtype, g); break;
      case KVQ_Q8_0: store_block_kernel<KVQ_Q8_0><<<blocks, 256, 0, st>>>(c, k_new, v_new, dtype, g); break;
      default: store_block_kernel<KVQ_ASYM4_G32><<<blocks, 256, 0, st>>>(c, k_new, v_new, dtype, g); break;
    }
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_store(const CacheView &c, const void *k_new, const void *v_new, int dtype, int n_new,
                         int pos0, cudaStream_t st, const int32_t *seq_pos, int pos_offset) {
  StoreGeom g;
  g.B = c.B; g.H = c.H; g.D = c.D; g.cap = c.cap; g.n_new = n_new; g.pos0 = pos0;
  g.seq_pos = seq_pos; g.pos_offset = pos_offset;
  g.nb = c.D / kBlock;
  g.rows_per_tensor = (long long)c.B * c.H * n_new;
  if (c.layout == c.v_layout) {                          // one launch for K and V
    g.row_bytes = c.row_bytes;
    g.n_rows = 2 * g.rows_per_tensor;
    g.kv_only = -1;
    return launch_store_plane(c, c.layout, k_new, v_new, dtype, g, st);
  }
  // mixed K/V precision: one launch per plane, each with its own layout
  g.n_rows = g.rows_per_tensor;
  g.kv_only = 0;
  g.row_bytes = c.row_bytes;
  cudaError_t e = launch_store_plane(c, c.layout, k_new, v_new, dtype, g, st);
  if (e != cudaSuccess) return e;
  g.kv_only = 1;
  g.row_bytes = c.v_row_bytes;
  return launch_store_plane(c, c.v_layout, k_new, v_new, dtype, g, st);
}

}  // namespace kvq
