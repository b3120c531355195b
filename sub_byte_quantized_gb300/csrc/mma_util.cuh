// Inline PTX helpers shared by the tensor-core phase-1 kernels: cp.async staging, ldmatrix,
// movmatrix, mma.sync m16n8k16 (f16 in, f32 accumulate), f16x2 arithmetic, lop3 and shared-memory
// mbarriers with bounded waits.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace kvq {
namespace mma {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// one token's scale (or zero-point) entry: N = 8 (four fp16) or 4 (one f32) bytes
template <int N>
__device__ __forceinline__ void cp_async_scale(uint32_t dst, const void *src, int src_bytes) {
  if (N == 8) cp_async8(dst, src, src_bytes);
  else cp_async4(dst, src, src_bytes);
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// m16n8k8: d += a . b, a0 / a1 = rows g / g+8 at k 2c, 2c+1; b0 = k 2c, 2c+1 of column g
__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}
// d = a . b + c with a separate accumulator input
__device__ __forceinline__ void mma16816_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                           float c0, float c1, float c2, float c3) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}
// m16n8k8 with tf32 operands (f32 bit patterns whose low 13 mantissa bits are zero), f32 accumulate:
// a0 / a1 = rows g / g+8 at k = c, a2 / a3 the same rows at k = c + 4; b0 / b1 = k = c / c + 4 of
// column g; d0, d1 = row g, columns 2c, 2c+1; d2, d3 = row g+8.
__device__ __forceinline__ void mma1688_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// x = hi + lo with hi = x rounded to tf32 (nearest, ties away) and lo = the remainder rounded to
// tf32: hi + lo carries 22 significant bits of x, and the products hi*hi + hi*lo + lo*hi of two
// split operands match their f32 product to about 2^-21 relative.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  const float r = x - __uint_as_float(hi);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
template <int LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, %4;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(LUT));
  return d;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// a * b - c in one rounding (the negation is an operand modifier of the f16x2 fma)
__device__ __forceinline__ uint32_t hfma2_negc(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("{\n.reg .b32 t;\nneg.f16x2 t, %3;\nfma.rn.f16x2 %0, %1, %2, t;\n}\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// f16x2 constants (bit patterns): 1/16, -1032, -72 in both halves.
constexpr uint32_t kH16th = 0x2C002C00u, kHm1032 = 0xE408E408u, kHm72 = 0xD480D480u;

// Q4_0 V operand: eight 4-bit fields n0..n7 of w (n0 = bits 0-3) -> four exact f16 pairs
// (n0,n4), (n1,n5), (n2,n6), (n3,n7) holding the signed code values (n ^ 8) - 8. One lop3 places
// a field in the mantissa under the exponent of 1024 (0x6400) with the sign flip folded in; one
// f16 add/fma removes the offset.
__device__ __forceinline__ void unpack8_q4(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  o[0] = hadd2(lop3<0x6a>(w, 0x000F000Fu, 0x64086408u), kHm1032);
  o[1] = hfma2(lop3<0x6a>(w, 0x00F000F0u, 0x64806480u), kH16th, kHm72);
  o[2] = hadd2(lop3<0x6a>(w8, 0x000F000Fu, 0x64086408u), kHm1032);
  o[3] = hfma2(lop3<0x6a>(w8, 0x00F000F0u, 0x64806480u), kH16th, kHm72);
}

// K operands: the same four pairs as unpack8_q4, but each code u (Q4_0 and Hadamard int4: u = n ^ 8,
// the code plus 8; asymmetric: u = n) is placed in the mantissa of an f16 with a zero exponent,
// i.e. the exact subnormal u * 2^-24 (high fields: 16 u * 2^-24). One lop3 per pair, no f16
// arithmetic. The query entries facing high fields are divided by 16, the 2^-24 goes into the
// row's scale and the offset -8 * sum(q) into the accumulator's initial value (asymmetric: the
// zero-point term is added to each block's partial). A score is one short dot product, so the
// offset costs no precision there; value paths take the exact signed forms instead, because their
// long accumulation would carry the offset's mass.
template <bool ASYM>
__device__ __forceinline__ void unpack8_sub(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  if (!ASYM) {
    o[0] = lop3<0x6a>(w, 0x000F000Fu, 0x00080008u);
    o[1] = lop3<0x6a>(w, 0x00F000F0u, 0x00800080u);
    o[2] = lop3<0x6a>(w8, 0x000F000Fu, 0x00080008u);
    o[3] = lop3<0x6a>(w8, 0x00F000F0u, 0x00800080u);
  } else {
    o[0] = w & 0x000F000Fu;
    o[1] = w & 0x00F000F0u;
    o[2] = w8 & 0x000F000Fu;
    o[3] = w8 & 0x00F000F0u;
  }
}

// Unsigned 4-bit fields n0..n7 of w -> four exact f16 pairs (n0,n4), (n1,n5), (n2,n6), (n3,n7)
// holding n: the field is placed in the mantissa under the exponent of 1024 (low fields: 1024 + n,
// high fields: 1024 + 16 n) and one f16 add / fma removes the offset.
__device__ __forceinline__ void unpack8_u4(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  o[0] = hadd2(lop3<0xEA>(w, 0x000F000Fu, 0x64006400u), 0xE400E400u);
  o[1] = hfma2(lop3<0xEA>(w, 0x00F000F0u, 0x64006400u), kH16th, 0xD400D400u);
  o[2] = hadd2(lop3<0xEA>(w8, 0x000F000Fu, 0x64006400u), 0xE400E400u);
  o[3] = hfma2(lop3<0xEA>(w8, 0x00F000F0u, 0x64006400u), kH16th, 0xD400D400u);
}

// Unsigned 4-bit fields n0..n7 of w -> four exact f16 pairs (n0,n4), (n1,n5), (n2,n6), (n3,n7)
// holding n - 8 (the asymmetric codes centred on the group's midpoint): like unpack8_q4, with the
// field ORed under the exponent of 1024 instead of XORed.
__device__ __forceinline__ void unpack8_u4m8(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  o[0] = hadd2(lop3<0xEA>(w, 0x000F000Fu, 0x64006400u), kHm1032);
  o[1] = hfma2(lop3<0xEA>(w, 0x00F000F0u, 0x64006400u), kH16th, kHm72);
  o[2] = hadd2(lop3<0xEA>(w8, 0x000F000Fu, 0x64006400u), kHm1032);
  o[3] = hfma2(lop3<0xEA>(w8, 0x00F000F0u, 0x64006400u), kH16th, kHm72);
}

// The midpoints x = z + 8 s of two asymmetric groups (f16 pairs of zero-points z and scales s)
// as f16 hi + lo parts: x is formed in f32 (exact but for the rare exponent spread beyond 24
// bits), hi = rn(x), lo = rn(x - hi).
__device__ __forceinline__ void midpoint_split(uint32_t z, uint32_t s, uint32_t &hi, uint32_t &lo) {
  const float2 zf = __half22float2(u32_as_h2(z)), sf = __half22float2(u32_as_h2(s));
  const float x0 = fmaf(8.0f, sf.x, zf.x), x1 = fmaf(8.0f, sf.y, zf.y);
  hi = pack_f16x2(x0, x1);
  const float2 hf = __half22float2(u32_as_h2(hi));
  lo = pack_f16x2(x0 - hf.x, x1 - hf.y);
}

// Signed 8-bit fields: a = values v0..v3, b = v4..v7 (byte i = value i, two's complement) ->
// four exact f16 pairs (v0,v4), (v1,v5), (v2,v6), (v3,v7). The two bytes of a pair are placed
// under the exponent of 1024 with the sign bit flipped (1024 + v + 128), then 1152 is removed.
__device__ __forceinline__ void unpack8_s8(uint32_t a, uint32_t b, uint32_t (&o)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = prmt(a, b, (uint32_t)(((4 + i) << 8) | i));
    o[i] = hadd2(lop3<0x6A>(t, 0x00FF00FFu, 0x64806480u), 0xE480E480u);
  }
}

// Signed 2-bit fields f0..f7 in the low 16 bits of h (field i at bits 2i, code (f ^ 2) - 2) ->
// four exact f16 pairs (c0,c4), (c1,c5), (c2,c6), (c3,c7): the fields' two bytes go to the two
// 16-bit lanes, each pair is masked under the exponent of 1024 with bit 1 flipped, then 1026 is
// removed.
__device__ __forceinline__ void unpack8_s2(uint32_t h, uint32_t (&o)[4]) {
  const uint32_t x = prmt(h, 0u, 0x4140u);
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = hadd2(lop3<0x6A>(x >> (2 * i), 0x00030003u, 0x64026402u), 0xE402E402u);
}

// Signed 6-bit codes of one 8-value chunk of a Q6_0 block: `lo` = the low-plane word (value i's
// low four bits at bits 4i), `h16` = the two high-plane bytes (value i's top two bits at bits 2i)
// -> four exact f16 pairs (c0,c4), (c1,c5), (c2,c6), (c3,c7) of the codes (v ^ 0x20) - 0x20. The
// low nibble goes under the exponent of 1024 with bit 5 set, the high field is XORed into bits
// 4-5 (so the f16 holds 1024 + (v ^ 0x20)), and one f16 add removes 1056.
__device__ __forceinline__ void unpack8_s6(uint32_t lo, uint32_t h16, uint32_t (&o)[4]) {
  const uint32_t x = prmt(h16, 0u, 0x4140u);           // values 0-3 -> low lane, 4-7 -> high lane
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t t = lop3<0x6A>(lo >> (4 * k), 0x000F000Fu, 0x64206420u);   // (a & b) ^ c
    const uint32_t xs = k < 3 ? x << (4 - 2 * k) : x >> 2;
    o[k] = hadd2(lop3<0x6A>(xs, 0x00300030u, t), 0xE420E420u);
  }
}

// ---- mbarriers in shared memory with bounded waits (a wait that gives up returns false; the
// caller then ends its work and reports the failure instead of hanging)
constexpr unsigned long long kWaitNs = 250ull * 1000 * 1000;   // give up on a wait after 250 ms

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint64_t *b, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count));
}
__device__ __forceinline__ void bar_arrive(uint64_t *b) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_addr(b)) : "memory");
}
// Wait for the completion of the phase with the given parity; false if it has not completed
// within kWaitNs. Each try suspends the warp for up to kSuspendNs unless the phase completes first,
// so waiting warps do not take issue slots from working ones; the clock is read every 64 tries.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool bar_wait(uint64_t *b, uint32_t parity) {
  uint64_t start = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done = 0;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(smem_addr(b)), "r"(parity), "r"(kSuspendNs) : "memory");
    if (done) return true;
    if ((it & 63) == 63) {
      const uint64_t now = global_ns();
      if (start == 0) start = now;
      else if (now - start > kWaitNs) return false;
    }
  }
}
// A wait off the critical path (a role that runs ahead of the one it feeds): between tries the
// warp sleeps, so that it does not take issue slots from the working warps.
__device__ __forceinline__ bool bar_wait_relaxed(uint64_t *b, uint32_t parity) {
  uint64_t start = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done = 0;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(smem_addr(b)), "r"(parity) : "memory");
    if (done) return true;
    __nanosleep(128);
    if ((it & 63) == 63) {
      const uint64_t now = global_ns();
      if (start == 0) start = now;
      else if (now - start > kWaitNs) return false;
    }
  }
}

}  // namespace mma
}  // namespace kvq
