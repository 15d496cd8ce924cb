// NVFP4 block encoding shared by the quantiser and the GEMM's NVFP4-output epilogue, and the
// byte offset of a scale in the swizzled 128x4 scale layout.
//
// Per 16-element block of a row, with the tensor's global scale s and d = RN(6 s) (the NVFP4
// recipe of the "[QST] Performance overhead ..." page's Nvf4 kernels, each step one float32
// operation rounded to nearest even): scale = UE4M3(RN(amax / d)) (0 when d == 0), saturating;
// den = RN(value(scale) * s); element = E2M1(RN(x / den)) (0 when den == 0), saturating.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace bsg {

// Byte offset of scale (r, c) in the swizzled buffer (cols4 = padded scale columns / 4): atoms of
// 128 rows x 4 columns, 512 bytes each, band by band; in an atom, byte (r % 32) * 16 +
// ((r % 128) / 32) * 4 + c % 4.
__device__ __forceinline__ size_t sf_swizzle_offset(int r, int c, int cols4) {
  const size_t atom = static_cast<size_t>(r >> 7) * cols4 + (c >> 2);
  return atom * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// E4M3 code with the sign bit clear -> exact float value.
__device__ __forceinline__ float ue4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  if (e == 0) return static_cast<float>(m) * 0x1p-9f;
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// E2M1 codes of RN(a / den) and RN(b / den), packed in one byte (a in the low nibble): the
// path of the block encoder below for blocks outside the range where the quotients are formed
// without a division, out of line (it is rarely taken, and inlined 16 times a block it multiplied
// the code size of the encoding epilogues).
static __device__ __noinline__ uint32_t e2m1_pair_div(float a, float b, float den) {
  return cvt_e2m1x2(__fdiv_rn(a, den), __fdiv_rn(b, den)) & 0xFFu;
}

// Packed float32 pairs, each lane exactly the scalar operation: (a0 b0, a1 b1) rounded to
// nearest even, and (a0 b0 + c0, a1 b1 + c1) with one rounding, to nearest even (rn) or toward
// minus infinity (rm).
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void fmul2_rn(float a0, float a1, float b0, float b1, float& r0, float& r1) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f32x2_pack(a0, a1)), "l"(f32x2_pack(b0, b1)));
  f32x2_unpack(r, r0, r1);
}
__device__ __forceinline__ void ffma2_rn(float a0, float a1, float b0, float b1, float c0, float c1, float& r0,
                                         float& r1) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(f32x2_pack(a0, a1)), "l"(f32x2_pack(b0, b1)), "l"(f32x2_pack(c0, c1)));
  f32x2_unpack(r, r0, r1);
}
__device__ __forceinline__ void ffma2_rm(float a0, float a1, float b0, float b1, float c0, float c1, float& r0,
                                         float& r1) {
  uint64_t r;
  asm("fma.rm.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(f32x2_pack(a0, a1)), "l"(f32x2_pack(b0, b1)), "l"(f32x2_pack(c0, c1)));
  f32x2_unpack(r, r0, r1);
}

// Quotients without a division, by Markstein's correction step (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990):
// with r = RN(1/y) the correctly rounded reciprocal, p = RN(x r) is within about an ulp of x / y,
// the remainder x - p y is exact as one fused multiply-add, and RN(p + (x - p y) r) is RN(x / y).
// The remainder is exact whenever it is a multiple of 2^-149: with y in [2^-64, 2^64] (the only
// divisors the encoder sends here), for every quotient at or above 2^-39.  Smaller quotients may
// come out a little off, but E4M3 and E2M1 send everything up to 2^-10 to code 0, so their codes
// do not change.  The remainder is formed rounding toward minus infinity, which changes no exact
// value but makes a zero remainder -0, so that x = -0 gives -0 (code 0x8) like RN(-0 / y).  p must
// not overflow: the encoder keeps |x| / y below about 2^64.  ny = -y.
__device__ __forceinline__ float div_markstein(float x, float r, float ny) {
  const float p = __fmul_rn(x, r);
  return __fmaf_rn(__fmaf_rd(p, ny, x), r, p);
}
__device__ __forceinline__ void div2_markstein(float x0, float x1, float r, float ny, float& q0, float& q1) {
  float p0, p1, e0, e1;
  fmul2_rn(x0, x1, r, r, p0, p1);
  ffma2_rm(p0, p1, ny, ny, x0, x1, e0, e1);
  ffma2_rn(e0, e1, r, r, p0, p1, q0, q1);
}

__device__ __forceinline__ bool markstein_range(float y) { return y >= 0x1p-64f && y <= 0x1p64f; }

// The per-tensor part: s, d = RN(6 s), and RN(1/d) when d is in the range above (fast).
struct NvTensorScale {
  float s, d, rd;
  bool fast;
};

__device__ __forceinline__ NvTensorScale nv_tensor_scale(float s) {
  NvTensorScale t;
  t.s = s;
  t.d = __fmul_rn(6.0f, s);
  t.fast = markstein_range(t.d);
  t.rd = t.fast ? __frcp_rn(t.d) : 0.0f;
  return t;
}

// The scale of one block from its amax, and what its elements' encoding needs.
struct NvBlockScale {
  uint32_t sc;  // UE4M3 scale code
  float den;    // RN(value(sc) * s)
  float inv;    // RN(1 / den) when fast
  bool fast;    // den in the range above and amax / den below about 2^64
};

__device__ __forceinline__ NvBlockScale nv_block_scale(float bmax, const NvTensorScale& t) {
  NvBlockScale b;
  float q;
  if (t.fast && __fmul_rn(bmax, t.rd) <= 0x1p64f) q = div_markstein(bmax, t.rd, -t.d);
  else q = t.d != 0.0f ? __fdiv_rn(bmax, t.d) : 0.0f;
  b.sc = cvt_e4m3x2(q, 0.0f) & 0x7Fu;
  b.den = __fmul_rn(ue4m3_value(b.sc), t.s);
  const bool in_range = markstein_range(b.den);
  b.inv = in_range ? __frcp_rn(b.den) : 0.0f;
  b.fast = in_range && __fmul_rn(bmax, b.inv) <= 0x1p64f;
  return b;
}

// E2M1 codes of RN(x0 / den) and RN(x1 / den) in one byte (x0 in the low nibble).
__device__ __forceinline__ uint32_t nv_pair_code(float x0, float x1, const NvBlockScale& b) {
  float q0, q1;
  div2_markstein(x0, x1, b.inv, -b.den, q0, q1);
  return cvt_e2m1x2(q0, q1);
}

// E2M1 codes of a block's pairs where the quotients cannot be formed as above: IEEE divisions,
// or 0 when den is 0.
__device__ __forceinline__ uint32_t nv_pair_code_slow(float x0, float x1, const NvBlockScale& b) {
  return b.den == 0.0f ? 0u : e2m1_pair_div(x0, x1, b.den);
}

// One block of 16 values v -> its UE4M3 scale code (returned) and 16 E2M1 codes packed two per
// byte, element 2j in the low nibble of byte j (lo: bytes 0..3, hi: bytes 4..7).
__device__ __forceinline__ uint32_t nv_encode_block16(const float (&v)[16], const NvTensorScale& t, uint32_t& lo,
                                                      uint32_t& hi) {
  float bmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) bmax = fmaxf(bmax, fabsf(v[j]));
  const NvBlockScale b = nv_block_scale(bmax, t);
  lo = 0;
  hi = 0;
  if (b.fast) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = nv_pair_code(v[2 * j], v[2 * j + 1], b);
      if (j < 4) lo |= byte << (8 * j);
      else hi |= byte << (8 * (j - 4));
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = nv_pair_code_slow(v[2 * j], v[2 * j + 1], b);
      if (j < 4) lo |= byte << (8 * j);
      else hi |= byte << (8 * (j - 4));
    }
  }
  return b.sc;
}

// The same encoding with the block's 16 values spread over four neighbouring lanes of a warp
// (lanes 4k .. 4k+3, all calling this together), four each: v holds elements 4q .. 4q+3 of the
// block, q = lane % 4.  Every lane gets the block's scale code (returned, from the amax of all 16)
// and its own four E2M1 codes in `codes` (16 bits: element 4q in the low nibble).
__device__ __forceinline__ uint32_t nv_encode_quad(const float (&v)[4], const NvTensorScale& t, uint32_t& codes) {
  const unsigned mask = 0xFu << (threadIdx.x & 28u);
  float bmax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  bmax = fmaxf(bmax, __shfl_xor_sync(mask, bmax, 1));
  bmax = fmaxf(bmax, __shfl_xor_sync(mask, bmax, 2));
  const NvBlockScale b = nv_block_scale(bmax, t);
  if (b.fast) codes = nv_pair_code(v[0], v[1], b) | (nv_pair_code(v[2], v[3], b) << 8);
  else codes = nv_pair_code_slow(v[0], v[1], b) | (nv_pair_code_slow(v[2], v[3], b) << 8);
  return b.sc;
}

}  // namespace bsg
