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
// exact path of the block encoder below, out of line (it is rarely taken, and inlined 16 times
// a block it multiplied the code size of the encoding epilogues).
static __device__ __noinline__ uint32_t e2m1_pair_div(float a, float b, float den) {
  return cvt_e2m1x2(__fdiv_rn(a, den), __fdiv_rn(b, den)) & 0xFFu;
}

// The scale of one block from its amax, and what its elements' encoding needs.
struct NvBlockScale {
  uint32_t sc;  // UE4M3 scale code
  float den;    // RN(value(sc) * s)
  float inv;    // RN(1 / den) when fast
  bool fast;    // den and 1 / den are normal float32 values
};

__device__ __forceinline__ NvBlockScale nv_block_scale(float bmax, float s, float d) {
  NvBlockScale b;
  const float t = (d != 0.0f) ? __fdiv_rn(bmax, d) : 0.0f;
  b.sc = cvt_e4m3x2(t, 0.0f) & 0x7Fu;
  b.den = __fmul_rn(ue4m3_value(b.sc), s);
  b.fast = b.den >= 0x1p-126f && b.den <= 0x1p126f;
  b.inv = b.fast ? __frcp_rn(b.den) : 0.0f;
  return b;
}

// E2M1 codes of RN(x0 / den) and RN(x1 / den) in one byte (x0 in the low nibble), reached without
// a division per element: p = RN(x * RN(1/den)) is within 2^-22.4 of x/den relative (and so of
// RN(x/den)), and E2M1 rounding is monotone, so when p (1 - 2^-21) and p (1 + 2^-21) round to the
// same code, that is the code of RN(x/den).  Pairs that straddle a rounding threshold, and blocks
// whose den or 1/den is not a normal float32, take the IEEE division.
__device__ __forceinline__ uint32_t nv_pair_code(float x0, float x1, const NvBlockScale& b) {
  if (b.den == 0.0f) return 0u;
  if (b.fast) {
    const float p0 = __fmul_rn(x0, b.inv), p1 = __fmul_rn(x1, b.inv);
    const uint32_t below = cvt_e2m1x2(__fmul_rn(p0, 1.0f - 0x1p-21f), __fmul_rn(p1, 1.0f - 0x1p-21f)) & 0xFFu;
    const uint32_t above = cvt_e2m1x2(__fmul_rn(p0, 1.0f + 0x1p-21f), __fmul_rn(p1, 1.0f + 0x1p-21f)) & 0xFFu;
    if (below == above) return below;
  }
  return e2m1_pair_div(x0, x1, b.den);
}

// One block of 16 values v -> its UE4M3 scale code (returned) and 16 E2M1 codes packed two per
// byte, element 2j in the low nibble of byte j (lo: bytes 0..3, hi: bytes 4..7).
__device__ __forceinline__ uint32_t nv_encode_block16(const float (&v)[16], float s, float d, uint32_t& lo,
                                                      uint32_t& hi) {
  float bmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) bmax = fmaxf(bmax, fabsf(v[j]));
  const NvBlockScale b = nv_block_scale(bmax, s, d);
  lo = 0;
  hi = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t byte = nv_pair_code(v[2 * j], v[2 * j + 1], b);
    if (j < 4) lo |= byte << (8 * j);
    else hi |= byte << (8 * (j - 4));
  }
  return b.sc;
}

// The same encoding with the block's 16 values spread over four neighbouring lanes of a warp
// (lanes 4k .. 4k+3, all calling this together), four each: v holds elements 4q .. 4q+3 of the
// block, q = lane % 4.  Every lane gets the block's scale code (returned, from the amax of all 16)
// and its own four E2M1 codes in `codes` (16 bits: element 4q in the low nibble).
__device__ __forceinline__ uint32_t nv_encode_quad(const float (&v)[4], float s, float d, uint32_t& codes) {
  const unsigned mask = 0xFu << (threadIdx.x & 28u);
  float bmax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  bmax = fmaxf(bmax, __shfl_xor_sync(mask, bmax, 1));
  bmax = fmaxf(bmax, __shfl_xor_sync(mask, bmax, 2));
  const NvBlockScale b = nv_block_scale(bmax, s, d);
  codes = nv_pair_code(v[0], v[1], b) | (nv_pair_code(v[2], v[3], b) << 8);
  return b.sc;
}

}  // namespace bsg
