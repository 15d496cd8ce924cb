// Test-only probe of the division-free quotients of the NVFP4 block encoder.
//
// The encoder forms RN(x / y) as RN(p + (x - p y) r) with r = RN(1/y) and p = RN(x r) (Markstein's
// correction step) for divisors y in [2^-64, 2^64] and |x| / y below about 2^64.  This probe draws
// divisors y, two dividends x each, from a counter-based generator (splitmix64 of seed + index),
// forms each quotient both ways, the encoder's (packed pair and scalar) and CUDA's IEEE division
// __fdiv_rn, and counts the quotients where they differ: in the float32 bits for quotients at or
// above 2^-39 (or zero), and in the E2M1 and E4M3 codes for every quotient.  Four kinds of
// divisors, a quarter each:
//   0: y with a random significand and exponent, x = y times a random value in 2^-45 .. 2^8;
//   1: x within 16 ulps of y times a value where an E2M1 or E4M3 code changes (a rounding
//      threshold), or times a code value;
//   2: like 0 with y's significand all ones;
//   3: y = RN(value(c) * s) for a random UE4M3 code c and a random s, the encoder's own divisors,
//      x a random BF16 value.
// Dividends and divisors outside the encoder's range are skipped.  out[0] counts quotients tested,
// out[1] quotient mismatches, out[2] code mismatches (over the pair and the scalar form both);
// out[3], out[4] hold the bits of x and y of one mismatch.
#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_codec.cuh"

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float make_float(int e, uint32_t mant, uint32_t sign) {
  return __uint_as_float((sign << 31) | (static_cast<uint32_t>(e + 127) << 23) | (mant & 0x7FFFFFu));
}

// x for divisor y (kind as above) from the 64 random bits h.
__device__ float draw_x(int kind, float y, uint64_t h) {
  const uint32_t sign = static_cast<uint32_t>(h >> 63);
  const int ey = static_cast<int>((__float_as_uint(y) >> 23) & 0xFF) - 127;
  if (kind == 1) {
    const float t[21] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f,
                         0x1p-10f, 0x1.2p-9f, 17.0f, 272.0f, 432.0f, 448.0f, 464.0f};
    const float base = __fmul_rn(t[(h & 0xFFFF) % 21], y);
    const int k = static_cast<int>((h >> 16) % 33) - 16;
    return __uint_as_float((__float_as_uint(base) + k) | (sign << 31));
  }
  if (kind == 3) {  // a BF16 value: 7 random significand bits
    const int e = ey + static_cast<int>((h & 0xFFFF) % 21) - 12;
    return make_float(e, static_cast<uint32_t>(h >> 16) & 0x7F0000u, sign);
  }
  const int eq = static_cast<int>((h & 0xFFFF) % 54) - 45;
  return make_float(ey + eq, static_cast<uint32_t>(h >> 16), sign);
}

// Pair j: one divisor y and two dividends.
__device__ void draw(uint64_t j, uint64_t seed, float& x0, float& x1, float& y) {
  const uint64_t h1 = splitmix64(seed + 3 * j), h2 = splitmix64(seed + 3 * j + 1), h3 = splitmix64(seed + 3 * j + 2);
  const int kind = static_cast<int>(j & 3);
  if (kind == 3) {
    const uint32_t c = 1 + static_cast<uint32_t>((h1 & 0xFFFF) % 126);
    const float s = make_float(static_cast<int>((h1 >> 16) % 81) - 40, static_cast<uint32_t>(h1 >> 24), 0);
    y = __fmul_rn(bsg::ue4m3_value(c), s);
  } else {
    const int ey = static_cast<int>((h1 & 0xFF) % 129) - 64;
    y = make_float(ey, kind == 2 ? 0x7FFFFFu : static_cast<uint32_t>(h1 >> 8), 0);
  }
  x0 = draw_x(kind, y, h2);
  x1 = draw_x(kind, y, h3);
}

__global__ void division_probe_kernel(uint64_t n, uint64_t seed, unsigned long long* out) {
  unsigned long long tested = 0, qbad = 0, cbad = 0;
  for (uint64_t j = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; 2 * j < n;
       j += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    float x0, x1, y;
    draw(j, seed, x0, x1, y);
    if (!bsg::markstein_range(y)) continue;
    const float r = __frcp_rn(y);
    if (!isfinite(x0) || !isfinite(x1) || fabsf(__fmul_rn(x0, r)) > 0x1p64f || fabsf(__fmul_rn(x1, r)) > 0x1p64f)
      continue;
    float q0, q1;
    bsg::div2_markstein(x0, x1, r, -y, q0, q1);
    const float s0 = bsg::div_markstein(x0, r, -y), s1 = bsg::div_markstein(x1, r, -y);
    const float w0 = __fdiv_rn(x0, y), w1 = __fdiv_rn(x1, y);
    tested += 2;
    const float got[4] = {q0, q1, s0, s1}, want[4] = {w0, w1, w0, w1}, xs[4] = {x0, x1, x0, x1};
    for (int k = 0; k < 4; ++k) {
      const bool big = fabsf(want[k]) >= 0x1p-39f || want[k] == 0.0f;
      const bool qdiff = big && __float_as_uint(got[k]) != __float_as_uint(want[k]);
      const bool cdiff = bsg::cvt_e2m1x2(got[k], 0.0f) != bsg::cvt_e2m1x2(want[k], 0.0f) ||
                         bsg::cvt_e4m3x2(got[k], 0.0f) != bsg::cvt_e4m3x2(want[k], 0.0f);
      if (qdiff) ++qbad;
      if (cdiff) ++cbad;
      if (qdiff || cdiff) {
        out[3] = __float_as_uint(xs[k]);
        out[4] = __float_as_uint(y);
      }
    }
  }
  atomicAdd(out + 0, tested);
  if (qbad) atomicAdd(out + 1, qbad);
  if (cbad) atomicAdd(out + 2, cbad);
}

}  // namespace

// n dividends (two per divisor), generator seed; out: 5 unsigned 64-bit counters in device
// memory, zeroed by the caller.  Returns the launch's cudaError_t.
extern "C" __attribute__((visibility("default"))) int division_probe(unsigned long long n, unsigned long long seed,
                                                                     void* out, void* stream) {
  division_probe_kernel<<<152 * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      n, seed, static_cast<unsigned long long*>(out));
  return static_cast<int>(cudaGetLastError());
}
