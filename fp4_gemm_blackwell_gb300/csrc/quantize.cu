// Quantisers: row-major float32 or BF16 -> block-scaled codes + swizzled 128x4 scale atoms.
// A BF16 input is widened to float32 exactly (its bits are the upper half of the float32's),
// so it quantises to the same bytes as its float32 value.
//
// MXFP8 ("Add Cutlass MxFp8 Block Scale Matrix Multiplication", test step
// pytorch_mxfp8_quantize with block size 32, then linear_to_swizzled_128_4): per 32-element
// K-block, scale 2^e with e the least integer such that amax <= 448 * 2^e, elements E4M3 of
// x * 2^-e rounded to nearest even with saturation.
// NVFP4 (the Nvf4 kernels of "[QST] Performance overhead ..."): s = amax / 2688 per tensor,
// per 16-element block UE4M3(amax_blk / (6 s)), elements E2M1(x / (scale * s)); each step one
// float32 operation rounded to nearest even.
//
// One thread per (row, block) of the PADDED scale matrix, so every byte of the swizzled scale
// buffer, padding included, is written by the call.
#include <cstdint>

#include "bsg_internal.h"
#include "nvfp4_codec.cuh"
#include "ptx.cuh"

namespace bsg {

// e = least integer with a <= 448 * 2^e, clamped to [-127, 127], for finite a >= 0.
// With a = (1 + f) 2^(E-127) (E the biased exponent field) and 448 = 1.75 * 2^8:
// a <= 448 * 2^e  <=>  e >= E - 135 when f <= 0.75, else e >= E - 134.
__device__ __forceinline__ int mx_exponent(float a) {
  const uint32_t bits = __float_as_uint(a);
  const int E = static_cast<int>(bits >> 23);
  const uint32_t frac = bits & 0x7FFFFFu;
  if (E == 0) return -127;  // zero or subnormal: far below 448 * 2^-127
  int e = E - 135 + (frac > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as float32 for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2_neg(int e) {
  const int be = 127 - e;
  return be >= 1 ? __uint_as_float(static_cast<uint32_t>(be) << 23) : __uint_as_float(0x00400000u);
}

// N consecutive input elements as float32: float4 loads, or 16-byte loads of eight BF16 each.
template <int N>
__device__ __forceinline__ void load_f32(const float* p, float (&v)[N]) {
  const float4* src = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    const float4 t = __ldg(src + j);
    v[4 * j] = t.x;
    v[4 * j + 1] = t.y;
    v[4 * j + 2] = t.z;
    v[4 * j + 3] = t.w;
  }
}
template <int N>
__device__ __forceinline__ void load_f32(const uint16_t* p, float (&v)[N]) {
  const uint4* src = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int j = 0; j < N / 8; ++j) {
    const uint4 t = __ldg(src + j);
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * j + 2 * h] = __uint_as_float(w[h] << 16);
      v[8 * j + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
    }
  }
}

// I: the index type of the (row, block) loop, 32-bit unsigned whenever the padded scale matrix has
// fewer than 2^32 entries (a 64-bit division per block costs about as much as the block's
// arithmetic).
template <typename T, typename I>
__global__ void __launch_bounds__(256) quantize_mx_kernel(const T* __restrict__ x, int rows, int K,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ sf, int rows_pad,
                                                          int cols4) {
  const int nblk = K / 32;
  const I cols_pad = static_cast<I>(cols4) * 4;
  const I total = static_cast<I>(rows_pad) * cols_pad;
  for (I i = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<I>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / cols_pad);
    const int c = static_cast<int>(i % cols_pad);
    uint8_t code = 0;
    if (r < rows && c < nblk) {
      float v[32];
      load_f32(x + static_cast<size_t>(r) * K + c * 32, v);
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
      const int e = mx_exponent(amax);
      const float inv = exp2_neg(e);
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(v[4 * j], inv), __fmul_rn(v[4 * j + 1], inv));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(v[4 * j + 2], inv), __fmul_rn(v[4 * j + 3], inv));
        w[j] = lo | (hi << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(codes + static_cast<size_t>(r) * K + c * 32);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      code = static_cast<uint8_t>(e + 127);
    }
    sf[sf_swizzle_offset(r, c, cols4)] = code;
  }
}

// amax(|x|) into *amax_bits (float bits; non-negative floats order like unsigned integers).
// n is a multiple of 32 (K % 32 == 0): eight elements per step.
template <typename T>
__global__ void __launch_bounds__(256) amax_kernel(const T* __restrict__ x, long long n,
                                                   unsigned* __restrict__ amax_bits) {
  float m = 0.0f;
  const long long n8 = n / 8;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  // four groups of eight per thread in flight at once, then the remainder one group at a time
  for (; i + 3 * step < n8; i += 4 * step) {
    float v[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) load_f32(x + (i + u * step) * 8, v[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[u][j]));
  }
  for (; i < n8; i += step) {
    float v[8];
    load_f32(x + i * 8, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.0f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) b = fmaxf(b, wmax[w]);
    atomicMax(amax_bits, __float_as_uint(b));
  }
}

// The (row, block) entries are visited from the end of the matrix backwards: the amax pass that
// precedes this one read the matrix from the start, so its last rows are the ones still in L2.
// SCALED: the global scale s is given (*scale_in, a float) instead of derived from the amax
// pass's result (*scale_in holding the amax's bits).
template <typename T, typename I, bool SCALED>
__global__ void __launch_bounds__(256) quantize_nv_kernel(const T* __restrict__ x, int rows, int K,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ sf, int rows_pad,
                                                          int cols4,
                                                          const unsigned* __restrict__ scale_in) {
  const float s = SCALED ? __uint_as_float(*scale_in) : __fdiv_rn(__uint_as_float(*scale_in), 2688.0f);
  const float d = __fmul_rn(6.0f, s);
  const int nblk = K / 16;
  const I cols_pad = static_cast<I>(cols4) * 4;
  const I total = static_cast<I>(rows_pad) * cols_pad;
  for (I j = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; j < total;
       j += static_cast<I>(gridDim.x) * blockDim.x) {
    const I i = total - 1 - j;
    const int r = static_cast<int>(i / cols_pad);
    const int c = static_cast<int>(i % cols_pad);
    uint8_t code = 0;
    if (r < rows && c < nblk) {
      float v[16];
      load_f32(x + static_cast<size_t>(r) * K + c * 16, v);
      uint32_t lo, hi;
      const uint32_t sc = nv_encode_block16(v, s, d, lo, hi);
      *reinterpret_cast<uint2*>(codes + static_cast<size_t>(r) * (K / 2) + c * 8) = make_uint2(lo, hi);
      code = static_cast<uint8_t>(sc);
    }
    sf[sf_swizzle_offset(r, c, cols4)] = code;
  }
}

__global__ void nv_finalize_kernel(float* global_scale) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned*>(global_scale));
  *global_scale = __fdiv_rn(amax, 2688.0f);
}

static int grid_for(long long n, int threads) {
  long long b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > 152 * 16) b = 152 * 16;
  return static_cast<int>(b);
}

template <typename T>
cudaError_t quantize_mx(const T* x, int rows, int K, uint8_t* codes, uint8_t* sf, cudaStream_t s) {
  const int rows_pad = (rows + 127) / 128 * 128;
  const int cols4 = (K / 32 + 3) / 4;
  const long long total = static_cast<long long>(rows_pad) * cols4 * 4;
  if (total < (1LL << 32))
    quantize_mx_kernel<T, uint32_t><<<grid_for(total, 256), 256, 0, s>>>(x, rows, K, codes, sf, rows_pad, cols4);
  else
    quantize_mx_kernel<T, unsigned long long><<<grid_for(total, 256), 256, 0, s>>>(x, rows, K, codes, sf, rows_pad,
                                                                                     cols4);
  return cudaGetLastError();
}

template <typename T>
cudaError_t quantize_nv(const T* x, int rows, int K, uint8_t* codes, uint8_t* sf, float* global_scale,
                        cudaStream_t s) {
  const int rows_pad = (rows + 127) / 128 * 128;
  const int cols4 = (K / 16 + 3) / 4;
  const long long total = static_cast<long long>(rows_pad) * cols4 * 4;
  cudaError_t e = cudaMemsetAsync(global_scale, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(rows) * K;
  amax_kernel<T><<<grid_for(n / 8, 256), 256, 0, s>>>(x, n, reinterpret_cast<unsigned*>(global_scale));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (total < (1LL << 32))
    quantize_nv_kernel<T, uint32_t, false><<<grid_for(total, 256), 256, 0, s>>>(
        x, rows, K, codes, sf, rows_pad, cols4, reinterpret_cast<unsigned*>(global_scale));
  else
    quantize_nv_kernel<T, unsigned long long, false><<<grid_for(total, 256), 256, 0, s>>>(
        x, rows, K, codes, sf, rows_pad, cols4, reinterpret_cast<unsigned*>(global_scale));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  nv_finalize_kernel<<<1, 1, 0, s>>>(global_scale);
  return cudaGetLastError();
}

// NVFP4 with the global scale given: one pass, no amax.
template <typename T>
cudaError_t quantize_nv_scaled(const T* x, int rows, int K, uint8_t* codes, uint8_t* sf, const float* global_scale,
                               cudaStream_t s) {
  const int rows_pad = (rows + 127) / 128 * 128;
  const int cols4 = (K / 16 + 3) / 4;
  const long long total = static_cast<long long>(rows_pad) * cols4 * 4;
  const unsigned* sc = reinterpret_cast<const unsigned*>(global_scale);
  if (total < (1LL << 32))
    quantize_nv_kernel<T, uint32_t, true><<<grid_for(total, 256), 256, 0, s>>>(x, rows, K, codes, sf, rows_pad,
                                                                               cols4, sc);
  else
    quantize_nv_kernel<T, unsigned long long, true><<<grid_for(total, 256), 256, 0, s>>>(x, rows, K, codes, sf,
                                                                                         rows_pad, cols4, sc);
  return cudaGetLastError();
}

cudaError_t launch_quantize_nv_scaled(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                                      const float* global_scale, cudaStream_t s) {
  return quantize_nv_scaled(x, rows, K, codes, sf, global_scale, s);
}
cudaError_t launch_quantize_nv_scaled(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                                      const float* global_scale, cudaStream_t s) {
  return quantize_nv_scaled(x, rows, K, codes, sf, global_scale, s);
}

cudaError_t launch_quantize_mx(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                               cudaStream_t s) {
  return quantize_mx(x, rows, K, codes, sf, s);
}
cudaError_t launch_quantize_mx(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                               cudaStream_t s) {
  return quantize_mx(x, rows, K, codes, sf, s);
}
cudaError_t launch_quantize_nv(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                               float* global_scale, cudaStream_t s) {
  return quantize_nv(x, rows, K, codes, sf, global_scale, s);
}
cudaError_t launch_quantize_nv(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                               float* global_scale, cudaStream_t s) {
  return quantize_nv(x, rows, K, codes, sf, global_scale, s);
}

}  // namespace bsg
