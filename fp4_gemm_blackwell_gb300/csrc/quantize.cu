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
// Every byte of the swizzled scale buffer, padding included, is written by the call.
#include <atomic>
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

// 16-byte words already loaded -> float32 elements (four per word for float32 input, eight for BF16).
template <typename T, int W, int N>
__device__ __forceinline__ void unpack_f32(const uint4 (&raw)[W], float (&v)[N]) {
  static_assert(N == W * 16 / static_cast<int>(sizeof(T)), "element count");
#pragma unroll
  for (int j = 0; j < W; ++j) {
    const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if constexpr (sizeof(T) == 4) {
        v[4 * j + h] = __uint_as_float(w[h]);
      } else {
        v[8 * j + 2 * h] = __uint_as_float(w[h] << 16);
        v[8 * j + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
      }
    }
  }
}

// Position (r, c) of a block in a rows x nblk matrix of blocks, moved by a fixed number of blocks
// (step = sr * nblk + sc, 0 <= sc < nblk) without a division.
struct BlockCursor {
  int r, c;
  __device__ __forceinline__ void forward(int sr, int sc, int nblk) {
    c += sc;
    r += sr;
    if (c >= nblk) {
      c -= nblk;
      ++r;
    }
  }
  __device__ __forceinline__ void backward(int sr, int sc, int nblk) {
    c -= sc;
    r -= sr;
    if (c < 0) {
      c += nblk;
      --r;
    }
  }
};

// Zero every scale byte of the padded (rows rounded up to 128) x (cols4 * 4) scale matrix outside
// the rows x nblk blocks: the columns past nblk of each row, then the rows past `rows`.  Thread t of
// `stride` takes entries t, t + stride, ...
__device__ __forceinline__ void sf_zero_padding(uint8_t* __restrict__ sf, int rows, int nblk, int cols4, long long t,
                                                long long stride) {
  const int cols_pad = cols4 * 4, padc = cols_pad - nblk;
  const int rows_pad = (rows + 127) / 128 * 128;
  const long long n_right = static_cast<long long>(rows) * padc;
  const long long n_all = n_right + static_cast<long long>(rows_pad - rows) * cols_pad;
  for (long long q = t; q < n_all; q += stride) {
    int r, c;
    if (q < n_right) {
      r = static_cast<int>(q / padc);
      c = nblk + static_cast<int>(q % padc);
    } else {
      const long long u = q - n_right;
      r = rows + static_cast<int>(u / cols_pad);
      c = static_cast<int>(u % cols_pad);
    }
    sf[sf_swizzle_offset(r, c, cols4)] = 0;
  }
}

// MXFP8, 64 bytes a thread: each thread reads 64 contiguous input bytes (the matrix read as one
// row-major run of 32-element blocks), a whole BF16 block or half of a float32 block (the two
// halves in neighbouring lanes share the amax by a shuffle), U blocks a grid stride apart loaded
// before any is encoded.  The loop runs while the first block of the thread's warp is in the
// matrix, so that every lane takes the shuffles.  (A warp reading 512 contiguous bytes an
// instruction, eight lanes to a float32 block, was measured slower: it repeats the block's
// exponent and shuffles in every lane.)
template <typename T, int U>
__global__ void __launch_bounds__(256) quantize_mx_kernel(const T* __restrict__ x, int rows, int K,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ sf, int cols4) {
  constexpr int LPB = static_cast<int>(sizeof(T)) / 2;  // threads per 32-element block
  constexpr int EPL = 32 / LPB;                          // elements per thread (64 bytes)
  const int nblk = K / 32;
  const long long nb = static_cast<long long>(rows) * nblk;
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x / LPB;  // blocks between iterations
  const int half = static_cast<int>(threadIdx.x) & (LPB - 1);
  const int sr = static_cast<int>(step / nblk), sc = static_cast<int>(step % nblk);
  BlockCursor cur{static_cast<int>((t / LPB) / nblk), static_cast<int>((t / LPB) % nblk)};
  for (long long first = (t & ~31LL) / LPB; first < nb; first += U * step) {
    BlockCursor at[U];
    uint4 raw[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      at[u] = cur;
      cur.forward(sr, sc, nblk);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (at[u].r < rows) {
        const uint4* src = reinterpret_cast<const uint4*>(
            x + (static_cast<long long>(at[u].r) * nblk + at[u].c) * 32 + half * EPL);
#pragma unroll
        for (int w = 0; w < 4; ++w) raw[u][w] = __ldg(src + w);
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) raw[u][w] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float v[EPL];
      unpack_f32<T, 4>(raw[u], v);
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < EPL; ++j) amax = fmaxf(amax, fabsf(v[j]));
      if constexpr (LPB == 2) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      const int e = mx_exponent(amax);
      const float inv = exp2_neg(e);
      uint32_t w[EPL / 4];
#pragma unroll
      for (int j = 0; j < EPL / 4; ++j) {
        float p0, p1, p2, p3;
        fmul2_rn(v[4 * j], v[4 * j + 1], inv, inv, p0, p1);
        fmul2_rn(v[4 * j + 2], v[4 * j + 3], inv, inv, p2, p3);
        w[j] = cvt_e4m3x2(p0, p1) | (cvt_e4m3x2(p2, p3) << 16);
      }
      if (at[u].r < rows) {
        uint4* dst = reinterpret_cast<uint4*>(codes + (static_cast<long long>(at[u].r) * nblk + at[u].c) * 32 +
                                              half * EPL);
#pragma unroll
        for (int q = 0; q < EPL / 16; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        if (half == 0) sf[sf_swizzle_offset(at[u].r, at[u].c, cols4)] = static_cast<uint8_t>(e + 127);
      }
    }
  }
  sf_zero_padding(sf, rows, nblk, cols4, t, static_cast<long long>(gridDim.x) * blockDim.x);
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

// NVFP4: one thread per 16-element block, U blocks (a grid stride apart) loaded before any is
// encoded.  The blocks are visited from the end of the matrix backwards: the amax pass that precedes
// this one read the matrix from the start, so its last rows are the ones still in L2.
// SCALED: the global scale s is given (*scale_in, a float) instead of derived from the amax
// pass's result (*scale_in holding the amax's bits).
template <typename T, bool SCALED, int U>
__global__ void __launch_bounds__(256) quantize_nv_kernel(const T* __restrict__ x, int rows, int K,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ sf, int cols4,
                                                          const unsigned* __restrict__ scale_in) {
  constexpr int W = static_cast<int>(sizeof(T));  // 16-byte words per block
  const NvTensorScale ts = nv_tensor_scale(SCALED ? __uint_as_float(*scale_in)
                                                  : __fdiv_rn(__uint_as_float(*scale_in), 2688.0f));
  const int nblk = K / 16;
  const long long nb = static_cast<long long>(rows) * nblk;
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const int sr = static_cast<int>(stride / nblk), sc = static_cast<int>(stride % nblk);
  BlockCursor cur{-1, 0};
  if (t < nb) {
    const long long b = nb - 1 - t;
    cur.r = static_cast<int>(b / nblk);
    cur.c = static_cast<int>(b % nblk);
  }
  while (cur.r >= 0) {
    BlockCursor at[U];
    uint4 raw[U][W];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      at[u] = cur;
      cur.backward(sr, sc, nblk);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (at[u].r >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(
            x + (static_cast<long long>(at[u].r) * nblk + at[u].c) * 16);
#pragma unroll
        for (int w = 0; w < W; ++w) raw[u][w] = __ldg(src + w);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (at[u].r >= 0) {
        float v[16];
        unpack_f32<T, W>(raw[u], v);
        uint32_t lo, hi;
        const uint32_t scode = nv_encode_block16(v, ts, lo, hi);
        *reinterpret_cast<uint2*>(codes + (static_cast<long long>(at[u].r) * nblk + at[u].c) * 8) =
            make_uint2(lo, hi);
        sf[sf_swizzle_offset(at[u].r, at[u].c, cols4)] = static_cast<uint8_t>(scode);
      }
    }
  }
  sf_zero_padding(sf, rows, nblk, cols4, t, stride);
}

__global__ void nv_finalize_kernel(float* global_scale) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned*>(global_scale));
  *global_scale = __fdiv_rn(amax, 2688.0f);
}

// CTAs of 256 threads of KERNEL resident on one SM, asked of the runtime once per kernel (a
// failed query gives 1 and is asked again next time; its error is cleared so that the launch
// reports its own).
template <auto KERNEL>
static int resident_ctas() {
  static std::atomic<int> cached{0};
  int n = cached.load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, KERNEL, 256, 0) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      return 1;
    }
    cached.store(n, std::memory_order_relaxed);
  }
  return n;
}

// A persistent grid: as many CTAs of 256 threads as are resident on `sms` SMs at once, fewer when
// `threads` are enough for the work.
template <auto KERNEL>
static int persistent_grid(long long threads, int sms) {
  const long long need = (threads + 255) / 256;
  const long long full = static_cast<long long>(resident_ctas<KERNEL>()) * (sms > 0 ? sms : 1);
  return static_cast<int>(need < 1 ? 1 : (need < full ? need : full));
}

// Blocks a thread loads before it encodes any: NVFP4 with BF16 input has the most arithmetic per
// input byte and gains from two; the others keep one (measured on 8192 x 8192 inputs).
template <typename T>
constexpr int nv_unroll() {
  return sizeof(T) == 2 ? 2 : 1;
}

// MXFP8: 16 CTAs of 256 threads per SM at most (several waves of the grid-stride loop), one
// 64-byte input segment a thread at a time.
template <typename T>
cudaError_t quantize_mx(const T* x, int rows, int K, uint8_t* codes, uint8_t* sf, int sms, cudaStream_t s) {
  const int cols4 = (K / 32 + 3) / 4;
  const long long threads = static_cast<long long>(rows) * (K / 32) * (static_cast<int>(sizeof(T)) / 2);
  long long grid = (threads + 255) / 256;
  const long long cap = 16LL * (sms > 0 ? sms : 1);
  grid = grid < 1 ? 1 : (grid < cap ? grid : cap);
  quantize_mx_kernel<T, 1><<<static_cast<int>(grid), 256, 0, s>>>(x, rows, K, codes, sf, cols4);
  return cudaGetLastError();
}

template <typename T, bool SCALED>
static cudaError_t launch_nv(const T* x, int rows, int K, uint8_t* codes, uint8_t* sf, const unsigned* scale_in,
                             int sms, cudaStream_t s) {
  const int cols4 = (K / 16 + 3) / 4;
  constexpr int U = nv_unroll<T>();
  const long long nb = static_cast<long long>(rows) * (K / 16);
  quantize_nv_kernel<T, SCALED, U><<<persistent_grid<quantize_nv_kernel<T, SCALED, U>>((nb + U - 1) / U, sms), 256, 0,
                                     s>>>(x, rows, K, codes, sf, cols4, scale_in);
  return cudaGetLastError();
}

template <typename T>
cudaError_t quantize_nv(const T* x, int rows, int K, uint8_t* codes, uint8_t* sf, float* global_scale, int sms,
                        cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(global_scale, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(rows) * K;
  const int grid = persistent_grid<amax_kernel<T>>(n / 32, sms);  // 32 elements a thread an iteration
  amax_kernel<T><<<grid, 256, 0, s>>>(x, n, reinterpret_cast<unsigned*>(global_scale));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_nv<T, false>(x, rows, K, codes, sf, reinterpret_cast<unsigned*>(global_scale), sms, s);
  if (e != cudaSuccess) return e;
  nv_finalize_kernel<<<1, 1, 0, s>>>(global_scale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_nv_scaled(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                                      const float* global_scale, int sms, cudaStream_t s) {
  return launch_nv<float, true>(x, rows, K, codes, sf, reinterpret_cast<const unsigned*>(global_scale), sms, s);
}
cudaError_t launch_quantize_nv_scaled(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                                      const float* global_scale, int sms, cudaStream_t s) {
  return launch_nv<uint16_t, true>(x, rows, K, codes, sf, reinterpret_cast<const unsigned*>(global_scale), sms, s);
}

cudaError_t launch_quantize_mx(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf, int sms,
                               cudaStream_t s) {
  return quantize_mx(x, rows, K, codes, sf, sms, s);
}
cudaError_t launch_quantize_mx(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf, int sms,
                               cudaStream_t s) {
  return quantize_mx(x, rows, K, codes, sf, sms, s);
}
cudaError_t launch_quantize_nv(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                               float* global_scale, int sms, cudaStream_t s) {
  return quantize_nv(x, rows, K, codes, sf, global_scale, sms, s);
}
cudaError_t launch_quantize_nv(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                               float* global_scale, int sms, cudaStream_t s) {
  return quantize_nv(x, rows, K, codes, sf, global_scale, sms, s);
}

}  // namespace bsg
