// Block-scaled GEMM kernel for sm_103a: D = alpha * (A . B^T) (+ bias[n]) (-> SiLU).
//
// One persistent CTA per SM, sixteen warps in four warpgroups with fixed roles:
//   warp 0       TMA producer of the A / B code tiles (128-byte swizzled) into a STAGES-deep
//                shared-memory ring (mbarrier full / empty pairs);
//   warp 1       owns tensor memory and issues the block-scaled tcgen05.mma chain into an FP32
//                accumulator;
//   warp 2       TMA producer of the matching 128x4 scale atoms (same stages, same barriers);
//   warps 4..7   scale warps: copy each stage's scale atoms into a TMEM slot (tcgen05.st);
//   warps 8..15  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes 32*(w%4)..,
//                warps 8..11 the first half of the columns, warps 12..15 the second half),
//                alpha, bias, SiLU, FP16/BF16 rounding and stores; with split-K, FP32 partial
//                tiles reduced inside a thread-block cluster or through the workspace.
// Tile 128 x BN x (128 bytes of K): MXFP8 = 128 E4M3 per row per stage (four K=32 MMAs, one
// UE8M0 scale each), NVFP4 = 256 E2M1 per row per stage (four K=64 MMAs, four UE4M3 each).
//
// The operation, formats and the 1-SM 128-row tile follow "Add Cutlass MxFp8 Block Scale
// Matrix Multiplication" (MxFp8GemmSm100, PerSmTileShape 128 x 256 x 256) and "[QST]
// Performance overhead ..." (KernelConfigM128: 1-SM 128 x 256 tiles; runNvfp4Gemm with the
// kEnableBias / kEnableSilu epilogue), re-derived for a persistent, warp-specialised schedule.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bsg_internal.h"
#include "nvfp4_codec.cuh"
#include "ptx.cuh"

namespace bsg {

// KC = k-slabs of 128 bytes of K per ring stage (one barrier wait and one commit per stage).
template <int KIND, int BN, int KC>
struct GemmCfg {
  static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 256, "tile width");
  static_assert(KC == 1 || KC == 2, "k-slabs per stage");
  static constexpr int BM = 128;
  static constexpr int BK_BYTES = 128;
  static constexpr int K_TILE = KC * (KIND == KIND_MX ? 128 : 256);  // elements per stage
  static constexpr int MMA_K = KIND == KIND_MX ? 32 : 64;            // elements per MMA
  static constexpr int STEPS = K_TILE / MMA_K;                       // MMAs per stage (4 a slab)
  static constexpr int SF_ATOMS = KC * (KIND == KIND_MX ? 1 : 4);    // 128x4 atoms per band per stage
  static constexpr int NB = BN >= 128 ? BN / 128 : 1;                // 128-row scale bands of B per tile
  static constexpr int SLAB_A = BM * BK_BYTES;                       // one 128-byte k-slab of A
  static constexpr int SLAB_B = BN * BK_BYTES;
  static constexpr int A_BYTES = KC * SLAB_A;
  static constexpr int B_BYTES = KC * SLAB_B;
  static constexpr int SFA_BYTES = SF_ATOMS * 512;
  static constexpr int SFB_BYTES = NB * SF_ATOMS * 512;
  static constexpr int STAGE_RAW = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_RAW + 1023) / 1024 * 1024;
  static constexpr int SMEM_LIMIT = 232448;  // 227 KB per CTA
  static constexpr int AUX_BYTES = 1024;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - AUX_BYTES - 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + AUX_BYTES + 1024;
  static constexpr int NACC = BN <= 128 ? 2 : 1;             // accumulator buffers in TMEM
  static constexpr int SFA_COLS = 4 * SF_ATOMS;
  static constexpr int SFB_COLS = 4 * SF_ATOMS * NB;
  static constexpr int SF_SLOT_COLS = SFA_COLS + SFB_COLS;
  static constexpr int SF_COL0 = NACC * BN;
  // Scale atoms reach TMEM through four scale warps that write them into a TMEM slot per ring
  // stage with tcgen05.st: a tcgen05.cp per atom would occupy the tensor pipe (about 84 cycles
  // each, 3 per MXFP8 and 12 per NVFP4 k-tile of a 256-wide tile) next to 512 cycles of MMAs.
  // Tiles narrower than a 128-row scale band use only a quarter or a half of each B atom, which
  // the scale warps move to the slot's first columns (every scale address the MMA gets stays a
  // multiple of four columns).
  static constexpr int SF_SLOTS = STAGES;
  static constexpr int TMEM_USED = SF_COL0 + SF_SLOTS * SF_SLOT_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
  static constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter, each owning half the columns
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  // Sixteen warps in four warpgroups: {A/B producer, MMA, scale producer, idle}, the four scale
  // warps, and the eight epilogue warps.  With 16 warps the launch gives every thread 128
  // registers; the first two warpgroups hand registers to the epilogue (setmaxnreg), whose
  // 256-wide tiles need about 180.
  static constexpr int SCALE_WARP0 = 4;
  static constexpr int EPI_WARP0 = 8;  // first epilogue warp
  static constexpr int THREADS = 32 * EPI_WARP0 + EPI_THREADS;
  static constexpr int REGS_CTRL = 56, REGS_SCALE = 80, REGS_EPI = 184;
  // per SM sub-partition (one warp of each warpgroup): 56 + 80 + 2 x 184 <= 512 registers a lane
  static_assert(REGS_CTRL + REGS_SCALE + 2 * REGS_EPI <= 512, "register split");
  static_assert(THREADS == 512, "warpgroup layout");
  // Instruction descriptor (block-scaled kinds): [4,6) B scale id, [7,10) A type,
  // [10,13) B type, [15]/[16] A/B major (0 = K), [17,23) N >> 3, [23] scale type
  // (1 = UE8M0, 0 = UE4M3), [24,29) M >> 4, [29,31) A scale id.
  static constexpr uint32_t IDESC =
      (KIND == KIND_MX ? ((0u << 7) | (0u << 10) | (1u << 23))    // E4M3 x E4M3, UE8M0
                       : ((1u << 7) | (1u << 10) | (0u << 23)))   // E2M1 x E2M1, UE4M3
      | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
  static_assert(STAGES >= 2, "ring too shallow");
  static_assert(STAGES <= 8, "barrier slots");
  static_assert(TMEM_USED <= 512, "tensor memory");
  static_assert(SF_ATOMS <= 4 || SF_ATOMS % 4 == 0, "scale-warp stores");
};

struct UnitCoord {
  int m_blk, n_blk, split, tile, kt0, kt1;
  int batch;  // entry of A, SFA, D and C
  int bsel;   // entry of B, SFB and alpha_dev: the batch entry, or the tile's group when grouped
  bool skip;  // grouped: the tile has no group (every role passes over it)
};

// Unit u (a tile, or one split of a tile, of batch entry u / units_per_batch) -> tile
// coordinates and k range.  `tile` is the tile's index over all entries (the workspace's).
// Batch entries and groups exist only in the EXT instantiations; elsewhere c.batch and c.bsel
// are the constant 0 and every entry offset folds away.  Grouped (1-SM tiles), the tile's group
// is that of its first row.
template <bool EXT>
__device__ __forceinline__ UnitCoord decode_unit(const GemmParams& p, int u) {
  UnitCoord c;
  c.batch = 0;
  int tile0 = 0;  // tiles of the entries before this one
  if (EXT && p.batches > 1) {
    c.batch = u / p.units_per_batch;
    u -= c.batch * p.units_per_batch;
    tile0 = c.batch * (p.units_per_batch / p.splits);
  }
  c.split = u % p.splits;
  const int t = u / p.splits;
  c.tile = tile0 + t;
  const int per_group = p.group_m * p.num_n_tiles;
  const int g = t / per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.num_m_tiles - first_m, p.group_m);
  const int r = t - g * per_group;
  c.m_blk = first_m + r % gm;
  c.n_blk = r / gm;
  c.kt0 = c.split * p.k_tiles_per_split;
  c.kt1 = min(c.kt0 + p.k_tiles_per_split, p.num_k_tiles);
  c.bsel = c.batch;
  c.skip = false;
  if (EXT && p.group_index != nullptr) {
    const int r0 = c.m_blk * 128;
    const int grp = r0 < p.M ? __ldg(p.group_index + r0) : -1;
    c.bsel = grp;
    c.skip = grp < 0 || grp >= p.b_entries;
  }
  return c;
}

// Whether output row m of unit c is stored: inside M and, grouped, in the unit's group.
template <bool EXT>
__device__ __forceinline__ bool row_live(const GemmParams& p, const UnitCoord& c, int m) {
  if (m >= p.M) return false;
  return !(EXT && p.group_index != nullptr) || __ldg(p.group_index + m) == c.bsel;
}

// The unit's alpha: the plan's, or (EXT, device alpha with several B entries) its entry's.
template <bool EXT>
__device__ __forceinline__ float unit_alpha(const GemmParams& p, const UnitCoord& c, float alpha) {
  return (EXT && (p.flags & F_ALPHA_DEVICE) && p.b_entries > 1) ? __ldg(p.alpha_dev + c.bsel) : alpha;
}

// Bounded mbarrier wait.  Gives up when another role flagged an abort, or after the
// plan's time limit (then flags the abort and records `who` in the status word).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             const GemmParams& p, unsigned who) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > p.wait_limit_ns) {
      *abort_flag = 1;
      atomicOr(p.status, who);
      return false;
    }
  }
}

// The same for barriers that threads of another CTA of the cluster arrive on (acquire at
// cluster scope).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                     const GemmParams& p, unsigned who) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > p.wait_limit_ns) {
      *abort_flag = 1;
      atomicOr(p.status, who);
      return false;
    }
  }
}

// The same wait performed by a whole warp, which leaves it together: every lane polls (each
// acquiring the barrier's phase for itself), and the loop's exit is decided by warp votes, so the
// warp stays converged and values computed after the wait stay warp-uniform.
__device__ __forceinline__ bool wait_bounded_cluster_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                          const GemmParams& p, unsigned who) {
  if (__all_sync(0xffffffffu, mbar_try_wait_cluster(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait_cluster(bar, parity))) return true;
    const bool aborted = *abort_flag != 0;
    const bool late = globaltimer_ns() - t0 > p.wait_limit_ns;
    if (__any_sync(0xffffffffu, aborted || late)) {
      if ((threadIdx.x & 31) == 0 && !aborted) {
        *abort_flag = 1;
        atomicOr(p.status, who);
      }
      __syncwarp();
      return false;
    }
  }
}

// The same at CTA scope (barriers only this CTA's threads and copies arrive on).
__device__ __forceinline__ bool wait_bounded_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  const GemmParams& p, unsigned who) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const bool aborted = *abort_flag != 0;
    const bool late = globaltimer_ns() - t0 > p.wait_limit_ns;
    if (__any_sync(0xffffffffu, aborted || late)) {
      if ((threadIdx.x & 31) == 0 && !aborted) {
        *abort_flag = 1;
        atomicOr(p.status, who);
      }
      __syncwarp();
      return false;
    }
  }
}

// Named-barrier AND over `nthreads` threads: every participant gets the same answer.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "barrier.cta.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Two values rounded to the 16-bit output type and packed (BF16 for OUT_BF16, and for OUT_NV4,
// whose bias and C are BF16).
template <int OUT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (OUT == OUT_F16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int OUT>
__device__ __forceinline__ float out_to_float(uint16_t bits) {
  if constexpr (OUT == OUT_F16) {
    return __half2float(__ushort_as_half(bits));
  } else {
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  }
}

// 16 output values (8 packed words) of one row at d: one 32-byte store when D is 32-byte aligned
// (a whole L2 sector per lane; n is a multiple of 16 and N % 16 == 0), else two 16-byte stores.
__device__ __forceinline__ void st_out16(uint16_t* d, const uint32_t (&o)[8], bool wide) {
  if (wide) {
    st_global_v8(d, o);
  } else {
    reinterpret_cast<uint4*>(d)[0] = make_uint4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<uint4*>(d)[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// Row m of D (C) of batch entry b.
__device__ __forceinline__ uint16_t* d_row(const GemmParams& p, int b, int m) {
  return static_cast<uint16_t*>(p.d) + static_cast<size_t>(b) * p.d_batch + static_cast<size_t>(m) * p.N;
}
__device__ __forceinline__ const uint16_t* c_row(const GemmParams& p, int b, int m) {
  return static_cast<const uint16_t*>(p.c) + static_cast<size_t>(b) * p.c_batch + static_cast<size_t>(m) * p.N;
}

// alpha * alpha_row[m]: the part of the epilogue factor shared by a whole output row.
__device__ __forceinline__ float row_alpha(const GemmParams& p, float alpha, int m) {
  return ((p.flags & F_ALPHA_ROW) && m < p.M) ? __fmul_rn(alpha, __ldg(p.alpha_row + m)) : alpha;
}

// y * sigmoid(y) in place.  The reciprocal uses the fast division: an IEEE division takes a slow
// path whenever 1 + e^-y overflows (y < -88), which is common for long K; __fdividef(1, d)
// returns 0 for d > 2^126, the correctly rounded sigmoid there.
template <int W>
__device__ __forceinline__ void silu_inplace(float (&y)[W]) {
#pragma unroll
  for (int i = 0; i < W; ++i) y[i] = y[i] * __fdividef(1.0f, 1.0f + __expf(-y[i]));
}

// W consecutive values of the bias (output type) at column n, as float32.
template <int OUT, int W>
__device__ __forceinline__ void load_bias(const GemmParams& p, int n, float (&b)[W]) {
  uint16_t raw[W];
  if constexpr (W == 8)
    *reinterpret_cast<uint4*>(raw) = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.bias) + n));
  else
    *reinterpret_cast<uint2*>(raw) = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.bias) + n));
#pragma unroll
  for (int i = 0; i < W; ++i) b[i] = out_to_float<OUT>(raw[i]);
}

// Epilogue of W consecutive accumulator values v of one output row, columns n..n+W-1:
//   y = alpha * v[i] (+ bias[n+i]);  SiLU;  rounded to the output type and packed two per word.
// Columns at or beyond N read no bias.  The path of every problem without C or per-column
// factors (epi_pack_ext covers those).
template <int OUT, int W>
__device__ __forceinline__ void epi_vals(const GemmParams& p, int n, const float* v, float alpha, float* y) {
  static_assert(W == 4 || W == 8, "group width");
  if ((p.flags & F_BIAS) && n < p.N) {
    float b[W];
    load_bias<OUT, W>(p, n, b);
#pragma unroll
    for (int i = 0; i < W; ++i) y[i] = __fmaf_rn(alpha, v[i], b[i]);
  } else {
#pragma unroll
    for (int i = 0; i < W; ++i) y[i] = __fmul_rn(alpha, v[i]);
  }
  if (p.flags & F_SILU) silu_inplace(reinterpret_cast<float(&)[W]>(*y));
}
template <int OUT, int W>
__device__ __forceinline__ void epi_pack(const GemmParams& p, int n, const float* v, float alpha, uint32_t* out) {
  float y[W];
  epi_vals<OUT, W>(p, n, v, alpha, y);
#pragma unroll
  for (int i = 0; i < W / 2; ++i) out[i] = pack2<OUT>(y[2 * i], y[2 * i + 1]);
}

// The epilogue with the residual and per-column factors, on W values of row m at columns n..:
//   y = alpha_m * alpha_col[n+i] * v[i] + bias[n+i] + beta * c[i];  SiLU;  packed.
// alpha_m = row_alpha(alpha, m); c = the W values of C[m, n..] already loaded (cw: W/2 words of
// two output-type values), read only with F_C.  Columns at or beyond N read nothing.
template <int OUT, int W>
__device__ __forceinline__ void epi_vals_ext(const GemmParams& p, int n, const float* v, float alpha_m,
                                             const uint32_t* cw, float* y) {
  static_assert(W == 4 || W == 8, "group width");
  const bool in = n < p.N;
  float a[W];
#pragma unroll
  for (int i = 0; i < W; ++i)
    a[i] = ((p.flags & F_ALPHA_COL) && in) ? __fmul_rn(alpha_m, __ldg(p.alpha_col + n + i)) : alpha_m;
  if ((p.flags & F_BIAS) && in) {
    float b[W];
    load_bias<OUT, W>(p, n, b);
#pragma unroll
    for (int i = 0; i < W; ++i) y[i] = __fmaf_rn(a[i], v[i], b[i]);
  } else {
#pragma unroll
    for (int i = 0; i < W; ++i) y[i] = __fmul_rn(a[i], v[i]);
  }
  if (p.flags & F_C) {
    const uint16_t* c = reinterpret_cast<const uint16_t*>(cw);
#pragma unroll
    for (int i = 0; i < W; ++i) y[i] = __fmaf_rn(p.beta, out_to_float<OUT>(c[i]), y[i]);
  }
  if (p.flags & F_SILU) silu_inplace(reinterpret_cast<float(&)[W]>(*y));
}
template <int OUT, int W>
__device__ __forceinline__ void epi_pack_ext(const GemmParams& p, int n, const float* v, float alpha_m,
                                             const uint32_t* cw, uint32_t* out) {
  float y[W];
  epi_vals_ext<OUT, W>(p, n, v, alpha_m, cw, y);
#pragma unroll
  for (int i = 0; i < W / 2; ++i) out[i] = pack2<OUT>(y[2 * i], y[2 * i + 1]);
}

// 16 consecutive values of C (output type) at row m, column n, as eight words: one 32-byte load
// when C is 32-byte aligned (wide), else two 16-byte loads.  Plain loads: C may be D itself, and
// every element is read by the thread that later stores it.
__device__ __forceinline__ void load_c16(const GemmParams& p, int b, int m, int n, bool wide, uint32_t (&w)[8]) {
  const uint16_t* src = c_row(p, b, m) + n;
  if (wide) {
    asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(src)
                 : "memory");
  } else {
    const uint4 a = reinterpret_cast<const uint4*>(src)[0];
    const uint4 b = reinterpret_cast<const uint4*>(src)[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
}

// NVFP4 output (OUT_NV4): a row segment of 16*G accumulator values r (row m, columns n0.., n0 a
// multiple of 16) through the epilogue (bias and C in BF16) and the NVFP4 block encoding with the
// global scale *d_scale: 8 code bytes per 16 columns into D (row-major, N/2 bytes a row) and one
// scale byte into SFD.  Every scale byte of the padded layout that the segment covers is written,
// 0 for rows at or beyond M and columns at or beyond N, and the thread holding the row's last
// block also zeroes the padding columns after its segment, so that the scale buffer is complete
// for a GEMM that reads it.  Rows past M rounded up to 128 (a pair tile's) touch nothing.
template <int G, bool EXT>
__device__ __forceinline__ void epilogue_row_nv4(const GemmParams& p, int m, bool row_in, int n0, const uint32_t* r,
                                                 float alpha) {
  if (m >= ((p.M + 127) & ~127)) return;
  const NvTensorScale ts = nv_tensor_scale(__ldg(p.d_scale));
  const int cols_pad = p.sfd_cols4 * 4;
  uint8_t* drow = static_cast<uint8_t*>(p.d) + static_cast<size_t>(m) * (p.N >> 1);
  const bool ext = EXT && (p.flags & (F_C | F_ALPHA_COL | F_ALPHA_ROW));
  const float alpha_m = ext ? row_alpha(p, alpha, m) : alpha;
  // In the swizzled layout the scales of blocks 4w .. 4w+3 of a row are the four bytes of one
  // 32-bit word, so the segment's scale bytes are gathered in `word` and each run within a word
  // goes out as one store (8192^3 with NVFP4 output: ~0.6 us faster than a byte store per block).
  // A padded column count is a multiple of 4: a word is inside the padded columns or wholly past
  // them.
  const int c0 = n0 >> 4;
  uint32_t word = 0;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int n = n0 + 16 * g;
    const int c = n >> 4;
    uint32_t sc = 0;
    if (row_in && n < p.N) {
      float y[16];
      const float* v = reinterpret_cast<const float*>(r + 16 * g);
      if (ext) {
        uint32_t cw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (p.flags & F_C) load_c16(p, 0, m, n, (p.flags & F_D32) != 0, cw);
        epi_vals_ext<OUT_NV4, 8>(p, n, v, alpha_m, cw, y);
        epi_vals_ext<OUT_NV4, 8>(p, n + 8, v + 8, alpha_m, cw + 4, y + 8);
      } else {
        epi_vals<OUT_NV4, 8>(p, n, v, alpha, y);
        epi_vals<OUT_NV4, 8>(p, n + 8, v + 8, alpha, y + 8);
      }
      uint32_t lo, hi;
      sc = nv_encode_block16(y, ts, lo, hi);
      *reinterpret_cast<uint2*>(drow + (n >> 1)) = make_uint2(lo, hi);
    }
    word |= sc << (8 * (c & 3));
    if (((c & 3) == 3 || g == G - 1) && (c & ~3) < cols_pad) {
      // the run of this word's bytes that the segment covers: first .. c % 4
      const int first = c0 > (c & ~3) ? (c0 & 3) : 0;
      const int len = (c & 3) - first + 1;
      uint8_t* dst = p.sfd + sf_swizzle_offset(m, (c & ~3) + first, p.sfd_cols4);
      const uint32_t bytes = word >> (8 * first);
      if (len == 4) {
        *reinterpret_cast<uint32_t*>(dst) = bytes;
      } else if (len == 2 && (first & 1) == 0) {
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(bytes);
      } else {
#pragma unroll
        for (int j = 0; j < 3; ++j)
          if (j < len) dst[j] = static_cast<uint8_t>(bytes >> (8 * j));
      }
      word = 0;
    }
  }
  const int last = (p.N >> 4) - 1;
  if (last >= (n0 >> 4) && last < (n0 >> 4) + G)
    for (int c = (n0 >> 4) + G; c < cols_pad; ++c) p.sfd[sf_swizzle_offset(m, c, p.sfd_cols4)] = 0;
}

// NVFP4 output of a thread's HC-column row segment straight from TMEM (t, its first column):
// 32-column chunks (16 when HC is 16) loaded, encoded and stored one after another, so that few
// values are live at once.  The caller releases the accumulator afterwards.
template <int HC, bool EXT>
__device__ __forceinline__ void nv4_segment(const GemmParams& p, uint32_t t, int m, bool row_in, int n0,
                                            float alpha) {
  if constexpr (HC < 32) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(t, r);
    tmem_ld_wait();
    epilogue_row_nv4<1, EXT>(p, m, row_in, n0, r, alpha);
  } else {
#pragma unroll 1
    for (int ch = 0; ch < HC / 32; ++ch) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t + ch * 32, r);
      tmem_ld_wait();
      epilogue_row_nv4<2, EXT>(p, m, row_in, n0 + ch * 32, r, alpha);
    }
  }
}

// A row segment of 16*G accumulator values r (row m, columns n0.., n0 a multiple of 16) through
// the epilogue into D: the NVFP4 output above, the plain path, or (C / per-column factors) the extended one, which loads
// C one group of 16 columns ahead of the arithmetic.  The row is stored only if row_in
// (row_live), and columns at or beyond N never.
template <int OUT, int G, bool EXT>
__device__ __forceinline__ void epilogue_row(const GemmParams& p, int b, int m, bool row_in, int n0,
                                             const uint32_t* r, float alpha) {
  if constexpr (OUT == OUT_NV4) {
    epilogue_row_nv4<G, EXT>(p, m, row_in, n0, r, alpha);
    return;
  }
  uint16_t* drow = d_row(p, b, m);
  const bool wide = p.flags & F_D32;
  if (!EXT || !(p.flags & (F_C | F_ALPHA_COL | F_ALPHA_ROW))) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int n = n0 + 16 * g;
      uint32_t o[8];
      epi_pack<OUT, 8>(p, n, reinterpret_cast<const float*>(r + 16 * g), alpha, o);
      epi_pack<OUT, 8>(p, n + 8, reinterpret_cast<const float*>(r + 16 * g + 8), alpha, o + 4);
      if (row_in && n < p.N) st_out16(drow + n, o, wide);
    }
    return;
  }
  const float alpha_m = row_alpha(p, alpha, m);
  const bool has_c = (p.flags & F_C) && row_in;
  uint32_t cnext[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (has_c && n0 < p.N) load_c16(p, b, m, n0, wide, cnext);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int n = n0 + 16 * g;
    uint32_t ccur[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ccur[i] = cnext[i];
    if (g + 1 < G && has_c && n + 16 < p.N) load_c16(p, b, m, n + 16, wide, cnext);
    uint32_t o[8];
    epi_pack_ext<OUT, 8>(p, n, reinterpret_cast<const float*>(r + 16 * g), alpha_m, ccur, o);
    epi_pack_ext<OUT, 8>(p, n + 8, reinterpret_cast<const float*>(r + 16 * g + 8), alpha_m, ccur + 4, o + 4);
    if (row_in && n < p.N) st_out16(drow + n, o, wide);
  }
}

// Epilogue of 32 consecutive columns n0.. of output row m held by this thread.
template <int OUT, bool EXT>
__device__ __forceinline__ void store_chunk32(const GemmParams& p, int b, int m, bool row_in, int n0,
                                              const float* v, float alpha) {
  if (!row_in) return;
  uint16_t* drow = d_row(p, b, m);
  const bool ext = EXT && (p.flags & (F_C | F_ALPHA_COL | F_ALPHA_ROW));
  const float alpha_m = ext ? row_alpha(p, alpha, m) : alpha;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int n = n0 + 16 * h;
    if (n >= p.N) break;  // N % 16 == 0: groups of 16 are whole
    uint32_t o[8];
    if (ext) {
      uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (p.flags & F_C) load_c16(p, b, m, n, (p.flags & F_D32) != 0, c);
      epi_pack_ext<OUT, 8>(p, n, v + 16 * h, alpha_m, c, o);
      epi_pack_ext<OUT, 8>(p, n + 8, v + 16 * h + 8, alpha_m, c + 4, o + 4);
    } else {
      epi_pack<OUT, 8>(p, n, v + 16 * h, alpha, o);
      epi_pack<OUT, 8>(p, n + 8, v + 16 * h + 8, alpha, o + 4);
    }
    st_out16(drow + n, o, (p.flags & F_D32) != 0);
  }
}

// The epilogue on 4 accumulator values of row m, columns n..n+3, with the bias preloaded
// (braw), into y before the output rounding.  EXT: the residual and per-column factors too
// (alpha_m is then row_alpha(alpha, m)); without it, the plain path's arithmetic exactly.
template <int OUT, bool EXT>
__device__ __forceinline__ void epi4_values(const GemmParams& p, int b, int m, int n, const float4& a, uint2 braw,
                                            float alpha_m, float (&y)[4]) {
  const uint16_t* bv = reinterpret_cast<const uint16_t*>(&braw);
  y[0] = a.x;
  y[1] = a.y;
  y[2] = a.z;
  y[3] = a.w;
  const bool has_bias = (p.flags & F_BIAS) != 0;
  if (!EXT || !(p.flags & F_ALPHA_COL)) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      y[i] = has_bias ? __fmaf_rn(alpha_m, y[i], out_to_float<OUT>(bv[i])) : __fmul_rn(alpha_m, y[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float ai = __fmul_rn(alpha_m, __ldg(p.alpha_col + n + i));
      y[i] = has_bias ? __fmaf_rn(ai, y[i], out_to_float<OUT>(bv[i])) : __fmul_rn(ai, y[i]);
    }
  }
  if (EXT && (p.flags & F_C)) {
    uint16_t c[4];
    *reinterpret_cast<uint2*>(c) = *reinterpret_cast<const uint2*>(c_row(p, b, m) + n);
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = __fmaf_rn(p.beta, out_to_float<OUT>(c[i]), y[i]);
  }
  if (p.flags & F_SILU) silu_inplace(y);
}

// The same, rounded to the output type and packed two per word.
template <int OUT, bool EXT>
__device__ __forceinline__ uint2 epi4_with_bias(const GemmParams& p, int b, int m, int n, const float4& a,
                                                uint2 braw, float alpha_m) {
  float y[4];
  epi4_values<OUT, EXT>(p, b, m, n, a, braw, alpha_m, y);
  return make_uint2(pack2<OUT>(y[0], y[1]), pack2<OUT>(y[2], y[3]));
}

// NVFP4 output (OUT_NV4) of 4 reduced accumulator values a of row m, columns n..n+3: a quarter
// of a 16-column block whose other quarters are in the three neighbouring lanes (lanes 4k ..
// 4k+3 of the warp, all calling this for the same row and block).  The epilogue in float32 (bias
// and C in BF16), then the quantiser's block encoding with the global scale *d_scale, the
// block's amax taken across the four lanes: 2 code bytes into D (row-major, N/2 bytes a row),
// and the scale byte from the block's first lane.  A row outside the problem stores no codes and
// a zero scale; a block past N (N % 16 == 0: blocks are whole) inside the padded scale columns
// a zero scale.
template <bool EXT>
__device__ __forceinline__ void nv4_quarter(const GemmParams& p, const UnitCoord& c, int m, int n, const float4& a,
                                            uint2 braw, float alpha) {
  const int blk = n >> 4;
  const bool first = (n & 15) == 0;
  if (n >= p.N) {
    if (first && blk < p.sfd_cols4 * 4) p.sfd[sf_swizzle_offset(m, blk, p.sfd_cols4)] = 0;
    return;
  }
  uint32_t sc = 0;
  if (row_live<EXT>(p, c, m)) {
    float y[4];
    epi4_values<OUT_NV4, EXT>(p, c.batch, m, n, a, braw, EXT ? row_alpha(p, alpha, m) : alpha, y);
    uint32_t codes;
    sc = nv_encode_quad(y, nv_tensor_scale(__ldg(p.d_scale)), codes);
    *reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(p.d) + static_cast<size_t>(m) * (p.N >> 1) + (n >> 1)) =
        static_cast<uint16_t>(codes);
  }
  if (first) p.sfd[sf_swizzle_offset(m, blk, p.sfd_cols4)] = static_cast<uint8_t>(sc);
}

// Split-K through a cluster, owner side: the S partial slabs of this CTA's 128/S rows are in
// shared memory, slot sp = split sp, [128/S rows][BN + 4] floats each.  The owner sums them in
// split order (deterministic), applies the epilogue and stores whole rows: epilogue thread t
// takes column group c4 = t % (BN/4) (4 consecutive columns) of rows t / (BN/4), + 1024/BN, ...
template <int OUT, int BN, int S, bool EXT>
__device__ __forceinline__ void cluster_reduce_s(const GemmParams& p, const float* slabs, const UnitCoord& c,
                                                 float alpha, uint2 braw, int t) {
  constexpr int R = 128 / S;
  constexpr int C4 = BN / 4;          // column groups per row
  constexpr int RP = 256 / C4;        // rows per pass of the 256 epilogue threads
  constexpr int NP = R / RP;          // passes (R is a multiple of RP for S <= 8)
  static_assert(R % RP == 0 && NP >= 1, "reduction passes");
  const int c4 = t % C4;
  const int col = 4 * c4;
  const int n = c.n_blk * BN + col;
  const int r0 = t / C4;
  // every shared-memory read first (a fixed number of passes, so all of them are in flight
  // together), then the sums in split order, the epilogue and the stores
  float4 part[NP][S];
#pragma unroll
  for (int i = 0; i < NP; ++i)
#pragma unroll
    for (int sp = 0; sp < S; ++sp)
      part[i][sp] = *reinterpret_cast<const float4*>(slabs + (sp * R + r0 + i * RP) * (BN + 4) + col);
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int rl = r0 + i * RP;
    float4 acc = part[i][0];
#pragma unroll
    for (int sp = 1; sp < S; ++sp) {
      acc.x += part[i][sp].x;
      acc.y += part[i][sp].y;
      acc.z += part[i][sp].z;
      acc.w += part[i][sp].w;
    }
    // slab row rl holds tile row (rl / LPO) * 32 + split * LPO + rl % LPO, LPO = 32 / S
    const int row = (rl / (32 / S)) * 32 + c.split * (32 / S) + rl % (32 / S);
    const int m = c.m_blk * 128 + row;
    if constexpr (OUT == OUT_NV4) {
      // four consecutive column groups (lanes 4k .. 4k+3: C4 is a multiple of 16) make a block
      nv4_quarter<EXT>(p, c, m, n, acc, braw, alpha);
    } else if (row_live<EXT>(p, c, m) && n < p.N) {  // N % 16 == 0: groups of 4 are whole
      *reinterpret_cast<uint2*>(d_row(p, c.batch, m) + n) =
          epi4_with_bias<OUT, EXT>(p, c.batch, m, n, acc, braw, EXT ? row_alpha(p, alpha, m) : alpha);
    }
  }
}

template <int OUT, int BN, bool EXT>
__device__ __forceinline__ void cluster_reduce(const GemmParams& p, const float* slabs, const UnitCoord& c,
                                               float alpha, uint2 braw, int t) {
  if (EXT && (p.flags & (F_C | F_ALPHA_COL | F_ALPHA_ROW))) {
    if (p.splits == 2) cluster_reduce_s<OUT, BN, 2, true>(p, slabs, c, alpha, braw, t);
    else if (p.splits == 4) cluster_reduce_s<OUT, BN, 4, true>(p, slabs, c, alpha, braw, t);
    else cluster_reduce_s<OUT, BN, 8, true>(p, slabs, c, alpha, braw, t);
  } else {
    if (p.splits == 2) cluster_reduce_s<OUT, BN, 2, false>(p, slabs, c, alpha, braw, t);
    else if (p.splits == 4) cluster_reduce_s<OUT, BN, 4, false>(p, slabs, c, alpha, braw, t);
    else cluster_reduce_s<OUT, BN, 8, false>(p, slabs, c, alpha, braw, t);
  }
}

// Word t of the result is word (t + r) % 4 of v (r uniform across the warp).
__device__ __forceinline__ uint4 rotate_words(uint4 v, int r) {
  if (r & 1) v = make_uint4(v.y, v.z, v.w, v.x);
  if (r & 2) v = make_uint4(v.z, v.w, v.x, v.y);
  return v;
}

// EXT: the instantiation with the residual and per-row / per-column factor epilogue and batch
// entries (single problems without those flags run the instantiation without their code).
template <int KIND, int BN, int KC, int OUT, bool EXT>
__global__ void __launch_bounds__(GemmCfg<KIND, BN, KC>::THREADS, 1) bsg_gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<KIND, BN, KC>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
  const uint32_t smem0 = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint8_t* aux = smem + C::STAGES * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux);
  // barrier slots: full[0..7], empty[8..15], tmem_full[16..17], tmem_empty[18..19], drain[20]
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + 8 + s); };
  auto bar_tfull = [&](int a) { return smem_u32(bars + 16 + a); };
  auto bar_tempty = [&](int a) { return smem_u32(bars + 18 + a); };
  const uint32_t bar_drain = smem_u32(bars + 20);
  auto bar_sf_full = [&](int s) { return smem_u32(bars + 24 + s); };  // scale atoms landed
  const uint32_t bar_recv = smem_u32(bars + 32);  // split-K cluster: peers' slabs have landed
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 21);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 22);
  volatile int* last_flag = reinterpret_cast<volatile int*>(bars + 23);

  auto stage_a = [&](int s) { return smem0 + s * C::STAGE_BYTES; };
  auto stage_b = [&](int s) { return smem0 + s * C::STAGE_BYTES + C::A_BYTES; };
  auto stage_sfa = [&](int s) { return smem0 + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES; };
  auto stage_sfb = [&](int s) {
    return smem0 + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES + C::SFA_BYTES;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // the code producer (with its bytes) and the four scale warps once the stage's scales are
      // in TMEM: one wait per k-tile for the MMA issuer
      mbar_init(bar_full(s), 1 + 4);
      mbar_init(bar_empty(s), 1);  // the MMA issuer's commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull(a), 1);
      mbar_init(bar_tempty(a), C::EPI_WARPS);  // one arrival per epilogue warp
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_recv, 1);
    for (int s = 0; s < C::STAGES; ++s) mbar_init(bar_sf_full(s), 1);  // the scale producer
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Split-K cluster: the peers store partial rows into this CTA's receive slots (shared memory
  // past the ring stages in use), so every CTA announces at start-up that its barriers are
  // initialised (fence.mbarrier_init above); a thread waits for the announcements before its
  // first remote store, or at teardown.
  bool cluster_waited = false;  // this thread has completed the start-up cluster barrier
  if (p.split_mode == SPLIT_CLUSTER) cluster_arrive_relaxed();
  const int u0 = static_cast<int>(blockIdx.x);     // first unit of this CTA
  const int ustep = static_cast<int>(gridDim.x);  // CTAs of the grid
  const uint32_t tmem_base = *tmem_slot;
  const int nst = p.ring_stages;  // ring stages in use (fewer than STAGES with a split-K cluster)
  // Pointer-agnostic run: the code producer's own copies of the tensor maps, written before the
  // wait below (they read only this launch's parameters, and the slot set is not the one the
  // plan's previous launch, which may still run, uses), so that their fences overlap it.
  const CUtensorMap* tma = &p.tmap_a;
  const CUtensorMap* tmb = &p.tmap_b;
  if (EXT && p.map_slots != nullptr) {
    CUtensorMap* slot = p.map_slots + MAP_SLOTS_PER_CTA * blockIdx.x;
    if (warp == 0 && lane == 0) {
      tmap_remap2(slot, &p.tmap_a, &p.tmap_b, p.remap_a, p.remap_b);
    }
    if (warp == 0) {  // every lane acquires them: the lane that issues the copies is elected
      __syncwarp();
      tmap_acquire2(slot);
    }
    tma = slot;
    tmb = slot + 1;
  }
  // Everything above touched only this CTA's own resources; from here on global memory is
  // read and written, so wait for the preceding grid in the stream (programmatic dependent
  // launch), and let the next grid start its launch while this one runs.
  griddep_wait();
  griddep_launch_dependents();

  // Roles by warpgroup; each warpgroup first sets its register budget (setmaxnreg is executed
  // by all four warps of a warpgroup at the same instruction).
  if (warp < C::SCALE_WARP0) {
    setmaxnreg_dec<C::REGS_CTRL>();
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer: code tiles
      // The whole warp runs the loop with warp-uniform values; one elected lane issues each copy
      // (a diverged lane was held ~100 cycles per copy).
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool first = true;
      for (int u = u0; ok && u < p.num_units; u += ustep) {
        const UnitCoord c = decode_unit<EXT>(p, u);
        if (EXT && c.skip) continue;
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          ok = wait_bounded_warp(bar_empty(stage), phase ^ 1u, abort_flag, p, ST_TIMEOUT_PRODUCER);
          if (!ok) break;
          if (first && p.debug_skip_first_load) {
            // test hook: leave this stage unfilled so that the MMA warp's wait runs out
          } else {
            const uint32_t fb = bar_full(stage);
            mbar_arrive_expect_tx_warp(fb, C::A_BYTES + C::B_BYTES);
#pragma unroll
            for (int j = 0; j < KC; ++j) {  // k-slabs past K read as zeros (their MMAs are skipped)
              const int x = (kt * KC + j) * C::BK_BYTES;
              const uint32_t sa = stage_a(stage) + j * C::SLAB_A, sb = stage_b(stage) + j * C::SLAB_B;
              if (EXT && p.batches > 1)
                tma_load_3d_warp(sa, tma, fb, x, c.m_blk * C::BM, c.batch);
              else
                tma_load_2d_warp(sa, tma, fb, x, c.m_blk * C::BM);
              if (EXT && p.b_entries > 1)
                tma_load_3d_warp(sb, tmb, fb, x, c.n_blk * BN, c.bsel);
              else
                tma_load_2d_warp(sb, tmb, fb, x, c.n_blk * BN);
            }
          }
          first = false;
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else if (warp == 2) {
      // ------------------------------------------------------------ TMA producer: scale atoms
      // A second issuing warp, so that the scale copies run beside the code-tile copies, into the
      // same stage, completing on the stage's `sf_full` barrier, which the scale warps wait for;
      // they in turn arrive on the stage's `full` barrier, so the MMA issuer waits once per
      // k-tile.  Whole-warp loop, one elected lane per copy.
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool first = true;
      for (int u = u0; ok && u < p.num_units; u += ustep) {
        const UnitCoord c = decode_unit<EXT>(p, u);
        if (EXT && c.skip) continue;
        const int band0 = c.n_blk * BN / 128;    // first scale band of the B tile
        const bool a_band = c.m_blk < p.sfa_bands;  // false only for a cluster's m-tile beyond M
        int bands = 0;
#pragma unroll
        for (int rb = 0; rb < C::NB; ++rb) bands += (band0 + rb < p.sfb_bands) ? 1 : 0;
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          ok = wait_bounded_warp(bar_empty(stage), phase ^ 1u, abort_flag, p, ST_TIMEOUT_PRODUCER);
          if (!ok) break;
          const int k_rem = p.K - kt * C::K_TILE;
          const int steps = min(C::STEPS, (k_rem + C::MMA_K - 1) / C::MMA_K);
          const int sf_atoms = KIND == KIND_MX ? (steps + 3) / 4 : steps;  // atoms K still covers
          if (first && p.debug_skip_first_load) {
            // test hook (see the code producer)
          } else {
            const uint32_t fb = bar_sf_full(stage);
            mbar_arrive_expect_tx_warp(fb, static_cast<uint32_t>(((a_band ? 1 : 0) + bands) * sf_atoms * 512));
            if (a_band) {
              const uint8_t* sa = p.sfa + c.batch * p.sfa_batch + (static_cast<size_t>(c.m_blk) * p.sfa_atoms_per_band +
                                           static_cast<size_t>(kt) * C::SF_ATOMS) * 512;
              bulk_load_warp(stage_sfa(stage), sa, sf_atoms * 512, fb);
            }
#pragma unroll
            for (int rb = 0; rb < C::NB; ++rb) {
              const int band = band0 + rb;
              if (band < p.sfb_bands) {
                const uint8_t* sb = p.sfb + c.bsel * p.sfb_batch + (static_cast<size_t>(band) * p.sfb_atoms_per_band +
                                             static_cast<size_t>(kt) * C::SF_ATOMS) * 512;
                bulk_load_warp(stage_sfb(stage) + rb * C::SF_ATOMS * 512, sb, sf_atoms * 512, fb);
              }
            }
          }
          first = false;
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the loop with warp-uniform values; one elected lane issues each MMA
      // and commit.
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = u0; ok && u < p.num_units; u += ustep) {
        const UnitCoord c = decode_unit<EXT>(p, u);
        if (EXT && c.skip) continue;
        ok = wait_bounded_warp(bar_tempty(acc), acc_phase ^ 1u, abort_flag, p, ST_TIMEOUT_MMA);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_t = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          ok = wait_bounded_warp(bar_full(stage), phase, abort_flag, p, ST_TIMEOUT_MMA);
          if (!ok) break;
          tc_fence_after();
          const int k_rem = p.K - kt * C::K_TILE;
          const int steps = min(C::STEPS, (k_rem + C::MMA_K - 1) / C::MMA_K);
          // the scale warps have put this stage's scales in its TMEM slot
          const uint32_t sfa_t = tmem_base + C::SF_COL0 + stage * C::SF_SLOT_COLS;
          const uint32_t sfb_t = sfa_t + C::SFA_COLS;
          const uint32_t sa = stage_a(stage), sb = stage_b(stage);
          const uint32_t acc0 = kt > c.kt0 ? 1u : 0u;
          // MMA j reads 32 bytes of K at offset 32 (j % 4) of k-slab j / 4; its scales are in
          // atom j / 4 (MXFP8, byte j % 4 of each word) or atom j (NVFP4)
          auto mma = [&](int j, uint32_t accumulate) {
            const uint32_t jj = static_cast<uint32_t>(j & 3), slab = static_cast<uint32_t>(j >> 2);
            if constexpr (KIND == KIND_MX)
              tc_mma_mxf8_warp(d_t, sdesc_kmajor_sw128(sa + slab * C::SLAB_A + 32 * jj),
                               sdesc_kmajor_sw128(sb + slab * C::SLAB_B + 32 * jj), C::IDESC | (jj << 4) | (jj << 29),
                               sfa_t + 4 * slab, sfb_t + 4 * C::NB * slab, accumulate);
            else
              tc_mma_nvf4_warp(d_t, sdesc_kmajor_sw128(sa + slab * C::SLAB_A + 32 * jj),
                               sdesc_kmajor_sw128(sb + slab * C::SLAB_B + 32 * jj), C::IDESC, sfa_t + 4 * j,
                               sfb_t + 4 * C::NB * j, accumulate);
          };
          if (steps == C::STEPS) {
#pragma unroll
            for (int j = 0; j < C::STEPS; ++j) mma(j, j == 0 ? acc0 : 1u);  // straight-line issue
          } else {
            for (int j = 0; j < steps; ++j) mma(j, j == 0 ? acc0 : 1u);  // the last, partial k-tile
          }
          tc_commit_warp(bar_empty(stage));
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_warp(bar_tfull(acc));
        if (C::NACC == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        // let every tensor-core operation issued so far finish before TMEM is released
        tc_commit_warp(bar_drain);
        if (lane == 0) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar_drain, 0)) {
            if (globaltimer_ns() - t0 > 10000000ull) {
              atomicOr(p.status, ST_TIMEOUT_DRAIN);
              break;
            }
          }
        }
        __syncwarp();
      }
    }
  } else if (warp < C::EPI_WARP0) {
    setmaxnreg_dec<C::REGS_SCALE>();
    // ------------------------------------------------------------ scale warps (warps 4..7)
    // Per stage, each warp writes its TMEM lane quarter of the stage's scale slot with the layout
    // a 32x128b.warpx4 copy of the atoms produces: lane i, column 4j + k holds the four scales
    // (one 32-bit word of the atom's row i) of A row 32k + i of atom j, and column
    // 4*NB*j + 4b + k those of B row 128b + 32k + i.  Of A's four columns the MMA reads, in lane
    // quarter q, only column 4j + q (the scales of its own rows 32q + i), so each warp writes only
    // that one.  A tile narrower than its 128-row band uses words jq.. of each B atom row, jq =
    // its first 32-row quarter of the band: they are rotated to the front.
    const int q = warp & 3;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = u0; ok && u < p.num_units; u += ustep) {
      const UnitCoord c = decode_unit<EXT>(p, u);
      if (EXT && c.skip) continue;
      const int jq = BN < 128 ? (c.n_blk * BN % 128) / 32 : 0;
      for (int kt = c.kt0; kt < c.kt1; ++kt) {
        ok = __all_sync(0xffffffffu, wait_bounded(bar_sf_full(stage), phase, abort_flag, p, ST_TIMEOUT_SCALES));
        if (!ok) break;
        const uint32_t slot = tmem_base + C::SF_COL0 + stage * C::SF_SLOT_COLS + (static_cast<uint32_t>(q * 32) << 16);
        // atoms in groups of up to four: 4 A columns and 4 * NB B columns per atom
        constexpr int NA = C::SF_ATOMS;
        constexpr int GA = NA < 4 ? NA : 4;
#pragma unroll
        for (int g0 = 0; g0 < NA; g0 += GA) {
          uint32_t a[GA], b[4 * C::NB * GA];
#pragma unroll
          for (int t = 0; t < GA; ++t) {
            a[t] = lds_u32(stage_sfa(stage) + 512 * (g0 + t) + 16 * lane + 4 * q);  // this quarter's word
#pragma unroll
            for (int rb = 0; rb < C::NB; ++rb) {
              const uint4 w = rotate_words(lds_u4(stage_sfb(stage) + rb * NA * 512 + 512 * (g0 + t) + 16 * lane), jq);
              b[(C::NB * t + rb) * 4] = w.x;
              b[(C::NB * t + rb) * 4 + 1] = w.y;
              b[(C::NB * t + rb) * 4 + 2] = w.z;
              b[(C::NB * t + rb) * 4 + 3] = w.w;
            }
          }
#pragma unroll
          for (int t = 0; t < GA; ++t) tmem_st_32x32b_x1(slot + 4 * (g0 + t) + q, a[t]);
          tmem_st_cols(slot + C::SFA_COLS + 4 * C::NB * g0, b);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_full(stage));
        if (++stage == nst) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    setmaxnreg_inc<C::REGS_EPI>();
    // ------------------------------------------------------------ epilogue (warps 8..15)
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;       // accumulator row = TMEM lane
    constexpr int HC = BN / 2;           // columns per thread
    const int col0 = ((warp - C::EPI_WARP0) >> 2) * HC;
    const float alpha0 = (p.flags & F_ALPHA_DEVICE) ? __ldg(p.alpha_dev) : p.alpha;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = u0; u < p.num_units; u += ustep) {
      const UnitCoord c = decode_unit<EXT>(p, u);
      if (EXT && c.skip) continue;
      const float alpha = unit_alpha<EXT>(p, c, alpha0);
      bool ok = wait_bounded(bar_tfull(acc), acc_phase, abort_flag, p, ST_TIMEOUT_EPILOGUE);
      ok = named_bar_and(1, C::EPI_THREADS, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(q * 32) << 16);
      const int m = c.m_blk * C::BM + row;
      const bool row_in = row_live<EXT>(p, c, m);
      const int nbase = c.n_blk * BN;
      if (p.split_mode == SPLIT_NONE) {
        uint16_t* drow = d_row(p, c.batch, m);
        if constexpr (OUT == OUT_NV4 && C::NACC == 2) {
          // NVFP4 output beside a second accumulator: chunk by chunk from TMEM, then the release
          // (with one accumulator the path below drains, releases, then encodes, so that the next
          // tile's MMAs do not wait for the encoding)
          nv4_segment<HC, EXT>(p, t_row + col0, m, row_in, nbase + col0, alpha);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(acc));
        } else if constexpr (C::NACC == 1) {
          // One accumulator: the whole row segment comes out of TMEM before any arithmetic and
          // the accumulator is released at once, since the next tile's MMAs need all of it.
          uint32_t r[HC];
#pragma unroll
          for (int ch = 0; ch < HC / 32; ++ch)
            tmem_ld_32x32b_x32(t_row + col0 + ch * 32, reinterpret_cast<uint32_t(&)[32]>(r[32 * ch]));
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(acc));
          epilogue_row<OUT, HC / 16, EXT>(p, c.batch, m, row_in, nbase + col0, r, alpha);
        } else {
          // Two accumulators: the next tile's MMAs run in the other one, so the segment is
          // rounded chunk by chunk (fewer live registers) and released before the stores.
          uint32_t packed[HC / 2];
          constexpr int W = HC < 32 ? HC : 32;
          auto load_chunk = [&](int ch, uint32_t (&r)[W]) {
            if constexpr (W == 16)
              tmem_ld_32x32b_x16(t_row + col0, r);
            else
              tmem_ld_32x32b_x32(t_row + col0 + ch * 32, r);
            tmem_ld_wait();
          };
          if (EXT && (p.flags & (F_C | F_ALPHA_COL | F_ALPHA_ROW))) {
            const float alpha_m = row_alpha(p, alpha, m);
#pragma unroll
            for (int ch = 0; ch < (HC + 31) / 32; ++ch) {
              uint32_t r[W];
              load_chunk(ch, r);
#pragma unroll
              for (int h = 0; h < W / 16; ++h) {
                const int n = nbase + col0 + ch * 32 + 16 * h;
                uint32_t cw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if ((p.flags & F_C) && row_in && n < p.N) load_c16(p, c.batch, m, n, (p.flags & F_D32) != 0, cw);
                epi_pack_ext<OUT, 8>(p, n, reinterpret_cast<const float*>(&r[16 * h]), alpha_m, cw,
                                     &packed[ch * 16 + 8 * h]);
                epi_pack_ext<OUT, 8>(p, n + 8, reinterpret_cast<const float*>(&r[16 * h + 8]), alpha_m, cw + 4,
                                     &packed[ch * 16 + 8 * h + 4]);
              }
            }
          } else {
#pragma unroll
            for (int ch = 0; ch < (HC + 31) / 32; ++ch) {
              uint32_t r[W];
              load_chunk(ch, r);
#pragma unroll
              for (int g = 0; g < W / 8; ++g)
                epi_pack<OUT, 8>(p, nbase + col0 + ch * 32 + 8 * g, reinterpret_cast<const float*>(&r[8 * g]), alpha,
                                 &packed[ch * 16 + 4 * g]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(acc));
          const bool wide = p.flags & F_D32;
#pragma unroll
          for (int g = 0; g < HC / 16; ++g) {
            const int n = nbase + col0 + 16 * g;
            if (row_in && n < p.N) st_out16(drow + n, reinterpret_cast<const uint32_t(&)[8]>(packed[8 * g]), wide);
          }
        }
      } else if constexpr (BN >= 64) {  // split-K: tiles 64 wide or more
        if (p.split_mode == SPLIT_CLUSTER) {
          // Split-K through the cluster (one unit per CTA).  Row `row` of the tile belongs to
          // split owner = lane / (32/S), so every warp holds rows of every owner.  Each thread
          // streams its partial row from TMEM through registers into slot `split` of the owner's
          // receive area: a peer's with st.async (counted on the peer's receive barrier), its own
          // with plain stores.  The receive area, S slots of 128/S rows, lies past the ring
          // stages in use, so peers write it while this CTA may still be running its MMAs.  Then
          // all epilogue threads of the owner sum the S slots in split order (deterministic) and
          // store whole rows.
          const int S = p.splits, LPO = 32 / S, R = 128 / S;
          const int owner = lane / LPO;
          const int lr = q * LPO + lane % LPO;  // row within the owner's slab
          const uint32_t slab_bytes = static_cast<uint32_t>(R * (BN + 4) * 4);
          const uint32_t recv0 = smem0 + static_cast<uint32_t>(nst * C::STAGE_BYTES);
          const int et = threadIdx.x - C::EPI_WARP0 * 32;  // epilogue thread index
          uint2 braw = make_uint2(0u, 0u);  // bias of the columns this thread reduces, loaded early
          {
            const int n = nbase + 4 * (et % (BN / 4));
            if ((p.flags & F_BIAS) && n < p.N)
              braw = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.bias) + n));
          }
          if (threadIdx.x == C::EPI_WARP0 * 32)
            mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>(S - 1) * slab_bytes);
          // Partial rows leave TMEM into shared memory: this CTA's own rows into its receive slot
          // `split`, every peer's rows into a staging slab of the ring (idle: the unit's MMAs have
          // completed and no copy is pending), laid out as the peer's slot.  Then one bulk copy per
          // peer moves a whole slab over DSMEM (complete-tx on the peer's receive barrier), which
          // runs several times faster than per-thread remote stores.
          const bool mine = owner == c.split;
          const uint32_t dst = (mine ? recv0 + static_cast<uint32_t>(c.split) * slab_bytes
                                     : smem0 + static_cast<uint32_t>(owner) * slab_bytes) +
                               static_cast<uint32_t>((lr * (BN + 4) + col0) * 4);
#pragma unroll 1
          for (int ch = 0; ch < HC / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(t_row + col0 + ch * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 8; ++g)
              sts_u4(dst + static_cast<uint32_t>((ch * 32 + 4 * g) * 4),
                     make_uint4(r[4 * g], r[4 * g + 1], r[4 * g + 2], r[4 * g + 3]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(acc));
          fence_proxy_async_smem();  // the staging slabs are read by the bulk copies (async proxy)
          named_bar_sync(1, C::EPI_THREADS);
          cluster_wait();  // every CTA of the cluster has initialised its receive barrier
          cluster_waited = true;
          const bool sender = et < S && et != c.split;  // one thread per peer
          if (sender) {
            bulk_copy_s2c(mapa_shared(recv0 + static_cast<uint32_t>(c.split) * slab_bytes, static_cast<uint32_t>(et)),
                          smem0 + static_cast<uint32_t>(et) * slab_bytes, slab_bytes,
                          mapa_shared(bar_recv, static_cast<uint32_t>(et)));
            bulk_commit_group();
          }
          const bool got = named_bar_and(1, C::EPI_THREADS,
                                         wait_bounded_cluster(bar_recv, 0, abort_flag, p, ST_TIMEOUT_EPILOGUE));
          if (got)
            cluster_reduce<OUT, BN, EXT>(p, reinterpret_cast<const float*>(smem + nst * C::STAGE_BYTES), c, alpha,
                                         braw, et);
          if (sender) bulk_wait_group0();  // the slab has reached the peer before this CTA may leave
        } else {
          // FP32 partial tile -> workspace as float4 [chunk][8][128 rows] (coalesced per warp)
          float4* part = reinterpret_cast<float4*>(
              p.partial + (static_cast<size_t>(c.split) * p.num_tiles + c.tile) * (C::BM * BN));
          const int ch0 = col0 / 32;
#pragma unroll 1
          for (int ch = ch0; ch < ch0 + HC / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(t_row + ch * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              float4 v4 = make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                      __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
              __stcg(part + (ch * 8 + g) * C::BM + row, v4);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty(acc));
          __threadfence();
          named_bar_sync(1, C::EPI_THREADS);
          if (threadIdx.x == C::EPI_WARP0 * 32) {
            const unsigned old = atomicAdd(p.counters + c.tile, 1u);
            const int last = (old == static_cast<unsigned>(p.splits - 1)) ? 1 : 0;
            if (last) p.counters[c.tile] = 0u;  // ready for the next launch
            *last_flag = last;
          }
          named_bar_sync(1, C::EPI_THREADS);
          if (*last_flag) {
            __threadfence();
            const float4* base = reinterpret_cast<const float4*>(
                p.partial + static_cast<size_t>(c.tile) * (C::BM * BN));
            const size_t split_stride = static_cast<size_t>(p.num_tiles) * (C::BM * BN) / 4;
#pragma unroll 1
            for (int ch = ch0; ch < ch0 + HC / 32; ++ch) {
              float v[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.0f;
              for (int s = 0; s < p.splits; ++s) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  const float4 t = __ldcg(base + s * split_stride + (ch * 8 + g) * C::BM + row);
                  v[4 * g] += t.x;
                  v[4 * g + 1] += t.y;
                  v[4 * g + 2] += t.z;
                  v[4 * g + 3] += t.w;
                }
              }
              if constexpr (OUT == OUT_NV4)
                epilogue_row_nv4<2, EXT>(p, m, row_in, nbase + ch * 32, reinterpret_cast<const uint32_t*>(v), alpha);
              else
                store_chunk32<OUT, EXT>(p, c.batch, m, row_in, nbase + ch * 32, v, alpha);
            }
          }
          named_bar_sync(1, C::EPI_THREADS);
        }
      }
      if (C::NACC == 2) {
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      } else {
        acc_phase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------ split-K cluster: lifetime
  if (p.split_mode == SPLIT_CLUSTER) {
    // Every thread completes the start-up barrier (the epilogue threads did before storing).  No
    // CTA needs to outlive another: a CTA leaves after its receive barrier saw every byte sent
    // to it, and what it sent came from registers.
    if (!cluster_waited) cluster_wait();
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // give copies that were already in flight time to land before the CTA's smem goes away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int KIND, int BN, int KC, int OUT, bool EXT = false>
bool fill_kernel_info(GemmKernelInfo* info) {
  using C = GemmCfg<KIND, BN, KC>;
  info->fn = reinterpret_cast<const void*>(&bsg_gemm_kernel<KIND, BN, KC, OUT, EXT>);
  info->smem_bytes = C::SMEM_BYTES;
  info->threads = C::THREADS;
  info->bn = BN;
  info->stages = C::STAGES;
  info->stage_bytes = C::STAGE_BYTES;
  info->kc = KC;
  return true;
}

}  // namespace bsg
