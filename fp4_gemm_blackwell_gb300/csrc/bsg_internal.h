// Internal declarations shared by the host side and the kernels of the block-scaled GEMM.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsg {

enum : int { KIND_MX = 0, KIND_NV = 1 };
enum : int { OUT_F16 = 0, OUT_BF16 = 1, OUT_NV4 = 2 };  // OUT_NV4: NVFP4 codes + scales
enum : unsigned {
  F_BIAS = 1u,
  F_SILU = 2u,
  F_ALPHA_DEVICE = 4u,
  F_C = 8u,
  F_ALPHA_ROW = 16u,
  F_ALPHA_COL = 32u,
  F_GROUPED = 64u,
  F_D32 = 1u << 30  // D (and C) 32-byte aligned: set by the host, not a caller flag
};

// How split-K partial tiles are combined: not split; FP32 partials in the plan's global
// workspace, summed by the last split to arrive; or the splits of a tile form one thread-block
// cluster and each CTA sums a slab of rows from the peers' shared memory (DSMEM).
enum : int { SPLIT_NONE = 0, SPLIT_WORKSPACE = 1, SPLIT_CLUSTER = 2 };

// Bits of the device status word (OR-ed in by a CTA that gives up a wait).
enum : unsigned {
  ST_TIMEOUT_PRODUCER = 1u << 0,
  ST_TIMEOUT_MMA = 1u << 1,
  ST_TIMEOUT_EPILOGUE = 1u << 2,
  ST_TIMEOUT_DRAIN = 1u << 3,
  ST_TIMEOUT_SCALES = 1u << 4,
};

// Kernel parameters, passed by value as a __grid_constant__ (the tensor maps must live in
// parameter space for the TMA instructions).
// Tensor-map slots per CTA of a pointer-agnostic run.
constexpr int MAP_SLOTS_PER_CTA = 4;

struct GemmParams {
  CUtensorMap tmap_a;  // A codes: bytes, dims {K bytes, M, batches}, box {128, 128, 1}, 128-byte swizzle
  CUtensorMap tmap_b;  // B codes: bytes, dims {K bytes, N, b_entries}, box {128, BN, 1}, 128-byte swizzle
  const uint8_t* sfa;  // swizzled 128x4 scale atoms of A
  const uint8_t* sfb;
  const void* bias;    // N values of the output type (flags & F_BIAS)
  void* d;             // M x N output, row-major
  const void* c;       // M x N residual input, row-major, output type (flags & F_C)
  const float* alpha_row;  // M factors (flags & F_ALPHA_ROW)
  const float* alpha_col;  // N factors (flags & F_ALPHA_COL)
  const float* alpha_dev;
  uint8_t* sfd;            // NVFP4 output: swizzled UE4M3 scales of D (M x N/16, padded)
  const float* d_scale;    // NVFP4 output: the global scale s of D (device memory)
  int sfd_cols4;           // NVFP4 output: padded scale columns / 4
  float* partial;      // split-K partial tiles (splits x tiles x 128 x BN floats)
  unsigned* counters;  // split-K arrival counter per tile (0 between launches)
  unsigned* status;    // device status word
  unsigned long long wait_limit_ns;
  float alpha;
  float beta;
  int M, N, K;
  unsigned flags;
  int sfa_atoms_per_band;  // padded scale columns / 4 of A
  int sfb_atoms_per_band;
  int sfb_bands;           // padded rows / 128 of B
  int sfa_bands;           // padded rows / 128 of A
  int num_m_tiles, num_n_tiles, num_k_tiles;
  int num_tiles;           // tiles of all batch entries (the workspace's tile count)
  int batches;             // entries of A, SFA, D and C: L >= 1 problems of this shape at the strides
                           // below (1 when grouped)
  int b_entries;           // entries of B and SFB: L when batched, the G groups when grouped, else 1
  const int* group_index;  // grouped (F_GROUPED): the group of each of the M rows, -1 = no group
  // Pointer-agnostic runs (EXT instantiations): when map_slots is set, each CTA copies its tensor
  // maps (tmap_a, tmap_b, and in the CTA-pair kernel PairParams::tmap_sfa, tmap_sfb) into its 128-byte global
  // slots (map_slots + MAP_SLOTS_PER_CTA * blockIdx.x), replaces their global addresses by
  // remap_a, remap_b (remap_sfa, remap_sfb) and loads through the copies.  The host alternates
  // between two slot sets from one such launch of a plan to the next.
  CUtensorMap* map_slots;
  const void* remap_a;
  const void* remap_b;
  const void* remap_sfa;
  const void* remap_sfb;
  int units_per_batch;     // num_m_tiles * num_n_tiles * splits
  long long sfa_batch, sfb_batch;  // bytes between the scale buffers of consecutive entries (groups)
  long long d_batch, c_batch;      // 16-bit elements between consecutive D (C) matrices
  int splits;              // split-K factor (every split owns >= 1 k-tile)
  int split_mode;          // SPLIT_NONE, SPLIT_WORKSPACE or SPLIT_CLUSTER
  int k_tiles_per_split;
  int num_units;           // units_per_batch * batches
  int group_m;             // tile rasterisation: m-blocks per group
  int ring_stages;         // shared-memory ring stages in use (the kernel's maximum, or fewer to
                           // make room for split-K receive slots)
  int debug_skip_first_load;  // test hook: the producer never loads its first stage
};
// The CTA-pair kernel's parameters: GemmParams, then the tiled maps of the scale atoms of A and B
// (32-bit words, dims {128 (one 512-byte atom), bands x atoms per band, entries}, box {128, atoms
// per ring stage, 1}, no swizzle; rows past the buffer read as zeros).  The host builds this
// superset for every plan; a 1-SM kernel, whose parameter is GemmParams, is launched with the
// same block and receives its first sizeof(GemmParams) bytes (the launch copies as many bytes
// as the kernel's parameter holds): 640 bytes instead of 896, a shorter launch (host time per
// launch of an empty cluster kernel: 1.47 us with 512 bytes of parameters, 1.56 with 768).
struct PairParams : GemmParams {
  CUtensorMap tmap_sfa;
  CUtensorMap tmap_sfb;
};
static_assert(sizeof(GemmParams) % 64 == 0 && sizeof(PairParams) == sizeof(GemmParams) + 2 * sizeof(CUtensorMap),
              "the pair kernel's parameter block extends the 1-SM one");


struct GemmKernelInfo {
  const void* fn;
  int smem_bytes;
  int threads;
  int bn;
  int stages;       // ring stages
  int stage_bytes;  // bytes of one ring stage
  int kc;           // k-tiles (128 bytes of K) per ring stage
};

// Look up a kernel instantiation: tile width bn (32, 64, 128 or 256), out (OUT_*), kc k-slabs per
// ring stage (1, or 2 for bn 64 and 128).
bool gemm_kernel_info_mx(int bn, int out, int kc, GemmKernelInfo* info);
bool gemm_kernel_info_nv(int bn, int out, int kc, GemmKernelInfo* info);
bool gemm_kernel_info_mx_narrow(int bn, int out, GemmKernelInfo* info);  // bn 32 or 64
bool gemm_kernel_info_nv_narrow(int bn, int out, GemmKernelInfo* info);
bool gemm_kernel_info_mx_kc2(int bn, int out, GemmKernelInfo* info);     // bn 64 or 128
bool gemm_kernel_info_nv_kc2(int bn, int out, GemmKernelInfo* info);
// CTA-pair kernels (256 x 256 pair tiles, launched in clusters of 2).
bool gemm_pair_kernel_info_mx(int out, GemmKernelInfo* info);  // BSG_PAIR_KC=1 or 2 (default 2)
bool gemm_pair_kernel_info_nv(int out, GemmKernelInfo* info);  // BSG_PAIR_KC=1 or 2 (default 2)
// The same lookups for the extended instantiations: the residual and per-row / per-column factor
// epilogue and batch entries (chosen when a problem sets BSG_F_C, BSG_F_ALPHA_ROW or
// BSG_F_ALPHA_COL, or has L > 1).
bool gemm_kernel_info_mx_ext(int bn, int out, int kc, GemmKernelInfo* info);
bool gemm_kernel_info_nv_ext(int bn, int out, int kc, GemmKernelInfo* info);
bool gemm_kernel_info_mx_narrow_ext(int bn, int out, GemmKernelInfo* info);
bool gemm_kernel_info_nv_narrow_ext(int bn, int out, GemmKernelInfo* info);
bool gemm_kernel_info_mx_kc2_ext(int bn, int out, GemmKernelInfo* info);
bool gemm_kernel_info_nv_kc2_ext(int bn, int out, GemmKernelInfo* info);
bool gemm_pair_kernel_info_mx_ext(int out, GemmKernelInfo* info);
bool gemm_pair_kernel_info_nv_ext(int out, GemmKernelInfo* info);

// The kernel of variant (pair, bn, kc) for a problem's format, output type, epilogue flags and
// batch count.
bool find_kernel(int kind, int out, unsigned flags, int batches, bool pair, int bn, int kc, GemmKernelInfo* info);
// The same with the instantiation named: EXT (ext) or plain.
bool find_kernel_variant(int kind, int out, bool ext, bool pair, int bn, int kc, GemmKernelInfo* info);

// Quantisers (stream-ordered).  See bsg_quantize / bsg_quantize_bf16 in include/bsgemm.h; the
// uint16_t forms read BF16 bit patterns; sms: the device's SM count (the grids are persistent).
cudaError_t launch_quantize_mx(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf, int sms,
                               cudaStream_t s);
cudaError_t launch_quantize_mx(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf, int sms,
                               cudaStream_t s);
cudaError_t launch_quantize_nv(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                               float* global_scale, int sms, cudaStream_t s);
cudaError_t launch_quantize_nv(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                               float* global_scale, int sms, cudaStream_t s);
// NVFP4 with the global scale given in device memory (one pass, no amax).
cudaError_t launch_quantize_nv_scaled(const float* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                                      const float* global_scale, int sms, cudaStream_t s);
cudaError_t launch_quantize_nv_scaled(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* sf,
                                      const float* global_scale, int sms, cudaStream_t s);

}  // namespace bsg
