/*
 * bsgemm.h -- block-scaled low-precision GEMM for GB300 (sm_103a), C ABI.
 *
 *     D = alpha * (A . B^T) (+ bias) (-> SiLU),  FP32 accumulation,  FP16 / BF16 output
 *
 * in two formats:
 *   MXFP8  E4M3 elements, one UE8M0 scale per 32 K-elements
 *          ("Add Cutlass MxFp8 Block Scale Matrix Multiplication": MxFp8GemmSm100,
 *           ElementA/B = mx_float8_t<float_e4m3_t>, ElementSFA/SFB = float_ue8m0_t);
 *   NVFP4  E2M1 elements (two per byte, element 2j in the low nibble of byte j), one
 *          UE4M3 scale per 16 K-elements, plus a float global factor alpha
 *          ("[QST] Performance overhead: Frequent cuTensorMapEncodeTiled and
 *           cudaGetDriverEntryPoint calls during Blackwell GEMM loops": runNvfp4Gemm<T,
 *           kEnableSilu, kEnableBias>(output, input_a, input_b, scales_a, scales_b, bias,
 *           alpha, M, N, K, stream)).
 *
 * Layouts (the MxFp8GemmSm100 element/layout configuration):
 *   A    M x K, row-major (K contiguous);  MXFP8 1 byte per element, NVFP4 K/2 bytes per row.
 *   B    N x K, row-major (K contiguous) -- the "ColumnMajor" K x N operand of the page.
 *   SFA  block scales of A in the swizzled 128x4 layout: rows padded to a multiple of 128,
 *        scale columns (K/32 or K/16) padded to a multiple of 4, cut into 512-byte atoms of
 *        128 rows x 4 columns stored band by band; inside an atom, scale (r, c) is at byte
 *        (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4).  Padding bytes must be 0.
 *        ("scales must be padded/swizzled to 128x4 blocks"; linear_to_swizzled_128_4.)
 *   SFB  the same for B (N rows).
 *   D    M x N, row-major, FP16 or BF16.   bias: N values of the output type.
 *
 * Ownership: the caller owns every device buffer and the stream.  The library owns the
 * plan, its TMA tensor maps and its workspace (allocated in bsg_plan_create, freed in
 * bsg_plan_destroy).  No call takes ownership of a caller pointer.
 *
 * Errors: every call returns a bsg_status; on failure bsg_last_error() holds a message
 * (thread-local).  Nothing is thrown across the ABI.  Validation happens before any device
 * work; an invalid argument never launches a kernel.  There is no CPU fallback: a device
 * that is not compute capability 10.3 gets BSG_ERR_ARCH.
 *
 * Asynchrony: run calls enqueue on the given stream and return; faults of a kernel surface
 * on a later synchronising call, and a kernel whose internal wait ran past its time limit
 * reports BSG_ERR_DEVICE_TIMEOUT through bsg_plan_check_status().
 */
#ifndef BSGEMM_H_
#define BSGEMM_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers (same type). */
typedef struct CUstream_st* bsg_stream_t;

typedef enum {
  BSG_OK = 0,
  BSG_ERR_INVALID_ARG = 1,   /* null pointer, null plan, bad enum, bad flags */
  BSG_ERR_SHAPE = 2,         /* M, N, K out of range, K / N not a multiple of the block,
                                or a buffer smaller than its shape needs */
  BSG_ERR_ALIGNMENT = 3,     /* a pointer not 16-byte aligned */
  BSG_ERR_SCALE_LAYOUT = 4,  /* scale buffer smaller than its padded 128x4 layout */
  BSG_ERR_DTYPE = 5,         /* output type / format combination not supported */
  BSG_ERR_ARCH = 6,          /* current device is not sm_103 */
  BSG_ERR_CUDA = 7,          /* a CUDA runtime / driver call failed (message holds it) */
  BSG_ERR_DEVICE_TIMEOUT = 8,/* a kernel's bounded internal wait expired */
  BSG_ERR_NOMEM = 9          /* a host or device allocation failed */
} bsg_status;

typedef enum { BSG_MXFP8 = 0, BSG_NVFP4 = 1 } bsg_kind;
/* NVFP4: D holds packed E2M1 codes (M x N/2 bytes, row-major, element 2j in the low nibble
 * of byte j) and SFD its UE4M3 block scales (one per 16 columns) in the swizzled 128x4 layout of
 * the scale operands (bsg_sf_bytes(BSG_NVFP4, M, N) bytes, padding written as zeros), quantised
 * with the global scale *d_scale by the recipe of bsg_quantize: ready to be the A operand of an
 * NVFP4 GEMM whose K is this N (its alpha then carries *d_scale). */
typedef enum { BSG_OUT_F16 = 0, BSG_OUT_BF16 = 1, BSG_OUT_NVFP4 = 2 } bsg_out;

/* Epilogue flags.  BIAS and SILU are the kEnableBias / kEnableSilu switches of
 * runNvfp4Gemm; ALPHA_DEVICE reads alpha from device memory at run time, the
 * fusion_args.alpha_ptr of the MXFP8 page.  C adds beta * C[m,n] from a separate matrix
 * (the MXFP8 page's LinearCombination epilogue with its C operand, there aliased to D);
 * ALPHA_ROW / ALPHA_COL multiply alpha by alpha_row[m] / alpha_col[n] (per-row and
 * per-column factors, e.g. per-token and per-channel global scales).  GROUPED makes the
 * problem a grouped GEMM (see bsg_desc). */
enum {
  BSG_F_BIAS = 1u,
  BSG_F_SILU = 2u,
  BSG_F_ALPHA_DEVICE = 4u,
  BSG_F_C = 8u,
  BSG_F_ALPHA_ROW = 16u,
  BSG_F_ALPHA_COL = 32u,
  BSG_F_GROUPED = 64u
};

typedef struct bsg_plan_s* bsg_plan_t;

/* One GEMM problem.  Pointers are device pointers, 16-byte aligned (alpha_dev, alpha_row
 * and alpha_col 4-byte aligned).
 *   M >= 1, N >= 16, K >= 32, N % 16 == 0, K % 32 == 0 (the MXFP8 page validates
 *   K % 16 and N % 16; K % 32 keeps every MXFP8 block whole and every NVFP4 row a
 *   whole number of 16-byte units).  M, N, K <= 2^20.
 *   bias is read only with BSG_F_BIAS; alpha_dev only with BSG_F_ALPHA_DEVICE (else the
 *   host value alpha is used); C (M x N, row-major, the output type; it may be D itself)
 *   and beta only with BSG_F_C; alpha_row (M floats) only with BSG_F_ALPHA_ROW; alpha_col
 *   (N floats) only with BSG_F_ALPHA_COL.  With every flag set
 *     D[m,n] = silu(alpha * alpha_row[m] * alpha_col[n] * acc[m,n] + bias[n] + beta * C[m,n]),
 *   the factors multiplied in float32 in that order, each term added in float32.
 * Batched (the L of the MXFP8 page's {m, n, k, l} problem shape): L >= 2 independent problems
 * of this shape in one launch, entry l at A + l*stride_A, B + l*stride_B, SFA + l*stride_SFA,
 * SFB + l*stride_SFB, D + l*stride_D and (with C) C + l*stride_C (strides in bytes, multiples
 * of 16, each at least one entry's size); bias, alpha, alpha_row and alpha_col are shared by all
 * entries, and with BSG_F_ALPHA_DEVICE alpha_dev holds one alpha per entry.  L = 0 or 1 is one
 * problem (the strides are then ignored); L <= 65535.
 * Grouped (BSG_F_GROUPED; a mixture-of-experts layer's expert GEMMs): L >= 1 groups share
 * N and K; group g has its own B (B + g*stride_B, SFB + g*stride_SFB) and, with
 * BSG_F_ALPHA_DEVICE, alpha_dev[g].  A, SFA, D and C hold the rows of every group: the M
 * rows of one matrix each, and group_index (M int32, device memory, read when the kernel
 * runs, so a preceding kernel may write it) gives each row's group, or -1 for a row that
 * belongs to none (not computed into D, D left as it was).  Each 128-row block of rows
 * (rows 128t .. 128t+127) must hold rows of at most one group plus rows of none; the group
 * of a block is that of its first row.  A block whose first row has no group (or a group
 * outside 0..L-1) is skipped whole, and a row whose group differs from its block's is not
 * stored.  So each group's rows start on a multiple of 128 and are padded with -1 rows to the
 * next one.  stride_A, stride_SFA, stride_D and stride_C are ignored.  Grouped problems run on
 * 128-row tiles (no CTA pairs).
 * NVFP4 output (out = BSG_OUT_NVFP4, single problems only): SFD (16-byte aligned) and d_scale
 * (one float, device memory, 4-byte aligned) are required; bias and C are BF16.  Each
 * 16-column block of y (the value before the output rounding above) is quantised in float32:
 * scale = UE4M3(amax / (6 s)), elements E2M1(y / (scale s)), s = *d_scale.  Such a problem is
 * never split along K. */
typedef struct {
  bsg_kind kind;
  bsg_out out;
  unsigned flags;
  int M, N, K;
  const void* A;
  const void* B;
  const void* SFA;
  const void* SFB;
  const void* bias;
  void* D;
  float alpha;
  const float* alpha_dev;
  const void* C;
  float beta;
  const float* alpha_row;
  const float* alpha_col;
  int L;
  long long stride_A, stride_B, stride_SFA, stride_SFB, stride_D, stride_C;
  const int* group_index;
  void* SFD;
  const float* d_scale;
} bsg_desc;

/* Validate d, choose the kernel variant (tile shape, split-K), encode the TMA tensor
 * maps once, allocate the plan's workspace and fill a launch configuration.  The plan
 * refers to d's pointers; it does not copy or own the buffers.  The device current at
 * this call is the plan's device.  Returns BSG_ERR_* without allocating on bad input.
 * (Split-K and variant choice may be forced with the BSG_FORCE_BN / BSG_FORCE_SPLITS
 * environment variables, read here.) */
bsg_status bsg_plan_create(bsg_plan_t* plan, const bsg_desc* d);

/* Enqueue the GEMM on `stream`: one kernel launch.  No tensor-map encoding, no driver
 * entry-point lookup, no allocation, no host synchronisation, so it can be captured in a
 * CUDA graph.  A plan may be in flight on one stream at a time (its split-K workspace is
 * shared between its launches). */
bsg_status bsg_plan_run(bsg_plan_t plan, bsg_stream_t stream);

/* The buffers of one run of a plan on operands other than those it was created with
 * (fields as in bsg_desc; those the plan's flags do not read are ignored). */
typedef struct {
  const void* A;
  const void* B;
  const void* SFA;
  const void* SFB;
  void* D;
  const void* bias;
  const float* alpha_dev;
  const void* C;
  const float* alpha_row;
  const float* alpha_col;
  const int* group_index;
  void* SFD;
  const float* d_scale;
} bsg_operands;

/* Pointer-agnostic run: enqueue the plan's GEMM on `ops`' buffers, which must have the
 * plan's shapes, strides and alignment (checked here as at plan creation, each buffer
 * against its allocation).  Nothing is re-encoded on the host: the new pointers travel as
 * kernel parameters.  Each CTA copies the plan's two TMA tensor maps into its own slot of
 * the plan's workspace and replaces their global addresses on the device (tensormap.replace,
 * the device-side form of re-encoding a tensor map that the launch-overhead page profiles
 * on the host), so a captured graph node of this call can be re-pointed by updating its
 * kernel parameters alone.  The plan's own buffers are untouched; bsg_plan_run still uses
 * them.  Same stream rule as bsg_plan_run. */
bsg_status bsg_plan_run_operands(bsg_plan_t plan, const bsg_operands* ops, bsg_stream_t stream);

/* Free the plan and its workspace.  Call after its last launch has completed. */
bsg_status bsg_plan_destroy(bsg_plan_t plan);

/* Synchronise the plan's device and read the plan's device status word: BSG_OK, or
 * BSG_ERR_DEVICE_TIMEOUT if a launch of this plan abandoned a wait.  Clears the word. */
bsg_status bsg_plan_check_status(bsg_plan_t plan);

/* Name of the kernel variant the plan chose, e.g. "mxfp8_bn256_s1" (owned by the plan). */
const char* bsg_plan_variant(bsg_plan_t plan);

/* One-shot calls: look the problem up in a process-wide plan cache (keyed on every
 * argument but alpha, and the device), create the plan on a miss, and run it.  After the first
 * call with given arguments, a call costs a lookup (lock-free when the calling thread used the
 * same arguments recently) and one launch. */
bsg_status mxfp8_gemm(void* D, const void* A, const void* B, const void* SFA, const void* SFB,
                      float alpha, int M, int N, int K, bsg_out out, bsg_stream_t stream);

bsg_status nvfp4_gemm(void* D, const void* A, const void* B, const void* SFA, const void* SFB,
                      const void* bias, float alpha, unsigned flags, int M, int N, int K,
                      bsg_out out, bsg_stream_t stream);

/* Allocation-free GEMM.  The pages have no counterpart of this call.  It is for callers that
 * cannot allocate device memory when they run a GEMM -- code running inside an allocator or
 * memory-pool callback, engines that forbid device allocation after start-up to keep a fixed
 * memory budget, hosts whose CUDA allocator belongs to someone else.  It computes exactly what
 * bsg_plan_create + bsg_plan_run compute for `d` (same validation, same kernel), but makes no
 * cudaMalloc, no cudaFree and no call to an allocating library routine.  Its status word,
 * split-K counters and split-K partial tiles live in one static device array of 16 MiB that
 * every GPU loading this library holds until the process exits; a problem whose split-K
 * partials would not fit is rejected with BSG_ERR_SHAPE (use a plan instead).
 * First use: the first call on a device looks up that array's device address (once per
 * device, with that device current), and the first call that runs a given kernel variant sets
 * its shared-memory attribute.  With CUDA's default lazy module loading, these first uses load
 * the library's device code and the array itself, which the driver does by allocating device
 * memory.  So make one call of each problem shape you will use outside the restricted context
 * and before any stream capture (or set CUDA_MODULE_LOADING=EAGER); calls after that allocate
 * nothing.  Every call clears the split-K counters at its start on `stream`; all calls share
 * the one array, so calls that overlap on the GPU (different streams, or concurrent host
 * threads) race.  A kernel that gives up a bounded wait records it in the array's status word,
 * which stays set until bsg_noalloc_check_status reads it.  Each call encodes its tensor maps
 * on the host, so it costs more host time than a plan's run. */
bsg_status bsg_gemm_noalloc(const bsg_desc* d, bsg_stream_t stream);

/* Status of the allocation-free calls on the current device: synchronise `stream` (the
 * stream of those calls), read the status word of the device's scratch array and clear it.
 * BSG_OK, or BSG_ERR_DEVICE_TIMEOUT if a bsg_gemm_noalloc launch on this device abandoned a
 * bounded wait since the last check (its output is then incomplete).  Allocates nothing. */
bsg_status bsg_noalloc_check_status(bsg_stream_t stream);

/* Drop every plan of the one-shot cache.  Call it after the work using them has completed and
 * while no other thread is inside a one-shot call. */
bsg_status bsg_cache_clear(void);

/* Bytes of the swizzled scale buffer of a rows x K operand: 128*ceil(rows/128) *
 * 4*ceil((K/blk)/4), blk = 32 (MXFP8) or 16 (NVFP4).  K must be a multiple of blk (so an
 * NVFP4 output's N, a multiple of 16, is accepted).  0 for invalid arguments. */
size_t bsg_sf_bytes(bsg_kind kind, int rows, int K);

/* Quantise a row-major float32 matrix x (rows x K, device) on `stream`:
 *   codes  rows x K bytes (MXFP8) or rows x K/2 bytes (NVFP4), device;
 *   sf     bsg_sf_bytes(kind, rows, K) bytes, written whole (padding zero), device;
 *   global_scale  NVFP4 only: device float receiving s = amax(|x|) / 2688 (it is used as
 *          the amax accumulator while the call runs); ignored for MXFP8.
 * MXFP8 per 32-block: e = least integer with amax <= 448 * 2^e (clamped to [-127, 127]),
 * scale code e + 127, element = E4M3 round-to-nearest-even saturating of x * 2^-e.
 * NVFP4: d = 6 s, block scale = UE4M3(amax_block / d), element = E2M1(x / (scale * s)),
 * each step one float32 operation rounded to nearest even (0 where a divisor is 0).
 * The GEMM factor of two NVFP4 operands is alpha = s_A * s_B.  The MXFP8 page's test
 * quantises with pytorch_mxfp8_quantize and swizzles with linear_to_swizzled_128_4 before
 * each GEMM.  rows >= 1, K >= 32, K % 32 == 0; x, codes, sf 16-byte aligned. */
bsg_status bsg_quantize(bsg_kind kind, const float* x, int rows, int K, void* codes, void* sf,
                        float* global_scale, bsg_stream_t stream);

/* bsg_quantize for a row-major BF16 matrix x (rows x K 16-bit BF16 values, device, 16-byte
 * aligned): each element is widened to float32 exactly (a BF16 value is the upper half of a
 * float32) and quantised as bsg_quantize quantises that float32, so the codes, the scale
 * buffer and the NVFP4 global scale are the bytes bsg_quantize writes for the widened matrix.
 * It reads half the bytes: the activation quantiser in front of a GEMM whose input comes out
 * of a BF16 layer (the MXFP8 page's test quantises its operands before every GEMM).  Same
 * arguments, ownership, stream ordering and errors as bsg_quantize. */
bsg_status bsg_quantize_bf16(bsg_kind kind, const void* x, int rows, int K, void* codes, void* sf,
                             float* global_scale, bsg_stream_t stream);

/* NVFP4 quantisation with the global scale s given by the caller: *global_scale (a device float,
 * read when the call runs, not written) takes the place of amax(|x|) / 2688, and steps 2-3 of the
 * NVFP4 recipe above run unchanged in one pass over x, with no amax pass: block scale =
 * UE4M3(amax_block / (6 s)), saturating at 448; element = E2M1(x / (scale * s)), saturating at 6;
 * s = 0 gives all-zero codes and scales.  The recipe's own s reproduces bsg_quantize's bytes.  This
 * is the quantiser in front of a GEMM whose activation scale is calibrated or carried over from the
 * previous step (as the NVFP4-output epilogue takes its s), the way the "[QST] Performance
 * overhead ..." page's Nvf4 GEMM receives a precomputed global alpha.  x holds rows x K float32
 * values (bf16_input = 0) or BF16 values (bf16_input != 0), 16-byte aligned; codes, sf as for
 * bsg_quantize.  Errors as bsg_quantize. */
bsg_status bsg_quantize_nvfp4_scaled(const void* x, int bf16_input, int rows, int K, void* codes, void* sf,
                                     const float* global_scale, bsg_stream_t stream);

/* Last error message of the calling thread ("" if none). */
const char* bsg_last_error(void);

/* Library version string. */
const char* bsg_version(void);

/* ---- test hooks (fault injection without a GPU fault) ----
 * Set the plan's bounded-wait limit (nanoseconds, 0 keeps the default of 2 s) and, with
 * skip_first_load != 0, make the producer of every CTA leave its first ring stage unfilled,
 * so that the tensor-core warp's wait runs out, the kernel flags BSG_ERR_DEVICE_TIMEOUT in
 * the plan's status word and returns cleanly.  With plan == NULL the setting applies to every
 * later bsg_gemm_noalloc call of the process (read back with bsg_noalloc_check_status).  For
 * tests of the failure path only. */
bsg_status bsg_plan_debug_set(bsg_plan_t plan, int skip_first_load, unsigned long long wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* BSGEMM_H_ */
