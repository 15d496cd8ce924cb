// C ABI of the block-scaled GEMM library: validation, plans, tensor maps, launch, plan cache.
//
// The pages' host path ("[QST] Performance overhead: Frequent cuTensorMapEncodeTiled and
// cudaGetDriverEntryPoint calls ...", runNvfp4Gemm; and the runGemm launcher of "Add Cutlass
// MxFp8 Block Scale Matrix Multiplication") allocates a workspace, checks the arguments and
// encodes the TMA descriptors on EVERY call, then launches.  Here all of that happens once,
// in bsg_plan_create; bsg_plan_run is a single cudaLaunchKernelExC.  The driver entry points
// are resolved once per process.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <unordered_map>
#include <unordered_set>

#include "bsg_internal.h"
#include "bsgemm.h"

#define BSG_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr uint32_t kPlanMagic = 0xB5C0FFEEu;
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kMaxDim = 1 << 20;

thread_local std::string g_err;

// State of the allocation-free entry point (bsg_gemm_noalloc): the lock of its per-device
// scratch lookup, and its test hook (bsg_plan_debug_set with a null plan).
std::mutex g_noalloc_mutex;
int g_noalloc_skip_first_load = 0;
unsigned long long g_noalloc_wait_limit_ns = kDefaultWaitLimitNs;

bsg_status fail(bsg_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

bsg_status cuda_fail(cudaError_t e, const char* what) {
  return fail(BSG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------- driver entry points
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuMemGetAddressRange_v3020 g_addr_range = nullptr;
PFN_cuLaunchKernelEx_v11060 g_launch = nullptr;  // plan runs (see LaunchCfg)
std::once_flag g_driver_once;

bool load_driver_entry_points() {
  std::call_once(g_driver_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    fn = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 3020, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_addr_range = reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(fn);
    fn = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuLaunchKernelEx", &fn, 11060, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_launch = reinterpret_cast<PFN_cuLaunchKernelEx_v11060>(fn);
    cudaGetLastError();
  });
  return g_encode != nullptr;
}

// ---------------------------------------------------------------- device info
struct DeviceInfo {
  int major = 0, minor = 0, sms = 0;
};
std::mutex g_dev_mutex;
std::unordered_map<int, DeviceInfo> g_dev;

bsg_status current_device(int* dev, DeviceInfo* info) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  auto it = g_dev.find(*dev);
  if (it == g_dev.end()) {
    DeviceInfo di;
    if ((e = cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, *dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, *dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    it = g_dev.emplace(*dev, di).first;
  }
  // bind the device's primary context to this thread so that the driver calls below see it
  if ((e = cudaSetDevice(*dev)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  *info = it->second;
  if (info->major != 10 || info->minor != 3)
    return fail(BSG_ERR_ARCH, "device %d is compute capability %d.%d; this library runs on sm_103 only",
                *dev, info->major, info->minor);
  return BSG_OK;
}

// [p, p + need) must lie inside one device allocation.
bsg_status check_range(const void* p, size_t need, bsg_status code, const char* name) {
  if (g_addr_range == nullptr) return BSG_OK;  // no way to check: trust the caller
  CUdeviceptr base = 0;
  size_t size = 0;
  const CUresult r = g_addr_range(&base, &size, reinterpret_cast<CUdeviceptr>(p));
  if (r != CUDA_SUCCESS)
    return fail(BSG_ERR_INVALID_ARG, "%s (%p) is not a device allocation (driver error %d)", name, p,
                static_cast<int>(r));
  const size_t avail = static_cast<size_t>(base + size - reinterpret_cast<CUdeviceptr>(p));
  if (need > avail)
    return fail(code, "%s needs %zu bytes but its allocation holds %zu from that address", name, need,
                avail);
  return BSG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t sf_bytes_of(int kind, int rows, int K) {
  const int blk = kind == bsg::KIND_MX ? 32 : 16;
  const size_t rp = (static_cast<size_t>(rows) + 127) / 128 * 128;
  const size_t cp = (static_cast<size_t>(K / blk) + 3) / 4 * 4;
  return rp * cp;
}

size_t code_row_bytes(int kind, int K) { return kind == bsg::KIND_MX ? K : K / 2; }

int out_type(int out) {
  return out == BSG_OUT_BF16 ? bsg::OUT_BF16 : (out == BSG_OUT_NVFP4 ? bsg::OUT_NV4 : bsg::OUT_F16);
}

bsg_status validate_desc(const bsg_desc* d) {
  if (d == nullptr) return fail(BSG_ERR_INVALID_ARG, "descriptor is null");
  if (d->kind != BSG_MXFP8 && d->kind != BSG_NVFP4) return fail(BSG_ERR_INVALID_ARG, "unknown kind %d", d->kind);
  if (d->out != BSG_OUT_F16 && d->out != BSG_OUT_BF16 && d->out != BSG_OUT_NVFP4)
    return fail(BSG_ERR_DTYPE, "unsupported output type %d (FP16, BF16 or NVFP4)", d->out);
  if (d->out == BSG_OUT_NVFP4) {
    if (!d->SFD || !d->d_scale) return fail(BSG_ERR_INVALID_ARG, "NVFP4 output needs SFD and d_scale");
    if (!aligned16(d->SFD) || (reinterpret_cast<uintptr_t>(d->d_scale) & 3u))
      return fail(BSG_ERR_ALIGNMENT, "SFD must be 16-byte and d_scale 4-byte aligned");
    if (d->L > 1 || (d->flags & BSG_F_GROUPED))
      return fail(BSG_ERR_SHAPE, "NVFP4 output is for single problems (no batches or groups)");
  }
  if (d->flags &
      ~(BSG_F_BIAS | BSG_F_SILU | BSG_F_ALPHA_DEVICE | BSG_F_C | BSG_F_ALPHA_ROW | BSG_F_ALPHA_COL | BSG_F_GROUPED))
    return fail(BSG_ERR_INVALID_ARG, "unknown flag bits 0x%x", d->flags);
  if (d->M < 1 || d->N < 16 || d->K < 32 || d->M > kMaxDim || d->N > kMaxDim || d->K > kMaxDim)
    return fail(BSG_ERR_SHAPE, "shape M=%d N=%d K=%d out of range (M>=1, N>=16, K>=32, each <= 2^20)",
                d->M, d->N, d->K);
  if (d->N % 16) return fail(BSG_ERR_SHAPE, "N=%d is not a multiple of 16", d->N);
  if (d->K % 32) return fail(BSG_ERR_SHAPE, "K=%d is not a multiple of 32", d->K);
  if (d->L < 0 || d->L > 65535) return fail(BSG_ERR_SHAPE, "L=%d out of range (0..65535)", d->L);
  const bool grouped = (d->flags & BSG_F_GROUPED) != 0;
  if (grouped) {
    if (d->L < 1) return fail(BSG_ERR_SHAPE, "GROUPED needs L >= 1 groups");
    if (!d->group_index) return fail(BSG_ERR_INVALID_ARG, "GROUPED set but group_index is null");
    if (reinterpret_cast<uintptr_t>(d->group_index) & 3u)
      return fail(BSG_ERR_ALIGNMENT, "group_index must be 4-byte aligned");
  }
  if (d->L > 1) {
    // batched: every operand has L entries; grouped: B and SFB have one per group
    const long long rb = static_cast<long long>(code_row_bytes(d->kind, d->K));
    const long long dm = 2LL * d->M * d->N;
    const struct {
      long long stride, need;
      const char* name;
      bool used;
    } st[] = {{d->stride_A, rb * d->M, "stride_A", !grouped},
              {d->stride_B, rb * d->N, "stride_B", true},
              {d->stride_SFA, static_cast<long long>(sf_bytes_of(d->kind, d->M, d->K)), "stride_SFA", !grouped},
              {d->stride_SFB, static_cast<long long>(sf_bytes_of(d->kind, d->N, d->K)), "stride_SFB", true},
              {d->stride_D, dm, "stride_D", !grouped},
              {d->stride_C, dm, "stride_C", !grouped && (d->flags & BSG_F_C)}};
    for (const auto& x : st)
      if (x.used && (x.stride % 16 || x.stride < x.need))
        return fail(BSG_ERR_SHAPE, "%s=%lld must be a multiple of 16 and at least one entry (%lld bytes)", x.name,
                    x.stride, x.need);
  }
  if (!d->A || !d->B || !d->SFA || !d->SFB || !d->D) return fail(BSG_ERR_INVALID_ARG, "null operand pointer");
  if ((d->flags & BSG_F_BIAS) && !d->bias) return fail(BSG_ERR_INVALID_ARG, "BIAS set but bias is null");
  if ((d->flags & BSG_F_ALPHA_DEVICE) && !d->alpha_dev)
    return fail(BSG_ERR_INVALID_ARG, "ALPHA_DEVICE set but alpha_dev is null");
  if (!aligned16(d->A) || !aligned16(d->B) || !aligned16(d->SFA) || !aligned16(d->SFB) || !aligned16(d->D) ||
      ((d->flags & BSG_F_BIAS) && !aligned16(d->bias)))
    return fail(BSG_ERR_ALIGNMENT, "operand pointers must be 16-byte aligned");
  if ((d->flags & BSG_F_ALPHA_DEVICE) && (reinterpret_cast<uintptr_t>(d->alpha_dev) & 3u))
    return fail(BSG_ERR_ALIGNMENT, "alpha_dev must be 4-byte aligned");
  if ((d->flags & BSG_F_C) && !d->C) return fail(BSG_ERR_INVALID_ARG, "C set but C is null");
  if ((d->flags & BSG_F_ALPHA_ROW) && !d->alpha_row)
    return fail(BSG_ERR_INVALID_ARG, "ALPHA_ROW set but alpha_row is null");
  if ((d->flags & BSG_F_ALPHA_COL) && !d->alpha_col)
    return fail(BSG_ERR_INVALID_ARG, "ALPHA_COL set but alpha_col is null");
  if ((d->flags & BSG_F_C) && !aligned16(d->C)) return fail(BSG_ERR_ALIGNMENT, "C must be 16-byte aligned");
  if (((d->flags & BSG_F_ALPHA_ROW) && (reinterpret_cast<uintptr_t>(d->alpha_row) & 3u)) ||
      ((d->flags & BSG_F_ALPHA_COL) && (reinterpret_cast<uintptr_t>(d->alpha_col) & 3u)))
    return fail(BSG_ERR_ALIGNMENT, "alpha_row and alpha_col must be 4-byte aligned");
  return BSG_OK;
}

bsg_status validate_ranges(const bsg_desc* d) {
  const size_t rb = code_row_bytes(d->kind, d->K);
  const bool grouped = (d->flags & BSG_F_GROUPED) != 0;
  // bytes of L entries at `stride`, one entry being `one` bytes (A, SFA, D and C have one entry
  // when grouped)
  const size_t L1 = d->L > 1 ? static_cast<size_t>(d->L - 1) : 0;
  auto span = [&](long long stride, size_t one) { return L1 * static_cast<size_t>(stride) + one; };
  auto span_a = [&](long long stride, size_t one) { return grouped ? one : span(stride, one); };
  bsg_status s;
  if ((s = check_range(d->A, span_a(d->stride_A, rb * d->M), BSG_ERR_SHAPE, "A")) != BSG_OK) return s;
  if ((s = check_range(d->B, span(d->stride_B, rb * d->N), BSG_ERR_SHAPE, "B")) != BSG_OK) return s;
  if ((s = check_range(d->SFA, span_a(d->stride_SFA, sf_bytes_of(d->kind, d->M, d->K)), BSG_ERR_SCALE_LAYOUT,
                       "SFA")) != BSG_OK)
    return s;
  if ((s = check_range(d->SFB, span(d->stride_SFB, sf_bytes_of(d->kind, d->N, d->K)), BSG_ERR_SCALE_LAYOUT, "SFB")) !=
      BSG_OK)
    return s;
  const size_t d_bytes = static_cast<size_t>(d->M) * d->N * (d->out == BSG_OUT_NVFP4 ? 1 : 4) / 2;
  if ((s = check_range(d->D, span_a(d->stride_D, d_bytes), BSG_ERR_SHAPE, "D")) != BSG_OK) return s;
  if (d->out == BSG_OUT_NVFP4 &&
      ((s = check_range(d->SFD, sf_bytes_of(bsg::KIND_NV, d->M, d->N), BSG_ERR_SCALE_LAYOUT, "SFD")) != BSG_OK ||
       (s = check_range(d->d_scale, 4, BSG_ERR_SHAPE, "d_scale")) != BSG_OK))
    return s;
  if ((d->flags & BSG_F_BIAS) && (s = check_range(d->bias, static_cast<size_t>(d->N) * 2, BSG_ERR_SHAPE, "bias")) != BSG_OK)
    return s;
  // one alpha per entry (group) when there are several, else one
  if ((d->flags & BSG_F_ALPHA_DEVICE) &&
      (s = check_range(d->alpha_dev, 4 * (L1 + 1), BSG_ERR_SHAPE, "alpha_dev")) != BSG_OK)
    return s;
  if ((d->flags & BSG_F_C) &&
      (s = check_range(d->C, span_a(d->stride_C, static_cast<size_t>(d->M) * d->N * 2), BSG_ERR_SHAPE, "C")) != BSG_OK)
    return s;
  if (grouped &&
      (s = check_range(d->group_index, static_cast<size_t>(d->M) * 4, BSG_ERR_SHAPE, "group_index")) != BSG_OK)
    return s;
  if ((d->flags & BSG_F_ALPHA_ROW) &&
      (s = check_range(d->alpha_row, static_cast<size_t>(d->M) * 4, BSG_ERR_SHAPE, "alpha_row")) != BSG_OK)
    return s;
  if ((d->flags & BSG_F_ALPHA_COL) &&
      (s = check_range(d->alpha_col, static_cast<size_t>(d->N) * 4, BSG_ERR_SHAPE, "alpha_col")) != BSG_OK)
    return s;
  return BSG_OK;
}

}  // namespace

// A kernel's launch configuration, built once: the driver-API form for cuLaunchKernelEx (about
// 0.1 us of host time cheaper per launch than the runtime's cudaLaunchKernelExC on GB300, which
// matters at a launch of 1.4 us beside kernels of ~15 us) and the runtime form, used when the
// driver entry point or a function handle is missing, or when the driver call fails (e.g. on a
// thread with no current context, which the runtime call binds).  The attribute pointers point
// into the struct itself: it is built in place and never copied.
struct LaunchCfg {
  cudaLaunchConfig_t rt;
  cudaLaunchAttribute rt_attrs[2];
  CUlaunchConfig drv;
  CUlaunchAttribute drv_attrs[2];
};

struct bsg_plan_s {
  uint32_t magic;
  bsg_desc desc;
  bsg::PairParams params;
  bsg::GemmKernelInfo info;
  const void* fn_ext;        // the EXT instantiation of the same variant (bsg_plan_run_operands)
  CUtensorMap* map_slots;    // two sets of MAP_SLOTS_PER_CTA 128-byte tensor-map slots per CTA, in the workspace
  unsigned remap_runs;       // pointer-agnostic launches so far (their parity picks the slot set)
  int device;
  int grid;
  int cluster;
  void* workspace;
  char variant[64];
  // launch configuration built once at plan creation (a run only sets the stream)
  LaunchCfg lc;
  CUfunction cu_fn;      // driver handles of info.fn and fn_ext in the plan's device context
  CUfunction cu_fn_ext;
};

namespace {

std::mutex g_attr_mutex;
std::unordered_set<const void*> g_attr_done;

bsg_status ensure_smem_attr(const bsg::GemmKernelInfo& info, int device) {
  std::lock_guard<std::mutex> lk(g_attr_mutex);
  const void* key = reinterpret_cast<const char*>(info.fn) + device;  // per (kernel, device)
  if (g_attr_done.count(key)) return BSG_OK;
  cudaError_t e = cudaFuncSetAttribute(info.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, info.smem_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  g_attr_done.insert(key);
  return BSG_OK;
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (v == nullptr || *v == 0) return dflt;
  return std::atoi(v);
}

// Kernel variant, from measurements on GB300 (NVFP4 and MXFP8, M from 1 to 8192):
//  - M > 256 and at least a quarter as many 256 x 256 tiles as SMs: the CTA-pair kernel (its
//    per-SM shared-memory traffic per MMA is two thirds of the 1-SM tile's);
//  - else 1-SM tiles: 256 wide when they alone give every SM a tile, 128 wide when they give at
//    least two thirds of the SMs one; otherwise, for K of at most four k-tiles, 32-wide tiles
//    (more CTAs loading at once; split-K would cost more than it saves), and for longer K,
//    128-wide tiles with K split so that tiles x splits fills at most one wave (2, 4 or 8
//    splits reduce inside a thread-block cluster; other factors, only reachable by forcing,
//    go through the plan's global workspace).
// Every TMA copy of these kernels lands in the shared memory of the CTA that issues it; a
// cluster exists only for split-K reductions (DSMEM) and CTA pairs.
struct Variant {
  int bn, splits, kps, mode, cluster;
  int kc;        // 128-byte k-slabs per ring stage (1-SM kernel; kps counts ring stages)
  bool pair;     // CTA-pair kernel: 256 x 256 tiles over 2-CTA clusters
};

Variant choose_variant(const bsg_desc* d, int sms) {
  const int k_tile = d->kind == BSG_MXFP8 ? 128 : 256;
  const int nkt = (d->K + k_tile - 1) / k_tile;
  const long long mt = (d->M + 127) / 128;
  // tiles of all batch entries compete for the SMs; grouped rows are all in M already
  const bool grouped = (d->flags & BSG_F_GROUPED) != 0;
  const long long L = d->L > 1 && !grouped ? d->L : 1;
  const long long t256 = mt * ((d->N + 255) / 256) * L;
  const long long t128 = mt * ((d->N + 127) / 128) * L;
  const long long pair_tiles = ((d->M + 255) / 256) * ((d->N + 255) / 256) * L;
  int b, s = 1;
  bool pair = false;
  if (d->M > 256 && 4 * pair_tiles >= sms && !grouped) {
    pair = true;
    b = 256;
  } else if (t256 >= sms) {
    b = 256;
  } else if (3 * t128 >= 2LL * sms) {
    b = 128;
  } else if (nkt <= 4) {
    b = 32;
  } else {
    // split-K: 128- or 64-wide tiles, s = the largest power of two <= min(k-tiles, 8,
    // #SMs / tiles); pick the cheaper by a per-CTA cost in KB moved (measured weights): per
    // k-tile 16 (A) + bn/8 (B) + 10 / kc (control, per ring stage of kc k-slabs: two for
    // 64-wide tiles, see below), plus 5 per KB of partial rows exchanged over DSMEM ((s-1)/s
    // of a 128 x bn FP32 tile), which moves ~5x slower than TMA fills.
    double best = 1e30;
    for (int cb : {128, 64}) {
      // the NVFP4-output kernels that reduce split-K partials are the 64-wide ones
      if (d->out == BSG_OUT_NVFP4 && cb != 64) continue;
      const long long tiles = mt * ((d->N + cb - 1) / cb) * L;
      const long long want = std::min<long long>(std::min<long long>(nkt, 8), std::max<long long>(1, sms / tiles));
      int cs = 1;
      while (cs * 2 <= want) cs *= 2;
      const int kps = (nkt + cs - 1) / cs;
      const double ckc = (cb == 64 || cs == 1) ? 2.0 : 1.0;
      const double cost = kps * (16.0 + cb / 8.0 + 10.0 / ckc) + 5.0 * (cs - 1) / cs * (cb / 2.0);
      if (cost < best) {
        best = cost;
        b = cb;
        s = cs;
      }
    }
  }
  const int fb = env_int("BSG_FORCE_BN", 0);
  const int fs = env_int("BSG_FORCE_SPLITS", 0);
  if (fb == 32 || fb == 64 || fb == 128 || fb == 256) {  // a forced width runs unsplit unless
    b = fb;                                               // the splits are forced too
    pair = false;
    s = 1;
  }
  if (fs >= 1) s = std::min(fs, nkt);
  if (b < 64) s = 1;  // 32-wide tiles never split K
  if (d->out == BSG_OUT_NVFP4 && s > 1 && b != 64) s = 1;  // a forced other width runs unsplit
  // Two 128-byte k-slabs per ring stage halve the per-stage control (one barrier wait, one
  // commit, one scale staging per 8 MMAs) where the ring keeps three stages of the doubled size:
  // 64-wide tiles, and 128-wide tiles without a split-K receive area (measured: 128x4096x4096
  // 9.1 -> 8.1 us with 64-wide split-K 2; 128-wide split-K 4, left with 2 stages, got slower).
  int kc = (b == 64 || (b == 128 && s == 1)) ? 2 : 1;
  const int fk = env_int("BSG_KC", 0);
  if (fk == 1 || (fk == 2 && (b == 64 || b == 128))) kc = fk;
  const int nst = (nkt + kc - 1) / kc;  // ring stages along K
  int k = (nst + s - 1) / s;
  s = (nst + k - 1) / k;
  Variant v;
  v.kc = kc;
  v.pair = pair && env_int("BSG_FORCE_SPLITS", 0) == 0;
  const int fp = env_int("BSG_FORCE_PAIR", -1);
  if (fp == 0 || fp == 1) v.pair = fp == 1;
  if (grouped) v.pair = false;  // a 256-row pair tile could span two groups
  if (v.pair) {
    v.bn = 256;
    v.kc = 1;
    v.splits = 1;
    v.kps = nkt;
    v.mode = bsg::SPLIT_NONE;
    v.cluster = 2;
    return v;
  }
  v.bn = b;
  v.splits = s;
  v.kps = k;
  // A cluster split keeps 128 x (bn + 4) floats of partial rows in shared memory next to the
  // ring, which leaves 64- and 128-wide tiles enough stages and a 256-wide tile too few.
  const bool cluster_ok = (s == 2 || s == 4 || s == 8) && (b == 64 || b == 128);
  v.mode = s == 1 ? bsg::SPLIT_NONE
                  : (cluster_ok && env_int("BSG_SPLIT_WORKSPACE", 0) == 0 ? bsg::SPLIT_CLUSTER
                                                                           : bsg::SPLIT_WORKSPACE);
  v.cluster = v.mode == bsg::SPLIT_CLUSTER ? s : 1;
  return v;
}

// Workspace layout: [status word | per-tile counters | split-K partials (workspace mode) |
// tensor-map slots (pointer-agnostic runs: two sets of MAP_SLOTS_PER_CTA 128-byte maps per CTA
// of a grid of `grid`)].
struct WorkspaceLayout {
  size_t cnt_off, part_off, part_bytes, slot_off, total;
};

WorkspaceLayout workspace_layout(const Variant& v, int num_tiles, int grid) {
  WorkspaceLayout w;
  w.cnt_off = 256;
  w.part_off = w.cnt_off + (static_cast<size_t>(num_tiles) * 4 + 255) / 256 * 256;
  w.part_bytes = v.mode == bsg::SPLIT_WORKSPACE ? static_cast<size_t>(v.splits) * num_tiles * 128 * v.bn * 4 : 0;
  w.slot_off = (w.part_off + w.part_bytes + 255) / 256 * 256;
  w.total = w.slot_off + static_cast<size_t>(grid) * 2 * bsg::MAP_SLOTS_PER_CTA * sizeof(CUtensorMap);
  return w;
}

// Tiled map of a row-major code matrix (2-D), or of `batches` > 1 of them `batch_bytes` apart (3-D:
// the kernels load batched operands with the 3-D form of the copy, single ones with the 2-D form).
bsg_status encode_operand(CUtensorMap* m, const void* ptr, uint64_t row_bytes, uint64_t rows,
                          uint32_t box_rows, uint64_t batches, uint64_t batch_bytes, const char* name) {
  cuuint64_t dims[3] = {row_bytes, rows, batches};
  cuuint64_t strides[2] = {row_bytes, batch_bytes};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const cuuint32_t rank = batches > 1 ? 3 : 2;
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(ptr), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(BSG_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with driver error %d", name, static_cast<int>(r));
  return BSG_OK;
}

// Tiled map of the scale atoms of one operand for the CTA-pair kernel: 512-byte atoms as rows of
// 128 32-bit words, `rows` atoms per entry, `entries` entries `entry_bytes` apart; a box is the
// `box_atoms` consecutive atoms of one ring stage of one 128-row band.
bsg_status encode_scales(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t box_atoms, uint64_t entries,
                         uint64_t entry_bytes, const char* name) {
  cuuint64_t dims[3] = {128, rows, entries};
  cuuint64_t strides[2] = {512, entry_bytes};
  cuuint32_t box[3] = {128, box_atoms, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const cuuint32_t rank = entries > 1 ? 3 : 2;
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, rank, const_cast<void*>(ptr), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(BSG_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with driver error %d", name, static_cast<int>(r));
  return BSG_OK;
}

// Kernel parameters of problem d under variant v (tensor maps encoded here), except the
// workspace pointers.  Grid: persistent (<= #SMs) unless the splits form clusters, in which
// case every unit is its own CTA.
bsg_status fill_params(bsg::PairParams* g, const bsg_desc* d, const Variant& v, const bsg::GemmKernelInfo& info,
                       int sms, int* grid) {
  std::memset(g, 0, sizeof(*g));
  const size_t rb = code_row_bytes(d->kind, d->K);
  bsg_status s;
  const bool grouped = (d->flags & BSG_F_GROUPED) != 0;
  const int LB = d->L > 1 ? d->L : 1;  // entries of B and SFB (batch entries or groups)
  const int L = grouped ? 1 : LB;      // entries of A, SFA, D and C
  if ((s = encode_operand(&g->tmap_a, d->A, rb, d->M, 128u, L, d->stride_A, "A")) != BSG_OK ||
      (s = encode_operand(&g->tmap_b, d->B, rb, d->N, static_cast<uint32_t>(v.pair ? 128 : v.bn), LB, d->stride_B,
                          "B")) != BSG_OK)
    return s;
  g->batches = L;
  g->b_entries = LB;
  g->group_index = grouped ? d->group_index : nullptr;
  g->sfa_batch = L > 1 ? d->stride_SFA : 0;
  g->sfb_batch = LB > 1 ? d->stride_SFB : 0;
  g->d_batch = L > 1 ? d->stride_D / 2 : 0;
  g->c_batch = (L > 1 && (d->flags & BSG_F_C)) ? d->stride_C / 2 : 0;
  const int k_tile = d->kind == BSG_MXFP8 ? 128 : 256;
  const int blk = d->kind == BSG_MXFP8 ? 32 : 16;
  g->sfa = static_cast<const uint8_t*>(d->SFA);
  g->sfb = static_cast<const uint8_t*>(d->SFB);
  g->bias = d->bias;
  g->d = d->D;
  g->alpha_dev = d->alpha_dev;
  g->wait_limit_ns = kDefaultWaitLimitNs;
  g->alpha = d->alpha;
  g->M = d->M;
  g->N = d->N;
  g->K = d->K;
  // 32-byte stores (and loads of C) when D (16-bit output) and, if read, C are 32-byte aligned
  const bool d32 = (d->out == BSG_OUT_NVFP4 || (reinterpret_cast<uintptr_t>(d->D) & 31u) == 0) &&
                   (!(d->flags & BSG_F_C) || (reinterpret_cast<uintptr_t>(d->C) & 31u) == 0);
  if (d->out == BSG_OUT_NVFP4) {
    g->sfd = static_cast<uint8_t*>(d->SFD);
    g->d_scale = d->d_scale;
    g->sfd_cols4 = (d->N / 16 + 3) / 4;
  }
  g->flags = d->flags | (d32 ? bsg::F_D32 : 0u);
  g->c = (d->flags & BSG_F_C) ? d->C : nullptr;
  g->beta = d->beta;
  g->alpha_row = (d->flags & BSG_F_ALPHA_ROW) ? d->alpha_row : nullptr;
  g->alpha_col = (d->flags & BSG_F_ALPHA_COL) ? d->alpha_col : nullptr;
  g->sfa_atoms_per_band = (d->K / blk + 3) / 4;
  g->sfb_atoms_per_band = g->sfa_atoms_per_band;
  g->sfb_bands = (d->N + 127) / 128;
  g->sfa_bands = (d->M + 127) / 128;
  if (v.pair) {
    // the pair kernel loads its scale atoms with the pair form of the tiled copy, so that both
    // CTAs' atoms complete on the leader's barrier
    const uint32_t box_atoms = static_cast<uint32_t>(info.kc * (d->kind == BSG_MXFP8 ? 1 : 4));
    const uint64_t apb = static_cast<uint64_t>(g->sfa_atoms_per_band);
    if ((s = encode_scales(&g->tmap_sfa, d->SFA, g->sfa_bands * apb, box_atoms, L,
                           L > 1 ? static_cast<uint64_t>(d->stride_SFA) : g->sfa_bands * apb * 512, "SFA")) != BSG_OK ||
        (s = encode_scales(&g->tmap_sfb, d->SFB, g->sfb_bands * apb, box_atoms, LB,
                           LB > 1 ? static_cast<uint64_t>(d->stride_SFB) : g->sfb_bands * apb * 512, "SFB")) != BSG_OK)
      return s;
  }
  g->num_m_tiles = v.pair ? (d->M + 255) / 256 : (d->M + 127) / 128;
  g->num_n_tiles = (d->N + v.bn - 1) / v.bn;
  g->num_k_tiles = (d->K + k_tile * info.kc - 1) / (k_tile * info.kc);  // ring stages of K
  g->num_tiles = g->num_m_tiles * g->num_n_tiles * L;  // over all entries
  g->splits = v.splits;
  g->split_mode = v.mode;
  g->k_tiles_per_split = v.pair ? g->num_k_tiles : v.kps;  // in ring stages
  g->units_per_batch = g->num_m_tiles * g->num_n_tiles * v.splits;
  g->num_units = g->units_per_batch * L;
  // m-tiles per rasterisation group: NVFP4 pair tiles 32 (8192^3: 168 us against 171.5 with 16),
  // otherwise 16 (MXFP8 pair tiles, whose operands are twice the bytes: 32 read 726 MB from DRAM
  // against 252 MB and took 323 us against 304)
  const int group_default = (v.pair && d->kind == BSG_NVFP4) ? 32 : 16;
  g->group_m = std::max(1, env_int("BSG_GROUP_M", group_default));
  g->debug_skip_first_load = 0;
  g->ring_stages = info.stages;
  if (v.mode == bsg::SPLIT_CLUSTER) {
    // the split-K receive area, splits x (128 / splits) rows x (bn + 4) floats, takes the place
    // of the last ring stages
    const long long recv = 128LL * (v.bn + 4) * 4;
    g->ring_stages = info.stages - static_cast<int>((recv + info.stage_bytes - 1) / info.stage_bytes);
    if (g->ring_stages < 2)
      return fail(BSG_ERR_SHAPE, "split-K cluster receive slots leave fewer than two ring stages");
    // the peers' partial rows are staged in the ring before their bulk copies
    if (recv > static_cast<long long>(g->ring_stages) * info.stage_bytes)
      return fail(BSG_ERR_SHAPE, "split-K cluster staging does not fit the ring");
  }
  if (v.pair) *grid = 2 * std::min(g->num_units, sms / 2);
  else *grid = v.mode == bsg::SPLIT_CLUSTER ? g->num_units : std::min(g->num_units, sms);
  return BSG_OK;
}

// Launch configuration: grid, block, dynamic shared memory, programmatic dependent launch
// (unless BSG_PDL=0, read when the configuration is built) and the cluster shape, in both forms.
void make_launch_config(LaunchCfg* lc, int grid, int threads, int smem, int cluster) {
  std::memset(lc, 0, sizeof(*lc));
  int n = 0;
  if (env_int("BSG_PDL", 1)) {
    lc->rt_attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    lc->rt_attrs[n].val.programmaticStreamSerializationAllowed = 1;
    lc->drv_attrs[n].id = CU_LAUNCH_ATTRIBUTE_PROGRAMMATIC_STREAM_SERIALIZATION;
    lc->drv_attrs[n].value.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    lc->rt_attrs[n].id = cudaLaunchAttributeClusterDimension;
    lc->rt_attrs[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    lc->rt_attrs[n].val.clusterDim.y = 1;
    lc->rt_attrs[n].val.clusterDim.z = 1;
    lc->drv_attrs[n].id = CU_LAUNCH_ATTRIBUTE_CLUSTER_DIMENSION;
    lc->drv_attrs[n].value.clusterDim.x = static_cast<unsigned>(cluster);
    lc->drv_attrs[n].value.clusterDim.y = 1;
    lc->drv_attrs[n].value.clusterDim.z = 1;
    ++n;
  }
  lc->rt.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  lc->rt.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  lc->rt.dynamicSmemBytes = static_cast<size_t>(smem);
  lc->rt.attrs = lc->rt_attrs;
  lc->rt.numAttrs = n;
  lc->drv.gridDimX = static_cast<unsigned>(grid);
  lc->drv.gridDimY = 1;
  lc->drv.gridDimZ = 1;
  lc->drv.blockDimX = static_cast<unsigned>(threads);
  lc->drv.blockDimY = 1;
  lc->drv.blockDimZ = 1;
  lc->drv.sharedMemBytes = static_cast<unsigned>(smem);
  lc->drv.attrs = lc->drv_attrs;
  lc->drv.numAttrs = static_cast<unsigned>(n);
}

// One launch of `fn` (its driver handle `cu`, or null) with `params` on `stream`.
bsg_status launch_with(LaunchCfg* lc, const void* fn, CUfunction cu, const bsg::PairParams& params,
                       cudaStream_t stream) {
  void* args[] = {const_cast<bsg::PairParams*>(&params)};
  if (cu != nullptr && g_launch != nullptr) {
    lc->drv.hStream = reinterpret_cast<CUstream>(stream);
    if (g_launch(&lc->drv, cu, args, nullptr) == CUDA_SUCCESS) return BSG_OK;
  }
  lc->rt.stream = stream;
  const cudaError_t e = cudaLaunchKernelExC(&lc->rt, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC");
  return BSG_OK;
}

bsg_status launch_gemm(const void* fn, const bsg::PairParams& params, int grid, int threads, int smem,
                       int cluster, cudaStream_t stream) {
  LaunchCfg lc;
  make_launch_config(&lc, grid, threads, smem, cluster);
  return launch_with(&lc, fn, nullptr, params, stream);
}

// The driver handle of kernel `fn` in the current context, or null (the runtime path is used).
CUfunction driver_function(const void* fn) {
  cudaFunction_t f = nullptr;
  if (cudaGetFuncBySymbol(&f, fn) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<CUfunction>(f);
}

}  // namespace

namespace bsg {
bool find_kernel(int kind, int out, unsigned flags, int batches, bool pair, int bn, int kc, GemmKernelInfo* info) {
  const bool ext =
      (flags & (BSG_F_C | BSG_F_ALPHA_ROW | BSG_F_ALPHA_COL | BSG_F_GROUPED)) != 0 || batches > 1 || out == OUT_NV4;
  return find_kernel_variant(kind, out, ext, pair, bn, kc, info);
}
bool find_kernel_variant(int kind, int out, bool ext, bool pair, int bn, int kc, GemmKernelInfo* info) {
  if (pair) {
    if (kind == KIND_MX) return ext ? gemm_pair_kernel_info_mx_ext(out, info) : gemm_pair_kernel_info_mx(out, info);
    return ext ? gemm_pair_kernel_info_nv_ext(out, info) : gemm_pair_kernel_info_nv(out, info);
  }
  if (kind == KIND_MX) return ext ? gemm_kernel_info_mx_ext(bn, out, kc, info) : gemm_kernel_info_mx(bn, out, kc, info);
  return ext ? gemm_kernel_info_nv_ext(bn, out, kc, info) : gemm_kernel_info_nv(bn, out, kc, info);
}
}  // namespace bsg

namespace {

bsg_status plan_create(bsg_plan_t* out, const bsg_desc* d) {
  if (out == nullptr) return fail(BSG_ERR_INVALID_ARG, "plan output pointer is null");
  *out = nullptr;
  bsg_status s = validate_desc(d);
  if (s != BSG_OK) return s;
  int dev = 0;
  DeviceInfo di;
  if ((s = current_device(&dev, &di)) != BSG_OK) return s;
  if (!load_driver_entry_points())
    return fail(BSG_ERR_CUDA, "cannot resolve cuTensorMapEncodeTiled from the driver");
  if ((s = validate_ranges(d)) != BSG_OK) return s;

  const Variant v = choose_variant(d, di.sms);
  bsg::GemmKernelInfo info{};
  const int out_t = out_type(d->out);
  const bool found = bsg::find_kernel(d->kind == BSG_MXFP8 ? bsg::KIND_MX : bsg::KIND_NV, out_t, d->flags, d->L,
                                      v.pair, v.bn, v.kc, &info);
  if (!found) return fail(BSG_ERR_DTYPE, "no kernel for this format / output type / variant");
  if ((s = ensure_smem_attr(info, dev)) != BSG_OK) return s;
  bsg::GemmKernelInfo info_ext{};
  if (!bsg::find_kernel_variant(d->kind == BSG_MXFP8 ? bsg::KIND_MX : bsg::KIND_NV, out_t, true, v.pair, v.bn, v.kc,
                                &info_ext))
    return fail(BSG_ERR_DTYPE, "no extended kernel for this format / output type");
  if ((s = ensure_smem_attr(info_ext, dev)) != BSG_OK) return s;

  bsg_plan_s* p = new (std::nothrow) bsg_plan_s();
  if (p == nullptr) return fail(BSG_ERR_NOMEM, "host allocation of the plan failed");
  p->magic = kPlanMagic;
  p->desc = *d;
  p->info = info;
  p->fn_ext = info_ext.fn;
  p->remap_runs = 0;
  p->device = dev;
  p->workspace = nullptr;
  p->cluster = v.cluster;
  bsg::PairParams& g = p->params;
  if ((s = fill_params(&g, d, v, info, di.sms, &p->grid)) != BSG_OK) {
    delete p;
    return s;
  }
  const WorkspaceLayout w = workspace_layout(v, g.num_tiles, p->grid);
  cudaError_t e = cudaMalloc(&p->workspace, w.total);
  if (e != cudaSuccess) {
    delete p;
    cudaGetLastError();
    return fail(BSG_ERR_NOMEM, "cudaMalloc of a %zu-byte workspace failed", w.total);
  }
  e = cudaMemset(p->workspace, 0, w.part_off);
  if (e != cudaSuccess) {
    cudaFree(p->workspace);
    delete p;
    return cuda_fail(e, "cudaMemset(workspace)");
  }
  char* ws = static_cast<char*>(p->workspace);
  g.status = reinterpret_cast<unsigned*>(ws);
  g.counters = reinterpret_cast<unsigned*>(ws + w.cnt_off);
  g.partial = w.part_bytes ? reinterpret_cast<float*>(ws + w.part_off) : nullptr;
  p->map_slots = reinterpret_cast<CUtensorMap*>(ws + w.slot_off);
  static const char* kModeName[] = {"", "w", "c"};
  if (v.pair) {
    std::snprintf(p->variant, sizeof(p->variant), "%s_pair256_st%d_g%d", d->kind == BSG_MXFP8 ? "mxfp8" : "nvfp4",
                  info.stages, p->grid);
  } else {
    std::snprintf(p->variant, sizeof(p->variant), "%s_bn%d_s%d%s%s_st%d_g%d", d->kind == BSG_MXFP8 ? "mxfp8" : "nvfp4",
                  v.bn, v.splits, kModeName[v.mode], v.kc == 2 ? "_kc2" : "", g.ring_stages, p->grid);
  }
  make_launch_config(&p->lc, p->grid, info.threads, info.smem_bytes, p->cluster);
  p->cu_fn = driver_function(info.fn);
  p->cu_fn_ext = driver_function(info_ext.fn);
  if (env_int("BSG_LOG", 0))
    std::fprintf(stderr, "[bsgemm] plan M=%d N=%d K=%d -> %s\n", d->M, d->N, d->K, p->variant);
  *out = p;
  return BSG_OK;
}

bool plan_ok(bsg_plan_t p) { return p != nullptr && p->magic == kPlanMagic; }

bsg_status plan_launch(bsg_plan_t p, const bsg::PairParams& params, cudaStream_t stream) {
  return launch_with(&p->lc, p->info.fn, p->cu_fn, params, stream);
}

}  // namespace

// ==================================================================== exported C ABI

BSG_API const char* bsg_last_error(void) { return g_err.c_str(); }

BSG_API const char* bsg_version(void) { return "bsgemm 0.1 (sm_103a)"; }

BSG_API size_t bsg_sf_bytes(bsg_kind kind, int rows, int K) {
  const int blk = kind == BSG_MXFP8 ? 32 : 16;
  if ((kind != BSG_MXFP8 && kind != BSG_NVFP4) || rows < 1 || K < blk || K % blk) return 0;
  return sf_bytes_of(kind, rows, K);
}

BSG_API bsg_status bsg_plan_create(bsg_plan_t* plan, const bsg_desc* d) { return plan_create(plan, d); }

BSG_API bsg_status bsg_plan_run(bsg_plan_t plan, bsg_stream_t stream) {
  if (!plan_ok(plan)) return fail(BSG_ERR_INVALID_ARG, "invalid plan handle");
  return plan_launch(plan, plan->params, reinterpret_cast<cudaStream_t>(stream));
}

BSG_API bsg_status bsg_plan_run_operands(bsg_plan_t plan, const bsg_operands* ops, bsg_stream_t stream) {
  if (!plan_ok(plan)) return fail(BSG_ERR_INVALID_ARG, "invalid plan handle");
  if (ops == nullptr) return fail(BSG_ERR_INVALID_ARG, "operands are null");
  bsg_desc d = plan->desc;
  d.A = ops->A;
  d.B = ops->B;
  d.SFA = ops->SFA;
  d.SFB = ops->SFB;
  d.D = ops->D;
  d.bias = ops->bias;
  d.alpha_dev = ops->alpha_dev;
  d.C = ops->C;
  d.alpha_row = ops->alpha_row;
  d.alpha_col = ops->alpha_col;
  d.group_index = ops->group_index;
  d.SFD = ops->SFD;
  d.d_scale = ops->d_scale;
  bsg_status s = validate_desc(&d);
  if (s != BSG_OK) return s;
  if ((s = validate_ranges(&d)) != BSG_OK) return s;
  bsg::PairParams g = plan->params;
  g.sfa = static_cast<const uint8_t*>(d.SFA);
  g.sfb = static_cast<const uint8_t*>(d.SFB);
  g.bias = d.bias;
  g.d = d.D;
  g.alpha_dev = d.alpha_dev;
  g.c = (d.flags & BSG_F_C) ? d.C : nullptr;
  g.alpha_row = (d.flags & BSG_F_ALPHA_ROW) ? d.alpha_row : nullptr;
  g.alpha_col = (d.flags & BSG_F_ALPHA_COL) ? d.alpha_col : nullptr;
  g.group_index = (d.flags & BSG_F_GROUPED) ? d.group_index : nullptr;
  const bool d32 = (d.out == BSG_OUT_NVFP4 || (reinterpret_cast<uintptr_t>(d.D) & 31u) == 0) &&
                   (!(d.flags & BSG_F_C) || (reinterpret_cast<uintptr_t>(d.C) & 31u) == 0);
  g.flags = (g.flags & ~bsg::F_D32) | (d32 ? bsg::F_D32 : 0u);
  if (d.out == BSG_OUT_NVFP4) {
    g.sfd = static_cast<uint8_t*>(d.SFD);
    g.d_scale = d.d_scale;
  }
  // The kernel writes its slots before its programmatic-launch wait, while the plan's previous
  // launch may still run: consecutive pointer-agnostic launches take alternate slot sets.
  g.map_slots = plan->map_slots + static_cast<size_t>(plan->remap_runs++ & 1u) * bsg::MAP_SLOTS_PER_CTA * plan->grid;
  g.remap_a = d.A;
  g.remap_b = d.B;
  g.remap_sfa = d.SFA;
  g.remap_sfb = d.SFB;
  return launch_with(&plan->lc, plan->fn_ext, plan->cu_fn_ext, g, reinterpret_cast<cudaStream_t>(stream));
}

BSG_API bsg_status bsg_plan_destroy(bsg_plan_t plan) {
  if (!plan_ok(plan)) return fail(BSG_ERR_INVALID_ARG, "invalid plan handle");
  plan->magic = 0;
  cudaError_t e = cudaSuccess;
  if (plan->workspace) e = cudaFree(plan->workspace);
  delete plan;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
  return BSG_OK;
}

BSG_API bsg_status bsg_plan_check_status(bsg_plan_t plan) {
  if (!plan_ok(plan)) return fail(BSG_ERR_INVALID_ARG, "invalid plan handle");
  int cur = 0;
  cudaGetDevice(&cur);
  cudaError_t e = cudaSetDevice(plan->device);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  unsigned word = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&word, plan->params.status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word != 0) e = cudaMemset(plan->params.status, 0, sizeof(word));
  cudaSetDevice(cur);
  if (e != cudaSuccess) return cuda_fail(e, "reading the plan status word");
  if (word != 0)
    return fail(BSG_ERR_DEVICE_TIMEOUT, "a launch of this plan gave up a wait (status 0x%x:%s%s%s%s%s)", word,
                (word & bsg::ST_TIMEOUT_PRODUCER) ? " producer" : "", (word & bsg::ST_TIMEOUT_MMA) ? " mma" : "",
                (word & bsg::ST_TIMEOUT_EPILOGUE) ? " epilogue" : "", (word & bsg::ST_TIMEOUT_DRAIN) ? " drain" : "",
                (word & bsg::ST_TIMEOUT_SCALES) ? " scales" : "");
  return BSG_OK;
}

BSG_API const char* bsg_plan_variant(bsg_plan_t plan) {
  if (!plan_ok(plan)) return "";
  return plan->variant;
}

BSG_API bsg_status bsg_plan_debug_set(bsg_plan_t plan, int skip_first_load, unsigned long long wait_limit_ns) {
  if (plan == nullptr) {  // the allocation-free path's setting (process-wide)
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    g_noalloc_skip_first_load = skip_first_load ? 1 : 0;
    g_noalloc_wait_limit_ns = wait_limit_ns ? wait_limit_ns : kDefaultWaitLimitNs;
    return BSG_OK;
  }
  if (!plan_ok(plan)) return fail(BSG_ERR_INVALID_ARG, "invalid plan handle");
  plan->params.debug_skip_first_load = skip_first_load ? 1 : 0;
  plan->params.wait_limit_ns = wait_limit_ns ? wait_limit_ns : kDefaultWaitLimitNs;
  return BSG_OK;
}

// ---------------------------------------------------------------- one-shot plan cache
namespace {

struct CacheKey {
  int kind, out, M, N, K, device;
  unsigned flags;
  const void *A, *B, *SFA, *SFB, *bias, *D;
  bool operator==(const CacheKey& o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};
static_assert(sizeof(CacheKey) % 8 == 0, "the key is hashed in 8-byte words");

// A hash of the key's 8-byte words (its padding is zeroed when it is built).
uint64_t key_hash(const CacheKey& k) {
  uint64_t w[sizeof(CacheKey) / 8];
  std::memcpy(w, &k, sizeof(k));
  uint64_t h = 0x9E3779B97F4A7C15ull;
  for (uint64_t x : w) {
    h ^= x + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
    h *= 0xFF51AFD7ED558CCDull;
  }
  return h ^ (h >> 29);
}

struct CacheKeyHash {
  size_t operator()(const CacheKey& k) const { return static_cast<size_t>(key_hash(k)); }
};

std::mutex g_cache_mutex;
std::unordered_map<CacheKey, bsg_plan_t, CacheKeyHash> g_cache;
// Bumped by bsg_cache_clear: a per-thread entry of an older generation names a destroyed plan.
std::atomic<unsigned> g_cache_gen{1};

// Per-thread front of the cache: 16 direct-mapped entries, looked up without the lock.  A loop
// that cycles over a few problems finds its plan here after the first call of each.
struct ThreadEntry {
  CacheKey key;
  bsg_plan_t plan;
  unsigned gen;
};
thread_local ThreadEntry t_cache[16];

bsg_status cached_run(const bsg_desc& d, cudaStream_t stream) {
  const bsg_status vs = validate_desc(&d);  // before any CUDA call
  if (vs != BSG_OK) return vs;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  CacheKey key;
  std::memset(&key, 0, sizeof(key));  // padding bytes take part in the hash
  key.kind = d.kind;
  key.out = d.out;
  key.M = d.M;
  key.N = d.N;
  key.K = d.K;
  key.device = dev;
  key.flags = d.flags;
  key.A = d.A;
  key.B = d.B;
  key.SFA = d.SFA;
  key.SFB = d.SFB;
  key.bias = (d.flags & BSG_F_BIAS) ? d.bias : nullptr;
  key.D = d.D;
  bsg_plan_t plan = nullptr;
  const uint64_t h = key_hash(key);
  ThreadEntry& te = t_cache[(h >> 7) & 15];
  const unsigned gen = g_cache_gen.load(std::memory_order_acquire);
  if (te.plan != nullptr && te.gen == gen && te.key == key) {
    plan = te.plan;
  } else {
    std::lock_guard<std::mutex> lk(g_cache_mutex);
    auto it = g_cache.find(key);
    if (it != g_cache.end()) {
      plan = it->second;
    } else {
      bsg_status s = plan_create(&plan, &d);
      if (s != BSG_OK) return s;
      g_cache.emplace(key, plan);
    }
    te.key = key;
    te.plan = plan;
    te.gen = g_cache_gen.load(std::memory_order_relaxed);
  }
  if (plan->params.alpha == d.alpha) return plan_launch(plan, plan->params, stream);
  bsg::PairParams params = plan->params;  // alpha is not part of the key
  params.alpha = d.alpha;
  return plan_launch(plan, params, stream);
}

}  // namespace

BSG_API bsg_status mxfp8_gemm(void* D, const void* A, const void* B, const void* SFA, const void* SFB,
                              float alpha, int M, int N, int K, bsg_out out, bsg_stream_t stream) {
  bsg_desc d;
  std::memset(&d, 0, sizeof(d));
  d.kind = BSG_MXFP8;
  d.out = out;
  d.flags = 0;
  d.M = M;
  d.N = N;
  d.K = K;
  d.A = A;
  d.B = B;
  d.SFA = SFA;
  d.SFB = SFB;
  d.D = D;
  d.alpha = alpha;
  return cached_run(d, reinterpret_cast<cudaStream_t>(stream));
}

BSG_API bsg_status nvfp4_gemm(void* D, const void* A, const void* B, const void* SFA, const void* SFB,
                              const void* bias, float alpha, unsigned flags, int M, int N, int K, bsg_out out,
                              bsg_stream_t stream) {
  if (flags & BSG_F_ALPHA_DEVICE)
    return fail(BSG_ERR_INVALID_ARG, "nvfp4_gemm takes a host alpha; use a plan for a device alpha");
  bsg_desc d;
  std::memset(&d, 0, sizeof(d));
  d.kind = BSG_NVFP4;
  d.out = out;
  d.flags = flags;
  d.M = M;
  d.N = N;
  d.K = K;
  d.A = A;
  d.B = B;
  d.SFA = SFA;
  d.SFB = SFB;
  d.bias = bias;
  d.D = D;
  d.alpha = alpha;
  return cached_run(d, reinterpret_cast<cudaStream_t>(stream));
}

BSG_API bsg_status bsg_cache_clear(void) {
  std::lock_guard<std::mutex> lk(g_cache_mutex);
  g_cache_gen.fetch_add(1, std::memory_order_acq_rel);
  bsg_status r = BSG_OK;
  for (auto& kv : g_cache) {
    const bsg_status s = bsg_plan_destroy(kv.second);
    if (s != BSG_OK) r = s;
  }
  g_cache.clear();
  return r;
}

// ---------------------------------------------------------------- quantiser
// Shared by both quantiser entry points: validation, then the launch for element type T
// (float32, or BF16 bit patterns as uint16_t).
template <typename T>
static bsg_status quantize_entry(bsg_kind kind, const T* x, int rows, int K, void* codes, void* sf,
                                 float* global_scale, bsg_stream_t stream) {
  if (kind != BSG_MXFP8 && kind != BSG_NVFP4) return fail(BSG_ERR_INVALID_ARG, "unknown kind %d", kind);
  if (rows < 1 || K < 32 || K % 32 || rows > kMaxDim || K > kMaxDim)
    return fail(BSG_ERR_SHAPE, "quantise shape rows=%d K=%d (rows>=1, K>=32, K%%32==0, each <= 2^20)", rows, K);
  if (!x || !codes || !sf || (kind == BSG_NVFP4 && !global_scale))
    return fail(BSG_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(codes) || !aligned16(sf) ||
      (kind == BSG_NVFP4 && (reinterpret_cast<uintptr_t>(global_scale) & 3u)))
    return fail(BSG_ERR_ALIGNMENT, "x, codes and sf must be 16-byte aligned, global_scale 4-byte aligned");
  int dev = 0;
  DeviceInfo di;
  bsg_status s = current_device(&dev, &di);
  if (s != BSG_OK) return s;
  load_driver_entry_points();
  if ((s = check_range(x, static_cast<size_t>(rows) * K * sizeof(T), BSG_ERR_SHAPE, "x")) != BSG_OK ||
      (s = check_range(codes, code_row_bytes(kind, K) * rows, BSG_ERR_SHAPE, "codes")) != BSG_OK ||
      (s = check_range(sf, sf_bytes_of(kind, rows, K), BSG_ERR_SCALE_LAYOUT, "sf")) != BSG_OK ||
      (kind == BSG_NVFP4 && (s = check_range(global_scale, 4, BSG_ERR_SHAPE, "global_scale")) != BSG_OK))
    return s;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      kind == BSG_MXFP8
          ? bsg::launch_quantize_mx(x, rows, K, static_cast<uint8_t*>(codes), static_cast<uint8_t*>(sf), di.sms,
                                    st)
          : bsg::launch_quantize_nv(x, rows, K, static_cast<uint8_t*>(codes), static_cast<uint8_t*>(sf),
                                    global_scale, di.sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "quantiser launch");
  return BSG_OK;
}

BSG_API bsg_status bsg_quantize(bsg_kind kind, const float* x, int rows, int K, void* codes, void* sf,
                                float* global_scale, bsg_stream_t stream) {
  return quantize_entry(kind, x, rows, K, codes, sf, global_scale, stream);
}

BSG_API bsg_status bsg_quantize_bf16(bsg_kind kind, const void* x, int rows, int K, void* codes, void* sf,
                                     float* global_scale, bsg_stream_t stream) {
  return quantize_entry(kind, static_cast<const uint16_t*>(x), rows, K, codes, sf, global_scale, stream);
}

BSG_API bsg_status bsg_quantize_nvfp4_scaled(const void* x, int bf16_input, int rows, int K, void* codes, void* sf,
                                             const float* global_scale, bsg_stream_t stream) {
  if (rows < 1 || K < 32 || K % 32 || rows > kMaxDim || K > kMaxDim)
    return fail(BSG_ERR_SHAPE, "quantise shape rows=%d K=%d (rows>=1, K>=32, K%%32==0, each <= 2^20)", rows, K);
  if (!x || !codes || !sf || !global_scale) return fail(BSG_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(codes) || !aligned16(sf) || (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return fail(BSG_ERR_ALIGNMENT, "x, codes and sf must be 16-byte aligned, global_scale 4-byte aligned");
  int dev = 0;
  DeviceInfo di;
  bsg_status s = current_device(&dev, &di);
  if (s != BSG_OK) return s;
  load_driver_entry_points();
  const size_t elem = bf16_input ? 2 : 4;
  if ((s = check_range(x, static_cast<size_t>(rows) * K * elem, BSG_ERR_SHAPE, "x")) != BSG_OK ||
      (s = check_range(codes, code_row_bytes(BSG_NVFP4, K) * rows, BSG_ERR_SHAPE, "codes")) != BSG_OK ||
      (s = check_range(sf, sf_bytes_of(BSG_NVFP4, rows, K), BSG_ERR_SCALE_LAYOUT, "sf")) != BSG_OK ||
      (s = check_range(global_scale, 4, BSG_ERR_SHAPE, "global_scale")) != BSG_OK)
    return s;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      bf16_input ? bsg::launch_quantize_nv_scaled(static_cast<const uint16_t*>(x), rows, K, static_cast<uint8_t*>(codes),
                                                  static_cast<uint8_t*>(sf), global_scale, di.sms, st)
                 : bsg::launch_quantize_nv_scaled(static_cast<const float*>(x), rows, K, static_cast<uint8_t*>(codes),
                                                  static_cast<uint8_t*>(sf), global_scale, di.sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "quantiser launch");
  return BSG_OK;
}

// ==================================================================== allocation-free GEMM
// Some callers cannot allocate device memory at the point where they run a GEMM: code that
// runs inside a custom allocator or memory-pool callback, an engine that forbids device
// allocation after start-up so that its memory budget stays fixed, or a host environment
// where the CUDA allocator is owned by someone else.  bsg_gemm_noalloc serves them: it runs
// the same kernel as bsg_plan_run, but its status word, split-K counters and split-K partial
// tiles live in the file-scope device array below (kNoAllocScratchBytes per GPU that loads
// this library, held until the process exits) instead of a plan's cudaMalloc'ed workspace.
// The status word (offset 0) is cleared only by bsg_noalloc_check_status, so that a wait a
// kernel gave up stays visible until it is read; every call clears the split-K counters.

namespace {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kNoAllocMaxDevices = 64;
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

unsigned char* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on `dev` (current device); looked up once per device.
bsg_status noalloc_scratch(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(BSG_ERR_INVALID_ARG, "device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(allocation-free scratch)");
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return BSG_OK;
}

}  // namespace

BSG_API bsg_status bsg_gemm_noalloc(const bsg_desc* d, bsg_stream_t stream) {
  bsg_status s = validate_desc(d);
  if (s != BSG_OK) return s;
  int dev = 0;
  DeviceInfo di;
  if ((s = current_device(&dev, &di)) != BSG_OK) return s;
  if (!load_driver_entry_points())
    return fail(BSG_ERR_CUDA, "cannot resolve cuTensorMapEncodeTiled from the driver");
  if ((s = validate_ranges(d)) != BSG_OK) return s;

  const Variant v = choose_variant(d, di.sms);
  bsg::GemmKernelInfo info{};
  const int out_t = out_type(d->out);
  const bool found = bsg::find_kernel(d->kind == BSG_MXFP8 ? bsg::KIND_MX : bsg::KIND_NV, out_t, d->flags, d->L,
                                      v.pair, v.bn, v.kc, &info);
  if (!found) return fail(BSG_ERR_DTYPE, "no kernel for this format / output type");
  bsg::PairParams g;
  int grid = 0;
  if ((s = fill_params(&g, d, v, info, di.sms, &grid)) != BSG_OK) return s;
  // the same layout a plan's workspace has for this variant and tile count (no map slots)
  const WorkspaceLayout w = workspace_layout(v, g.num_tiles, 0);
  if (w.total > kNoAllocScratchBytes)
    return fail(BSG_ERR_SHAPE,
                "this problem needs %zu bytes of scratch (split-K %d over %d tiles); the allocation-free "
                "entry point has %zu; use a plan",
                w.total, v.splits, g.num_tiles, kNoAllocScratchBytes);
  unsigned char* scratch = nullptr;
  if ((s = noalloc_scratch(dev, &scratch)) != BSG_OK) return s;
  if ((s = ensure_smem_attr(info, dev)) != BSG_OK) return s;
  g.status = reinterpret_cast<unsigned*>(scratch);
  g.counters = reinterpret_cast<unsigned*>(scratch + w.cnt_off);
  g.partial = w.part_bytes ? reinterpret_cast<float*>(scratch + w.part_off) : nullptr;
  g.debug_skip_first_load = g_noalloc_skip_first_load;
  g.wait_limit_ns = g_noalloc_wait_limit_ns;

  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the split-K counters must start at zero (a launch that gave up a wait can leave them
  // set); the partial tiles are written whole by their split before they are read
  const cudaError_t e = cudaMemsetAsync(scratch + w.cnt_off, 0, w.part_off - w.cnt_off, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(allocation-free scratch)");
  return launch_gemm(info.fn, g, grid, info.threads, info.smem_bytes, v.cluster, st);
}

BSG_API bsg_status bsg_noalloc_check_status(bsg_stream_t stream) {
  int dev = 0;
  DeviceInfo di;
  bsg_status s = current_device(&dev, &di);
  if (s != BSG_OK) return s;
  unsigned char* scratch = nullptr;
  if ((s = noalloc_scratch(dev, &scratch)) != BSG_OK) return s;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned word = 0;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word != 0) e = cudaMemset(scratch, 0, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "reading the allocation-free status word");
  if (word != 0)
    return fail(BSG_ERR_DEVICE_TIMEOUT,
                "an allocation-free launch on this device gave up a wait (status 0x%x:%s%s%s%s%s)", word,
                (word & bsg::ST_TIMEOUT_PRODUCER) ? " producer" : "", (word & bsg::ST_TIMEOUT_MMA) ? " mma" : "",
                (word & bsg::ST_TIMEOUT_EPILOGUE) ? " epilogue" : "", (word & bsg::ST_TIMEOUT_DRAIN) ? " drain" : "",
                (word & bsg::ST_TIMEOUT_SCALES) ? " scales" : "");
  return BSG_OK;
}
