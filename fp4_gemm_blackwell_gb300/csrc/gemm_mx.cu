// MXFP8 (E4M3 elements, UE8M0 per-32 scales) instantiations of the block-scaled GEMM kernel.
#include "gemm_kernel.cuh"

// Instantiated twice: here without the residual / factor epilogue and batch entries, and by the
// _ext twin of this file (which defines these two macros and includes it) with them.
#ifndef BSG_INST_EXT
#define BSG_INST_EXT false
#define BSG_INST_NAME(f) f
#endif

namespace bsg {

bool BSG_INST_NAME(gemm_kernel_info_mx)(int bn, int out, int kc, GemmKernelInfo* info) {
  if (kc == 2) return BSG_INST_NAME(gemm_kernel_info_mx_kc2)(bn, out, info);
  if (bn < 128) return BSG_INST_NAME(gemm_kernel_info_mx_narrow)(bn, out, info);
  if (bn == 128 && out == OUT_F16) return fill_kernel_info<KIND_MX, 128, 1, OUT_F16, BSG_INST_EXT>(info);
  if (bn == 128 && out == OUT_BF16) return fill_kernel_info<KIND_MX, 128, 1, OUT_BF16, BSG_INST_EXT>(info);
  if (bn == 256 && out == OUT_F16) return fill_kernel_info<KIND_MX, 256, 1, OUT_F16, BSG_INST_EXT>(info);
  if (bn == 256 && out == OUT_BF16) return fill_kernel_info<KIND_MX, 256, 1, OUT_BF16, BSG_INST_EXT>(info);
#ifdef BSG_INST_NV4
  if (bn == 256 && out == OUT_NV4) return fill_kernel_info<KIND_MX, 256, 1, OUT_NV4, true>(info);
#endif
  return false;
}

}  // namespace bsg
