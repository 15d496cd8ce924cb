// NVFP4 (E2M1 elements, UE4M3 per-16 scales) instantiations of the block-scaled GEMM kernel with
// 32- and 64-wide tiles (few row tiles: every SM gets a tile without splitting K).
#include "gemm_kernel.cuh"

// Instantiated twice: here without the residual / factor epilogue and batch entries, and by the
// _ext twin of this file (which defines these two macros and includes it) with them.
#ifndef BSG_INST_EXT
#define BSG_INST_EXT false
#define BSG_INST_NAME(f) f
#endif

namespace bsg {

bool BSG_INST_NAME(gemm_kernel_info_nv_narrow)(int bn, int out, GemmKernelInfo* info) {
  if (bn == 32 && out == OUT_F16) return fill_kernel_info<KIND_NV, 32, 1, OUT_F16, BSG_INST_EXT>(info);
  if (bn == 32 && out == OUT_BF16) return fill_kernel_info<KIND_NV, 32, 1, OUT_BF16, BSG_INST_EXT>(info);
  if (bn == 64 && out == OUT_F16) return fill_kernel_info<KIND_NV, 64, 1, OUT_F16, BSG_INST_EXT>(info);
  if (bn == 64 && out == OUT_BF16) return fill_kernel_info<KIND_NV, 64, 1, OUT_BF16, BSG_INST_EXT>(info);
#ifdef BSG_INST_NV4
  if (bn == 32 && out == OUT_NV4) return fill_kernel_info<KIND_NV, 32, 1, OUT_NV4, true>(info);
#endif
  return false;
}

}  // namespace bsg
