// NVFP4 (E2M1 elements, UE4M3 per-16 scales) instantiations of the block-scaled GEMM kernel with
// two 128-byte k-slabs per ring stage (64- and 128-wide tiles).
#include "gemm_kernel.cuh"

namespace bsg {

bool gemm_kernel_info_nv_kc2(int bn, int out, GemmKernelInfo* info) {
  if (bn == 64 && out == OUT_F16) return fill_kernel_info<KIND_NV, 64, 2, OUT_F16>(info);
  if (bn == 64 && out == OUT_BF16) return fill_kernel_info<KIND_NV, 64, 2, OUT_BF16>(info);
  if (bn == 128 && out == OUT_F16) return fill_kernel_info<KIND_NV, 128, 2, OUT_F16>(info);
  if (bn == 128 && out == OUT_BF16) return fill_kernel_info<KIND_NV, 128, 2, OUT_BF16>(info);
  return false;
}

}  // namespace bsg
