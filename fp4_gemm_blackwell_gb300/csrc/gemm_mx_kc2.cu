// MXFP8 (E4M3 elements, UE8M0 per-32 scales) instantiations of the block-scaled GEMM kernel with
// two 128-byte k-slabs per ring stage (64- and 128-wide tiles).
#include "gemm_kernel.cuh"

namespace bsg {

bool gemm_kernel_info_mx_kc2(int bn, int out, GemmKernelInfo* info) {
  if (bn == 64 && out == OUT_F16) return fill_kernel_info<KIND_MX, 64, 2, OUT_F16>(info);
  if (bn == 64 && out == OUT_BF16) return fill_kernel_info<KIND_MX, 64, 2, OUT_BF16>(info);
  if (bn == 128 && out == OUT_F16) return fill_kernel_info<KIND_MX, 128, 2, OUT_F16>(info);
  if (bn == 128 && out == OUT_BF16) return fill_kernel_info<KIND_MX, 128, 2, OUT_BF16>(info);
  return false;
}

}  // namespace bsg
