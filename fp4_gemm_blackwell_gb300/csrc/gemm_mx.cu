// MXFP8 (E4M3 elements, UE8M0 per-32 scales) instantiations of the block-scaled GEMM kernel.
#include <cstdlib>

#include "gemm_pair_kernel.cuh"

namespace bsg {

bool gemm_kernel_info_mx(int bn, int out, int kc, GemmKernelInfo* info) {
  if (kc == 2) return gemm_kernel_info_mx_kc2(bn, out, info);
  if (bn < 128) return gemm_kernel_info_mx_narrow(bn, out, info);
  if (bn == 128 && out == OUT_F16) return fill_kernel_info<KIND_MX, 128, 1, OUT_F16>(info);
  if (bn == 128 && out == OUT_BF16) return fill_kernel_info<KIND_MX, 128, 1, OUT_BF16>(info);
  if (bn == 256 && out == OUT_F16) return fill_kernel_info<KIND_MX, 256, 1, OUT_F16>(info);
  if (bn == 256 && out == OUT_BF16) return fill_kernel_info<KIND_MX, 256, 1, OUT_BF16>(info);
  return false;
}

bool gemm_pair_kernel_info_mx(int out, GemmKernelInfo* info) {
  const char* e = std::getenv("BSG_PAIR_KC");
  const int kc = (e != nullptr && std::atoi(e) == 1) ? 1 : 2;  // two k-tiles per stage unless forced
  if (kc == 2 && out == OUT_F16) return fill_pair_kernel_info<KIND_MX, 2, OUT_F16>(info);
  if (kc == 2 && out == OUT_BF16) return fill_pair_kernel_info<KIND_MX, 2, OUT_BF16>(info);
  if (out == OUT_F16) return fill_pair_kernel_info<KIND_MX, 1, OUT_F16>(info);
  if (out == OUT_BF16) return fill_pair_kernel_info<KIND_MX, 1, OUT_BF16>(info);
  return false;
}

}  // namespace bsg
