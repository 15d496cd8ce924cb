// NVFP4 (E2M1 elements, UE4M3 per-16 scales) instantiations of the block-scaled GEMM kernel.
#include <cstdlib>

#include "gemm_pair_kernel.cuh"

namespace bsg {

bool gemm_kernel_info_nv(int bn, int out, int kc, GemmKernelInfo* info) {
  if (kc == 2) return gemm_kernel_info_nv_kc2(bn, out, info);
  if (bn < 128) return gemm_kernel_info_nv_narrow(bn, out, info);
  if (bn == 128 && out == OUT_F16) return fill_kernel_info<KIND_NV, 128, 1, OUT_F16>(info);
  if (bn == 128 && out == OUT_BF16) return fill_kernel_info<KIND_NV, 128, 1, OUT_BF16>(info);
  if (bn == 256 && out == OUT_F16) return fill_kernel_info<KIND_NV, 256, 1, OUT_F16>(info);
  if (bn == 256 && out == OUT_BF16) return fill_kernel_info<KIND_NV, 256, 1, OUT_BF16>(info);
  return false;
}

bool gemm_pair_kernel_info_nv(int out, GemmKernelInfo* info) {
  const char* e = std::getenv("BSG_PAIR_KC");
  const int kc = (e != nullptr && std::atoi(e) == 1) ? 1 : 2;  // two k-slabs per stage unless forced
  if (kc == 2 && out == OUT_F16) return fill_pair_kernel_info<KIND_NV, 2, OUT_F16>(info);
  if (kc == 2 && out == OUT_BF16) return fill_pair_kernel_info<KIND_NV, 2, OUT_BF16>(info);
  if (out == OUT_F16) return fill_pair_kernel_info<KIND_NV, 1, OUT_F16>(info);
  if (out == OUT_BF16) return fill_pair_kernel_info<KIND_NV, 1, OUT_BF16>(info);
  return false;
}

}  // namespace bsg
