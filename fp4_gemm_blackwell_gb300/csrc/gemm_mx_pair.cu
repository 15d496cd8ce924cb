// MXFP8 (E4M3 elements, UE8M0 per-32 scales) instantiations of the CTA-pair kernel
// (256 x 256 tiles over 2-CTA clusters), in a translation unit of their own so that the build
// compiles them beside the 1-SM kernels.
#include <cstdlib>

#include "gemm_pair_kernel.cuh"

// Instantiated twice: here without the residual / factor epilogue and batch entries, and by the
// _ext twin of this file (which defines these macros and includes it) with them.
#ifndef BSG_INST_EXT
#define BSG_INST_EXT false
#define BSG_INST_NAME(f) f
#endif

namespace bsg {

bool BSG_INST_NAME(gemm_pair_kernel_info_mx)(int out, GemmKernelInfo* info) {
  const char* e = std::getenv("BSG_PAIR_KC");
  const int kc = (e != nullptr && std::atoi(e) == 2) ? 2 : 1;  // one k-slab per stage unless forced (more, smaller stages)
  if (kc == 2 && out == OUT_F16) return fill_pair_kernel_info<KIND_MX, 2, OUT_F16, BSG_INST_EXT>(info);
  if (kc == 2 && out == OUT_BF16) return fill_pair_kernel_info<KIND_MX, 2, OUT_BF16, BSG_INST_EXT>(info);
  if (out == OUT_F16) return fill_pair_kernel_info<KIND_MX, 1, OUT_F16, BSG_INST_EXT>(info);
  if (out == OUT_BF16) return fill_pair_kernel_info<KIND_MX, 1, OUT_BF16, BSG_INST_EXT>(info);
#ifdef BSG_INST_NV4
  if (out == OUT_NV4) return kc == 2 ? fill_pair_kernel_info<KIND_MX, 2, OUT_NV4, true>(info)
                                     : fill_pair_kernel_info<KIND_MX, 1, OUT_NV4, true>(info);
#endif
  return false;
}

}  // namespace bsg
