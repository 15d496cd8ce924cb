// Instantiations of gemm_nv_kc2.cu with the residual and per-row / per-column factor epilogue and
// batch entries (EXT): the same lookups, named with an _ext suffix.
#define BSG_INST_EXT true
#define BSG_INST_NV4 1  // the NVFP4-output kernels live in the extended units only
#define BSG_INST_NAME(f) f##_ext
#include "gemm_nv_kc2.cu"
