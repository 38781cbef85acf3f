// Kernel instantiations and launchers for the __nv_bfloat16 element type.
#include "ks_kernels.cuh"

KS_DEFINE_LAUNCHERS(bf16, __nv_bfloat16)
