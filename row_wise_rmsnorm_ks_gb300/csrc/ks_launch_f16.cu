// Kernel instantiations and launchers for the __half element type.
#include "ks_kernels.cuh"

KS_DEFINE_LAUNCHERS(f16, __half)
