// Kernel instantiations and launchers for the float element type.
#include "ks_kernels.cuh"

KS_DEFINE_LAUNCHERS(f32, float)
