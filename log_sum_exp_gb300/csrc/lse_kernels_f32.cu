// Kernels of the row-wise log-sum-exp for f32 elements (see lse_kernels.cuh).
#include "lse_kernels.cuh"

LSE_DEFINE_TYPE_ENTRY_POINTS(lse::kF32, f32, false, false)
