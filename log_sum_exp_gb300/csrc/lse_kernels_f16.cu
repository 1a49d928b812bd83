// Kernels of the row-wise log-sum-exp for f16 elements (see lse_kernels.cuh).
#include "lse_kernels.cuh"

LSE_DEFINE_TYPE_ENTRY_POINTS(lse::kF16, f16, false, false)
