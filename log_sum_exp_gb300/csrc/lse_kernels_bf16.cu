// Kernels of the row-wise log-sum-exp for bf16 elements (see lse_kernels.cuh).
#include "lse_kernels.cuh"

LSE_DEFINE_TYPE_ENTRY_POINTS(lse::kBF16, bf16, false, false)
