// Kernels of the row-wise log-sum-exp with reduced-bit (packed bf16)
// exponentials, for bf16 elements (see lse_kernels.cuh).
#include "lse_kernels.cuh"

LSE_DEFINE_TYPE_ENTRY_POINTS(lse::kBF16, e16_bf16, false, true)
