// Kernels of the row-wise log-sum-exp with reduced-bit (packed bf16)
// exponentials, for f16 elements (see lse_kernels.cuh).
#include "lse_kernels.cuh"

LSE_DEFINE_TYPE_ENTRY_POINTS(lse::kF16, e16_f16, false, true)
