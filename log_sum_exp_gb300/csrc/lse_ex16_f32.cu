// Kernels of the row-wise log-sum-exp with reduced-bit (packed bf16)
// exponentials, for f32 elements (see lse_kernels.cuh).
#include "lse_kernels.cuh"

LSE_DEFINE_TYPE_ENTRY_POINTS(lse::kF32, e16_f32, false, true)
