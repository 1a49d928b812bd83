// Kernels of the row-wise log-sum-exp with the fused token log-probability
// epilogue, for f32 elements (see lse_kernels.cuh).
#include "lse_kernels.cuh"

LSE_DEFINE_TYPE_ENTRY_POINTS(lse::kF32, lp_f32, true, false)
