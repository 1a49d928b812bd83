// Kernels of the row-wise log-sum-exp with the fused token log-probability
// epilogue, for bf16 elements (see lse_kernels.cuh).
#include "lse_kernels.cuh"

LSE_DEFINE_TYPE_ENTRY_POINTS(lse::kBF16, lp_bf16, true, false)
