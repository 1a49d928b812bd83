"""GB300-native row-wise log-sum-exp: out[b] = log sum_n exp(x[b, n]).

The compute path is liblse (hand-written sm_103a CUDA kernels behind the C ABI
in include/lse.h); this package only builds it and marshals arguments to it.
Source of the method: "Speeding up Log-Sum-Exp: Kernel Fusion at the Memory
Wall, Integer Arithmetic at the Compute Wall" (Sec. 3.1, FuseLSE).
"""
from ._binding import (  # noqa: F401
    ABI_FUNCTIONS,
    DEFAULT_WAIT_POLLS,
    DTYPES,
    PATHS,
    LseError,
    LsePlan,
    library_path,
    load,
    logsumexp,
    lse_backward,
    lse_backward_ptr,
    lse_backward_strided_ptr,
    lse_forward,
    lse_forward16,
    lse_forward16_ptr,
    lse_forward_host,
    lse_forward_host_ptr,
    lse_forward_plan,
    lse_forward_plan_ptr,
    lse_forward_ptr,
    lse_forward_split_static_ptr,
    lse_forward_strided_ptr,
    lse_plan_query,
    lse_plan_query_ptr,
    lse_set_wait_limit,
    lse_token_logprob,
    lse_token_logprob_ptr,
    lse_trim_memory,
    lse_wait_timeouts,
    status_string,
)
