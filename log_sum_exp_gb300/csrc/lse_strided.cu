// lse_strided.cu -- log-sum-exp over a non-last dimension (sm_103a).
//
//     out[a * C + c] = log sum_{r < R} exp(x[a * stride_a + r * stride_r + c])
//
// The reduction a probabilistic-circuit sum layer performs over the children
// of each node ("Speeding up Log-Sum-Exp: Kernel Fusion at the Memory Wall,
// Integer Arithmetic at the Compute Wall", Sec. 5.2), or a column LSE of a
// matrix.  One pass over x, per-column online (m, s) accumulators, the same
// pairwise merge and finalize as the row kernels (lse_device.cuh).
//
// Mapping: a CTA of 8 warps covers one column tile of 32 lanes x EPV columns
// (EPV = elements per 16-byte vector, or 1 when the layout is not 16-byte
// aligned) of one index a.  Warp w reads rows w, w + 8, ... so each load
// instruction covers one contiguous stretch of a row; a thread folds U rows
// per batch into EPV accumulators with one rescale per batch.  Shared memory
// merges the 8 warps.  With P > 1 the rows are split across blockIdx.z and
// the (m, s) partials [A * C, P] go to the row path's merge kernel.
#include <cstdint>

#include <cuda_runtime.h>

#include "lse_device.cuh"
#include "lse_internal.h"

namespace lse {
namespace {

constexpr int kColWarps = 8;
constexpr int kColThreads = 32 * kColWarps;

template <int DT, bool VEC>
__global__ void __launch_bounds__(kColThreads)
lse_cols_kernel(const void* __restrict__ x, int64_t A, int64_t R, int64_t C, int64_t stride_a,
                int64_t stride_r, int64_t rows_per_split, float* __restrict__ out,
                float2* __restrict__ partial, int64_t P) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int EPV = VEC ? 16 / EB : 1;
    constexpr int U = VEC ? 4 : 8;  // rows per batch per thread
    __shared__ float2 part[kColWarps][32][EPV];

    pdl_trigger();
    pdl_wait();

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * 32 + lane) * EPV;
    const bool active = c0 < C;  // VEC: C is a multiple of EPV, whole vectors only
    const int64_t split = blockIdx.z;
    const int64_t r_begin = split * rows_per_split;
    const int64_t r_end = r_begin + rows_per_split < R ? r_begin + rows_per_split : R;
    const char* xb = reinterpret_cast<const char*>(x);

    for (int64_t a = blockIdx.y; a < A; a += gridDim.y) {
        const char* base = xb + (a * stride_a + c0) * EB;
        Acc acc[EPV];
        float mu[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            acc[e] = acc_identity();
            mu[e] = 0.0f;
        }
        for (int64_t r = r_begin + wid; r < r_end; r += static_cast<int64_t>(kColWarps) * U) {
            float v[U][EPV];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t rr = r + j * kColWarps;
                const bool ok = active && rr < r_end;
                if constexpr (VEC) {
                    uint4 u = make_uint4(neg_inf_word<DT>(), neg_inf_word<DT>(), neg_inf_word<DT>(),
                                         neg_inf_word<DT>());
                    if (ok) u = ldg_stream16(base + rr * stride_r * EB);
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < EPV; ++e) v[j][e] = word_elem<DT>(w4, e);
                } else {
                    v[j][0] = ok ? load_elem<DT>(base, rr * stride_r) : __int_as_float(kNegInfF32);
                }
            }
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                float cm = v[0][e];
#pragma unroll
                for (int j = 1; j < U; ++j) cm = fmaxf(cm, v[j][e]);
                acc_raise(acc[e], mu[e], cm);
                float sum = 0.0f;
#pragma unroll
                for (int j = 0; j < U; ++j) sum += ex2((v[j][e] - mu[e]) * kLog2e);
                acc[e].s += sum;
            }
        }
#pragma unroll
        for (int e = 0; e < EPV; ++e) part[wid][lane][e] = make_float2(acc[e].m, acc[e].s);
        __syncthreads();
        if (wid == 0 && active) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                Acc t = acc_identity();
#pragma unroll
                for (int w = 0; w < kColWarps; ++w) t = acc_merge(t, Acc{part[w][lane][e].x, part[w][lane][e].y});
                const int64_t c = c0 + e;
                if (c < C) {
                    if (P == 1)
                        out[a * C + c] = acc_finalize(t);
                    else
                        partial[(a * C + c) * P + split] = make_float2(t.m, t.s);
                }
            }
        }
        __syncthreads();  // part[] is reused by the next a
    }
}

template <int DT, bool VEC>
cudaError_t launch_cols_t(const StridedArgs& a) {
    return launch_pdl(lse_cols_kernel<DT, VEC>, a.grid, dim3(kColThreads), a.stream, a.x, a.A, a.R,
                      a.C, a.stride_a, a.stride_r, a.rows_per_split, a.out, a.partial, a.P);
}

template <int DT, bool VEC>
int cols_occupancy_t() {
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, lse_cols_kernel<DT, VEC>, kColThreads,
                                                      0) != cudaSuccess)
        return 1;
    return blocks > 0 ? blocks : 1;
}

}  // namespace

cudaError_t launch_cols(int dt, bool vec, const StridedArgs& a) {
    switch (dt) {
    case kF32: return vec ? launch_cols_t<kF32, true>(a) : launch_cols_t<kF32, false>(a);
    case kBF16: return vec ? launch_cols_t<kBF16, true>(a) : launch_cols_t<kBF16, false>(a);
    default: return vec ? launch_cols_t<kF16, true>(a) : launch_cols_t<kF16, false>(a);
    }
}

int cols_occupancy(int dt, bool vec) {
    switch (dt) {
    case kF32: return vec ? cols_occupancy_t<kF32, true>() : cols_occupancy_t<kF32, false>();
    case kBF16: return vec ? cols_occupancy_t<kBF16, true>() : cols_occupancy_t<kBF16, false>();
    default: return vec ? cols_occupancy_t<kF16, true>() : cols_occupancy_t<kF16, false>();
    }
}

int cols_columns_per_cta(bool vec, int dt) { return 32 * (vec ? 16 / (dt == kF32 ? 4 : 2) : 1); }
int cols_rows_per_batch(bool vec) { return kColWarps * (vec ? 4 : 8); }

}  // namespace lse
