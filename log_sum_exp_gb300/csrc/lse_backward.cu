// lse_backward.cu -- gradient of the row-wise log-sum-exp (sm_103a).
//
// d lse[b] / d x[b, n] = exp(x[b, n] - lse[b]), so with the upstream gradient
// g[b] of each row value,
//
//     dx[b, n] = g[b] * exp(x[b, n] - lse[b]),
//
// one read of x and one write of dx ("Speeding up Log-Sum-Exp: Kernel Fusion
// at the Memory Wall, Integer Arithmetic at the Compute Wall", Table 3 lists
// backward support; lse[b] is the saved forward result).  The exponential is
// ex2.approx.ftz on (x - lse) * log2 e, computed in f32 and rounded once to
// the element type (nearest-even) on store.
//
// Mapping: a CTA is TX x TY threads; TY rows, TX threads across a row, each
// thread moving U = 4 slots (16-byte vectors, or single elements when rows are
// not 16-byte aligned) per iteration with every load issued before any store.
// blockIdx.x picks a segment of seg_slots slots of the row; rows beyond
// gridDim.y * TY are covered by a grid-stride loop.
#include <cstdint>

#include <cuda_runtime.h>

#include "lse_device.cuh"
#include "lse_internal.h"

namespace lse {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdU = 4;

// Two floats -> packed 16-bit pair, nearest-even.
template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (DT == kBF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int DT>
__device__ __forceinline__ void store_elem(void* row, int64_t i, float v) {
    if constexpr (DT == kF32) {
        reinterpret_cast<float*>(row)[i] = v;
    } else {
        const uint32_t p = pack2<DT>(v, 0.0f);
        reinterpret_cast<unsigned short*>(row)[i] = static_cast<unsigned short>(p & 0xffffu);
    }
}

__device__ __forceinline__ float grad_term(float x, float lse, float g) {
    return g * ex2((x - lse) * kLog2e);
}

// One 16-byte vector: 4 f32 or 8 16-bit elements.
template <int DT>
__device__ __forceinline__ uint4 grad_vector(uint4 u, float lse, float g) {
    if constexpr (DT == kF32) {
        return make_uint4(__float_as_uint(grad_term(__uint_as_float(u.x), lse, g)),
                          __float_as_uint(grad_term(__uint_as_float(u.y), lse, g)),
                          __float_as_uint(grad_term(__uint_as_float(u.z), lse, g)),
                          __float_as_uint(grad_term(__uint_as_float(u.w), lse, g)));
    } else {
        const uint32_t in[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = pack2<DT>(grad_term(word_lo<DT>(in[i]), lse, g),
                             grad_term(word_hi<DT>(in[i]), lse, g));
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kBwdThreads)
lse_backward_kernel(const void* __restrict__ x, int64_t B, int64_t N, int64_t row_stride,
                    const float* __restrict__ lse, const float* __restrict__ grad,
                    void* __restrict__ dx, int64_t dx_row_stride, int64_t seg_slots) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int EPV = VEC ? 16 / EB : 1;
    pdl_trigger();
    pdl_wait();
    const int TX = blockDim.x;
    const int64_t nv = N / EPV;            // full slots per row
    const int tail = static_cast<int>(N - nv * EPV);
    const int64_t k_begin = static_cast<int64_t>(blockIdx.x) * seg_slots;
    int64_t k_end = k_begin + seg_slots;
    const int64_t nvt = nv + (tail > 0 ? 1 : 0);
    if (k_end > nvt) k_end = nvt;

    for (int64_t row = static_cast<int64_t>(blockIdx.y) * blockDim.y + threadIdx.y; row < B;
         row += static_cast<int64_t>(gridDim.y) * blockDim.y) {
        const float l = __ldg(lse + row);
        const float g = __ldg(grad + row);
        const char* xr = reinterpret_cast<const char*>(x) + row * row_stride * EB;
        char* dr = reinterpret_cast<char*>(dx) + row * dx_row_stride * EB;
        for (int64_t k = k_begin + threadIdx.x; k < k_end; k += static_cast<int64_t>(TX) * kBwdU) {
            if constexpr (VEC) {
                uint4 v[kBwdU];
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t kk = k + j * TX;
                    if (kk < nv && kk < k_end) v[j] = ldg_stream16(xr + kk * 16);
                }
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t kk = k + j * TX;
                    if (kk < nv && kk < k_end) {
                        __stcs(reinterpret_cast<uint4*>(dr + kk * 16), grad_vector<DT>(v[j], l, g));
                    } else if (kk == nv && kk < k_end) {  // the < EPV tail elements
                        for (int i = 0; i < tail; ++i)
                            store_elem<DT>(dr, nv * EPV + i,
                                           grad_term(load_elem<DT>(xr, nv * EPV + i), l, g));
                    }
                }
            } else {
                float v[kBwdU];
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t kk = k + j * TX;
                    if (kk < k_end) v[j] = load_elem<DT>(xr, kk);
                }
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t kk = k + j * TX;
                    if (kk < k_end) store_elem<DT>(dr, kk, grad_term(v[j], l, g));
                }
            }
        }
    }
}

template <int DT, bool VEC>
cudaError_t launch_backward_t(const BackwardArgs& a) {
    return launch_pdl(lse_backward_kernel<DT, VEC>, a.grid, a.block, a.stream, a.x, a.B, a.N,
                      a.row_stride, a.lse, a.grad, a.dx, a.dx_row_stride, a.seg_slots);
}

}  // namespace

cudaError_t launch_backward(int dt, bool vec, const BackwardArgs& a) {
    switch (dt) {
    case kF32: return vec ? launch_backward_t<kF32, true>(a) : launch_backward_t<kF32, false>(a);
    case kBF16: return vec ? launch_backward_t<kBF16, true>(a) : launch_backward_t<kBF16, false>(a);
    default: return vec ? launch_backward_t<kF16, true>(a) : launch_backward_t<kF16, false>(a);
    }
}

int backward_slots_per_thread() { return kBwdU; }
int backward_threads() { return kBwdThreads; }

}  // namespace lse
