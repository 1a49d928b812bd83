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
// lse_backward_strided_kernel is the same gradient for the value over a
// non-last dimension (lse_forward_strided), with lse and grad per column.
//
// Mapping: a CTA is TX x TY threads; TY rows, TX threads across a row, each
// thread moving U = 4 slots per iteration with every load issued before any
// store.  A slot is a 16-byte vector, or a single element when x and dx rows
// do not share their offset from a 16-byte boundary.  With PEEL, rows that do
// share it but do not start on a boundary read and write their head (the
// elements before the first boundary) and their tail element by element, in
// two more slots, and the rest as aligned vectors.  blockIdx.x picks a segment
// of seg_slots slots of the row; rows beyond gridDim.y * TY are covered by a
// grid-stride loop.
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

// grad_term on two elements at once (packed FP32, the same rounding), each
// with its own lse and gradient.
__device__ __forceinline__ void grad_term2(float x0, float x1, uint64_t l2, uint64_t g2, float& d0,
                                           float& d1) {
    const uint64_t t = f2_mul(f2_sub(f2_pack(x0, x1), l2), f2_pack(kLog2e, kLog2e));
    f2_unpack(f2_mul(g2, f2_ex2(t)), d0, d1);
}

// One 16-byte vector, l2[i] and g2[i] the lse and gradient pairs of its
// elements 2i and 2i + 1 (f32: i < 2; 16-bit: the halves of word i).  The row
// gradient passes one pair throughout, the column gradient its columns'.
template <int DT>
__device__ __forceinline__ uint4 grad_vector_pairs(uint4 u, const uint64_t (&l2)[4],
                                                   const uint64_t (&g2)[4]) {
    float d[8];
    if constexpr (DT == kF32) {
        grad_term2(__uint_as_float(u.x), __uint_as_float(u.y), l2[0], g2[0], d[0], d[1]);
        grad_term2(__uint_as_float(u.z), __uint_as_float(u.w), l2[1], g2[1], d[2], d[3]);
        return make_uint4(__float_as_uint(d[0]), __float_as_uint(d[1]), __float_as_uint(d[2]),
                          __float_as_uint(d[3]));
    } else {
        const uint32_t in[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            grad_term2(word_lo<DT>(in[i]), word_hi<DT>(in[i]), l2[i], g2[i], d[2 * i], d[2 * i + 1]);
            o[i] = pack2<DT>(d[2 * i], d[2 * i + 1]);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// One 16-byte vector of a row: 4 f32 or 8 16-bit elements, one lse and gradient.
template <int DT>
__device__ __forceinline__ uint4 grad_vector(uint4 u, float lse, float g) {
    const uint64_t l2 = f2_pack(lse, lse), g2 = f2_pack(g, g);
    const uint64_t lp[4] = {l2, l2, l2, l2}, gp[4] = {g2, g2, g2, g2};
    return grad_vector_pairs<DT>(u, lp, gp);
}

// Elements of row `rp` before its first 16-byte boundary, at most N.
template <int DT>
__device__ __forceinline__ int64_t head_elems_of(const void* rp, int64_t N) {
    const int64_t h = static_cast<int64_t>((16u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(rp)) & 15u)) & 15u) /
                      DType<DT>::bytes;
    return N < h ? N : h;
}

// The elements [i0, i0 + n) of a row, n < 16 / element bytes (a head or a
// tail): every load issued before the first store, so the loads overlap and
// dx may be x.
template <int DT>
__device__ __forceinline__ void grad_elems(const char* xr, char* dr, int64_t i0, int n,
                                           float l, float g) {
    constexpr int M = 16 / DType<DT>::bytes - 1;
    float v[M];
#pragma unroll
    for (int i = 0; i < M; ++i)
        if (i < n) v[i] = load_elem<DT>(xr, i0 + i);
#pragma unroll
    for (int i = 0; i < M; ++i)
        if (i < n) store_elem<DT>(dr, i0 + i, grad_term(v[i], l, g));
}

// At most 64 registers: 4 CTAs (32 warps) per SM.
template <int DT, bool VEC, bool PEEL>
__global__ void __launch_bounds__(kBwdThreads, 4)
lse_backward_kernel(const void* __restrict__ x, int64_t B, int64_t N, int64_t row_stride,
                    const float* __restrict__ lse, const float* __restrict__ grad,
                    void* __restrict__ dx, int64_t dx_row_stride, int64_t seg_slots) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int EPV = VEC ? 16 / EB : 1;
    pdl_trigger();
    pdl_wait();
    const int TX = blockDim.x;
    const int64_t nv0 = N / EPV;  // full slots of a row on a 16-byte boundary
    const int tail0 = static_cast<int>(N - nv0 * EPV);
    // Slots per row: full vectors, then the tail slot, then (PEEL) the head slot.
    const int64_t nvt = PEEL ? nv0 + 2 : nv0 + (tail0 > 0 ? 1 : 0);
    const int64_t k_begin = static_cast<int64_t>(blockIdx.x) * seg_slots;
    int64_t k_end = k_begin + seg_slots;
    if (k_end > nvt) k_end = nvt;

    for (int64_t row = static_cast<int64_t>(blockIdx.y) * blockDim.y + threadIdx.y; row < B;
         row += static_cast<int64_t>(gridDim.y) * blockDim.y) {
        const float l = __ldg(lse + row);
        const float g = __ldg(grad + row);
        const char* xr = reinterpret_cast<const char*>(x) + row * row_stride * EB;
        char* dr = reinterpret_cast<char*>(dx) + row * dx_row_stride * EB;
        int head = 0;
        int64_t nv = nv0;
        int tail = tail0;
        if constexpr (PEEL) {
            head = static_cast<int>(head_elems_of<DT>(xr, N));
            nv = (N - head) / EPV;
            tail = static_cast<int>(N - head - nv * EPV);
        }
        const char* xv = xr + head * EB;  // 16-byte aligned, as is dv
        char* dv = dr + head * EB;
        for (int64_t k = k_begin + threadIdx.x; k < k_end; k += static_cast<int64_t>(TX) * kBwdU) {
            if constexpr (VEC) {
                uint4 v[kBwdU];
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t kk = k + j * TX;
                    if (kk < nv && kk < k_end) v[j] = ldg_stream16(xv + kk * 16);
                }
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t kk = k + j * TX;
                    if (kk >= k_end) continue;
                    if (kk < nv)
                        __stcs(reinterpret_cast<uint4*>(dv + kk * 16), grad_vector<DT>(v[j], l, g));
                    else if (kk == nv && tail > 0)  // the < EPV tail elements
                        grad_elems<DT>(xv, dv, nv * EPV, tail, l, g);
                    else if (PEEL && kk == nv + (tail > 0 ? 1 : 0) && head > 0)  // the head
                        grad_elems<DT>(xr, dr, 0, head, l, g);
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

// One 16-byte vector whose elements belong to different columns, each with
// its own lse and gradient.
template <int DT, int EPV>
__device__ __forceinline__ uint4 grad_vector_cols(uint4 u, const float (&l)[EPV],
                                                  const float (&g)[EPV]) {
    if constexpr (DT == kF32) {
        // f32 columns stay scalar: the pairs cost the one-warp tiles 16
        // registers and two CTAs per SM (pcsum [512, 64, 1024] 41.3 -> 45.5 us).
        return make_uint4(__float_as_uint(grad_term(__uint_as_float(u.x), l[0], g[0])),
                          __float_as_uint(grad_term(__uint_as_float(u.y), l[1], g[1])),
                          __float_as_uint(grad_term(__uint_as_float(u.z), l[2], g[2])),
                          __float_as_uint(grad_term(__uint_as_float(u.w), l[3], g[3])));
    }
    uint64_t lp[4], gp[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = 2 * i < EPV ? 2 * i : 0;  // f32: pairs 0 and 1 only
        lp[i] = f2_pack(l[e], l[e + 1 < EPV ? e + 1 : 0]);
        gp[i] = f2_pack(g[e], g[e + 1 < EPV ? e + 1 : 0]);
    }
    return grad_vector_pairs<DT>(u, lp, gp);
}

// Gradient of the value over a non-last dimension:
//     dx[a, r, c] = grad[a, c] * exp(x[a, r, c] - lse[a, c]),
// lse and grad dense [A, C].  A unit is one (a, column tile) pair, the tile
// LPT lanes x EPV columns (a 16-byte vector per lane, or one element when the
// layout is not 16-byte aligned); a lane loads its columns' lse and gradient
// once per unit.  LPT is 32, or 16 or 8 for one-warp units of narrow C (the
// column kernel's rule), a warp then taking 32 / LPT units side by side.  WT
// warps (1 or kStrWarps) share a unit and interleave the rows of blockIdx.z's
// split, each with kBwdU rows in flight (all loads before any store, so dx
// may be x).  A CTA's warps take consecutive units (several a when C is
// narrow) and CTAs stride over the units; nothing is merged, so every warp
// loops on its own.
constexpr int kStrWarps = 4;

template <int DT, bool VEC, int WT, int LPT>
__global__ void __launch_bounds__(32 * kStrWarps)
lse_backward_strided_kernel(const void* __restrict__ x, int64_t A, int64_t R, int64_t C,
                            int64_t stride_a, int64_t stride_r, const float* __restrict__ lse,
                            const float* __restrict__ grad, void* __restrict__ dx,
                            int64_t dx_stride_a, int64_t dx_stride_r, int64_t rows_per_split) {
    static_assert(LPT == 32 || ((LPT == 16 || LPT == 8) && WT == 1), "narrow tiles are one-warp units");
    constexpr int EB = DType<DT>::bytes;
    constexpr int EPV = VEC ? 16 / EB : 1;
    constexpr int UPW = 32 / LPT;             // units per warp
    constexpr int UPC = kStrWarps / WT * UPW;  // units per CTA
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int phase = wid % WT;
    const int64_t r_begin = static_cast<int64_t>(blockIdx.z) * rows_per_split;
    const int64_t r_end = r_begin + rows_per_split < R ? r_begin + rows_per_split : R;
    const int64_t wtiles = (C + LPT * EPV - 1) / (LPT * EPV);
    const int64_t units = A * wtiles;
    for (int64_t u0 = static_cast<int64_t>(blockIdx.x) * UPC + (wid / WT) * UPW; u0 < units;
         u0 += static_cast<int64_t>(gridDim.x) * UPC) {
        const int64_t unit = u0 + (UPW > 1 ? lane / LPT : 0);
        const int64_t a = unit < units ? unit / wtiles : 0;
        const int64_t c0 = ((unit - a * wtiles) * LPT + (lane & (LPT - 1))) * EPV;
        // VEC: C is a multiple of EPV, whole vectors only
        const bool active = unit < units && c0 < C;
        float l[EPV], g[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            l[e] = active ? __ldg(lse + a * C + c0 + e) : 0.0f;
            g[e] = active ? __ldg(grad + a * C + c0 + e) : 0.0f;
        }
        const char* xa = reinterpret_cast<const char*>(x) + (a * stride_a + (active ? c0 : 0)) * EB;
        char* da = reinterpret_cast<char*>(dx) + (a * dx_stride_a + (active ? c0 : 0)) * EB;
        for (int64_t r = r_begin + phase; r < r_end; r += static_cast<int64_t>(WT) * kBwdU) {
            if constexpr (VEC) {
                uint4 v[kBwdU];
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t rr = r + j * WT;
                    if (active && rr < r_end) v[j] = ldg_stream16(xa + rr * stride_r * EB);
                }
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t rr = r + j * WT;
                    if (active && rr < r_end)
                        __stcs(reinterpret_cast<uint4*>(da + rr * dx_stride_r * EB),
                               grad_vector_cols<DT, EPV>(v[j], l, g));
                }
            } else {
                float v[kBwdU];
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t rr = r + j * WT;
                    if (active && rr < r_end) v[j] = load_elem<DT>(xa, rr * stride_r);
                }
#pragma unroll
                for (int j = 0; j < kBwdU; ++j) {
                    const int64_t rr = r + j * WT;
                    if (active && rr < r_end)
                        store_elem<DT>(da, rr * dx_stride_r, grad_term(v[j], l[0], g[0]));
                }
            }
        }
    }
}

template <int DT, bool VEC>
cudaError_t launch_backward_strided_t(const BackwardStridedArgs& a) {
#define LSE_SBWD_LAUNCH(WT, LPT)                                                                     \
    return launch_pdl(lse_backward_strided_kernel<DT, VEC, WT, LPT>, a.grid, dim3(32 * kStrWarps), \
                      a.stream, a.x, a.A, a.R, a.C, a.stride_a, a.stride_r, a.lse, a.grad, a.dx,    \
                      a.dx_stride_a, a.dx_stride_r, a.rows_per_split)
    if (a.warps_per_unit != 1) LSE_SBWD_LAUNCH(kStrWarps, 32);
    switch (a.lanes_per_tile) {
    case 8: LSE_SBWD_LAUNCH(1, 8);
    case 16: LSE_SBWD_LAUNCH(1, 16);
    case 32: LSE_SBWD_LAUNCH(1, 32);
    default: return cudaErrorInvalidValue;
    }
#undef LSE_SBWD_LAUNCH
}

// Rows of at most kBwdU slots: the (row, slot) pairs are flattened and each
// thread keeps kBwdU of them in flight (slot q, q + stride, ...), so
// consecutive threads touch consecutive vectors whatever the row length.  A
// slot is a 16-byte vector (VEC; slot nv of a row holds its < EPV tail
// elements and, with PEEL, the next one its head) or one element.  lse and
// grad are read per slot; a row's slots share them in L1.
template <int DT, bool VEC, bool PEEL>
__global__ void __launch_bounds__(kBwdThreads, PEEL ? 3 : 4)
lse_backward_small_kernel(const void* __restrict__ x, int64_t B, int64_t N, int64_t row_stride,
                          const float* __restrict__ lse, const float* __restrict__ grad,
                          void* __restrict__ dx, int64_t dx_row_stride) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int EPV = VEC ? 16 / EB : 1;
    pdl_trigger();
    pdl_wait();
    const int nv0 = static_cast<int>(N / EPV);  // full slots of a row on a 16-byte boundary
    const int tail0 = static_cast<int>(N - static_cast<int64_t>(nv0) * EPV);
    const int nvt = PEEL ? nv0 + 2 : nv0 + (tail0 > 0 ? 1 : 0);  // slots per row (a few)
    const int64_t slots = B * nvt;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const char* xb = reinterpret_cast<const char*>(x);
    char* db = reinterpret_cast<char*>(dx);
    for (int64_t q0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q0 < slots;
         q0 += stride * kBwdU) {
        int64_t row[kBwdU];
        int k[kBwdU], head[kBwdU];
        float l[kBwdU], g[kBwdU];
        uint4 v[kBwdU];
#pragma unroll
        for (int j = 0; j < kBwdU; ++j) {
            const int64_t q = q0 + j * stride;
            row[j] = q < slots ? q / nvt : -1;
            k[j] = static_cast<int>(q - row[j] * nvt);
            head[j] = 0;
            if (row[j] >= 0) {
                l[j] = __ldg(lse + row[j]);
                g[j] = __ldg(grad + row[j]);
                const char* xr = xb + row[j] * row_stride * EB;
                if constexpr (VEC) {
                    if constexpr (PEEL) head[j] = static_cast<int>(head_elems_of<DT>(xr, N));
                    const int nv = PEEL ? static_cast<int>((N - head[j]) / EPV) : nv0;
                    if (k[j] < nv) v[j] = ldg_stream16(xr + head[j] * EB + k[j] * 16);
                } else {
                    v[j].x = __float_as_uint(load_elem<DT>(xr, k[j]));
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kBwdU; ++j) {
            if (row[j] < 0) continue;
            char* dr = db + row[j] * dx_row_stride * EB;
            if constexpr (VEC) {
                const char* xr = xb + row[j] * row_stride * EB;
                const int nv = PEEL ? static_cast<int>((N - head[j]) / EPV) : nv0;
                const int tail = PEEL ? static_cast<int>(N - head[j] - nv * EPV) : tail0;
                if (k[j] < nv)
                    __stcs(reinterpret_cast<uint4*>(dr + head[j] * EB + k[j] * 16),
                           grad_vector<DT>(v[j], l[j], g[j]));
                else if (k[j] == nv && tail > 0)  // the < EPV tail elements
                    grad_elems<DT>(xr, dr, head[j] + nv * EPV, tail, l[j], g[j]);
                else if (PEEL && k[j] == nv + (tail > 0 ? 1 : 0) && head[j] > 0)  // the head
                    grad_elems<DT>(xr, dr, 0, head[j], l[j], g[j]);
            } else {
                store_elem<DT>(dr, k[j], grad_term(__uint_as_float(v[j].x), l[j], g[j]));
            }
        }
    }
}

// One 16-byte vector whose elements [0, sp) belong to one row (l0, g0) and
// [sp, EPV) to the next (l1, g1).
template <int DT>
__device__ __forceinline__ uint4 grad_vector_split(uint4 u, int sp, float l0, float g0, float l1,
                                                   float g1) {
    if constexpr (DT == kF32) {
        const uint32_t in[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o[e] = __float_as_uint(grad_term(__uint_as_float(in[e]), e < sp ? l0 : l1,
                                             e < sp ? g0 : g1));
        return make_uint4(o[0], o[1], o[2], o[3]);
    } else {
        const uint32_t in[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = 2 * i;
            o[i] = pack2<DT>(grad_term(word_lo<DT>(in[i]), e < sp ? l0 : l1, e < sp ? g0 : g1),
                             grad_term(word_hi<DT>(in[i]), e + 1 < sp ? l0 : l1,
                                       e + 1 < sp ? g0 : g1));
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
}

constexpr int kFlatU = 4;  // vectors in flight per thread in the flat backward

// Back-to-back rows of x and dx (row stride N for both) at the same offset
// from a 16-byte boundary, N >= EPV: the [B, N] block is one flat array of
// B*N elements streamed as 16-byte vectors, whatever N is; the < EPV elements
// before the array's first boundary (all in row 0) and after its last one
// (all in row B - 1) are done element by element.  A vector holds elements of
// at most two rows.  One wave of CTAs strides through the vectors; each
// thread finds the row and in-row offset of its first vector with one
// division and then steps them by the stride incrementally.
// kFlatU vectors are in flight per thread, all loads before any store, so dx
// may be x.
template <int DT>
__global__ void __launch_bounds__(kBwdThreads, 4)
lse_backward_flat_kernel(const void* __restrict__ x, int64_t B, int64_t N,
                         const float* __restrict__ lse, const float* __restrict__ grad,
                         void* __restrict__ dx) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int EPV = 16 / EB;
    pdl_trigger();
    pdl_wait();
    const int64_t total = B * N;
    const int64_t head = head_elems_of<DT>(x, total);
    const int64_t nvec = (total - head) / EPV;
    const int tail = static_cast<int>(total - head - nvec * EPV);
    const char* xv = reinterpret_cast<const char*>(x) + head * EB;  // 16-byte aligned, as is dv
    char* dv = reinterpret_cast<char*>(dx) + head * EB;
    const int64_t T = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t == 0) {
        if (head > 0) grad_elems<DT>(reinterpret_cast<const char*>(x), reinterpret_cast<char*>(dx),
                                     0, static_cast<int>(head), __ldg(lse), __ldg(grad));
        if (tail > 0) grad_elems<DT>(reinterpret_cast<const char*>(x), reinterpret_cast<char*>(dx),
                                     total - tail, tail, __ldg(lse + B - 1), __ldg(grad + B - 1));
    }
    int64_t row = (head + t * EPV) / N;
    int64_t off = head + t * EPV - row * N;
    const int64_t qS = T * EPV / N;
    const int64_t rS = T * EPV - qS * N;  // a stride of T vectors: qS rows and rS elements
    for (int64_t v = t; v < nvec; v += kFlatU * T) {
        uint4 u[kFlatU];
        float l0[kFlatU], g0[kFlatU], l1[kFlatU], g1[kFlatU];
        int sp[kFlatU];
#pragma unroll
        for (int j = 0; j < kFlatU; ++j) {
            const int64_t vj = v + j * T;
            if (vj < nvec) {
                u[j] = ldg_stream16(xv + vj * 16);
                sp[j] = off + EPV > N ? static_cast<int>(N - off) : EPV;
                l0[j] = __ldg(lse + row);
                g0[j] = __ldg(grad + row);
                l1[j] = sp[j] < EPV ? __ldg(lse + row + 1) : l0[j];
                g1[j] = sp[j] < EPV ? __ldg(grad + row + 1) : g0[j];
            }
            row += qS;
            off += rS;
            if (off >= N) {
                off -= N;
                ++row;
            }
        }
#pragma unroll
        for (int j = 0; j < kFlatU; ++j) {
            const int64_t vj = v + j * T;
            if (vj < nvec)
                __stcs(reinterpret_cast<uint4*>(dv + vj * 16),
                       grad_vector_split<DT>(u[j], sp[j], l0[j], g0[j], l1[j], g1[j]));
        }
    }
}

template <int DT, bool VEC, bool PEEL>
cudaError_t launch_backward_dt(const BackwardArgs& a) {
    if (a.small)
        return launch_pdl(lse_backward_small_kernel<DT, VEC, PEEL>, a.grid, a.block, a.stream, a.x,
                          a.B, a.N, a.row_stride, a.lse, a.grad, a.dx, a.dx_row_stride);
    return launch_pdl(lse_backward_kernel<DT, VEC, PEEL>, a.grid, a.block, a.stream, a.x, a.B, a.N,
                      a.row_stride, a.lse, a.grad, a.dx, a.dx_row_stride, a.seg_slots);
}

template <int DT>
cudaError_t launch_backward_mode(int mode, const BackwardArgs& a) {
    switch (mode) {
    case kBwdFlat:
        return launch_pdl(lse_backward_flat_kernel<DT>, a.grid, a.block, a.stream, a.x, a.B, a.N,
                          a.lse, a.grad, a.dx);
    case kBwdVector: return launch_backward_dt<DT, true, false>(a);
    case kBwdPeel: return launch_backward_dt<DT, true, true>(a);
    default: return launch_backward_dt<DT, false, false>(a);
    }
}

}  // namespace

cudaError_t launch_backward(int dt, int mode, const BackwardArgs& a) {
    switch (dt) {
    case kF32: return launch_backward_mode<kF32>(mode, a);
    case kBF16: return launch_backward_mode<kBF16>(mode, a);
    default: return launch_backward_mode<kF16>(mode, a);
    }
}

cudaError_t launch_backward_strided(int dt, bool vec, const BackwardStridedArgs& a) {
    switch (dt) {
    case kF32:
        return vec ? launch_backward_strided_t<kF32, true>(a) : launch_backward_strided_t<kF32, false>(a);
    case kBF16:
        return vec ? launch_backward_strided_t<kBF16, true>(a)
                   : launch_backward_strided_t<kBF16, false>(a);
    default:
        return vec ? launch_backward_strided_t<kF16, true>(a) : launch_backward_strided_t<kF16, false>(a);
    }
}

int backward_strided_warps() { return kStrWarps; }
int backward_slots_per_thread() { return kBwdU; }
int backward_threads() { return kBwdThreads; }
int backward_flat_vectors_per_thread() { return kFlatU; }

}  // namespace lse
