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
// Mapping: a column tile is 32 lanes x EPV columns (EPV = elements per
// 16-byte vector, or 1 when the layout is not 16-byte aligned) of one index a,
// or 16 or 8 lanes when C is narrow;
// every load instruction of a warp covers one contiguous stretch of a row, and
// a thread folds U rows per batch into EPV accumulators with one rescale per
// batch.  WT = 1, 2, 4 or 8 warps share a tile, interleaving its rows and
// merging in shared memory (see lse_cols_kernel).  The (a, tile) pairs are
// flattened into units; a CTA's warps take consecutive units and CTAs stride
// over them.  With P > 1 the rows are also split across blockIdx.z; the
// (m, s) partials are stored split-major, [P, A * C], and
// merge_columns_kernel combines them with one thread per output.
#include <cstdint>

#include <cuda_runtime.h>

#include "lse_device.cuh"
#include "lse_internal.h"

namespace lse {
namespace {

// Warps per CTA for WT warps per tile: 4 (small CTAs balance better across
// SMs) unless the tile itself takes 8.  f32 variants keep 32 warps per SM
// resident (<= 64 registers per thread); 16-bit tiles hold 8 accumulators per
// lane and keep 28 (<= 73 registers; capping them at 64 measured 15 % slower
// on long reductions, 6 CTAs of one-warp tiles instead of 7 5-10 % slower on
// short ones).
// How far a column's maximum may rise above the shift its terms are taken
// against before the sum is rescaled: terms stay below e^8 (2^11.5).
constexpr float kLazyShift = 8.0f;

template <int WT> struct ColCta {
    static constexpr int warps = WT > 4 ? WT : 4;
    static constexpr int min_blocks(int elem_bytes) {
        return elem_bytes == 4 ? 1024 / (32 * warps) : 896 / (32 * warps);
    }
};

// WT warps share one column tile and interleave its rows (merged in shared
// memory); the CTA's warps cover warps / WT tiles.  WT = 1: each warp walks
// all rows of its own tile (short reductions, no merge); WT = 8: the whole CTA
// works on one tile (long reductions with few tiles).  LPT lanes make a tile:
// 32, or 16 or 8 when the wider tile would leave a quarter or more of its
// lanes without a column (narrow C); a warp then folds 32 / LPT tiles, one per
// group of LPT lanes, and WT warps share that group of tiles (each lane
// merges with the same lane of the group's other warps).
template <int DT, bool VEC, int WT, int LPT>
__global__ void __launch_bounds__(32 * ColCta<WT>::warps, ColCta<WT>::min_blocks(DType<DT>::bytes))
lse_cols_kernel(const void* __restrict__ x, int64_t A, int64_t R, int64_t C, int64_t stride_a,
                int64_t stride_r, int64_t rows_per_split, float* __restrict__ out,
                float2* __restrict__ partial, int64_t P) {
    static_assert(LPT == 32 || LPT == 16 || LPT == 8, "tiles of 32, 16 or 8 lanes");
    constexpr int EB = DType<DT>::bytes;
    constexpr int EPV = VEC ? 16 / EB : 1;
    constexpr int U = VEC ? 4 : 8;  // rows per batch per thread
    constexpr int NW = ColCta<WT>::warps;
    constexpr int UPW = 32 / LPT;         // tiles per warp
    constexpr int TPC = NW / WT * UPW;    // tiles per CTA
    __shared__ float2 part[WT > 1 ? NW : 1][32][EPV];

    pdl_trigger();
    pdl_wait();

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int phase = wid % WT;  // row interleave position within the tile's warps
    const int64_t split = blockIdx.z;
    const int64_t r_begin = split * rows_per_split;
    const int64_t r_end = r_begin + rows_per_split < R ? r_begin + rows_per_split : R;
    const char* xb = reinterpret_cast<const char*>(x);
    // Work units are (a, tile) pairs in a-major order; a CTA's TPC tile slots
    // take consecutive units (several a when C is narrow), and CTAs stride
    // over the units (the loop bound is the same for every warp of the CTA).
    const int64_t wtiles = (C + LPT * EPV - 1) / (LPT * EPV);
    const int64_t units = A * wtiles;
    const bool small = units <= 0xffffffffll;  // unit indices divide in 32 bits
    // 16-byte output stores: out on a 16-byte boundary (C % EPV == 0 and
    // c0 % EPV == 0 keep every lane's EPV outputs on one).
    const bool out_vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;

    constexpr int64_t kStep = static_cast<int64_t>(WT) * U;  // rows per batch of one warp
#pragma unroll 1
    for (int64_t u0 = static_cast<int64_t>(blockIdx.x) * TPC; u0 < units;
         u0 += static_cast<int64_t>(gridDim.x) * TPC) {
        const int64_t unit = u0 + (wid / WT) * UPW + (UPW > 1 ? lane / LPT : 0);
        // (past the last unit: the last a, whose rows the neighbouring units read)
        const int64_t a = unit >= units ? A - 1
                          : small ? static_cast<int64_t>(static_cast<uint32_t>(unit) / static_cast<uint32_t>(wtiles))
                                  : unit / wtiles;
        const int64_t tile = unit - a * wtiles;
        const int64_t c0 = (tile * LPT + (lane & (LPT - 1))) * EPV;
        const bool active = unit < units && c0 < C;  // VEC: whole vectors only (C % EPV == 0)
        const char* base = xb + (a * stride_a + (active ? c0 : 0)) * EB;
        Acc acc[EPV];
        float mu[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            acc[e] = acc_identity();
            mu[e] = 0.0f;
        }
        // VEC, 16-bit: acc[e].s is taken against the lazy shift mu[e], which
        // moves when a batch maximum exceeds thr[e]: -inf until column e has
        // met a value above -inf, then mu[e] + kLazyShift (acc[e].m is set
        // from mu and thr once the rows are done).
        float thr[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) thr[e] = __int_as_float(kNegInfF32);
        // PIPE: the next batch's loads are issued before the current batch is
        // folded, so two batches per warp are in flight.  For one warp per
        // tile (short reductions, which otherwise wait a full memory round
        // trip per batch; +5 % on bf16 [512, 64, 1024]).
        constexpr bool PIPE = VEC && WT == 1;
        const int64_t srb = stride_r * EB;  // bytes from one row to the next
        // A batch of U rows r0 + j * WT.  When all of them are in range (every
        // batch but a split's last, uniform per warp) the loads go without a
        // per-row test or -inf defaults; lanes without a column read the
        // column-0 rows of their a (in bounds, never stored).
        auto load_batch = [&](int64_t r0, const char* q, uint4 (&u)[U]) {
            if (r0 + (U - 1) * WT < r_end) {
#pragma unroll
                for (int j = 0; j < U; ++j) u[j] = ldg_stream16(q + j * WT * srb);
            } else {
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    u[j] = make_uint4(neg_inf_word<DT>(), neg_inf_word<DT>(), neg_inf_word<DT>(),
                                      neg_inf_word<DT>());
                    if (r0 + j * WT < r_end) u[j] = ldg_stream16(q + j * WT * srb);
                }
            }
        };
        auto fold = [&](const uint4 (&cur)[U]) {
            if constexpr (EB == 4) {
                // f32: four columns per lane; the eager rescale measured
                // faster here than the lazy one below (5.8 vs 5.5 TB/s on
                // [512, 64, 1024]).
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    float v[U];
#pragma unroll
                    for (int j = 0; j < U; ++j) v[j] = __uint_as_float(e == 0 ? cur[j].x : e == 1 ? cur[j].y
                                                                       : e == 2 ? cur[j].z : cur[j].w);
                    float cm = v[0];
#pragma unroll
                    for (int j = 1; j < U; ++j) cm = fmaxf(cm, v[j]);
                    acc_raise(acc[e], mu[e], cm);
                    float sum = 0.0f;
#pragma unroll
                    for (int j = 0; j < U; ++j) sum += ex2((v[j] - mu[e]) * kLog2e);
                    acc[e].s += sum;
                }
            } else {
                uint32_t w[U][4];
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    w[j][0] = cur[j].x; w[j][1] = cur[j].y; w[j][2] = cur[j].z; w[j][3] = cur[j].w;
                }
                // Column maxima of the batch, packed over the rows (NaN
                // lanes ignored, as fmaxf does), kept as 4 words.
                uint32_t cmw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t t = w[0][i];
#pragma unroll
                    for (int j = 1; j < U; ++j)
                        t = DT == kBF16 ? hmax2_bf16(t, w[j][i]) : hmax2_f16(t, w[j][i]);
                    cmw[i] = t;
                }
                auto cm = [&](int e) { return word_elem<DT>(cmw, e); };
                // Lazy shifts: a column's terms are taken relative to a shift
                // mu that only moves when the batch maximum exceeds it by more
                // than kLazyShift (or is the column's first value above -inf),
                // so terms stay below e^kLazyShift and most batches skip the
                // rescale; the warp branches over it uniformly.  The rescale
                // exponent is clamped to [-126, 0]: a sum that is already
                // +inf (the column met +inf) stays +inf instead of meeting a
                // factor flushed to 0, the first move scales the empty sum 0
                // by at most 1, and an older sum cut to 2^-126 of itself
                // instead of 0 is below any term that can follow (>= 1 for
                // the new maximum; the older sum holds < R e^8).
                bool any = false;
#pragma unroll
                for (int e = 0; e < EPV; ++e) any = any || cm(e) > thr[e];
                if (__any_sync(0xffffffffu, any)) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        if (cm(e) > thr[e]) {
                            const float mn = shift_of(cm(e));
                            acc[e].s *= ex2(fminf(fmaxf((mu[e] - mn) * kLog2e, -126.0f), 0.0f));
                            mu[e] = mn;
                            thr[e] = mn + kLazyShift;
                        }
                    }
                }
                // Columns 2i and 2i + 1 (the halves of word i) as packed pairs
                // (sub/mul/add .f32x2); each column's terms still summed in
                // row order.  +1-5 % on bf16 reductions of 64-4096 rows; the
                // f32 tiles above keep scalar sums (no gain there).
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t mu2 = f2_pack(mu[2 * i], mu[2 * i + 1]);
                    uint64_t sum2 = 0ull;
#pragma unroll
                    for (int j = 0; j < U; ++j) {
                        const uint64_t x2 = f2_pack(word_lo<DT>(w[j][i]), word_hi<DT>(w[j][i]));
                        sum2 = f2_add(sum2, f2_ex2(f2_mul(f2_sub(x2, mu2), f2_pack(kLog2e, kLog2e))));
                    }
                    float s0, s1;
                    f2_unpack(sum2, s0, s1);
                    acc[2 * i].s += s0;
                    acc[2 * i + 1].s += s1;
                }
            }
        };
        if constexpr (VEC) {
            const char* q = base + (r_begin + phase) * srb;
            const int64_t qstep = kStep * srb;
            int64_t r = r_begin + phase;
            if constexpr (PIPE) {
                // Two batches in flight, in two buffers used in turn (no copy
                // from the prefetched batch to the folded one).
                uint4 b0[U], b1[U];
                if (r < r_end) load_batch(r, q, b0);
                while (r < r_end) {
                    if (r + kStep < r_end) load_batch(r + kStep, q + qstep, b1);
                    fold(b0);
                    r += kStep;
                    q += qstep;
                    if (r >= r_end) break;
                    if (r + kStep < r_end) load_batch(r + kStep, q + qstep, b0);
                    fold(b1);
                    r += kStep;
                    q += qstep;
                }
            } else {
                for (; r < r_end; r += kStep, q += qstep) {
                    uint4 cur[U];
                    load_batch(r, q, cur);
                    fold(cur);
                }
            }
        } else {
            for (int64_t r = r_begin + phase; r < r_end; r += kStep) {
                float v[U];
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const int64_t rr = r + j * WT;
                    v[j] = active && rr < r_end ? load_elem<DT>(base, rr * stride_r)
                                                : __int_as_float(kNegInfF32);
                }
                float cm = v[0];
#pragma unroll
                for (int j = 1; j < U; ++j) cm = fmaxf(cm, v[j]);
                acc_raise(acc[0], mu[0], cm);
                float sum = 0.0f;
#pragma unroll
                for (int j = 0; j < U; ++j) sum += ex2((v[j] - mu[0]) * kLog2e);
                acc[0].s += sum;
            }
        }
        if constexpr (VEC && EB == 2) {
            // (shift, sum) as an accumulator: the shift stands in for the
            // maximum (it is within kLazyShift below it, and the merge and
            // the finalize only use m as a shift); -inf for a column of -inf,
            // +inf for a column holding +inf (its sum is +inf: the terms, at
            // most e^kLazyShift each, cannot overflow it otherwise), so that
            // merging it with other partials keeps +inf.
#pragma unroll
            for (int e = 0; e < EPV; ++e)
                acc[e].m = thr[e] == __int_as_float(kNegInfF32)      ? __int_as_float(kNegInfF32)
                           : acc[e].s == __int_as_float(0x7f800000) ? __int_as_float(0x7f800000)
                                                                     : mu[e];
        }
        if constexpr (WT > 1) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) part[wid][lane][e] = make_float2(acc[e].m, acc[e].s);
            __syncthreads();
            if (phase == 0 && active) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    Acc t = acc_identity();
#pragma unroll
                    for (int w = 0; w < WT; ++w)
                        t = acc_merge(t, Acc{part[wid + w][lane][e].x, part[wid + w][lane][e].y});
                    acc[e] = t;
                }
            }
            __syncthreads();  // part[] is reused by the next a
        }
        if (phase == 0 && active) {
            if constexpr (VEC) {
                // EPV consecutive outputs (C % EPV == 0, so all in range): 16-byte
                // stores where the destination allows (the scratch always does).
                if (P == 1) {
                    float* o = out + a * C + c0;
                    float r[EPV];
#pragma unroll
                    for (int e = 0; e < EPV; ++e) r[e] = acc_finalize(acc[e]);
                    if (out_vec) {
#pragma unroll
                        for (int e = 0; e < EPV; e += 4)
                            *reinterpret_cast<float4*>(o + e) = make_float4(r[e], r[e + 1], r[e + 2], r[e + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < EPV; ++e) o[e] = r[e];
                    }
                } else {  // split-major: coalesced here and in merge_columns_kernel
                    float2* o = partial + split * (A * C) + a * C + c0;
#pragma unroll
                    for (int e = 0; e < EPV; e += 2)
                        *reinterpret_cast<float4*>(o + e) = make_float4(acc[e].m, acc[e].s, acc[e + 1].m, acc[e + 1].s);
                }
            } else {
                if (P == 1)
                    out[a * C + c0] = acc_finalize(acc[0]);
                else
                    partial[split * (A * C) + a * C + c0] = make_float2(acc[0].m, acc[0].s);
            }
        }
    }
}

// One thread per output (a, c): merges its P partials in split order.
__global__ void __launch_bounds__(256)
merge_columns_kernel(const float2* __restrict__ partial, int64_t outputs, int64_t P,
                     float* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < outputs;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        Acc t = acc_identity();
        for (int64_t p = 0; p < P; ++p) {
            const float2 v = partial[p * outputs + i];
            t = acc_merge(t, Acc{v.x, v.y});
        }
        out[i] = acc_finalize(t);
    }
}

// Short reductions (R = RR <= 8 rows, the 16-byte vector layout): one thread
// per 16-byte vector of EPV columns of one a loads all RR rows at once, takes
// each column's maximum and then its exp-sum against it (two passes over
// registers, no online state, no rescale), and stores its EPV values, with
// 16-byte stores where out allows.  Threads stride over the A * C / EPV
// vectors in a-major order, so a warp's loads cover consecutive vectors of
// one row.
template <int DT, int RR>
__global__ void __launch_bounds__(kColsShortThreads)
lse_cols_short_kernel(const void* __restrict__ x, int64_t A, int64_t C, int64_t stride_a,
                      int64_t stride_r, float* __restrict__ out) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int EPV = 16 / EB;
    pdl_trigger();
    pdl_wait();
    const int64_t cv = C / EPV;  // vectors per row (C % EPV == 0)
    const int64_t nvec = A * cv;
    const bool small = nvec <= 0xffffffffll;  // indices divide in 32 bits
    const bool out_vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    const int64_t srb = stride_r * EB;
    const char* xb = reinterpret_cast<const char*>(x);
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < nvec;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t a = small ? static_cast<int64_t>(static_cast<uint32_t>(t) / static_cast<uint32_t>(cv))
                                : t / cv;
        const int64_t c0 = (t - a * cv) * EPV;
        const char* p = xb + (a * stride_a + c0) * EB;
        uint32_t w[RR][4];
#pragma unroll
        for (int r = 0; r < RR; ++r) {
            const uint4 u = ldg_stream16(p + r * srb);
            w[r][0] = u.x; w[r][1] = u.y; w[r][2] = u.z; w[r][3] = u.w;
        }
        // Column maxima (NaN ignored, as fmaxf does), as 4 words: f32 one
        // column per word, 16-bit two.
        uint32_t cmw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t t4 = w[0][i];
#pragma unroll
            for (int r = 1; r < RR; ++r) {
                if constexpr (DT == kF32) t4 = __float_as_uint(fmaxf(__uint_as_float(t4), __uint_as_float(w[r][i])));
                else t4 = DT == kBF16 ? hmax2_bf16(t4, w[r][i]) : hmax2_f16(t4, w[r][i]);
            }
            cmw[i] = t4;
        }
        float res[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const float m = word_elem<DT>(cmw, e);
            const float mu = shift_of(m);
            float sum = 0.0f;
#pragma unroll
            for (int r = 0; r < RR; ++r) sum += ex2((word_elem<DT>(w[r], e) - mu) * kLog2e);
            res[e] = acc_finalize(Acc{m, sum});
        }
        float* o = out + a * C + c0;
        if (out_vec) {
#pragma unroll
            for (int e = 0; e < EPV; e += 4)
                *reinterpret_cast<float4*>(o + e) = make_float4(res[e], res[e + 1], res[e + 2], res[e + 3]);
        } else {
#pragma unroll
            for (int e = 0; e < EPV; ++e) o[e] = res[e];
        }
    }
}

template <int DT>
cudaError_t launch_cols_short_t(const StridedArgs& a) {
#define LSE_COLS_SHORT(RR)                                                                          \
    return launch_pdl(lse_cols_short_kernel<DT, RR>, a.grid, dim3(kColsShortThreads), a.stream, a.x, \
                      a.A, a.C, a.stride_a, a.stride_r, a.out)
    switch (a.R) {
    case 1: LSE_COLS_SHORT(1);
    case 2: LSE_COLS_SHORT(2);
    case 3: LSE_COLS_SHORT(3);
    case 4: LSE_COLS_SHORT(4);
    case 5: LSE_COLS_SHORT(5);
    case 6: LSE_COLS_SHORT(6);
    case 7: LSE_COLS_SHORT(7);
    case 8: LSE_COLS_SHORT(8);
    default: return cudaErrorInvalidValue;
    }
#undef LSE_COLS_SHORT
}

template <int DT, bool VEC>
cudaError_t launch_cols_t(const StridedArgs& a) {
#define LSE_COLS_LAUNCH_L(WT, LPT)                                                                       \
    return launch_pdl(lse_cols_kernel<DT, VEC, WT, LPT>, a.grid, dim3(32 * ColCta<WT>::warps), a.stream, \
                      a.x, a.A, a.R, a.C, a.stride_a, a.stride_r, a.rows_per_split, a.out,               \
                      a.partial, a.P)
#define LSE_COLS_LAUNCH(WT) LSE_COLS_LAUNCH_L(WT, 32)
#define LSE_COLS_LAUNCH_W(WT)                                     \
    switch (cols_lanes_per_tile(DT, VEC, a.C, 1)) {               \
    case 8: LSE_COLS_LAUNCH_L(WT, 8);                             \
    case 16: LSE_COLS_LAUNCH_L(WT, 16);                           \
    default: LSE_COLS_LAUNCH(WT);                                 \
    }
    switch (a.warps_per_tile) {
    case 1: LSE_COLS_LAUNCH_W(1);
    case 2: LSE_COLS_LAUNCH_W(2);
    case 4: LSE_COLS_LAUNCH_W(4);
    case 8: LSE_COLS_LAUNCH_W(8);
    default: return cudaErrorInvalidValue;
    }
#undef LSE_COLS_LAUNCH_W
#undef LSE_COLS_LAUNCH
#undef LSE_COLS_LAUNCH_L
}

template <int DT, bool VEC, int WT>
int cols_occupancy_w() {
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, lse_cols_kernel<DT, VEC, WT, 32>,
                                                      32 * ColCta<WT>::warps, 0) != cudaSuccess)
        return 1;
    return blocks > 0 ? blocks : 1;
}

template <int DT, bool VEC>
int cols_occupancy_t(int wt) {
    switch (wt) {
    case 1: return cols_occupancy_w<DT, VEC, 1>();
    case 2: return cols_occupancy_w<DT, VEC, 2>();
    case 4: return cols_occupancy_w<DT, VEC, 4>();
    default: return cols_occupancy_w<DT, VEC, 8>();
    }
}

}  // namespace

cudaError_t launch_cols(int dt, bool vec, const StridedArgs& a) {
    switch (dt) {
    case kF32: return vec ? launch_cols_t<kF32, true>(a) : launch_cols_t<kF32, false>(a);
    case kBF16: return vec ? launch_cols_t<kBF16, true>(a) : launch_cols_t<kBF16, false>(a);
    default: return vec ? launch_cols_t<kF16, true>(a) : launch_cols_t<kF16, false>(a);
    }
}

int cols_occupancy(int dt, bool vec, int wt) {
    switch (dt) {
    case kF32: return vec ? cols_occupancy_t<kF32, true>(wt) : cols_occupancy_t<kF32, false>(wt);
    case kBF16: return vec ? cols_occupancy_t<kBF16, true>(wt) : cols_occupancy_t<kBF16, false>(wt);
    default: return vec ? cols_occupancy_t<kF16, true>(wt) : cols_occupancy_t<kF16, false>(wt);
    }
}

cudaError_t launch_cols_short(int dt, const StridedArgs& a) {
    switch (dt) {
    case kF32: return launch_cols_short_t<kF32>(a);
    case kBF16: return launch_cols_short_t<kBF16>(a);
    default: return launch_cols_short_t<kF16>(a);
    }
}

cudaError_t launch_merge_columns(const float2* partial, int64_t outputs, int64_t P, float* out,
                                 cudaStream_t stream) {
    int64_t grid = (outputs + 255) / 256;
    if (grid > 1048576) grid = 1048576;
    return launch_pdl(merge_columns_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), stream,
                      partial, outputs, P, out);
}

int cols_columns_per_warp(bool vec, int dt) { return 32 * (vec ? 16 / (dt == kF32 ? 4 : 2) : 1); }
int cols_lanes_per_tile(int dt, bool vec, int64_t C, int warps_per_tile) {
    // One-warp tiles narrow to 16 or 8 lanes while the wider tile would leave
    // a quarter or more of its lanes without a column: the widest tile that
    // keeps more than three quarters of them busy, else 8 lanes.
    if (warps_per_tile != 1) return 32;
    for (int lanes = 32; lanes > 8; lanes /= 2) {
        const int64_t w = cols_columns_per_warp(vec, dt) * lanes / 32;
        const int64_t padded = (C + w - 1) / w * w;
        if (4 * C > 3 * padded) return lanes;
    }
    return 8;
}
int cols_rows_per_batch(bool vec) { return vec ? 4 : 8; }
int cols_warps_per_cta(int wt) { return wt > 4 ? wt : 4; }

}  // namespace lse
