// lse_kernels.cuh -- the row-wise log-sum-exp kernels over strided rows (sm_103a).
//
// One pass over x: every element is loaded once with coalesced 128-bit loads
// (scalar loads when rows are not 16-byte aligned), folded into a register
// accumulator, and each row writes one float ("Speeding up Log-Sum-Exp ...",
// Sec. 3.1).  Two mappings live here:
//   subwarp  rows of at most 32*4 vectors: G lanes per row hold the whole row
//            in registers; max first, then the exp-sum (two passes over
//            registers, one over HBM); lanes combine by xor shuffles.
//   segment  one CTA per (row, segment): online (m, s) accumulation over
//            batches of 8 vectors per thread, then warp shuffles and shared
//            memory.  With one segment per row it writes out[row]; with P > 1
//            segments it writes an (m, s) partial that merge_kernel
//            (lse_api.cu) combines -- the split-row mapping for long or few rows.
// Both take an optional fused epilogue (TL) for the token log-probability, and
// E16 selects the reduced-bit exponentials of lse_device.cuh (two terms per
// packed bf16 SFU operation) in place of the f32 ones.
// Back-to-back short rows have a bulk-copy mapping of their own
// (lse_rowtile.cu).  This header is included by one translation unit per
// element type and epilogue.
#pragma once

#include "lse_device.cuh"
#include "lse_edges.cuh"
#include "lse_internal.h"

namespace lse {

// ---------------------------------------------------------------------------
// subwarp: G lanes per row, V slots per lane, R row-groups per warp iteration.
// VEC: a slot is one 16-byte vector of the aligned span covering the row; a
// row that does not start or end on a 16-byte boundary takes one or two more
// slots than its full vectors, whose outside elements are masked.  !VEC: a
// slot is one element.
// V = 8 (a whole warp per row of up to 256 slots, or 4-16 lanes per row of
// vectors: twice the rows in flight of V = 4 with half the lanes) keeps 32
// words per lane and runs at 4 CTAs per SM; a whole warp per row also takes
// V = 5 or 7, so a row of 129-256 slots pads to the next multiple of 32.
// ---------------------------------------------------------------------------
// The token log-probability epilogue keeps the targets and the peel state of
// every row group live: one CTA per SM less, so it does not spill.
template <int V, bool TL> struct SubwarpOccupancy {
    static constexpr int min_blocks = (V >= 5 ? 4 : kSubwarpMinBlocks) - (TL ? 1 : 0);
};

template <int DT, int G, int V, bool VEC, bool TL, bool E16>
__global__ void __launch_bounds__(kSubwarpThreads, SubwarpOccupancy<V, TL>::min_blocks)
lse_subwarp_kernel(const void* __restrict__ x, int64_t B, int64_t N, int64_t row_stride,
                   float* __restrict__ out, const int64_t* __restrict__ target,
                   float* __restrict__ logprob) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int RPW = 32 / G;             // rows per warp per row-group
    constexpr int R = V >= 3 ? 1 : (V == 2 ? 2 : 4);
    const int lane = threadIdx.x & 31;
    const int sub = lane & (G - 1);
    const int grp = lane / G;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const char* xb = reinterpret_cast<const char*>(x);
    pdl_trigger();
    pdl_wait();

    for (int64_t row0 = warp * (RPW * R); row0 < B; row0 += nwarps * (RPW * R)) {
        // Targets, loaded with the rows (token log-probability only); rows on
        // this path hold at most 32 * 8 * 8 elements, so an in-range target
        // fits in 32 bits and -1 marks an invalid one.
        int t[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = row0 + r * RPW + grp;
            const int64_t tt = (TL && row < B) ? __ldg(target + row) : -1;
            t[r] = (tt >= 0 && tt < N) ? static_cast<int>(tt) : -1;
        }
        if constexpr (VEC) {
            // Slot k of a row is the k-th 16-byte vector of the aligned span
            // covering the row, [rp - off, rp + N * EB) rounded out to 16
            // bytes: the first and the last vectors may hold bytes of the
            // neighbouring rows or of padding, masked to -inf.  A 16-byte block
            // holding a byte of the row lies in the row's memory page, so the
            // wider read cannot fault.
            uint32_t w[R][4 * V];
            uint32_t off[R];  // byte offset of each row from the 16-byte boundary below it
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r * RPW + grp;
                const char* rp = xb + (row < B ? row : 0) * row_stride * EB;
                off[r] = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(rp) & 15u);
                const char* a0 = rp - off[r];  // 16-byte aligned
                const uint32_t rb1 = off[r] + static_cast<uint32_t>(N) * EB;  // row end in the span
                const int nvc = static_cast<int>((rb1 + 15u) >> 4);           // vectors in the span
#pragma unroll
                for (int j = 0; j < V; ++j) {  // every load issued before any mask
                    const int k = sub + j * G;
                    uint4 u = make_uint4(neg_inf_word<DT>(), neg_inf_word<DT>(), neg_inf_word<DT>(),
                                         neg_inf_word<DT>());
                    if (row < B && k < nvc) u = ldg_stream16(a0 + k * 16);
                    w[r][4 * j] = u.x; w[r][4 * j + 1] = u.y; w[r][4 * j + 2] = u.z; w[r][4 * j + 3] = u.w;
                }
                if (off[r] != 0 || (rb1 & 15u) != 0) {
#pragma unroll
                    for (int j = 0; j < V; ++j) {
                        const int k = sub + j * G;
                        if (k == 0 || k == nvc - 1) {
                            uint32_t q[4] = {w[r][4 * j], w[r][4 * j + 1], w[r][4 * j + 2], w[r][4 * j + 3]};
                            if (k == 0) mask_prefix<DT>(q, static_cast<int>(off[r]));
                            if (k == nvc - 1) mask_suffix<DT>(q, static_cast<int>(rb1) - 16 * k);
#pragma unroll
                            for (int i = 0; i < 4; ++i) w[r][4 * j + i] = q[i];
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r * RPW + grp;
                float m = words_max<DT, 4 * V>(w[r]);
#pragma unroll
                for (int off = G / 2; off > 0; off >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                const float mu = shift_of(m);
                // FFMA form for the 4- and 8-slot variants (every row longer than
                // two vectors); same decision for the whole group.  Not with E16:
                // there the maximum's own argument must be exactly 0 (its bf16
                // term exactly 1), not the rounding residual of mu log2 e.
                const bool scaled = !E16 && V >= 3 && ffma_shift_ok(mu);
                const float c = mu * kLog2e;
                float s = scaled ? words_expsum_scaled<DT, 4 * V>(w[r], c)
                                 : expsum_words<DT, 4 * V, E16>(w[r], mu);
#pragma unroll
                for (int off = G / 2; off > 0; off >>= 1)
                    s += __shfl_xor_sync(0xffffffffu, s, off);
                // x[row, t] is already in the group's registers: the lane holding
                // it contributes it, the others 0, and a shuffle-sum combines.
                float xt = 0.0f;
                if constexpr (TL) {
                    const bool valid = t[r] >= 0;
                    if (valid) {
                        // slot and position of x[row, t] in the covering span
                        const int tb = static_cast<int>(off[r]) + t[r] * EB;
                        const int slot = tb >> 4;
                        const int pos = (tb & 15) / EB;
#pragma unroll
                        for (int j = 0; j < V; ++j)
                            if (sub + j * G == slot) xt = word_elem<DT>(&w[r][4 * j], pos);
                    }
#pragma unroll
                    for (int off = G / 2; off > 0; off >>= 1)
                        xt += __shfl_xor_sync(0xffffffffu, xt, off);
                    if (!valid) xt = __int_as_float(0x7fc00000);
                }
                if (sub == 0 && row < B) {
                    const float lse = scaled ? finalize_scaled(m, s, mu, c) : acc_finalize(Acc{m, s});
                    store_row(out, TL ? logprob : nullptr, row, lse, xt);
                }
            }
        } else {
            float v[R][V];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r * RPW + grp;
                const char* rp = xb + row * row_stride * EB;
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const int64_t k = sub + j * G;
                    v[r][j] = (row < B && k < N) ? load_elem<DT>(rp, k)
                                                 : __int_as_float(kNegInfF32);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r * RPW + grp;
                float m = v[r][0];
#pragma unroll
                for (int j = 1; j < V; ++j) m = fmaxf(m, v[r][j]);
#pragma unroll
                for (int off = G / 2; off > 0; off >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                const float mu = shift_of(m);
                float s = 0.0f;
                if constexpr (E16) {
#pragma unroll
                    for (int j = 0; j < V; j += 2) {
                        const float hi = j + 1 < V ? e16_arg(v[r][j + 1], mu)
                                                   : __int_as_float(kNegInfF32);
                        s = add_bf16_pair(s, ex2_bf16_pair(e16_arg(v[r][j], mu), hi));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < V; ++j) s += ex2((v[r][j] - mu) * kLog2e);
                }
#pragma unroll
                for (int off = G / 2; off > 0; off >>= 1)
                    s += __shfl_xor_sync(0xffffffffu, s, off);
                float xt = 0.0f;
                if constexpr (TL) {
                    const bool valid = t[r] >= 0;
#pragma unroll
                    for (int j = 0; j < V; ++j)
                        if (valid && sub + j * G == t[r]) xt = v[r][j];
#pragma unroll
                    for (int off = G / 2; off > 0; off >>= 1)
                        xt += __shfl_xor_sync(0xffffffffu, xt, off);
                    if (!valid) xt = __int_as_float(0x7fc00000);
                }
                if (sub == 0 && row < B) store_row(out, TL ? logprob : nullptr, row, acc_finalize(Acc{m, s}), xt);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// segment: blockIdx.x = row * P + seg.  VEC: the row's slots are the 16-byte
// vectors of the aligned span covering it (as in subwarp: the first and the
// last may be partly outside the row and are masked by the one thread that
// loads each).  Segment seg covers slots [seg * seg_slots, (seg + 1) *
// seg_slots); the last segment runs to the row's last slot.  !VEC: slots are
// elements.
// ---------------------------------------------------------------------------
// A 32-thread plan runs 8 units per CTA, one per warp (single-warp CTAs are
// launched too slowly to keep up with 4 KB rows); wider plans one unit per CTA.
template <int T> struct SegmentOccupancy {
    static constexpr int cta_threads = T == 32 ? 32 * kSegmentWarpUnitsPerCta : T;
    static constexpr int units_per_cta = cta_threads / T;
    static constexpr int min_blocks = 2048 / cta_threads / 2;
};

template <int DT, int T, bool VEC, bool TL, bool E16>
__global__ void __launch_bounds__(SegmentOccupancy<T>::cta_threads, SegmentOccupancy<T>::min_blocks)
lse_segment_kernel(const void* __restrict__ x, int64_t B, int64_t N, int64_t row_stride, int64_t P,
                   int64_t seg_slots, float* __restrict__ out, float2* __restrict__ partial,
                   const int64_t* __restrict__ target, float* __restrict__ logprob,
                   float* __restrict__ xt_buf) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int U = VEC ? 8 : 16;  // slots per thread per batch
    constexpr int NW = T / 32;
    constexpr int UPC = SegmentOccupancy<T>::units_per_cta;

    pdl_trigger();
    pdl_wait();

    const int tid = UPC > 1 ? static_cast<int>(threadIdx.x & (T - 1)) : static_cast<int>(threadIdx.x);
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * UPC + (UPC > 1 ? threadIdx.x / T : 0);
    if (UPC > 1 && unit >= B * P) return;  // uniform per warp; no CTA-wide barrier follows
    const int64_t row = unit / P;
    const int64_t seg = unit - row * P;
    const char* rp = reinterpret_cast<const char*>(x) + row * row_stride * EB;
    // VEC: the span [rp - off, rp + N * EB) rounded up to 16 bytes.
    const uint32_t off = VEC ? static_cast<uint32_t>(reinterpret_cast<uintptr_t>(rp) & 15u) : 0u;
    const char* a0 = rp - off;
    const int64_t rb1 = off + N * EB;                      // row end in the span, bytes
    const int64_t nslots = VEC ? (rb1 + 15) >> 4 : N;      // slots of the row
    const int64_t s_begin = seg * seg_slots;
    const int64_t s_end = seg == P - 1 || s_begin + seg_slots > nslots ? nslots : s_begin + seg_slots;
    // The threads that load the row's first or last vector when it is partly
    // outside the row.
    const bool edge = VEC && ((off != 0 && seg == 0 && tid == 0) ||
                              ((rb1 & 15) != 0 && s_end == nslots &&
                               (nslots - 1 - s_begin) % T == tid));
    auto mask_edge = [&](uint32_t* w4, int64_t kk) {
        if (kk == 0 || kk == nslots - 1) {
            uint32_t q[4] = {w4[0], w4[1], w4[2], w4[3]};
            if (kk == 0) mask_prefix<DT>(q, static_cast<int>(off));
            if (kk == nslots - 1) mask_suffix<DT>(q, static_cast<int>(rb1 - kk * 16));
#pragma unroll
            for (int i = 0; i < 4; ++i) w4[i] = q[i];
        }
    };

    Acc acc = acc_identity();
    float mu = 0.0f;
    int64_t k = s_begin + tid;

    // Token log-probability: thread 0 of the row's first segment gathers
    // x[row, target[row]] once, issued behind its first batch of loads.
    const bool gather = TL && seg == 0 && tid == 0;
    const int64_t t = gather ? __ldg(target + row) : -1;
    bool xt_pending = gather;
    float xt = __int_as_float(0x7fc00000);

    if constexpr (VEC) {
        for (; k + (U - 1) * T < s_end; k += U * T) {
            uint32_t w[4 * U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const uint4 u = ldg_stream16(a0 + (k + j * T) * 16);
                w[4 * j] = u.x; w[4 * j + 1] = u.y; w[4 * j + 2] = u.z; w[4 * j + 3] = u.w;
            }
            if (edge) {
#pragma unroll
                for (int j = 0; j < U; ++j) mask_edge(&w[4 * j], k + j * T);
            }
            if (xt_pending) {
                if (t >= 0 && t < N) xt = load_elem<DT>(rp, t);
                xt_pending = false;
            }
            acc_add_words<DT, 4 * U, E16>(acc, mu, w);
        }
        if (k < s_end) {
            // One-warp units take the last, partial batch with 1, 2, 4 or U
            // slots per thread, as few as cover what is left of the segment,
            // so a row just past a whole batch does not pay a full batch of
            // arithmetic on -inf.
            auto partial_batch = [&](auto n) {
                constexpr int UU = decltype(n)::value;
                uint32_t w[4 * UU];
#pragma unroll
                for (int j = 0; j < UU; ++j) {
                    const int64_t kk = k + j * T;
                    if (kk < s_end) {
                        const uint4 u = ldg_stream16(a0 + kk * 16);
                        w[4 * j] = u.x; w[4 * j + 1] = u.y; w[4 * j + 2] = u.z; w[4 * j + 3] = u.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) w[4 * j + i] = neg_inf_word<DT>();
                    }
                }
                if (edge) {  // after every load is issued
#pragma unroll
                    for (int j = 0; j < UU; ++j)
                        if (k + j * T < s_end) mask_edge(&w[4 * j], k + j * T);
                }
                acc_add_words<DT, 4 * UU, E16>(acc, mu, w);
            };
            const int64_t left = s_end - (k - tid);  // slots from this batch's first on
            if constexpr (T == 32) {  // short segments, where the last batch is much of the work
                if (left <= T) partial_batch(IntConst<1>{});
                else if (left <= 2 * T) partial_batch(IntConst<2>{});
                else if (left <= 4 * T) partial_batch(IntConst<4>{});
                else partial_batch(IntConst<U>{});
            } else {  // (wider CTAs: one more variant would spill at their 64 registers)
                partial_batch(IntConst<U>{});
            }
        }
    } else {
        for (; k + (U - 1) * T < s_end; k += U * T) {
            float v[U];
#pragma unroll
            for (int j = 0; j < U; ++j) v[j] = load_elem<DT>(rp, k + j * T);
            acc_add_floats<U, E16>(acc, mu, v);
        }
        if (k < s_end) {
            float v[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t kk = k + j * T;
                v[j] = kk < s_end ? load_elem<DT>(rp, kk) : __int_as_float(kNegInfF32);
            }
            acc_add_floats<U, E16>(acc, mu, v);
        }
    }

    if (xt_pending && t >= 0 && t < N) xt = load_elem<DT>(rp, t);

    acc = warp_merge<32>(acc);
    if constexpr (NW > 1) {
        __shared__ float2 part[NW];
        const int wid = threadIdx.x >> 5;
        const int lane = threadIdx.x & 31;
        if (lane == 0) part[wid] = make_float2(acc.m, acc.s);
        __syncthreads();
        if (wid == 0) {
            acc = lane < NW ? Acc{part[lane].x, part[lane].y} : acc_identity();
            acc = warp_merge<NW>(acc);
        }
    }
    if (tid == 0) {
        if (P == 1) {
            store_row(out, TL ? logprob : nullptr, row, acc_finalize(acc), xt);
        } else {
            partial[unit] = make_float2(acc.m, acc.s);
            if (gather) xt_buf[row] = xt;
        }
    }
}

// ---------------------------------------------------------------------------
// Host-side launchers for one element type.
// ---------------------------------------------------------------------------
template <int DT, int G, int V, bool VEC, bool TL, bool E16>
cudaError_t launch_subwarp_gv(const LaunchArgs& a, int64_t grid) {
    return launch_pdl(lse_subwarp_kernel<DT, G, V, VEC, TL, E16>, dim3(static_cast<unsigned>(grid)),
                      dim3(kSubwarpThreads), a.stream, a.x, a.B, a.N, a.row_stride, a.out,
                      a.tl.target, a.tl.logprob);
}

template <int DT, int G, bool VEC, bool TL, bool E16>
cudaError_t launch_subwarp_g(const LaunchArgs& a, int V, int64_t grid) {
    switch (V) {
    case 1: return launch_subwarp_gv<DT, G, 1, VEC, TL, E16>(a, grid);
    case 2: return launch_subwarp_gv<DT, G, 2, VEC, TL, E16>(a, grid);
    case 3: return launch_subwarp_gv<DT, G, 3, VEC, TL, E16>(a, grid);
    case 4: return launch_subwarp_gv<DT, G, 4, VEC, TL, E16>(a, grid);
    case 5:  // 5 or 7 slots per lane: a whole warp per row
        if constexpr (G == 32) return launch_subwarp_gv<DT, G, 5, VEC, TL, E16>(a, grid);
        else return cudaErrorInvalidValue;
    case 7:
        if constexpr (G == 32) return launch_subwarp_gv<DT, G, 7, VEC, TL, E16>(a, grid);
        else return cudaErrorInvalidValue;
    case 6:  // 6 or 8 slots per lane: a whole warp per row, or 4-16 lanes per row of vectors
        if constexpr (G == 32 || (VEC && G >= 4)) return launch_subwarp_gv<DT, G, 6, VEC, TL, E16>(a, grid);
        else return cudaErrorInvalidValue;
    case 8:
        if constexpr (G == 32 || (VEC && G >= 4)) return launch_subwarp_gv<DT, G, 8, VEC, TL, E16>(a, grid);
        else return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

template <int DT, bool VEC, bool TL, bool E16>
cudaError_t launch_subwarp_dt(const LaunchArgs& a, int G, int V, int64_t grid) {
    switch (G) {
    case 1: return launch_subwarp_g<DT, 1, VEC, TL, E16>(a, V, grid);
    case 2: return launch_subwarp_g<DT, 2, VEC, TL, E16>(a, V, grid);
    case 4: return launch_subwarp_g<DT, 4, VEC, TL, E16>(a, V, grid);
    case 8: return launch_subwarp_g<DT, 8, VEC, TL, E16>(a, V, grid);
    case 16: return launch_subwarp_g<DT, 16, VEC, TL, E16>(a, V, grid);
    case 32: return launch_subwarp_g<DT, 32, VEC, TL, E16>(a, V, grid);
    default: return cudaErrorInvalidValue;
    }
}

template <int DT, int T, bool VEC, bool TL, bool E16>
cudaError_t launch_segment_t(const LaunchArgs& a, int64_t P, int64_t seg_slots, float2* partial,
                             float* xt_buf) {
    using Occ = SegmentOccupancy<T>;
    const int64_t grid = (a.B * P + Occ::units_per_cta - 1) / Occ::units_per_cta;
    return launch_pdl(lse_segment_kernel<DT, T, VEC, TL, E16>, dim3(static_cast<unsigned>(grid)),
                      dim3(Occ::cta_threads), a.stream, a.x, a.B, a.N, a.row_stride, P, seg_slots,
                      a.out, partial, a.tl.target, a.tl.logprob, xt_buf);
}

template <int DT, int T, bool VEC, bool TL, bool E16>
int segment_occupancy_t() {
    // Resident units of T threads per SM.
    using Occ = SegmentOccupancy<T>;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, lse_segment_kernel<DT, T, VEC, TL, E16>,
                                                      Occ::cta_threads, 0) != cudaSuccess)
        return 0;
    return blocks * Occ::units_per_cta;
}

}  // namespace lse

// Instantiates the per-type entry points declared in lse_internal.h; TL selects
// the kernels with the fused token log-probability epilogue, E16 the
// reduced-bit exponentials.
#define LSE_DEFINE_TYPE_ENTRY_POINTS(DT, SUFFIX, TL, E16)                                               \
    namespace lse {                                                                            \
    cudaError_t launch_subwarp_##SUFFIX(const LaunchArgs& a, bool vec, int G, int V,           \
                                        int64_t grid) {                                        \
        return vec ? launch_subwarp_dt<DT, true, TL, E16>(a, G, V, grid)                                \
                   : launch_subwarp_dt<DT, false, TL, E16>(a, G, V, grid);                              \
    }                                                                                          \
    cudaError_t launch_segment_##SUFFIX(const LaunchArgs& a, bool vec, int threads, int64_t P, \
                                        int64_t seg_slots, float2* partial, float* xt_buf) {   \
        switch (threads) {                                                                     \
        case 32: return vec ? launch_segment_t<DT, 32, true, TL, E16>(a, P, seg_slots, partial, xt_buf)         \
                            : launch_segment_t<DT, 32, false, TL, E16>(a, P, seg_slots, partial, xt_buf);       \
        case 64: return vec ? launch_segment_t<DT, 64, true, TL, E16>(a, P, seg_slots, partial, xt_buf)         \
                            : launch_segment_t<DT, 64, false, TL, E16>(a, P, seg_slots, partial, xt_buf);       \
        case 128: return vec ? launch_segment_t<DT, 128, true, TL, E16>(a, P, seg_slots, partial, xt_buf)       \
                             : launch_segment_t<DT, 128, false, TL, E16>(a, P, seg_slots, partial, xt_buf);     \
        case 256: return vec ? launch_segment_t<DT, 256, true, TL, E16>(a, P, seg_slots, partial, xt_buf)       \
                             : launch_segment_t<DT, 256, false, TL, E16>(a, P, seg_slots, partial, xt_buf);     \
        case 512: return vec ? launch_segment_t<DT, 512, true, TL, E16>(a, P, seg_slots, partial, xt_buf)       \
                             : launch_segment_t<DT, 512, false, TL, E16>(a, P, seg_slots, partial, xt_buf);     \
        default: return cudaErrorInvalidValue;                                                 \
        }                                                                                      \
    }                                                                                          \
    int segment_occupancy_##SUFFIX(bool vec, int threads) {                                    \
        switch (threads) {                                                                     \
        case 32: return vec ? segment_occupancy_t<DT, 32, true, TL, E16>()                              \
                            : segment_occupancy_t<DT, 32, false, TL, E16>();                            \
        case 64: return vec ? segment_occupancy_t<DT, 64, true, TL, E16>()                              \
                            : segment_occupancy_t<DT, 64, false, TL, E16>();                            \
        case 128: return vec ? segment_occupancy_t<DT, 128, true, TL, E16>()                            \
                             : segment_occupancy_t<DT, 128, false, TL, E16>();                          \
        case 256: return vec ? segment_occupancy_t<DT, 256, true, TL, E16>()                            \
                             : segment_occupancy_t<DT, 256, false, TL, E16>();                          \
        case 512: return vec ? segment_occupancy_t<DT, 512, true, TL, E16>()                            \
                             : segment_occupancy_t<DT, 512, false, TL, E16>();                          \
        default: return 0;                                                                     \
        }                                                                                      \
    }                                                                                          \
    }
