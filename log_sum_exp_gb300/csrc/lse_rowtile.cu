// lse_rowtile.cu -- back-to-back rows fed by 1-D bulk copies (sm_103a).
//
// Rows of 16..128 bytes (a multiple of 16) stored back to back (row_stride ==
// N, 16-byte aligned): one persistent CTA per SM of kRingWarps warps, and every
// warp runs a ring of its own.  Lane 0 streams the warp's 4 KB chunks of whole
// rows from HBM into shared memory with cp.async.bulk (the Tensor Memory
// Accelerator's 1-D copy; completion tracked by an mbarrier transaction
// count); each lane reduces its rows out of shared memory: max, then one FFMA +
// ex2 per element (or, with E16, one packed bf16 ex2 per two elements), then
// the finalize of lse_device.cuh.  A stage is refilled as soon as its own 32
// lanes have read it, so no warp waits for another.  ("Speeding up
// Log-Sum-Exp ...", Sec. 3.1: one pass, a register accumulator per row.)
//
// With TL the same pass writes the token log-probability x[row, target[row]] -
// lse[row]: each lane loads its rows' targets before the chunk lands and reads
// the target element from the staged row in shared memory.
//
// Rows of other widths (not a multiple of 16 bytes, or longer than 128 bytes,
// up to 4 KB) take 32 KB chunks per CTA that start and end on 16-byte
// boundaries; each thread folds its row (rows of <= 128 bytes), or a group of
// G lanes folds each row, from 16-byte reads of the staged chunk, masking the
// elements of the neighbouring rows that share the row's first and last
// vectors.
//
// Waits are bounded: a stage that does not complete within the poll limit
// (kWaitPolls, or lower through lse_set_wait_limit) counts a timeout in a
// device counter (read by lse_wait_timeouts); the warp (or CTA) stops, waits
// with the default limit for the copies it issued and nobody consumed, and
// returns.  Such a timeout does not happen in correct operation.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "lse_device.cuh"
#include "lse_edges.cuh"
#include "lse_internal.h"

namespace lse {
namespace {

constexpr int kTileThreads = 256;      // any-width ring: threads per CTA
constexpr int kChunkBytes = 32 * 1024;  // any-width ring: bytes per stage
constexpr int kStages = 2;              // any-width ring: stages per CTA
constexpr int kWarpChunkBytes = 4096;   // vector ring: bytes per warp stage
constexpr int kRingWarps = 24;          // vector ring: warps per CTA
constexpr int kRingStages = 1;          // vector ring: stages per warp
constexpr int kRingCtasPerSm = 1;       // 96 KB of stages per SM
constexpr uint32_t kWaitPolls = 1u << 26;
constexpr int kAnyThreadRowBytes = 128;  // rows up to this: 256 per chunk, one per thread
constexpr int kAnyThreadRowVectors = 9;  // 16-byte vectors such a row can touch

__device__ unsigned long long g_wait_timeouts;

// Element i of a row staged in shared memory (plain loads: the read-only
// global path must not see a shared-memory address).
template <int DT>
__device__ __forceinline__ float staged_elem(const unsigned char* row, int i) {
    if constexpr (DT == kF32) {
        return reinterpret_cast<const float*>(row)[i];
    } else {
        const unsigned short h = reinterpret_cast<const unsigned short*>(row)[i];
        if constexpr (DT == kBF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
        else return __half2float(__ushort_as_half(h));
    }
}

// Lanes per repeat of the 16-byte bank group at which consecutive rows of NV
// vectors start: 8 / gcd(NV, 8).
template <int NV>
constexpr int kRotationPeriod = 8 / (NV % 8 == 0 ? 8 : (NV % 4 == 0 ? 4 : (NV % 2 == 0 ? 2 : 1)));

// NV (1..8) 16-byte vectors per row.  Every warp runs a ring of its own:
// S stages of one warp chunk each, a warp chunk being 32 * RPL rows
// (RPL = floor(8 / NV) rows per lane, at most 4 KB).  Lane 0 issues the bulk
// copy of each chunk into a free stage of its warp and every lane waits on
// that stage's mbarrier; once the 32 lanes have read the stage into registers
// (a __syncwarp), lane 0 refills it with the warp's next chunk, so a warp
// never waits for another one.  Warp chunks are dealt round-robin to the
// warps of the grid.  `polls` bounds every stage wait (kWaitPolls unless a
// caller lowered it through lse_set_wait_limit).
// E16: reduced-bit exponentials; TL: token log-probability epilogue (out may
// then be null).
template <int DT, int NV, bool E16, bool TL, int W, int S>
__global__ void __launch_bounds__(W * 32)
lse_rowtile_kernel(const void* __restrict__ x, int64_t B, float* __restrict__ out,
                   const int64_t* __restrict__ target, float* __restrict__ logprob,
                   uint32_t polls) {
    constexpr int RB = NV * 16;                // bytes per row
    constexpr int RPL = 8 / NV;                // rows per lane per chunk
    constexpr int CR = 32 * RPL;               // rows per warp chunk
    constexpr int NE = RB / DType<DT>::bytes;  // elements per row
    static_assert(NV >= 1 && NV <= 8 && CR * RB <= kWarpChunkBytes, "a chunk must fit one stage");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bars[W * S];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    unsigned char* ring = smem + wid * (S * kWarpChunkBytes);
    uint64_t* full = full_bars + wid * S;
    const int64_t nchunks = (B + CR - 1) / CR;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * W;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * W + wid;
    const char* xb = reinterpret_cast<const char*>(x);

    // The barriers live in this CTA's shared memory: set them up before
    // waiting for the previous kernel in the stream.
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    pdl_trigger();
    pdl_wait();

    auto issue = [&](int64_t chunk, int s) {  // lane 0 only
        const int64_t r0 = chunk * CR;
        const int64_t rows = B - r0 < CR ? B - r0 : CR;
        const uint32_t bytes = static_cast<uint32_t>(rows * RB);
        mbar_expect_tx(&full[s], bytes);
        bulk_load(ring + s * kWarpChunkBytes, xb + r0 * RB, bytes, &full[s]);
    };
    if (lane == 0)
        for (int s = 0; s < S; ++s) {
            const int64_t c = gw + static_cast<int64_t>(s) * nwarps;
            if (c < nchunks) issue(c, s);
        }

    int64_t k = 0;  // chunks consumed by this warp
    int64_t c = gw;
    bool timed_out = false;
    for (; c < nchunks; c += nwarps, ++k) {
        const int s = static_cast<int>(k % S);
        // Targets of this lane's rows (coalesced), loaded while the chunk lands.
        int tq[TL ? RPL : 1];
        if constexpr (TL) {
#pragma unroll
            for (int q = 0; q < RPL; ++q) {
                const int64_t row = c * CR + q * 32 + lane;
                const int64_t t = row < B ? __ldg(target + row) : -1;
                tq[q] = (t >= 0 && t < NE) ? static_cast<int>(t) : -1;
            }
        }
        const bool ok = __all_sync(0xffffffffu,
                                   mbar_wait(&full[s], static_cast<uint32_t>((k / S) & 1), polls));
        if (!ok) {  // every lane stops; lane 0 drains the copies below
            timed_out = true;
            break;
        }
        uint32_t w[RPL][4 * NV];
        float xt[TL ? RPL : 1];
#pragma unroll
        for (int q = 0; q < RPL; ++q) {
            const unsigned char* rowp = ring + s * kWarpChunkBytes + (q * 32 + lane) * RB;
            const uint4* rp = reinterpret_cast<const uint4*>(rowp);
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                // A 16-byte read by a warp is served a quarter-warp (8 lanes)
                // at a time: conflict free when the 8 lanes hit the 8
                // different 16-byte bank groups of a 128-byte line.  Lane l's
                // row starts at group NV * l (mod 8), a pattern of period
                // P = 8 / gcd(NV, 8) lanes, so lanes P apart start at the same
                // group; rotating the vector order by (l mod 8) / P moves them
                // apart.  Max and sum do not depend on the order.
                const uint4 u = rp[(j + (lane & 7) / kRotationPeriod<NV>) % NV];
                w[q][4 * j] = u.x; w[q][4 * j + 1] = u.y; w[q][4 * j + 2] = u.z; w[q][4 * j + 3] = u.w;
            }
            if constexpr (TL)
                xt[q] = tq[q] >= 0 ? staged_elem<DT>(rowp, tq[q]) : __int_as_float(0x7fc00000);
        }
        __syncwarp();  // every lane has read stage s: it may be refilled
        if (lane == 0) {
            const int64_t cn = c + static_cast<int64_t>(S) * nwarps;
            if (cn < nchunks) issue(cn, s);
        }
#pragma unroll
        for (int q = 0; q < RPL; ++q) {
            const int64_t row = c * CR + q * 32 + lane;
            if (row < B) {
                const float m = words_max<DT, 4 * NV>(w[q]);
                const float mu = shift_of(m);
                float lse;
                if (!E16 && ffma_shift_ok(mu)) {  // E16: exact 0 argument for the maximum
                    const float cc = mu * kLog2e;
                    lse = finalize_scaled(m, words_expsum_scaled<DT, 4 * NV>(w[q], cc), mu, cc);
                } else {
                    lse = acc_finalize(Acc{m, expsum_words<DT, 4 * NV, E16>(w[q], mu)});
                }
                store_row(out, TL ? logprob : nullptr, row, lse, TL ? xt[TL ? q : 0] : 0.0f);
            }
        }
    }
    if (timed_out && lane == 0) {
        atomicAdd(&g_wait_timeouts, 1ull);
        // Chunks c, c + nwarps, ..., c + (S-1) nwarps were issued and not yet
        // consumed: let each land (bounded) before the shared memory is released.
        for (int j = 0; j < S; ++j) {
            const int64_t kk = k + j;
            if (c + j * nwarps < nchunks)
                mbar_wait(&full[kk % S], static_cast<uint32_t>((kk / S) & 1), kWaitPolls);
        }
    }
    __syncwarp();
}

// Back-to-back rows whose width RB = N * elem bytes is not a multiple of 16
// or is above 128 bytes (up to kChunkBytes / 8; row value only).  A chunk of
// CR rows starts and ends on a 16-byte boundary as long as CR is a multiple of
// k = 16 / gcd(RB, 16): the copies cover the first Bm = B - B % k rows, and
// the < k rows after them are read from global memory by CTA 0 at the end.
// G == 1 (rows of <= 128 bytes plus one element): CR = 256 * floor(32 KB /
// (256 * RB)) up to 128 bytes, else as for G > 1, and each thread folds whole
// rows from vector reads (max, then the exp-sum).
// G > 1: CR = floor(32 KB / RB) rounded down to a multiple of k; the 256 / G
// groups of G lanes take the chunk's rows in turn, a lane reading every G-th
// 16-byte vector of its row from shared memory (conflict-free: a group reads
// consecutive vectors), the two vectors the row shares with its neighbours
// masked, folded online and merged over the group with shuffles.  A stage is
// released for the next copy only after every thread is done with it.  TL:
// the token log-probability epilogue (out may then be null): each row's target
// is loaded before its fold, and x[row, target] read from the staged row.
template <int DT, int G, bool TL, int NVT = kAnyThreadRowVectors>
__global__ void __launch_bounds__(kTileThreads)
lse_rowtile_any_kernel(const void* __restrict__ x, int64_t B, int64_t N, float* __restrict__ out,
                       const int64_t* __restrict__ target, float* __restrict__ logprob,
                       uint32_t polls) {
    constexpr int EB = DType<DT>::bytes;
    constexpr int GROUPS = kTileThreads / G;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ __align__(8) uint64_t full[kStages];
    const int tid = threadIdx.x;
    const int RB = static_cast<int>(N) * EB;
    int g = RB;  // gcd(RB, 16)
    for (int t = 16; t != 0;) {
        const int r = g % t;
        g = t;
        t = r;
    }
    const int64_t k = 16 / g;
    const int64_t CR = RB <= kAnyThreadRowBytes
                           ? static_cast<int64_t>(kTileThreads) * (kChunkBytes / (kTileThreads * RB))
                           : (kChunkBytes / RB) - (kChunkBytes / RB) % k;
    const int64_t Bm = B - B % k;
    const int64_t nchunks = (Bm + CR - 1) / CR;
    const char* xb = reinterpret_cast<const char*>(x);

    pdl_trigger();
    pdl_wait();
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    auto issue = [&](int64_t chunk, int s) {  // thread 0 only
        const int64_t r0 = chunk * CR;
        const int64_t rows = Bm - r0 < CR ? Bm - r0 : CR;
        const uint32_t bytes = static_cast<uint32_t>(rows * RB);  // a multiple of 16
        mbar_expect_tx(&full[s], bytes);
        bulk_load(stage + s * kChunkBytes, xb + r0 * RB, bytes, &full[s]);
    };
    if (tid == 0)
        for (int s = 0; s < kStages; ++s) {
            const int64_t c = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (c < nchunks) issue(c, s);
        }

    auto fold = [&](auto elem) {  // elem(n) -> float; the row value (G == 1)
        float m = __int_as_float(kNegInfF32);
        for (int n = 0; n < N; ++n) m = fmaxf(m, elem(n));
        const float mu = shift_of(m);
        float acc[2] = {0.0f, 0.0f};
        for (int n = 0; n < N; ++n) acc[n & 1] += ex2((elem(n) - mu) * kLog2e);
        return acc_finalize(Acc{m, acc[0] + acc[1]});
    };
    const int sub = tid & (G - 1);
    const int grp = tid / G;

    int64_t kc = 0;  // chunks consumed by this CTA
    int64_t c = blockIdx.x;
    bool timed_out = false;
    for (; c < nchunks; c += gridDim.x, ++kc) {
        const int s = static_cast<int>(kc % kStages);
        const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((kc / kStages) & 1), polls);
        const unsigned char* st = stage + s * kChunkBytes;
        // Results are stored as soon as they are computed; the stage is only
        // read before the barrier below.
        if constexpr (G == 1) {
            for (int64_t q = tid; q < CR; q += kTileThreads) {
                const int64_t row = c * CR + q;
                if (ok && row < Bm) {
                    const int64_t t = TL ? __ldg(target + row) : -1;
                    // The aligned 16-byte vectors holding the row's <= 128 bytes
                    // (at most NVT: 9, or 5 for rows of <= 64 + elem bytes; only
                    // those are read and folded), the
                    // neighbours' elements in the first and the last masked to
                    // -inf, folded from registers (max, then exp-sum).
                    const uint32_t rb0 = static_cast<uint32_t>(q * RB);
                    const uint32_t rb1 = rb0 + static_cast<uint32_t>(RB);
                    const uint32_t v0 = rb0 >> 4;
                    const int nvec = static_cast<int>(((rb1 + 15u) >> 4) - v0);
                    uint32_t w[4 * NVT];
#pragma unroll
                    for (int j = 0; j < NVT; ++j) {
                        uint4 u = make_uint4(neg_inf_word<DT>(), neg_inf_word<DT>(), neg_inf_word<DT>(),
                                             neg_inf_word<DT>());
                        if (j < nvec) u = *reinterpret_cast<const uint4*>(st + (v0 + j) * 16u);
                        w[4 * j] = u.x; w[4 * j + 1] = u.y; w[4 * j + 2] = u.z; w[4 * j + 3] = u.w;
                    }
#pragma unroll
                    for (int j = 0; j < NVT; ++j) {
                        if (j == 0 || j == nvec - 1) {
                            uint32_t q4[4] = {w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]};
                            if (j == 0) mask_prefix<DT>(q4, static_cast<int>(rb0 & 15u));
                            if (j == nvec - 1) mask_suffix<DT>(q4, static_cast<int>(rb1 - (v0 + j) * 16u));
#pragma unroll
                            for (int i = 0; i < 4; ++i) w[4 * j + i] = q4[i];
                        }
                    }
                    const float m = words_max<DT, 4 * NVT>(w);
                    const float mu = shift_of(m);
                    float sum = 0.0f;
#pragma unroll
                    for (int j = 0; j < NVT; ++j) {
                        if (j < nvec) {
                            const uint32_t q4[4] = {w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]};
                            sum += words_expsum<DT, 4>(q4, mu);
                        }
                    }
                    const float lse = acc_finalize(Acc{m, sum});
                    const float xt = TL && t >= 0 && t < N ? staged_elem<DT>(st + q * RB, static_cast<int>(t))
                                                           : __int_as_float(0x7fc00000);
                    store_row(out, TL ? logprob : nullptr, row, lse, xt);
                }
            }
        } else {
            const int64_t rows = Bm - c * CR < CR ? Bm - c * CR : CR;
            // Every lane runs the same number of passes (the group merge is a
            // warp-wide shuffle); rows past the chunk fold nothing.
            for (int64_t q0 = 0; q0 < rows; q0 += GROUPS) {
                const int64_t q = q0 + grp;
                const bool live = ok && q < rows;
                const uint32_t rb0 = live ? static_cast<uint32_t>(q * RB) : 0u;
                const uint32_t rb1 = live ? rb0 + static_cast<uint32_t>(RB) : 0u;
                const int64_t t = TL && live && sub == 0 ? __ldg(target + c * CR + q) : -1;
                Acc acc = acc_identity();
                float mu = 0.0f;
                const uint32_t v_end = (rb1 + 15u) >> 4;
                for (uint32_t v = (rb0 >> 4) + sub; v < v_end; v += 2 * G) {
                    uint32_t w[8];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t vh = v + h * G;
                        uint32_t q4[4] = {neg_inf_word<DT>(), neg_inf_word<DT>(), neg_inf_word<DT>(),
                                          neg_inf_word<DT>()};
                        if (vh < v_end) {
                            const uint4 u = *reinterpret_cast<const uint4*>(st + vh * 16u);
                            q4[0] = u.x; q4[1] = u.y; q4[2] = u.z; q4[3] = u.w;
                            // (the two-sided mask: one-sided ones measured slower in this
                            // loop, bf16 N = 520 0.838 -> 0.812 of the copy peak)
                            if (vh * 16u < rb0 || vh * 16u + 16u > rb1) mask_words<DT>(q4, vh * 16u, rb0, rb1);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) w[4 * h + i] = q4[i];
                    }
                    acc_add_words<DT, 8>(acc, mu, w);
                }
                acc = warp_merge<G>(acc);
                if (live && sub == 0) {
                    const float xt = TL && t >= 0 && t < N
                                         ? staged_elem<DT>(st + rb0, static_cast<int>(t))
                                         : __int_as_float(0x7fc00000);
                    store_row(out, TL ? logprob : nullptr, c * CR + q, acc_finalize(acc), xt);
                }
            }
        }
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        if (tid == 0) {
            const int64_t cn = c + static_cast<int64_t>(kStages) * gridDim.x;
            if (cn < nchunks) issue(cn, s);
        }
    }
    if (timed_out) {
        if (tid == 0) {
            atomicAdd(&g_wait_timeouts, 1ull);
            // Chunks c, c + grid, ..., c + (kStages-1) grid were issued and not
            // yet consumed: let each land (bounded) before the shared memory
            // is released.
            for (int j = 0; j < kStages; ++j) {
                const int64_t kk = kc + j;
                if (c + j * static_cast<int64_t>(gridDim.x) < nchunks)
                    mbar_wait(&full[kk % kStages], static_cast<uint32_t>((kk / kStages) & 1), kWaitPolls);
            }
        }
        __syncthreads();
        return;
    }
    if (blockIdx.x == 0 && Bm + tid < B) {  // the < k rows after the last copy
        const int64_t row = Bm + tid;
        const char* rowp = xb + row * RB;
        const int64_t t = TL ? __ldg(target + row) : -1;
        const float lse = fold([&](int n) { return load_elem<DT>(rowp, n); });
        const float xt = TL && t >= 0 && t < N ? load_elem<DT>(rowp, t) : __int_as_float(0x7fc00000);
        store_row(out, TL ? logprob : nullptr, row, lse, xt);
    }
}

// The poll limit of the stage waits (lse_set_wait_limit; kWaitPolls by default).
std::atomic<uint32_t> g_stage_polls{kWaitPolls};

// Raise kernel K's dynamic shared-memory limit once per device (the
// attribute belongs to the function in the current device's context).
template <auto K>
cudaError_t allow_smem(int bytes) {
    static std::atomic<uint64_t> done{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <int DT, int G, bool TL, int NVT = kAnyThreadRowVectors>
cudaError_t launch_rowtile_any_g(const LaunchArgs& a, int grid) {
    const int smem = kStages * kChunkBytes;
    cudaError_t e = allow_smem<lse_rowtile_any_kernel<DT, G, TL, NVT>>(smem);
    if (e != cudaSuccess) return e;
    return launch_pdl_smem(lse_rowtile_any_kernel<DT, G, TL, NVT>, dim3(static_cast<unsigned>(grid)),
                           dim3(kTileThreads), static_cast<size_t>(smem), a.stream, a.x, a.B, a.N,
                           a.out, a.tl.target, a.tl.logprob, g_stage_polls.load(std::memory_order_relaxed));
}

template <int DT, bool TL>
cudaError_t launch_rowtile_any_t(const LaunchArgs& a, int lanes, int grid) {
    switch (lanes) {
    case 1:  // a thread per row: 5 vector slots cover rows of <= 64 + elem bytes
        if (a.N * DType<DT>::bytes <= 64 + DType<DT>::bytes) return launch_rowtile_any_g<DT, 1, TL, 5>(a, grid);
        return launch_rowtile_any_g<DT, 1, TL>(a, grid);
    case 4: return launch_rowtile_any_g<DT, 4, TL>(a, grid);
    case 8: return launch_rowtile_any_g<DT, 8, TL>(a, grid);
    case 16: return launch_rowtile_any_g<DT, 16, TL>(a, grid);
    case 32: return launch_rowtile_any_g<DT, 32, TL>(a, grid);
    default: return cudaErrorInvalidValue;
    }
}

template <bool TL>
cudaError_t launch_rowtile_any(int dt, int lanes, const LaunchArgs& a, int grid) {
    switch (dt) {
    case kF32: return launch_rowtile_any_t<kF32, TL>(a, lanes, grid);
    case kBF16: return launch_rowtile_any_t<kBF16, TL>(a, lanes, grid);
    default: return launch_rowtile_any_t<kF16, TL>(a, lanes, grid);
    }
}

template <int DT, int NV, bool E16, bool TL>
cudaError_t launch_rowtile_t(const LaunchArgs& a, int grid) {
    constexpr int W = kRingWarps, S = kRingStages;
    const int smem = W * S * kWarpChunkBytes;
    cudaError_t e = allow_smem<lse_rowtile_kernel<DT, NV, E16, TL, W, S>>(smem);
    if (e != cudaSuccess) return e;
    return launch_pdl_smem(lse_rowtile_kernel<DT, NV, E16, TL, W, S>, dim3(static_cast<unsigned>(grid)),
                           dim3(W * 32), static_cast<size_t>(smem), a.stream, a.x, a.B,
                           a.out, a.tl.target, a.tl.logprob, g_stage_polls.load(std::memory_order_relaxed));
}

template <int DT, bool E16, bool TL>
cudaError_t launch_rowtile_dt(int nv, const LaunchArgs& a, int grid) {
    switch (nv) {
    case 1: return launch_rowtile_t<DT, 1, E16, TL>(a, grid);
    case 2: return launch_rowtile_t<DT, 2, E16, TL>(a, grid);
    case 3: return launch_rowtile_t<DT, 3, E16, TL>(a, grid);
    case 4: return launch_rowtile_t<DT, 4, E16, TL>(a, grid);
    case 5: return launch_rowtile_t<DT, 5, E16, TL>(a, grid);
    case 6: return launch_rowtile_t<DT, 6, E16, TL>(a, grid);
    case 7: return launch_rowtile_t<DT, 7, E16, TL>(a, grid);
    case 8: return launch_rowtile_t<DT, 8, E16, TL>(a, grid);
    default: return cudaErrorInvalidValue;
    }
}

template <bool E16, bool TL>
cudaError_t launch_rowtile_e(int dt, int nv, const LaunchArgs& a, int grid) {
    switch (dt) {
    case kF32: return launch_rowtile_dt<kF32, E16, TL>(nv, a, grid);
    case kBF16: return launch_rowtile_dt<kBF16, E16, TL>(nv, a, grid);
    default: return launch_rowtile_dt<kF16, E16, TL>(nv, a, grid);
    }
}

}  // namespace

cudaError_t launch_rowtile(int dt, int nv, int lanes, const LaunchArgs& a, int grid) {
    if (nv == 0) {  // any row width: row value or token log-probability, f32 exponentials
        if (a.e16) return cudaErrorInvalidValue;
        if ((lanes == 1) != (a.N * (dt == kF32 ? 4 : 2) <= rowtile_any_thread_row_max_bytes(dt == kF32 ? 4 : 2)) ||
            a.N * (dt == kF32 ? 4 : 2) > kChunkBytes / 8)
            return cudaErrorInvalidValue;
        return a.tl.logprob ? launch_rowtile_any<true>(dt, lanes, a, grid)
                            : launch_rowtile_any<false>(dt, lanes, a, grid);
    }
    if (a.tl.logprob) return launch_rowtile_e<false, true>(dt, nv, a, grid);
    return a.e16 ? launch_rowtile_e<true, false>(dt, nv, a, grid)
                 : launch_rowtile_e<false, false>(dt, nv, a, grid);
}

int rowtile_ctas_per_sm() { return kRingCtasPerSm; }
int rowtile_threads() { return kRingWarps * 32; }
int rowtile_rows_per_chunk(int nv) { return kRingWarps * 32 * (8 / nv); }  // one chunk per warp
int rowtile_any_ctas_per_sm() { return 3; }  // 3 x 64 KB of stages per SM
int rowtile_any_rows_per_chunk(int row_bytes) {
    if (row_bytes <= kAnyThreadRowBytes) return kTileThreads * (kChunkBytes / (kTileThreads * row_bytes));
    int g = row_bytes;  // gcd(row_bytes, 16)
    for (int t = 16; t != 0;) {
        const int r = g % t;
        g = t;
        t = r;
    }
    const int rows = kChunkBytes / row_bytes;
    return rows - rows % (16 / g);
}
int rowtile_any_max_row_bytes() { return kChunkBytes / 8; }

cudaError_t read_wait_timeouts(unsigned long long* count) {
    return cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(*count));
}

void set_stage_wait_polls(uint32_t polls) { g_stage_polls.store(polls, std::memory_order_relaxed); }
uint32_t stage_wait_polls() { return g_stage_polls.load(std::memory_order_relaxed); }
uint32_t default_stage_wait_polls() { return kWaitPolls; }

}  // namespace lse
