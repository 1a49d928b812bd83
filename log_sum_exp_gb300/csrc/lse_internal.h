// lse_internal.h -- declarations shared by the host dispatcher and the
// per-element-type kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "../../include/lse.h"

namespace lse {

constexpr int kSubwarpThreads = 256;
// Five resident CTAs per SM (<= 48 registers, no spills): one-shot CTAs whose
// 16-byte loads are all in flight at once; occupancy sets the bytes in flight.
constexpr int kSubwarpMinBlocks = 5;
// Segment plans of 32 threads per unit run this many units (one per warp) in a CTA.
constexpr int kSegmentWarpUnitsPerCta = 8;

// Optional fused consumer of the row value, the token log-probability
// logprob[b] = x[b, target[b]] - lse[b] (NaN when target[b] is not in [0, N)).
struct TokenLogprob {
    const int64_t* target = nullptr;  // device, one per row; nullptr = not requested
    float* logprob = nullptr;         // device, one per row
};

struct LaunchArgs {
    const void* x;
    int64_t B;
    int64_t N;
    int64_t row_stride;  // elements
    float* out;          // row values; may be nullptr when tl.logprob is set
    cudaStream_t stream;
    TokenLogprob tl;
    bool e16 = false;  // reduced-bit exponentials (row value only)
};

// Launch with programmatic stream serialization (see pdl_trigger / pdl_wait in
// lse_device.cuh): the kernel may start while its predecessor in the stream is
// finishing, and waits for it on the device before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args&&... args) {
    cudaLaunchAttribute attr[1] = {};
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// launch_pdl_smem without dynamic shared memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                       Args&&... args) {
    return launch_pdl_smem(kernel, grid, block, 0, stream, std::forward<Args>(args)...);
}

// Per element type (f32 / bf16 / f16): launchers and occupancy queries.
#define LSE_DECLARE_TYPE_ENTRY_POINTS(SUFFIX)                                                  \
    cudaError_t launch_subwarp_##SUFFIX(const LaunchArgs& a, bool vec, int G, int V,           \
                                        int64_t grid);                                         \
    cudaError_t launch_segment_##SUFFIX(const LaunchArgs& a, bool vec, int threads, int64_t P, \
                                        int64_t seg_slots, float2* partial, float* xt_buf);    \
    int segment_occupancy_##SUFFIX(bool vec, int threads);

LSE_DECLARE_TYPE_ENTRY_POINTS(f32)
LSE_DECLARE_TYPE_ENTRY_POINTS(bf16)
LSE_DECLARE_TYPE_ENTRY_POINTS(f16)
// The same kernels with the fused token log-probability epilogue.
LSE_DECLARE_TYPE_ENTRY_POINTS(lp_f32)
LSE_DECLARE_TYPE_ENTRY_POINTS(lp_bf16)
LSE_DECLARE_TYPE_ENTRY_POINTS(lp_f16)
// The same kernels with reduced-bit (packed bf16) exponentials.
LSE_DECLARE_TYPE_ENTRY_POINTS(e16_f32)
LSE_DECLARE_TYPE_ENTRY_POINTS(e16_bf16)
LSE_DECLARE_TYPE_ENTRY_POINTS(e16_f16)

// Type-independent kernels (lse_api.cu).
cudaError_t launch_fill_neg_inf(float* out, float* logprob, int64_t B, cudaStream_t stream);
cudaError_t launch_merge(const float2* partial, const float* xt_buf, int64_t B, int64_t P,
                         float* out, float* logprob, cudaStream_t stream);
// Backward (lse_backward.cu).
struct BackwardArgs {
    const void* x;
    int64_t B;
    int64_t N;
    int64_t row_stride;
    const float* lse;
    const float* grad;
    void* dx;
    int64_t dx_row_stride;
    int64_t seg_slots;  // slots (16-byte vectors or elements) per blockIdx.x segment
    bool small;         // rows of <= backward_slots_per_thread() slots: flattened mapping
    dim3 grid;
    dim3 block;
    cudaStream_t stream;
};
// Slots of the row backward: elements (x and dx rows at different offsets
// from a 16-byte boundary), 16-byte vectors (every row on a boundary),
// vectors with each row's head and tail peeled into element slots, or (flat)
// back-to-back rows streamed as one array of vectors that may span two rows.
enum BackwardMode { kBwdScalar = 0, kBwdVector = 1, kBwdPeel = 2, kBwdFlat = 3 };
cudaError_t launch_backward(int dt, int mode, const BackwardArgs& a);
// Backward of the value over a non-last dimension (lse_backward.cu).
struct BackwardStridedArgs {
    const void* x;
    int64_t A;
    int64_t R;
    int64_t C;
    int64_t stride_a;
    int64_t stride_r;
    const float* lse;   // [A, C]
    const float* grad;  // [A, C]
    void* dx;
    int64_t dx_stride_a;
    int64_t dx_stride_r;
    int64_t rows_per_split;
    int warps_per_unit;  // 1, or backward_strided_warps(): warps sharing one (a, tile) unit
    int lanes_per_tile;  // 32; 16 or 8 for one-warp units of narrow C (cols_lanes_per_tile)
    dim3 grid;           // (CTAs striding over the (a, tile) units, 1, row splits)
    cudaStream_t stream;
};
cudaError_t launch_backward_strided(int dt, bool vec, const BackwardStridedArgs& a);
int backward_strided_warps();
int backward_slots_per_thread();
int backward_threads();
int backward_flat_vectors_per_thread();

// Strided / column reduction (lse_strided.cu).
struct StridedArgs {
    const void* x;
    int64_t A;
    int64_t R;
    int64_t C;
    int64_t stride_a;
    int64_t stride_r;
    int64_t rows_per_split;
    float* out;
    float2* partial;  // [P, A * C] when P > 1
    int64_t P;
    int warps_per_tile;  // 1, 2, 4 or 8 warps interleave the rows of one column tile
    dim3 grid;           // (CTAs striding over the (a, tile) units, 1, row splits)
    cudaStream_t stream;
};
cudaError_t launch_cols(int dt, bool vec, const StridedArgs& a);
// R <= kColsShortMaxRows rows of 16-byte column vectors, a thread per vector
// (lse_cols_short_kernel); a.grid is the 1-D grid, a.R the rows.
constexpr int kColsShortThreads = 256;
constexpr int kColsShortMaxRows = 8;
cudaError_t launch_cols_short(int dt, const StridedArgs& a);
cudaError_t launch_merge_columns(const float2* partial, int64_t outputs, int64_t P, float* out,
                                 cudaStream_t stream);
int cols_occupancy(int dt, bool vec, int warps_per_tile);  // CTAs per SM
int cols_columns_per_warp(bool vec, int dt);
// Lanes per column tile: 32, or 16 for one-warp tiles of narrow C (a warp then
// folds two tiles).
int cols_lanes_per_tile(int dt, bool vec, int64_t C, int warps_per_tile);
int cols_rows_per_batch(bool vec);  // per warp per iteration
int cols_warps_per_cta(int warps_per_tile);

// Short contiguous rows through the bulk-copy ring (lse_rowtile.cu).
// Reads a.x, a.B, a.out, a.tl (token log-probability) and a.e16 (reduced-bit
// exponentials; not together with a.tl).  nv = 1..8 vectors per row, or 0 for
// rows of any width up to 128 bytes (a.N elements; row value only).
// nv 0: rows of any width; lanes per row 1 (rows of <= 128 bytes) or 4..32.
cudaError_t launch_rowtile(int dt, int nv, int lanes, const LaunchArgs& a, int grid);
int rowtile_ctas_per_sm();
int rowtile_threads();  // threads per CTA of the vector ring (one ring per warp)
// Widest back-to-back row the any-width ring folds with one thread: 128 bytes
// plus one element (such a row, from any element offset, touches at most
// nine 16-byte vectors).
inline int rowtile_any_thread_row_max_bytes(int elem_bytes) { return 128 + elem_bytes; }
int rowtile_rows_per_chunk(int nv);  // rows a CTA takes per round (one chunk per warp)
int rowtile_any_ctas_per_sm();
int rowtile_any_rows_per_chunk(int row_bytes);  // nv == 0: rows of any width
int rowtile_any_max_row_bytes();
cudaError_t read_wait_timeouts(unsigned long long* count);
// Poll limit of the rings' stage waits (the drain after a timeout keeps the
// default limit).
void set_stage_wait_polls(uint32_t polls);
uint32_t default_stage_wait_polls();

// Sets the calling thread's error reported by lse_last_cuda_error.
void record_cuda_error(cudaError_t e);

// The argument checks of the row entry points (lse_api.cu): dtype, B, N,
// row_stride, NULL and alignment of x and out, int64 byte extent.
lse_status check_args(const void* x, int dt, int64_t B, int64_t N, int64_t row_stride,
                      const void* out);

}  // namespace lse
