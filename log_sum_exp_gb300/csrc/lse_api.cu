// lse_api.cu -- the C ABI of liblse: argument checks, the choice of kernel
// mapping, stream-ordered scratch, and the two type-independent kernels (the
// N == 0 fill and the split-row merge).  See include/lse.h for the contract.
//
// Source of the operation: "Speeding up Log-Sum-Exp: Kernel Fusion at the
// Memory Wall, Integer Arithmetic at the Compute Wall", Sec. 3.1 (one fused
// pass; partial results combined with the pairwise LSE operation).
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/lse.h"
#include "lse_device.cuh"
#include "lse_internal.h"

namespace lse {
namespace {

thread_local int g_last_cuda_error = 0;

// Report a CUDA failure through the status code and lse_last_cuda_error, and
// clear the runtime's per-thread last error so it does not surface later in
// the caller's own error checks (sticky device errors cannot be cleared).
lse_status cuda_fail(cudaError_t e, lse_status st = LSE_ERR_CUDA) {
    g_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();
    return st;
}

constexpr int kMaxDevices = 64;
constexpr int kSubwarpMaxSlots = 4;    // slots per lane in the subwarp kernel (G < 32)
constexpr int kSubwarpWarpSlots = 8;   // slots per lane when a whole warp holds a row
constexpr int kSegmentBatchVec = 8;    // slots per thread per batch (16-byte loads)
constexpr int kSegmentBatchScalar = 16;
constexpr int kMergeRowsPerCta = 8;    // one warp per row
constexpr int kSplitMinBatches = 8;    // batches per thread a split segment keeps (when it can)

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int seg_occ[3][2][5] = {};  // [dtype][vec][log2(threads / 32)]
    // Library-owned stream-ordered pool: freed blocks stay mapped for reuse by
    // later calls (release threshold = max) until lse_trim_memory().
    cudaMemPool_t pool = nullptr;
};

std::mutex g_info_mutex;
DeviceInfo g_info[kMaxDevices];

int segment_occupancy(int dt, bool vec, int threads) {
    switch (dt) {
    case LSE_F32: return segment_occupancy_f32(vec, threads);
    case LSE_BF16: return segment_occupancy_bf16(vec, threads);
    default: return segment_occupancy_f16(vec, threads);
    }
}

lse_status device_info(int* dev_out, const DeviceInfo** info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return LSE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_info_mutex);
    DeviceInfo& d = g_info[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        for (int dt = 0; dt < 3; ++dt)
            for (int v = 0; v < 2; ++v)
                for (int t = 0; t < 5; ++t) {
                    const int occ = segment_occupancy(dt, v != 0, 32 << t);
                    d.seg_occ[dt][v][t] = occ > 0 ? occ : 1;
                }
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof props);
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        e = cudaMemPoolCreate(&d.pool, &props);
        if (e != cudaSuccess) return cuda_fail(e);
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) return cuda_fail(e);
        d.ready = true;
    }
    *dev_out = dev;
    *info = &d;
    return LSE_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int elem_bytes(lse_dtype dt) { return dt == LSE_F32 ? 4 : 2; }

// Stream-ordered device allocation from the library pool.  While `stream` is
// being captured into a CUDA graph the device's default pool is used instead,
// so the allocation becomes a graph memory node.
cudaError_t scratch_alloc(const DeviceInfo& info, void** p, size_t bytes, cudaStream_t stream) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return e;
    if (cap != cudaStreamCaptureStatusNone) return cudaMallocAsync(p, bytes, stream);
    return cudaMallocFromPoolAsync(p, bytes, info.pool, stream);
}

bool valid_dtype(int dt) { return dt == LSE_F32 || dt == LSE_BF16 || dt == LSE_F16; }

int pow2_ceil(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Slots per lane the sub-warp kernel is built for that hold v: 1, 2, 3, 4, and
// 6 or 8 in groups that may hold more than 4 (a whole warp, or 4-16 lanes of
// 16-byte vectors).  Rows just above a power of two of slots (an unaligned row
// adds up to two) waste less on -inf padding with 3 or 6 than with 4 or 8: on
// those the kernel is bound by instruction issue, not memory.
int64_t subwarp_slot_count(int64_t v, bool wide, bool warp) {
    if (v <= 4 || warp) return v;  // a whole warp per row: 5 and 7 slots too
    return wide && v <= 6 ? 6 : 8;
}

// Lanes per row of the automatic sub-warp plan for rows of nvt slots: the
// fewest that keep <= kSubwarpMaxSlots slots per lane (four independent loads
// per thread), at most a warp.  Vector rows of more than 16 slots take half
// the lanes with 8 slots each, so a warp holds twice the rows: measured on
// 256 MB of rows of 65-1024 elements (f32, bf16; aligned and peeled), faster
// for every length, +1-11 % on full groups, up to +40 % where a row fills
// half its slots.
int subwarp_auto_lanes(int64_t nvt, bool vec) {
    int G = pow2_ceil(ceil_div(nvt, kSubwarpMaxSlots));
    if (G > 32) G = 32;
    if (vec && nvt > 4 * kSubwarpMaxSlots) {
        G = pow2_ceil(ceil_div(nvt, kSubwarpWarpSlots));
        if (G < 4) G = 4;
    }
    return G;
}

// Slots per row of that plan (lanes x slots per lane) as the grouped-ring rule
// below was measured: slots per lane padded to 6 or 8 even for a whole warp
// (whose plans now take 5 and 7 too: f32 N = 520, 132 slots in 160, still
// measured faster on the ring, 1.018 against 0.971 of the copy peak; N = 600,
// 152 in 160, faster on the warp, 1.037 against 1.015).
int64_t subwarp_auto_slots(int64_t nvt, bool vec) {
    const int G = subwarp_auto_lanes(nvt, vec);
    return G * subwarp_slot_count(ceil_div(nvt, G), G == 32 || (vec && G >= 4), false);
}

// Fill in (or check) a plan.  `req` may be null (automatic).
lse_status make_plan(const void* x, lse_dtype dt, int64_t B, int64_t N, int64_t row_stride,
                     const DeviceInfo& info, const lse_plan* req, bool with_logprob,
                     lse_plan* plan, bool e16 = false) {
    lse_plan p;
    std::memset(&p, 0, sizeof p);
    const int eb = elem_bytes(dt);
    // Every row starts on a 16-byte boundary when x and the row stride do;
    // otherwise the vector path peels each row's head (and tail) into scalar
    // loads, which needs only element-aligned x.
    const bool aligned = (reinterpret_cast<uintptr_t>(x) % 16u == 0) &&
                         ((row_stride * eb) % 16 == 0);
    const bool peelable = reinterpret_cast<uintptr_t>(x) % static_cast<uintptr_t>(eb) == 0;
    bool vec = peelable;
    if (req && req->vector_bytes != 0) {
        if (req->vector_bytes == 16) {
            if (!peelable) return LSE_ERR_INVALID_ARG;
            vec = true;
        } else if (req->vector_bytes == 1) {
            vec = false;
        } else {
            return LSE_ERR_INVALID_ARG;
        }
    }
    p.vector_bytes = vec ? 16 : 1;
    const int64_t epv = vec ? 16 / eb : 1;
    const int64_t nv = N / epv;  // full slots per row (at most)
    // Slots including the tail vector, and the head slot of peeled rows.
    const int64_t nvt = vec && !aligned ? nv + 2 : ceil_div(N, epv);
    int path = req ? req->path : LSE_PATH_AUTO;

    if (N == 0) {
        if (path != LSE_PATH_AUTO && path != LSE_PATH_EMPTY) return LSE_ERR_INVALID_ARG;
        p.path = LSE_PATH_EMPTY;
        p.splits = 1;
        p.grid = ceil_div(B, 256);
        p.launches = B > 0 ? 1 : 0;
        *plan = p;
        return LSE_OK;
    }
    if (path == LSE_PATH_EMPTY || path < 0 || path > LSE_PATH_ROWTILE ||
        path == LSE_PATH_COLUMNS_WARP || path == LSE_PATH_COLUMNS_CTA)
        return LSE_ERR_INVALID_ARG;

    const int64_t sub_capacity = 32 * kSubwarpWarpSlots;  // slots per row
    // Bulk-copy ring for short back-to-back rows: contiguous 16-byte aligned
    // rows of 16..128 bytes, enough rows for every CTA.  Chosen automatically
    // where it measured faster than the sub-warp mapping (256 MB of rows per
    // width): every width but f32 rows of 2 vectors (sub-warp 6.94 TB/s, ring
    // 6.67); e.g. bf16 rows of 8 vectors 6.58 against 5.99.
    const int64_t row_bytes = N * eb;
    const bool rowtile_ok = vec && aligned && row_stride == N && row_bytes % 16 == 0 &&
                            row_bytes >= 16 && row_bytes <= 128;
    const int64_t row_vecs = row_bytes / 16;
    const bool rowtile_auto = !(eb == 4 && row_vecs == 2);
    // Rows of other widths up to 128 bytes plus one element, still back to
    // back from a 16-byte aligned base: the same ring, one thread per row (row
    // value or token log-probability, f32 exponentials).  Chosen automatically
    // for rows of at least 32 bytes (f32 N = 13: 5.06 against 3.93 TB/s, bf16
    // N = 31: 3.28 against 2.63); shorter rows measured faster on the sub-warp
    // mapping (f32 N = 7: 4.56 against 3.02).
    const int64_t thread_row_max = rowtile_any_thread_row_max_bytes(eb);
    const bool rowtile_any_ok = !rowtile_ok && !e16 && row_stride == N &&
                                row_bytes <= rowtile_any_max_row_bytes() &&
                                reinterpret_cast<uintptr_t>(x) % 16u == 0 &&
                                (!req || req->vector_bytes == 0 ||
                                 req->vector_bytes == (row_bytes <= thread_row_max ? 1 : 16));
    // Lanes per row of that ring: one thread per row up to thread_row_max, else a
    // group of 4-32 lanes, the largest power of two giving each lane >= 8 of
    // the row's 16-byte vectors (f32) or >= 16 (16-bit): the best group size
    // measured for rows of 129 bytes to 4 KB.
    int any_lanes = 1;
    if (row_bytes > thread_row_max) {
        const int64_t per_lane = eb == 4 ? 8 : 16;
        any_lanes = 4;
        while (any_lanes < 32 && ceil_div(row_bytes, 16) >= 2 * any_lanes * per_lane) any_lanes *= 2;
    }
    if (path == LSE_PATH_AUTO) {
        const int64_t chunk_rows = rowtile_ok ? rowtile_rows_per_chunk(static_cast<int>(row_bytes / 16)) : 1;
        const int64_t any_rows =
            rowtile_any_ok ? rowtile_any_rows_per_chunk(static_cast<int>(row_bytes)) : 1;
        if (rowtile_ok && rowtile_auto && B >= chunk_rows * info.sms * rowtile_ctas_per_sm())
            path = LSE_PATH_ROWTILE;
        else if (rowtile_any_ok && row_bytes >= 32 && row_bytes <= thread_row_max &&
                 B >= any_rows * info.sms * rowtile_any_ctas_per_sm())
            path = LSE_PATH_ROWTILE;
        // Back-to-back rows of more than 512 bytes take the grouped ring where
        // the sub-warp mapping cannot hold them, or would leave a quarter or
        // more of its slots empty (a row just past a power of two of slots)
        // and the row is f32 or at most 1.5 KB: measured f32 N = 129 6.14
        // against 5.51 TB/s, N = 257 5.74 / 5.46, N = 520 6.29 / 5.89, bf16
        // N = 520 5.09 / 4.93; with fuller slots the sub-warp mapping wins
        // (f32 N = 300 6.44 / 6.37, bf16 N = 300 4.47 / 4.29), and so it does
        // on longer 16-bit rows (bf16 N = 1025 4.06 / 3.02).
        else if (rowtile_any_ok && row_bytes > 512 && B >= any_rows * info.sms * rowtile_any_ctas_per_sm() &&
                 (nvt > sub_capacity ||
                  (4 * nvt < 3 * subwarp_auto_slots(nvt, vec) && (eb == 4 || row_bytes <= 1536))))
            path = LSE_PATH_ROWTILE;
        else
            path = nvt <= sub_capacity ? LSE_PATH_SUBWARP : LSE_PATH_CTA;
    }
    if (path == LSE_PATH_ROWTILE && !rowtile_ok && rowtile_any_ok) {
        if (req && req->lanes_per_row) {
            const int L = req->lanes_per_row;
            if (row_bytes <= thread_row_max ? L != 1 : (L < 4 || L > 32 || (L & (L - 1)) != 0))
                return LSE_ERR_INVALID_ARG;
            any_lanes = L;
        }
        const int64_t chunks = ceil_div(B, rowtile_any_rows_per_chunk(static_cast<int>(row_bytes)));
        int64_t grid = static_cast<int64_t>(info.sms) * rowtile_any_ctas_per_sm();
        if (grid > chunks) grid = chunks;
        if (grid < 1) grid = 1;
        p.path = LSE_PATH_ROWTILE;
        p.vector_bytes = row_bytes <= thread_row_max ? 1 : 16;
        p.lanes_per_row = any_lanes;
        p.threads = 256;
        p.slots_per_lane = 0;  // any row width
        p.splits = 1;
        p.grid = grid;
        p.launches = B > 0 ? 1 : 0;
        *plan = p;
        return LSE_OK;
    }
    if (path == LSE_PATH_ROWTILE) {
        if (!rowtile_ok) return LSE_ERR_INVALID_ARG;
        const int nvec = static_cast<int>(row_bytes / 16);
        const int64_t chunks = ceil_div(B, rowtile_rows_per_chunk(nvec));
        int64_t grid = static_cast<int64_t>(info.sms) * rowtile_ctas_per_sm();
        if (grid > chunks) grid = chunks;
        p.path = LSE_PATH_ROWTILE;
        p.threads = rowtile_threads();
        p.slots_per_lane = nvec;
        p.splits = 1;
        p.grid = grid;
        p.launches = B > 0 ? 1 : 0;
        *plan = p;
        return LSE_OK;
    }

    if (path == LSE_PATH_SUBWARP) {
        if (nvt > sub_capacity) return LSE_ERR_INVALID_ARG;
        int G = req && req->lanes_per_row ? req->lanes_per_row : subwarp_auto_lanes(nvt, vec);
        if (G < 1 || G > 32 || (G & (G - 1)) != 0) return LSE_ERR_INVALID_ARG;
        int64_t V = ceil_div(nvt, G);
        const bool wide = G == 32 || (vec && G >= 4);  // groups that may hold 8 slots per lane
        if (V > (wide ? kSubwarpWarpSlots : kSubwarpMaxSlots)) return LSE_ERR_INVALID_ARG;
        V = subwarp_slot_count(V, wide, G == 32);
        const int64_t R = V >= 3 ? 1 : (V == 2 ? 2 : 4);
        const int64_t rows_per_warp_iter = (32 / G) * R;
        const int64_t warps = ceil_div(B, rows_per_warp_iter);
        int64_t grid = ceil_div(warps, kSubwarpThreads / 32);
        if (grid > INT_MAX) grid = INT_MAX;  // grid-stride loop covers the rest
        p.path = LSE_PATH_SUBWARP;
        p.lanes_per_row = G;
        p.threads = kSubwarpThreads;
        p.splits = 1;
        p.grid = grid;
        p.slots_per_lane = static_cast<int32_t>(V);
        p.launches = B > 0 ? 1 : 0;
        *plan = p;
        return LSE_OK;
    }

    // CTA / SPLIT: the segment kernel.  Threads per CTA: the most (<= 512)
    // that still give every thread >= 2 batches; at most 128 when rows are
    // plentiful (B >= 16 per SM); with fewer rows than SMs at least 256, or
    // 128 where that is one full batch per thread for the whole row (64 rows
    // of 4096 f32: 2.07 against 2.47 us per call in a CUDA graph, 3.44 against
    // 3.45-3.59 back to back).  Rows are split only when B * threads would not cover half the
    // GPU's resident threads (a split adds a merge kernel).  Splits (measured
    // on 256 MB - 1 GB of few long rows): up to 8x the resident threads, but
    // every thread keeps >= kSplitMinBatches batches (short-lived CTAs cost
    // 5-15 %), and never fewer CTAs than one full wave.
    const int U = vec ? kSegmentBatchVec : kSegmentBatchScalar;
    const int64_t slots = vec ? nv : N;  // slots the segments cover (tail handled separately)
    int T = req && req->threads ? req->threads : 0;
    if (T == 0) {
        T = 512;
        while (T > 32 && slots < 2LL * U * T) T /= 2;
        if (B >= 16LL * info.sms && T > 128) T = 128;
        if (B < info.sms && T < 256) T = slots <= 128LL * U ? 128 : 256;
    }
    int t_index = -1;
    for (int t = 0; t < 5; ++t)
        if (T == (32 << t)) t_index = t;
    if (t_index < 0) return LSE_ERR_INVALID_ARG;
    const int64_t batch = static_cast<int64_t>(T) * U;
    const int64_t resident_threads = static_cast<int64_t>(info.sms) * T *
                                     info.seg_occ[dt][vec ? 1 : 0][t_index];
    int64_t P = 1;
    if (path == LSE_PATH_SPLIT) {
        if (req && req->splits) {
            P = req->splits;
            if (P < 2 || P > (slots > 0 ? slots : 1)) return LSE_ERR_INVALID_ARG;
        } else {
            P = ceil_div(8 * resident_threads, B * T);
            const int64_t max_p = slots / batch;
            if (P > max_p) P = max_p;
            if (P < 2) P = 2;
            if (P > slots) P = slots;
            if (P < 2) return LSE_ERR_INVALID_ARG;
        }
    } else {
        if (req && req->splits > 1) return LSE_ERR_INVALID_ARG;
        if ((!req || req->path == LSE_PATH_AUTO) && 2 * B * T < resident_threads) {
            int64_t want = ceil_div(8 * resident_threads, B * T);
            const int64_t long_p = slots / (kSplitMinBatches * batch);  // long-lived CTAs
            const int64_t wave_p = ceil_div(resident_threads, B * T);    // one full wave
            if (want > long_p) want = long_p > wave_p ? long_p : wave_p;
            const int64_t max_p = slots / (2 * batch);  // >= 2 batches per thread at least
            if (want > max_p) want = max_p;
            if (want >= 2) P = want;
        }
    }
    // Rows shorter than one vector have no full slots: one segment whose CTA
    // reads only the tail.
    const int64_t seg_slots = slots > 0 ? ceil_div(slots, P) : 1;
    P = slots > 0 ? ceil_div(slots, seg_slots) : 1;  // no empty trailing segments
    if (B > INT_MAX / P) return LSE_ERR_INVALID_ARG;  // grid.x = B * P must fit
    p.path = P > 1 ? LSE_PATH_SPLIT : LSE_PATH_CTA;
    p.threads = T;
    p.splits = P;
    p.grid = T == 32 ? ceil_div(B * P, kSegmentWarpUnitsPerCta) : B * P;  // CTAs
    // Split scratch: B*P (m, s) partials, then (token log-probability) the
    // gathered x[b, target[b]] per row.
    p.scratch_bytes = P > 1 ? B * P * static_cast<int64_t>(sizeof(float2)) +
                                  (with_logprob ? B * static_cast<int64_t>(sizeof(float)) : 0)
                            : 0;
    p.launches = B > 0 ? (P > 1 ? 2 : 1) : 0;
    p.segment_slots = seg_slots;
    *plan = p;
    return LSE_OK;
}

// The launch shape of lse_backward for x and dx rows (host logic only):
// fills the mode and a's grid, block, seg_slots and small fields.
lse_status plan_backward(const void* x, int eb, int64_t B, int64_t N, int64_t row_stride,
                         const void* dx, int64_t dx_row_stride, const DeviceInfo& info,
                         BackwardArgs* a, int* mode_out) {
    // 16-byte vectors when every row of x and dx starts on a 16-byte boundary;
    // vectors with a peeled head and tail when each x row and its dx row sit
    // at the same offset from one (same base offset, strides equal mod 16
    // bytes) and hold at least 4 vectors; elements otherwise.  Rows of fewer
    // vectors measured faster as elements (f32 N = 5: 2.8 vs 1.4 TB/s; N = 13:
    // 3.3 vs 3.1), longer ones faster peeled (N = 33: 3.2 vs 2.6; bf16 N = 50257:
    // 6.5 vs 2.7).
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), da = reinterpret_cast<uintptr_t>(dx);
    const bool aligned = xa % 16u == 0 && (row_stride * eb) % 16 == 0 && da % 16u == 0 &&
                         (dx_row_stride * eb) % 16 == 0;
    const bool coaligned = (xa - da) % 16u == 0 && ((row_stride - dx_row_stride) * eb) % 16 == 0;
    int mode = aligned ? kBwdVector : (coaligned && N / (16 / eb) >= 4 ? kBwdPeel : kBwdScalar);
    // Back-to-back rows of x and dx at the same offset from a boundary, not
    // all on one, from one vector up to 16 KB long: one flat array of vectors
    // (1.2-2.4x the peeled rows up to 4 K elements; longer rows peel faster).
    const bool flat_ok = row_stride == N && dx_row_stride == N && coaligned && N >= 16 / eb &&
                         N * eb <= 16384;
    if (flat_ok && !aligned) mode = kBwdFlat;
    const bool vec = mode != kBwdScalar;
    const int64_t epv = vec ? 16 / eb : 1;
    // Slots per row: the tail vector, and with the peel the head slot too.
    const int64_t nvt = mode == kBwdPeel ? N / epv + 2 : ceil_div(N, epv);
    const int U = backward_slots_per_thread();
    const int threads = backward_threads();
    // Threads across a row: just enough for U slots each (not rounded to a
    // power of two: rows of 33-257 peeled slots measured 1.1-1.3x faster).
    const int64_t tx = ceil_div(nvt, U);
    const int TX = tx > threads ? threads : static_cast<int>(tx);
    const int TY = threads / TX;
    const int64_t seg = nvt <= static_cast<int64_t>(TX) * U * 4 ? nvt : static_cast<int64_t>(TX) * U * 4;
    const int64_t P = ceil_div(nvt, seg);
    if (P > INT_MAX) return LSE_ERR_INVALID_ARG;
    int64_t gy = ceil_div(B, TY);
    if (gy > 65535) gy = 65535;  // grid-stride over the remaining rows

    a->seg_slots = seg;
    a->grid = dim3(static_cast<unsigned>(P), static_cast<unsigned>(gy));
    a->block = dim3(static_cast<unsigned>(TX), static_cast<unsigned>(TY));
    // Short rows: flattened (row, slot) pairs, U per thread in flight, at most
    // 4 waves of 256-thread CTAs striding over them.  Up to 2U slots for
    // aligned vectors (f32 rows of 6 and 8 vectors: +1.8 %; 16 vectors: -7 %),
    // up to U with the peel or with elements.
    a->small = nvt <= (mode == kBwdVector ? 2 * U : U);
    if (a->small) {
        int64_t ctas = ceil_div(ceil_div(B * nvt, U), threads);
        const int64_t cap = static_cast<int64_t>(info.sms) * 8 * 4;
        if (ctas > cap) ctas = cap;
        a->grid = dim3(static_cast<unsigned>(ctas));
        a->block = dim3(static_cast<unsigned>(threads));
    }
    if (mode == kBwdFlat) {  // one wave of resident CTAs (4 per SM) striding over the vectors
        int64_t ctas = ceil_div(ceil_div(B * N, 16 / eb),
                                static_cast<int64_t>(threads) * backward_flat_vectors_per_thread());
        const int64_t cap = static_cast<int64_t>(info.sms) * 4;
        if (ctas > cap) ctas = cap;
        if (ctas < 1) ctas = 1;
        a->small = false;
        a->grid = dim3(static_cast<unsigned>(ctas));
        a->block = dim3(static_cast<unsigned>(threads));
    }
    *mode_out = mode;
    return LSE_OK;
}

cudaError_t launch_subwarp(lse_dtype dt, const LaunchArgs& a, bool vec, int G, int V, int64_t grid) {
    const bool tl = a.tl.logprob != nullptr;
    if (a.e16) {
        switch (dt) {
        case LSE_F32: return launch_subwarp_e16_f32(a, vec, G, V, grid);
        case LSE_BF16: return launch_subwarp_e16_bf16(a, vec, G, V, grid);
        default: return launch_subwarp_e16_f16(a, vec, G, V, grid);
        }
    }
    switch (dt) {
    case LSE_F32: return tl ? launch_subwarp_lp_f32(a, vec, G, V, grid) : launch_subwarp_f32(a, vec, G, V, grid);
    case LSE_BF16: return tl ? launch_subwarp_lp_bf16(a, vec, G, V, grid) : launch_subwarp_bf16(a, vec, G, V, grid);
    default: return tl ? launch_subwarp_lp_f16(a, vec, G, V, grid) : launch_subwarp_f16(a, vec, G, V, grid);
    }
}

cudaError_t launch_segment(lse_dtype dt, const LaunchArgs& a, bool vec, int T, int64_t P,
                           int64_t seg_slots, float2* partial, float* xt_buf) {
    const bool tl = a.tl.logprob != nullptr;
    if (a.e16) {
        switch (dt) {
        case LSE_F32: return launch_segment_e16_f32(a, vec, T, P, seg_slots, partial, xt_buf);
        case LSE_BF16: return launch_segment_e16_bf16(a, vec, T, P, seg_slots, partial, xt_buf);
        default: return launch_segment_e16_f16(a, vec, T, P, seg_slots, partial, xt_buf);
        }
    }
    switch (dt) {
    case LSE_F32:
        return tl ? launch_segment_lp_f32(a, vec, T, P, seg_slots, partial, xt_buf)
                  : launch_segment_f32(a, vec, T, P, seg_slots, partial, xt_buf);
    case LSE_BF16:
        return tl ? launch_segment_lp_bf16(a, vec, T, P, seg_slots, partial, xt_buf)
                  : launch_segment_bf16(a, vec, T, P, seg_slots, partial, xt_buf);
    default:
        return tl ? launch_segment_lp_f16(a, vec, T, P, seg_slots, partial, xt_buf)
                  : launch_segment_f16(a, vec, T, P, seg_slots, partial, xt_buf);
    }
}

// N == 0: every row value is log(0) = -inf, and no target is in range.
__global__ void fill_neg_inf_kernel(float* __restrict__ out, float* __restrict__ logprob,
                                    int64_t B) {
    pdl_trigger();
    pdl_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t b = i; b < B; b += stride)
        store_row(out, logprob, b, __int_as_float(kNegInfF32), __int_as_float(0x7fc00000));
}

// One warp per row: lane l folds partials l, l+32, ... in order, then a fixed
// butterfly merges the lanes.  pdl_wait() returns once the segment kernel that
// produced the partials has completed and its writes are visible.
__global__ void __launch_bounds__(32 * kMergeRowsPerCta)
merge_kernel(const float2* __restrict__ partial, const float* __restrict__ xt_buf, int64_t B,
             int64_t P, float* __restrict__ out, float* __restrict__ logprob) {
    pdl_trigger();
    pdl_wait();
    const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= B) return;  // uniform per warp
    Acc a = acc_identity();
    const float2* pr = partial + row * P;
    for (int64_t p = lane; p < P; p += 32) {
        const float2 v = pr[p];
        a = acc_merge(a, Acc{v.x, v.y});
    }
    a = warp_merge<32>(a);
    if (lane == 0) store_row(out, logprob, row, acc_finalize(a), logprob ? xt_buf[row] : 0.0f);
}

}  // namespace

// Argument checks shared by every row entry point (lse_internal.h).
lse_status check_args(const void* x, int dt, int64_t B, int64_t N, int64_t row_stride,
                      const void* out) {
    if (!valid_dtype(dt)) return LSE_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || N < 0 || row_stride < N) return LSE_ERR_INVALID_ARG;
    if (B > 0 && out == nullptr) return LSE_ERR_INVALID_ARG;
    if (B > 0 && N > 0 && x == nullptr) return LSE_ERR_INVALID_ARG;
    // Every load is at least one whole element: x must be element aligned.
    if (B > 0 && N > 0 &&
        reinterpret_cast<uintptr_t>(x) % static_cast<uintptr_t>(elem_bytes(static_cast<lse_dtype>(dt))) != 0)
        return LSE_ERR_INVALID_ARG;
    if (out != nullptr && (reinterpret_cast<uintptr_t>(out) & 3u) != 0) return LSE_ERR_INVALID_ARG;
    // Byte extent of x and of out must fit in int64.
    int64_t extent = 0;
    if (B > 0 && __builtin_mul_overflow(B - 1, row_stride, &extent)) return LSE_ERR_INVALID_ARG;
    if (__builtin_add_overflow(extent, N, &extent)) return LSE_ERR_INVALID_ARG;
    if (__builtin_mul_overflow(extent, static_cast<int64_t>(elem_bytes(static_cast<lse_dtype>(dt))),
                               &extent))
        return LSE_ERR_INVALID_ARG;
    if (B > INT64_MAX / 4) return LSE_ERR_INVALID_ARG;
    return LSE_OK;
}

void record_cuda_error(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();
}

cudaError_t launch_fill_neg_inf(float* out, float* logprob, int64_t B, cudaStream_t stream) {
    int64_t grid = ceil_div(B, 256);
    if (grid > 65536) grid = 65536;
    return launch_pdl(fill_neg_inf_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), stream, out,
                      logprob, B);
}

cudaError_t launch_merge(const float2* partial, const float* xt_buf, int64_t B, int64_t P,
                         float* out, float* logprob, cudaStream_t stream) {
    return launch_pdl(merge_kernel, dim3(static_cast<unsigned>(ceil_div(B, kMergeRowsPerCta))),
                      dim3(32 * kMergeRowsPerCta), stream, partial, xt_buf, B, P, out, logprob);
}

}  // namespace lse

using namespace lse;

extern "C" {

const char* lse_status_string(lse_status status) {
    switch (status) {
    case LSE_OK: return "ok";
    case LSE_ERR_INVALID_ARG: return "invalid argument";
    case LSE_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case LSE_ERR_ALLOC: return "device scratch allocation failed";
    case LSE_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
    }
}

lse_status lse_last_cuda_error(int* cuda_err) {
    if (cuda_err == nullptr) return LSE_ERR_INVALID_ARG;
    *cuda_err = g_last_cuda_error;
    return LSE_OK;
}

lse_status lse_plan_query(const void* x, lse_dtype dtype, int64_t B, int64_t N,
                          int64_t row_stride, lse_plan* plan) {
    if (plan == nullptr) return LSE_ERR_INVALID_ARG;
    // Only the shape is checked here: stand-in non-null pointers for x and out.
    const void* stand_in = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
    lse_status st = check_args(x ? x : stand_in, dtype, B, N, row_stride, stand_in);
    if (st != LSE_OK) return st;
    int dev = 0;
    const DeviceInfo* info = nullptr;
    if ((st = device_info(&dev, &info)) != LSE_OK) return st;
    return make_plan(x, dtype, B, N, row_stride, *info, nullptr, false, plan);
}

}  // extern "C"

namespace {

// The forward pass behind lse_forward_plan, lse_token_logprob_plan and
// lse_forward16 (e16: reduced-bit exponentials).  `out` may be null when
// `tl.logprob` is set; arguments are already checked.
lse_status run_forward(const void* x, lse_dtype dtype, int64_t B, int64_t N, int64_t row_stride,
                       float* out, TokenLogprob tl, cudaStream_t stream, lse_plan* plan,
                       lse_event_t ev_begin, lse_event_t ev_end, bool e16 = false) {
    if (B == 0) return LSE_OK;  // no work, no device access
    int dev = 0;
    const DeviceInfo* info = nullptr;
    lse_status st = device_info(&dev, &info);
    if (st != LSE_OK) return st;
    lse_plan p;
    if ((st = make_plan(x, dtype, B, N, row_stride, *info, plan, tl.logprob != nullptr, &p, e16)) !=
        LSE_OK)
        return st;
    if (plan) *plan = p;

    const LaunchArgs a{x, B, N, row_stride, out, stream, tl, e16};
    cudaError_t e = cudaSuccess;
    char* scratch = nullptr;
    if (p.scratch_bytes > 0) {
        e = scratch_alloc(*info, reinterpret_cast<void**>(&scratch),
                          static_cast<size_t>(p.scratch_bytes), stream);
        if (e != cudaSuccess) return cuda_fail(e, LSE_ERR_ALLOC);
    }
    float2* partial = reinterpret_cast<float2*>(scratch);
    float* xt_buf = tl.logprob && scratch
                        ? reinterpret_cast<float*>(scratch + B * p.splits * sizeof(float2))
                        : nullptr;
    if (ev_begin && (e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev_begin), stream)) != cudaSuccess)
        goto fail;
    switch (p.path) {
    case LSE_PATH_EMPTY:
        e = launch_fill_neg_inf(out, tl.logprob, B, stream);
        break;
    case LSE_PATH_SUBWARP:
        e = launch_subwarp(dtype, a, p.vector_bytes == 16, p.lanes_per_row, p.slots_per_lane, p.grid);
        break;
    case LSE_PATH_ROWTILE:
        e = launch_rowtile(dtype, p.slots_per_lane, p.lanes_per_row, a, static_cast<int>(p.grid));
        break;
    default:
        e = launch_segment(dtype, a, p.vector_bytes == 16, p.threads, p.splits, p.segment_slots,
                           partial, xt_buf);
        break;
    }
    if (e != cudaSuccess) goto fail;
    if (ev_end && (e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev_end), stream)) != cudaSuccess)
        goto fail;
    if (p.path == LSE_PATH_SPLIT) {
        e = launch_merge(partial, xt_buf, B, p.splits, out, tl.logprob, stream);
        if (e != cudaSuccess) goto fail;
    }
    if (scratch && (e = cudaFreeAsync(scratch, stream)) != cudaSuccess) return cuda_fail(e);
    return LSE_OK;

fail:
    if (scratch) cudaFreeAsync(scratch, stream);
    return cuda_fail(e);
}

}  // namespace

extern "C" {

lse_status lse_forward_plan(const void* x, lse_dtype dtype, int64_t B, int64_t N,
                            int64_t row_stride, float* out, lse_stream_t stream,
                            lse_plan* plan, lse_event_t ev_begin, lse_event_t ev_end) {
    const lse_status st = check_args(x, dtype, B, N, row_stride, out);
    if (st != LSE_OK) return st;
    return run_forward(x, dtype, B, N, row_stride, out, TokenLogprob{},
                       reinterpret_cast<cudaStream_t>(stream), plan, ev_begin, ev_end);
}

lse_status lse_forward16(const void* x, lse_dtype dtype, int64_t B, int64_t N, int64_t row_stride,
                         float* out, lse_stream_t stream, lse_plan* plan) {
    const lse_status st = check_args(x, dtype, B, N, row_stride, out);
    if (st != LSE_OK) return st;
    return run_forward(x, dtype, B, N, row_stride, out, TokenLogprob{},
                       reinterpret_cast<cudaStream_t>(stream), plan, nullptr, nullptr, true);
}

lse_status lse_token_logprob_plan(const void* x, lse_dtype dtype, int64_t B, int64_t N,
                                  int64_t row_stride, const int64_t* target, float* logprob,
                                  float* lse_out, lse_stream_t stream, lse_plan* plan) {
    const void* stand_in = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
    lse_status st = check_args(x, dtype, B, N, row_stride, lse_out ? lse_out : stand_in);
    if (st != LSE_OK) return st;
    if (B > 0 && (target == nullptr || logprob == nullptr)) return LSE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(target) & 7u) != 0 ||
        (reinterpret_cast<uintptr_t>(logprob) & 3u) != 0)
        return LSE_ERR_INVALID_ARG;
    TokenLogprob tl;
    tl.target = target;
    tl.logprob = logprob;
    return run_forward(x, dtype, B, N, row_stride, lse_out, tl,
                       reinterpret_cast<cudaStream_t>(stream), plan, nullptr, nullptr);
}

lse_status lse_backward(const void* x, lse_dtype dtype, int64_t B, int64_t N, int64_t row_stride,
                        const float* lse_in, const float* grad, void* dx, int64_t dx_row_stride,
                        lse_stream_t stream) {
    const void* stand_in = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
    lse_status st = check_args(x, dtype, B, N, row_stride, stand_in);
    if (st != LSE_OK) return st;
    if (dx_row_stride < N) return LSE_ERR_INVALID_ARG;
    const int eb = elem_bytes(dtype);
    int64_t extent = 0;
    if (B > 0 && __builtin_mul_overflow(B - 1, dx_row_stride, &extent)) return LSE_ERR_INVALID_ARG;
    if (__builtin_add_overflow(extent, N, &extent) ||
        __builtin_mul_overflow(extent, static_cast<int64_t>(eb), &extent))
        return LSE_ERR_INVALID_ARG;
    if (B == 0 || N == 0) return LSE_OK;
    if (lse_in == nullptr || grad == nullptr || dx == nullptr) return LSE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(lse_in) & 3u) || (reinterpret_cast<uintptr_t>(grad) & 3u) ||
        (reinterpret_cast<uintptr_t>(dx) % static_cast<uintptr_t>(eb)))
        return LSE_ERR_INVALID_ARG;
    int dev = 0;
    const DeviceInfo* info = nullptr;
    if ((st = device_info(&dev, &info)) != LSE_OK) return st;

    BackwardArgs a;
    int mode = kBwdScalar;
    if ((st = plan_backward(x, eb, B, N, row_stride, dx, dx_row_stride, *info, &a, &mode)) != LSE_OK)
        return st;
    a.x = x;
    a.B = B;
    a.N = N;
    a.row_stride = row_stride;
    a.lse = lse_in;
    a.grad = grad;
    a.dx = dx;
    a.dx_row_stride = dx_row_stride;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = launch_backward(dtype, mode, a);
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

namespace {

// The plan of lse_forward_strided for R > 0 (host logic only): load width,
// warps per column tile, row splits and grid.  occ(dtype, vec, warps per
// tile) gives the resident CTAs per SM of a column-kernel variant.
lse_status plan_columns(const void* x, lse_dtype dtype, int64_t A, int64_t R, int64_t C,
                        int64_t stride_a, int64_t stride_r, int sms, int (*occ)(int, bool, int),
                        const lse_plan* req, lse_plan* plan) {
    const int eb = elem_bytes(dtype);
    const int64_t outputs = A * C;
    const int rpath = req ? req->path : LSE_PATH_AUTO;
    lse_plan p;
    std::memset(&p, 0, sizeof p);
    const int64_t epv16 = 16 / eb;
    const bool aligned = reinterpret_cast<uintptr_t>(x) % 16u == 0 && (stride_r * eb) % 16 == 0 &&
                         (stride_a * eb) % 16 == 0 && C % epv16 == 0;
    bool vec = aligned;
    if (req && req->vector_bytes) {
        if (req->vector_bytes == 16) {
            if (!aligned) return LSE_ERR_INVALID_ARG;
        } else if (req->vector_bytes != 1) {
            return LSE_ERR_INVALID_ARG;
        }
        vec = req->vector_bytes == 16;
    }
    // Short reductions of the vector layout: a thread per 16-byte column
    // vector folds all R rows from registers (automatic for R <= 8 unless a
    // split or warps per tile are asked for).
    const bool short_ok = vec && R <= kColsShortMaxRows;
    if (rpath == LSE_PATH_COLUMNS_SHORT ||
        (rpath == LSE_PATH_AUTO && short_ok && (!req || (req->splits <= 1 && req->lanes_per_row == 0)))) {
        if (!short_ok || (req && (req->splits > 1 || req->lanes_per_row != 0))) return LSE_ERR_INVALID_ARG;
        const int64_t nvec = outputs / epv16;
        int64_t grid = ceil_div(nvec, kColsShortThreads);
        const int64_t cap = static_cast<int64_t>(sms) * 32;  // 4 waves of 8 CTAs per SM
        if (grid > cap) grid = cap;
        p.path = LSE_PATH_COLUMNS_SHORT;
        p.vector_bytes = 16;
        p.threads = kColsShortThreads;
        p.lanes_per_row = 0;
        p.splits = 1;
        p.segment_slots = R;
        p.grid = grid;
        p.scratch_bytes = 0;
        p.launches = 1;
        *plan = p;
        return LSE_OK;
    }
    const int64_t wtiles = ceil_div(C, cols_columns_per_warp(vec, dtype));  // 32-lane column tiles
    int64_t units = 0;  // (a, tile) pairs
    if (__builtin_mul_overflow(A, wtiles, &units)) return LSE_ERR_INVALID_ARG;
    // Resident warps of the single-warp-tile variant (used to pick WT).
    const int64_t resident_warps = static_cast<int64_t>(sms) * cols_warps_per_cta(1) *
                                   occ(dtype, vec, 1);
    const int64_t batch = cols_rows_per_batch(vec);
    // Warps per tile (measured on 256 MB of [A, R, C] for R = 2..4096, C =
    // 128..16384): one warp walks each tile up to R = 64, or whenever the
    // units alone give every resident warp two; 2 warps up to R = 128 and 4
    // beyond share a tile (a shared-memory merge is cheaper than a split);
    // row splits below fill the GPU only where that is still not enough.
    int WT = req && req->lanes_per_row ? req->lanes_per_row : 0;
    int path = rpath;
    if (path == LSE_PATH_COLUMNS_WARP) {
        if (WT > 1) return LSE_ERR_INVALID_ARG;
        WT = 1;
    }
    // Narrow C (32-lane tiles would leave a quarter or more of their lanes
    // without a column) takes tiles of 16 or 8 lanes.  16-bit ones keep one
    // warp per tile at any R (with row splits): bf16 [8192, 128, 128] 4.55
    // against 2.14 TB/s with two warps per 32-lane tile, and one warp still
    // beats 2 or 4 per narrow tile at R = 128-4096 (C = 64, 192: 0.87-0.95
    // against 0.77-0.85 of the copy peak).  f32 narrow tiles take warps per
    // tile by the rule for wide ones: [A, R, 64] f32 at R = 256 / 512 / 4096
    // 0.978 / 0.956 / 0.933 with 4 warps against 0.856 / 0.862 / 0.859 with
    // one warp and splits; C = 192 0.92-0.97 against 0.87-0.93.
    const bool narrow16 = eb != 4 && cols_lanes_per_tile(dtype, vec, C, 1) != 32;
    if (WT == 0) {
        if (path == LSE_PATH_COLUMNS_CTA)
            WT = 8;
        else
            WT = (R <= 64 || units >= 2 * resident_warps || narrow16) ? 1 : (R <= 128 ? 2 : 4);
    }
    if (WT != 1 && WT != 2 && WT != 4 && WT != 8) return LSE_ERR_INVALID_ARG;
    path = WT == 1 ? LSE_PATH_COLUMNS_WARP : LSE_PATH_COLUMNS_CTA;
    const int W = cols_warps_per_cta(WT);
    // Narrow C: 16- or 8-lane tiles, 2 or 4 per warp (any warps per tile).
    const int lpt = cols_lanes_per_tile(dtype, vec, C, 1);
    if (lpt != 32) units = A * ceil_div(C, cols_columns_per_warp(vec, dtype) * lpt / 32);
    int64_t gx = ceil_div(units, W / WT * (32 / lpt));  // CTAs if each took one group of units
    const int64_t rows_per_warp_batch = WT * batch;
    const int64_t resident_ctas = static_cast<int64_t>(sms) * occ(dtype, vec, WT);
    int64_t P = req ? req->splits : 0;
    if (P == 0) {
        // No split while the CTAs already fill half the resident slots (a
        // split costs a merge kernel); otherwise as many splits as fit in ONE
        // wave of resident CTAs -- a partial second wave of these long-lived
        // CTAs would nearly double the time -- keeping >= 4 batches per warp.
        const int64_t base = gx;
        P = 2 * base >= resident_ctas ? 1 : resident_ctas / base;
        const int64_t max_p = R / (4 * rows_per_warp_batch);
        if (P > max_p) P = max_p;
        if (P < 1) P = 1;
    }
    if (P > R) return LSE_ERR_INVALID_ARG;
    const int64_t rows_per_split = ceil_div(R, P);
    P = ceil_div(R, rows_per_split);
    if (P > 65535) return LSE_ERR_INVALID_ARG;
    // Beyond a few waves CTAs loop over the units instead of being launched
    // one per group (tiny groups made the launch itself the bottleneck).
    if (gx > 4 * resident_ctas) gx = 4 * resident_ctas;
    if (P > 1 && outputs > INT64_MAX / (8 * P)) return LSE_ERR_INVALID_ARG;
    p.path = path;
    p.vector_bytes = vec ? 16 : 1;
    p.threads = 32 * W;
    p.lanes_per_row = WT;
    p.splits = P;
    p.segment_slots = rows_per_split;
    p.grid = gx * P;
    p.scratch_bytes = P > 1 ? outputs * P * static_cast<int64_t>(sizeof(float2)) : 0;
    p.launches = P > 1 ? 2 : 1;
    *plan = p;
    return LSE_OK;
}

// Elements spanned by an [A, R, C] layout with the given strides (0 when
// empty), or -1 when its byte extent overflows.
int64_t strided_extent(int64_t A, int64_t R, int64_t C, int64_t sa, int64_t sr, int eb) {
    if (A == 0 || R == 0 || C == 0) return 0;
    int64_t extent = 0, t = 0;
    if (__builtin_mul_overflow(A - 1, sa, &extent) || __builtin_mul_overflow(R - 1, sr, &t) ||
        __builtin_add_overflow(extent, t, &extent) || __builtin_add_overflow(extent, C, &extent) ||
        __builtin_mul_overflow(extent, static_cast<int64_t>(eb), &t))
        return -1;
    return extent;
}

}  // namespace

lse_status lse_backward_strided(const void* x, lse_dtype dtype, int64_t A, int64_t R, int64_t C,
                                int64_t stride_a, int64_t stride_r, const float* lse_in,
                                const float* grad, void* dx, int64_t dx_stride_a,
                                int64_t dx_stride_r, lse_stream_t stream) {
    if (!valid_dtype(dtype)) return LSE_ERR_UNSUPPORTED_DTYPE;
    if (A < 0 || R < 0 || C < 0 || stride_a < 0 || stride_r < 0 || dx_stride_a < 0 ||
        dx_stride_r < 0)
        return LSE_ERR_INVALID_ARG;
    const int eb = elem_bytes(dtype);
    int64_t outputs = 0;
    if (__builtin_mul_overflow(A, C, &outputs) || outputs > INT64_MAX / 8) return LSE_ERR_INVALID_ARG;
    if (strided_extent(A, R, C, stride_a, stride_r, eb) < 0 ||
        strided_extent(A, R, C, dx_stride_a, dx_stride_r, eb) < 0)
        return LSE_ERR_INVALID_ARG;
    if (A == 0 || R == 0 || C == 0) return LSE_OK;
    if (x == nullptr || lse_in == nullptr || grad == nullptr || dx == nullptr)
        return LSE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(lse_in) & 3u) || (reinterpret_cast<uintptr_t>(grad) & 3u) ||
        (reinterpret_cast<uintptr_t>(x) % static_cast<uintptr_t>(eb)) ||
        (reinterpret_cast<uintptr_t>(dx) % static_cast<uintptr_t>(eb)))
        return LSE_ERR_INVALID_ARG;
    int dev = 0;
    const DeviceInfo* info = nullptr;
    lse_status st = device_info(&dev, &info);
    if (st != LSE_OK) return st;

    const int64_t epv16 = 16 / eb;
    const auto al16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16u == 0; };
    const bool vec = al16(x) && al16(dx) && C % epv16 == 0 && (stride_a * eb) % 16 == 0 &&
                     (stride_r * eb) % 16 == 0 && (dx_stride_a * eb) % 16 == 0 &&
                     (dx_stride_r * eb) % 16 == 0;
    // Warps per unit: a warp takes a whole unit when rows are few (one batch
    // of rows per warp would leave a shared unit's warps idle) or C is narrow
    // (16- or 8-lane tiles, as the column kernel takes them), else the CTA's
    // warps share it.  Row splits only while the units cannot cover the GPU
    // 4x, keeping >= 2 batches per warp; beyond 4 waves CTAs loop over units.
    const int64_t W = backward_strided_warps();
    const int64_t U = backward_slots_per_thread();
    const int narrow_lanes = cols_lanes_per_tile(dtype, vec, C, 1);
    const int wpu = R <= 2 * W * U || narrow_lanes != 32 ? 1 : static_cast<int>(W);
    const int lpt = wpu == 1 ? narrow_lanes : 32;
    const int64_t wtiles = ceil_div(C, lpt * (vec ? epv16 : 1));  // column tiles of lpt lanes
    int64_t units = 0;  // (a, tile) pairs
    if (__builtin_mul_overflow(A, wtiles, &units)) return LSE_ERR_INVALID_ARG;
    const int64_t upc = W / wpu * (32 / lpt);  // units per CTA
    const int64_t resident_ctas = static_cast<int64_t>(info->sms) * (64 / W);
    int64_t gx = ceil_div(units, upc);
    int64_t P = ceil_div(4 * resident_ctas, gx);
    const int64_t max_p = ceil_div(R, 2 * wpu * U);
    if (P > max_p) P = max_p;
    if (P > 65535) P = 65535;
    if (P < 1) P = 1;
    const int64_t rows_per_split = ceil_div(R, P);
    P = ceil_div(R, rows_per_split);
    if (gx > 4 * resident_ctas) gx = 4 * resident_ctas;

    BackwardStridedArgs a;
    a.x = x;
    a.A = A;
    a.R = R;
    a.C = C;
    a.stride_a = stride_a;
    a.stride_r = stride_r;
    a.lse = lse_in;
    a.grad = grad;
    a.dx = dx;
    a.dx_stride_a = dx_stride_a;
    a.dx_stride_r = dx_stride_r;
    a.rows_per_split = rows_per_split;
    a.warps_per_unit = wpu;
    a.lanes_per_tile = lpt;
    a.grid = dim3(static_cast<unsigned>(gx), 1, static_cast<unsigned>(P));
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = launch_backward_strided(dtype, vec, a);
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

lse_status lse_forward_strided(const void* x, lse_dtype dtype, int64_t A, int64_t R, int64_t C,
                               int64_t stride_a, int64_t stride_r, float* out,
                               lse_stream_t stream_, lse_plan* plan) {
    if (!valid_dtype(dtype)) return LSE_ERR_UNSUPPORTED_DTYPE;
    if (A < 0 || R < 0 || C < 0 || stride_a < 0 || stride_r < 0) return LSE_ERR_INVALID_ARG;
    const int eb = elem_bytes(dtype);
    int64_t outputs = 0, extent = 0, t = 0;
    if (__builtin_mul_overflow(A, C, &outputs) || outputs > INT64_MAX / 8) return LSE_ERR_INVALID_ARG;
    if (A > 0 && R > 0 && C > 0) {
        if (__builtin_mul_overflow(A - 1, stride_a, &extent) ||
            __builtin_mul_overflow(R - 1, stride_r, &t) || __builtin_add_overflow(extent, t, &extent) ||
            __builtin_add_overflow(extent, C, &extent) ||
            __builtin_mul_overflow(extent, static_cast<int64_t>(eb), &extent))
            return LSE_ERR_INVALID_ARG;
    }
    const lse_plan* req = plan;
    const int rpath = req ? req->path : LSE_PATH_AUTO;
    if (rpath != LSE_PATH_AUTO && rpath != LSE_PATH_COLUMNS_WARP && rpath != LSE_PATH_COLUMNS_CTA &&
        rpath != LSE_PATH_COLUMNS_SHORT && rpath != LSE_PATH_EMPTY)
        return LSE_ERR_INVALID_ARG;
    if (req && req->splits < 0) return LSE_ERR_INVALID_ARG;
    if (outputs == 0) return LSE_OK;
    if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 3u)) return LSE_ERR_INVALID_ARG;
    if (R > 0 && (x == nullptr || reinterpret_cast<uintptr_t>(x) % static_cast<uintptr_t>(eb) != 0))
        return LSE_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    const DeviceInfo* info = nullptr;
    lse_status st = device_info(&dev, &info);
    if (st != LSE_OK) return st;
    lse_plan p;
    std::memset(&p, 0, sizeof p);
    if (R == 0) {
        if (rpath != LSE_PATH_AUTO && rpath != LSE_PATH_EMPTY) return LSE_ERR_INVALID_ARG;
        p.path = LSE_PATH_EMPTY;
        p.splits = 1;
        p.launches = 1;
        p.grid = ceil_div(outputs, 256);
        if (plan) *plan = p;
        const cudaError_t e = launch_fill_neg_inf(out, nullptr, outputs, stream);
        return e == cudaSuccess ? LSE_OK : cuda_fail(e);
    }
    if (rpath == LSE_PATH_EMPTY) return LSE_ERR_INVALID_ARG;
    if ((st = plan_columns(x, dtype, A, R, C, stride_a, stride_r, info->sms, cols_occupancy, req,
                           &p)) != LSE_OK)
        return st;
    if (plan) *plan = p;
    if (p.path == LSE_PATH_COLUMNS_SHORT) {
        StridedArgs a;
        std::memset(&a, 0, sizeof a);
        a.x = x;
        a.A = A;
        a.R = R;
        a.C = C;
        a.stride_a = stride_a;
        a.stride_r = stride_r;
        a.out = out;
        a.P = 1;
        a.grid = dim3(static_cast<unsigned>(p.grid));
        a.stream = stream;
        const cudaError_t e = launch_cols_short(dtype, a);
        return e == cudaSuccess ? LSE_OK : cuda_fail(e);
    }
    const bool vec = p.vector_bytes == 16;
    const int WT = p.lanes_per_row;
    const int64_t P = p.splits;
    const int64_t rows_per_split = p.segment_slots;
    const int64_t gx = p.grid / P;

    float2* scratch = nullptr;
    cudaError_t e = cudaSuccess;
    if (P > 1) {
        e = scratch_alloc(*info, reinterpret_cast<void**>(&scratch),
                          static_cast<size_t>(p.scratch_bytes), stream);
        if (e != cudaSuccess) return cuda_fail(e, LSE_ERR_ALLOC);
    }
    StridedArgs a;
    a.x = x;
    a.A = A;
    a.R = R;
    a.C = C;
    a.stride_a = stride_a;
    a.stride_r = stride_r;
    a.rows_per_split = rows_per_split;
    a.out = out;
    a.partial = scratch;
    a.P = P;
    a.warps_per_tile = WT;
    a.grid = dim3(static_cast<unsigned>(gx), 1, static_cast<unsigned>(P));
    a.stream = stream;
    e = launch_cols(dtype, vec, a);
    if (e == cudaSuccess && P > 1) e = launch_merge_columns(scratch, outputs, P, out, stream);
    if (scratch) {
        const cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e == cudaSuccess) e = ef;
    }
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

lse_status lse_token_logprob(const void* x, lse_dtype dtype, int64_t B, int64_t N,
                             int64_t row_stride, const int64_t* target, float* logprob,
                             float* lse_out, lse_stream_t stream) {
    return lse_token_logprob_plan(x, dtype, B, N, row_stride, target, logprob, lse_out, stream,
                                  nullptr);
}

lse_status lse_forward(const void* x, lse_dtype dtype, int64_t B, int64_t N, int64_t row_stride,
                       float* out, lse_stream_t stream) {
    return lse_forward_plan(x, dtype, B, N, row_stride, out, stream, nullptr, nullptr, nullptr);
}

// Device address of a page-locked (registered or cudaHostAlloc'ed) host
// buffer, or nullptr for pageable memory.
static void* mapped_host_pointer(const void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of an unknown pointer
        return nullptr;
    }
    return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}

lse_status lse_forward_host(const void* x_host, lse_dtype dtype, int64_t B, int64_t N,
                            int64_t row_stride, float* out_host, lse_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    lse_status st = check_args(x_host, dtype, B, N, row_stride, out_host);
    if (st != LSE_OK) return st;
    if (B == 0) return LSE_OK;
    int dev = 0;
    const DeviceInfo* info = nullptr;
    if ((st = device_info(&dev, &info)) != LSE_OK) return st;
    const size_t x_bytes =
        N > 0 ? static_cast<size_t>(((B - 1) * row_stride + N) * elem_bytes(dtype)) : 0;
    const size_t out_bytes = static_cast<size_t>(B) * sizeof(float);

    // Page-locked buffers are used in place: the kernel streams x over the
    // host link and writes out directly.  Pageable ones go through pooled
    // device buffers with cudaMemcpyAsync.
    const void* x_mapped = x_bytes ? mapped_host_pointer(x_host) : nullptr;
    float* out_mapped = static_cast<float*>(mapped_host_pointer(out_host));
    const void* d_x = x_mapped;
    float* d_out = out_mapped;
    void* x_staged = nullptr;
    float* out_staged = nullptr;
    cudaError_t e = cudaSuccess;
    if (x_bytes && !x_mapped) {
        if ((e = scratch_alloc(*info, &x_staged, x_bytes, stream)) != cudaSuccess)
            return cuda_fail(e, LSE_ERR_ALLOC);
        d_x = x_staged;
    }
    if (!out_mapped) {
        if ((e = scratch_alloc(*info, reinterpret_cast<void**>(&out_staged), out_bytes, stream)) !=
            cudaSuccess) {
            if (x_staged) cudaFreeAsync(x_staged, stream);
            return cuda_fail(e, LSE_ERR_ALLOC);
        }
        d_out = out_staged;
    }
    if (x_staged) e = cudaMemcpyAsync(x_staged, x_host, x_bytes, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) {
        st = lse_forward(d_x, dtype, B, N, row_stride, d_out, stream_);
        if (st == LSE_OK && out_staged)
            e = cudaMemcpyAsync(out_host, out_staged, out_bytes, cudaMemcpyDeviceToHost, stream);
    }
    if (x_staged) cudaFreeAsync(x_staged, stream);
    if (out_staged) cudaFreeAsync(out_staged, stream);
    const cudaError_t es = cudaStreamSynchronize(stream);
    if (st != LSE_OK) return st;
    if (e != cudaSuccess) return cuda_fail(e);
    if (es != cudaSuccess) return cuda_fail(es);
    return LSE_OK;
}

lse_status lse_set_wait_limit(uint32_t polls) {
    set_stage_wait_polls(polls);
    return LSE_OK;
}

lse_status lse_wait_timeouts(unsigned long long* count) {
    if (count == nullptr) return LSE_ERR_INVALID_ARG;
    const cudaError_t e = read_wait_timeouts(count);
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

lse_status lse_trim_memory(void) {
    int dev = 0;
    const DeviceInfo* info = nullptr;
    lse_status st = device_info(&dev, &info);
    if (st != LSE_OK) return st;
    const cudaError_t e = cudaMemPoolTrimTo(info->pool, 0);
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

}  // extern "C"
