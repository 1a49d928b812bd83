// lse_noalloc.cu -- lse_forward_split_static: the split-row mapping with its
// scratch in a fixed, statically allocated device array instead of memory
// allocated per call.
//
// Who needs it: callers that must not allocate device memory while they run.
// Examples are code that runs under a strict memory budget reserved up front,
// real-time or embedded loops where an allocator call (and the synchronisation
// or page mapping it can trigger) is not allowed, and hosts whose allocator is
// owned by another runtime that must see every byte.  This entry point calls
// no cudaMalloc / cudaFree / stream-ordered allocator and no allocating library
// routine.
//
// The scratch is kScratchPartials (m, s) pairs (1 MiB) in a file-scope
// __device__ array.  Every GPU that loads the library holds that 1 MiB until
// the process exits.  Host code cannot use the array's name as a device
// address, so the first call on each device, with that device current, looks
// the address up with cudaGetSymbolAddress and caches it; that first call
// should therefore happen before any stream capture.  All calls share the one
// array: two calls whose kernels overlap on the GPU (different streams, or
// different host threads without ordering) race and give wrong results.
// Calls on one stream are ordered and safe.  Nothing in the array needs to
// start at zero: each call writes every partial slot it later reads.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/lse.h"
#include "lse_internal.h"

namespace lse {
namespace {

constexpr int64_t kScratchPartials = LSE_STATIC_SCRATCH_BYTES / static_cast<int64_t>(sizeof(float2));
constexpr int kMaxDevices = 64;
constexpr int kThreads = 256;
constexpr int kBatchVec = 8;       // 16-byte slots per thread per batch
constexpr int kBatchScalar = 16;   // element slots per thread per batch

static __device__ __align__(256) float2 g_static_partials[kScratchPartials];

struct StaticScratch {
    bool ready = false;
    float2* ptr = nullptr;  // device address of g_static_partials on this device
    int sms = 0;
    int occ[3][2] = {};     // resident 256-thread segment CTAs per SM [dtype][vec]
};

std::mutex g_mutex;
StaticScratch g_devices[kMaxDevices];

lse_status fail(cudaError_t e) {
    record_cuda_error(e);
    return LSE_ERR_CUDA;
}

int occupancy(int dt, bool vec) {
    switch (dt) {
    case LSE_F32: return segment_occupancy_f32(vec, kThreads);
    case LSE_BF16: return segment_occupancy_bf16(vec, kThreads);
    default: return segment_occupancy_f16(vec, kThreads);
    }
}

// Once per device, with the device current: the array's device address.
lse_status setup(const StaticScratch** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(e);
    if (dev < 0 || dev >= kMaxDevices) return LSE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    StaticScratch& s = g_devices[dev];
    if (!s.ready) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_partials);
        if (e != cudaSuccess) return fail(e);
        e = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(e);
        for (int dt = 0; dt < 3; ++dt)
            for (int v = 0; v < 2; ++v) {
                const int o = occupancy(dt, v != 0);
                s.occ[dt][v] = o > 0 ? o : 1;
            }
        s.ptr = static_cast<float2*>(p);
        s.ready = true;
    }
    *out = &s;
    return LSE_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace lse

using namespace lse;

extern "C" lse_status lse_forward_split_static(const void* x, lse_dtype dtype, int64_t B,
                                               int64_t N, int64_t row_stride, float* out,
                                               lse_stream_t stream_) {
    lse_status st = check_args(x, dtype, B, N, row_stride, out);
    if (st != LSE_OK) return st;
    if (B == 0) return LSE_OK;
    if (B > kScratchPartials / 2) return LSE_ERR_INVALID_ARG;  // needs >= 2 partials per row
    const int eb = dtype == LSE_F32 ? 4 : 2;
    // 16-byte vectors; rows off a 16-byte boundary peel their head and tail
    // into element loads, unless they hold fewer than two vectors.
    const bool aligned = (reinterpret_cast<uintptr_t>(x) % 16u == 0) && ((row_stride * eb) % 16 == 0);
    const bool vec = aligned || N / (16 / eb) >= 2;
    const int64_t slots = vec ? N / (16 / eb) : N;  // segments cover these; head and tail ride along
    if (slots < 2) return LSE_ERR_INVALID_ARG;     // too short to split

    const StaticScratch* s = nullptr;
    st = setup(&s);
    if (st != LSE_OK) return st;

    // Splits per row: cover the GPU ~4 times over, >= 1 batch per segment,
    // >= 2 segments, and within the static array.
    const int64_t batch = static_cast<int64_t>(kThreads) * (vec ? kBatchVec : kBatchScalar);
    const int64_t resident = static_cast<int64_t>(s->sms) * kThreads * s->occ[dtype][vec ? 1 : 0];
    int64_t P = ceil_div(4 * resident, B * kThreads);
    if (P > slots / batch) P = slots / batch;
    if (P > kScratchPartials / B) P = kScratchPartials / B;
    if (P > slots) P = slots;
    if (P < 2) P = 2;
    const int64_t seg_slots = ceil_div(slots, P);
    P = ceil_div(slots, seg_slots);

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const LaunchArgs a{x, B, N, row_stride, out, stream, TokenLogprob{}, false};
    cudaError_t e;
    switch (dtype) {
    case LSE_F32: e = launch_segment_f32(a, vec, kThreads, P, seg_slots, s->ptr, nullptr); break;
    case LSE_BF16: e = launch_segment_bf16(a, vec, kThreads, P, seg_slots, s->ptr, nullptr); break;
    default: e = launch_segment_f16(a, vec, kThreads, P, seg_slots, s->ptr, nullptr); break;
    }
    if (e == cudaSuccess) e = launch_merge(s->ptr, nullptr, B, P, out, nullptr, stream);
    if (e != cudaSuccess) return fail(e);
    return LSE_OK;
}
