// lse_edges.cuh -- one-sided masks for the 16-byte vectors that hold a row's
// first and last bytes (sm_103a).
#pragma once

#include <cstdint>

#include "lse_device.cuh"

namespace lse {

// One-sided edge masks of a 16-byte vector held as 4 words: the elements in
// its first nb bytes (a row's first vector, nb = the row's offset from the
// 16-byte boundary) or from byte t on (its last vector, t = the row's bytes in
// it) set to -inf.  Element boundaries fall on nb and t, so a word's keep mask
// is one clamped shift of all-ones (shl/shr.b32 give 0 for shifts of 32 or
// more), about 4 instructions per word against about 10 for the two-sided
// 16-bit mask_words.
__device__ __forceinline__ uint32_t shl_clamped(uint32_t a, int s) {
    uint32_t d;
    asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(static_cast<uint32_t>(s < 0 ? 0 : s)));
    return d;
}
__device__ __forceinline__ uint32_t shr_clamped(uint32_t a, int s) {
    uint32_t d;
    asm("shr.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(static_cast<uint32_t>(s < 0 ? 0 : s)));
    return d;
}
template <int DT>
__device__ __forceinline__ void mask_prefix(uint32_t (&w)[4], int nb) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t keep = shl_clamped(0xffffffffu, 8 * nb - 32 * i);  // bytes >= nb
        w[i] = (w[i] & keep) | (neg_inf_word<DT>() & ~keep);
    }
}
template <int DT>
__device__ __forceinline__ void mask_suffix(uint32_t (&w)[4], int t) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t keep = shr_clamped(0xffffffffu, 32 * i + 32 - 8 * t);  // bytes < t
        w[i] = (w[i] & keep) | (neg_inf_word<DT>() & ~keep);
    }
}

}  // namespace lse
