// lse_device.cuh -- device building blocks of the row-wise log-sum-exp.
//
// The method ("Speeding up Log-Sum-Exp: Kernel Fusion at the Memory Wall,
// Integer Arithmetic at the Compute Wall", Sec. 3.1) folds a row into a
// register accumulator with the pairwise LSE operation and evaluates exp/log on
// the special function unit.  Sec. 2.2 names the streaming form used here: a
// running maximum m plus an exp-sum s rescaled whenever m grows.
//
// Accumulator (m, s): m is the largest element seen (NaN-free: max ignores
// NaN), and s = sum 2^((x - mu) * log2 e) over the elements seen, where the
// shift mu = m if m is finite and 0 otherwise.  With that choice
//   * -inf elements add ex2(-inf) = 0, an all -inf row keeps (m, s) = (-inf, 0);
//   * a +inf element adds ex2(+inf) = +inf, so s = +inf whenever m = +inf;
//   * a NaN element makes s NaN, and NaN survives every rescale and merge;
//   * no inf - inf or 0 * inf can occur, so s is NaN exactly when the row holds
//     a NaN.
// The pairwise operation on two accumulators (the merge below) is the paper's
// associative, commutative LSE operation written in this (m, s) form.
//
// Exponentials use base 2 (ex2.approx.ftz.f32, one SFU op) on the argument
// (x - mu) * log2 e; the final log uses lg2.approx.ftz.f32 times ln 2.  These
// are PTX instructions, not CUDA math-library routines.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace lse {

enum : int { kF32 = 0, kBF16 = 1, kF16 = 2 };

template <int DT> struct DType;
template <> struct DType<kF32>  { static constexpr int bytes = 4; };
template <> struct DType<kBF16> { static constexpr int bytes = 2; };
template <> struct DType<kF16>  { static constexpr int bytes = 2; };

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)

// Bit patterns of -inf: one f32, or two packed 16-bit elements.
constexpr uint32_t kNegInfF32 = 0xff800000u;
constexpr uint32_t kNegInfBF16x2 = 0xff80ff80u;
constexpr uint32_t kNegInfF16x2 = 0xfc00fc00u;

template <int DT> __device__ __forceinline__ constexpr uint32_t neg_inf_word() {
    return DT == kF32 ? kNegInfF32 : (DT == kBF16 ? kNegInfBF16x2 : kNegInfF16x2);
}

// A compile-time int carried by value (template arguments of generic lambdas).
template <int V> struct IntConst {
    static constexpr int value = V;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed FP32 (add/sub/mul/fma .f32x2, PTX ISA 8.6 on sm_100 and later): two
// f32 operations in one instruction, each rounded as its scalar form rounds
// it (round to nearest, no flush), so pairing two independent sums halves the
// issue slots of their FP32 work without changing a bit of the result.  A
// pair is one 64-bit register, the low word the first element.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t p, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// 2^t for both elements of a pair (two SFU operations; the SFU has no f32 pair form).
__device__ __forceinline__ uint64_t f2_ex2(uint64_t t) {
    float lo, hi;
    f2_unpack(t, lo, hi);
    return f2_pack(ex2(lo), ex2(hi));
}

// Three-input maximum (sm_100+ PTX); a NaN operand is ignored like in max.f32.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed maxima of two 16-bit lanes; NaN lanes are ignored.
__device__ __forceinline__ uint32_t hmax2_bf16(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hmax2_f16(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 16-byte streaming load through the read-only path, no L1 allocation, with a
// 256-byte L2 prefetch hint (rows are read exactly once).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Exact conversion of one element at element index i of a row.
template <int DT> __device__ __forceinline__ float load_elem(const void* row, int64_t i);
template <> __device__ __forceinline__ float load_elem<kF32>(const void* row, int64_t i) {
    return __ldg(reinterpret_cast<const float*>(row) + i);
}
template <> __device__ __forceinline__ float load_elem<kBF16>(const void* row, int64_t i) {
    const uint32_t h = __ldg(reinterpret_cast<const unsigned short*>(row) + i);
    return __uint_as_float(h << 16);
}
template <> __device__ __forceinline__ float load_elem<kF16>(const void* row, int64_t i) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + i);
    return __half2float(__ushort_as_half(h));
}

// Low / high element of a 32-bit word holding one f32 or two 16-bit elements.
template <int DT> __device__ __forceinline__ float word_lo(uint32_t w);
template <int DT> __device__ __forceinline__ float word_hi(uint32_t w);
template <> __device__ __forceinline__ float word_lo<kBF16>(uint32_t w) { return __uint_as_float(w << 16); }
template <> __device__ __forceinline__ float word_hi<kBF16>(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
template <> __device__ __forceinline__ float word_lo<kF16>(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
template <> __device__ __forceinline__ float word_hi<kF16>(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// Programmatic dependent launch.  Every kernel of the library lets the next
// kernel in its stream launch early (its CTAs become resident and wait), and
// waits for the previous kernel in its stream to complete, with its memory
// visible, before the first global access.  Without a programmatic predecessor
// the wait returns at once.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The shift mu for a maximum m (see the header comment).
__device__ __forceinline__ float shift_of(float m) {
    return fabsf(m) < __int_as_float(0x7f800000) ? m : 0.0f;
}

struct Acc {
    float m;  // running maximum (never NaN)
    float s;  // sum of 2^((x - shift_of(m)) log2 e)
};

__device__ __forceinline__ Acc acc_identity() { return Acc{__int_as_float(kNegInfF32), 0.0f}; }

// Pairwise LSE on two accumulators.
__device__ __forceinline__ Acc acc_merge(Acc a, Acc b) {
    const float m = fmaxf(a.m, b.m);
    const float mu = shift_of(m);
    const float s = a.s * ex2((a.m - mu) * kLog2e) + b.s * ex2((b.m - mu) * kLog2e);
    return Acc{m, s};
}

// log(sum exp) of a finished accumulator, with the special-value rules.
__device__ __forceinline__ float acc_finalize(Acc a) {
    if (a.s != a.s) return a.s;                       // NaN in the row
    if (a.m == __int_as_float(0x7f800000)) return a.m;  // +inf
    if (a.m == __int_as_float(kNegInfF32)) return a.m;  // all -inf, or empty
    return a.m + kLn2 * lg2(a.s);
}

// Write a finished row: the row value, and the token log-probability when
// requested (xt is x[row, target[row]], NaN for an invalid target).
__device__ __forceinline__ void store_row(float* out, float* logprob, int64_t row, float lse,
                                          float xt) {
    if (out) out[row] = lse;
    if (logprob) logprob[row] = xt - lse;
}

// The words of one 16-byte vector that starts at byte vb of a row's
// surroundings, with every element outside the row's bytes [rb0, rb1)
// replaced by -inf (f32 words whole, 16-bit elements by halves).
template <int DT>
__device__ __forceinline__ void mask_words(uint32_t (&w)[4], uint32_t vb, uint32_t rb0,
                                           uint32_t rb1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t b = vb + 4u * i;
        if constexpr (DT == kF32) {
            if (b < rb0 || b >= rb1) w[i] = kNegInfF32;
        } else {
            const uint32_t ninf = neg_inf_word<DT>();  // -inf in both halves
            const uint32_t lo = (b < rb0 || b >= rb1) ? (ninf & 0xffffu) : (w[i] & 0xffffu);
            const uint32_t hi = (b + 2 < rb0 || b + 2 >= rb1) ? (ninf & 0xffff0000u) : (w[i] & 0xffff0000u);
            w[i] = lo | hi;
        }
    }
}

// ---------------------------------------------------------------------------
// Shared-memory staging with 1-D bulk copies (cp.async.bulk, the Tensor Memory
// Accelerator's untiled copy) and mbarrier transaction counts.  Waits are
// bounded: mbar_wait returns false after `polls` unsuccessful polls.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// false when the phase did not complete within `polls` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t polls) {
    for (uint32_t i = 0; i < polls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Element i (0 .. elements-per-vector - 1) of a 16-byte vector held as 4 words.
template <int DT>
__device__ __forceinline__ float word_elem(const uint32_t* w4, int i) {
    if constexpr (DT == kF32) {
        return __uint_as_float(i == 0 ? w4[0] : i == 1 ? w4[1] : i == 2 ? w4[2] : w4[3]);
    } else {
        const int q = i >> 1;
        const uint32_t w = q == 0 ? w4[0] : q == 1 ? w4[1] : q == 2 ? w4[2] : w4[3];
        return (i & 1) ? word_hi<DT>(w) : word_lo<DT>(w);
    }
}

// Butterfly merge across `width` lanes (power of two <= 32); every lane of the
// group ends with the group's accumulator.  The merge order is fixed, so the
// result is deterministic.
template <int WIDTH>
__device__ __forceinline__ Acc warp_merge(Acc a) {
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) {
        Acc b;
        b.m = __shfl_xor_sync(0xffffffffu, a.m, off);
        b.s = __shfl_xor_sync(0xffffffffu, a.s, off);
        a = acc_merge(a, b);
    }
    return a;
}

// Raise the running maximum to cm (a chunk maximum), rescaling s once.
__device__ __forceinline__ void acc_raise(Acc& a, float& mu, float cm) {
    if (cm > a.m) {
        const float mu_new = shift_of(cm);
        a.s *= ex2((a.m - mu_new) * kLog2e);
        a.m = cm;
        mu = mu_new;
    }
}

// ---------------------------------------------------------------------------
// Chunks of raw 32-bit words (one f32 or two packed 16-bit elements each).
// ---------------------------------------------------------------------------

// Maximum over W raw words.
template <int DT, int W>
__device__ __forceinline__ float words_max(const uint32_t (&w)[W]) {
    if constexpr (DT == kF32) {
        float m = __uint_as_float(w[0]);
        int i = 1;
#pragma unroll
        for (; i + 1 < W; i += 2) m = fmax3(m, __uint_as_float(w[i]), __uint_as_float(w[i + 1]));
#pragma unroll
        for (; i < W; ++i) m = fmaxf(m, __uint_as_float(w[i]));
        return m;
    } else {
        // Packed pairwise tree on the 16-bit lanes, then the two halves.
        uint32_t t[W];
#pragma unroll
        for (int i = 0; i < W; ++i) t[i] = w[i];
#pragma unroll
        for (int stride = 1; stride < W; stride *= 2) {
#pragma unroll
            for (int i = 0; i + stride < W; i += 2 * stride)
                t[i] = DT == kBF16 ? hmax2_bf16(t[i], t[i + stride]) : hmax2_f16(t[i], t[i + stride]);
        }
        return fmaxf(word_lo<DT>(t[0]), word_hi<DT>(t[0]));
    }
}

// sum of 2^((x - mu) log2 e) over W raw words, into four interleaved
// accumulators (few live registers, short dependent add chains).
// Accumulator k takes words i with i % 4 == k (f32), or the low and high
// halves of word i as accumulators 2i % 4 and 2i % 4 + 1 (16-bit); the work is
// done on pairs (accumulators 0-1 and 2-3, elements two at a time) with the
// packed FP32 operations.
template <int DT, int W>
__device__ __forceinline__ float words_expsum(const uint32_t (&w)[W], float mu) {
    static_assert(W % 2 == 0, "whole word pairs");
    const uint64_t mu2 = f2_pack(mu, mu);
    const uint64_t log2e2 = f2_pack(kLog2e, kLog2e);
    uint64_t acc[2] = {0ull, 0ull};  // (+0, +0)
#pragma unroll
    for (int i = 0; i < W; ++i) {
        if constexpr (DT == kF32) {
            if (i & 1) continue;
            const uint64_t x = f2_pack(__uint_as_float(w[i]), __uint_as_float(w[i + 1]));
            acc[(i >> 1) & 1] = f2_add(acc[(i >> 1) & 1], f2_ex2(f2_mul(f2_sub(x, mu2), log2e2)));
        } else {
            const uint64_t x = f2_pack(word_lo<DT>(w[i]), word_hi<DT>(w[i]));
            acc[i & 1] = f2_add(acc[i & 1], f2_ex2(f2_mul(f2_sub(x, mu2), log2e2)));
        }
    }
    float a0, a1, a2, a3;
    f2_unpack(acc[0], a0, a1);
    f2_unpack(acc[1], a2, a3);
    return (a0 + a1) + (a2 + a3);
}

// Short rows with their shift mu known in advance: the same exp-sum with one
// FFMA per element, t = x log2 e - c where c = fl(mu log2 e).  Every term then
// carries the same factor 2^r, r = mu log2 e - c, which finalize_scaled takes
// back out exactly.  r is the rounding residual of c, up to half its ulp, so
// it grows with |mu| (r = 6e21 at mu = -1e30, overflowing every term): the
// form is used while |mu| <= 2^24, where |r| <= 1 and the terms keep the
// range of the two-step form.
__device__ __forceinline__ bool ffma_shift_ok(float mu) { return fabsf(mu) <= 0x1.0p24f; }

template <int DT, int W>
__device__ __forceinline__ float words_expsum_scaled(const uint32_t (&w)[W], float c) {
    static_assert(W % 2 == 0, "whole word pairs");
    const uint64_t nc2 = f2_pack(-c, -c);
    const uint64_t log2e2 = f2_pack(kLog2e, kLog2e);
    uint64_t acc[2] = {0ull, 0ull};  // accumulators as in words_expsum
#pragma unroll
    for (int i = 0; i < W; ++i) {
        if constexpr (DT == kF32) {
            if (i & 1) continue;
            const uint64_t x = f2_pack(__uint_as_float(w[i]), __uint_as_float(w[i + 1]));
            acc[(i >> 1) & 1] = f2_add(acc[(i >> 1) & 1], f2_ex2(f2_fma(x, log2e2, nc2)));
        } else {
            const uint64_t x = f2_pack(word_lo<DT>(w[i]), word_hi<DT>(w[i]));
            acc[i & 1] = f2_add(acc[i & 1], f2_ex2(f2_fma(x, log2e2, nc2)));
        }
    }
    float a0, a1, a2, a3;
    f2_unpack(acc[0], a0, a1);
    f2_unpack(acc[1], a2, a3);
    return (a0 + a1) + (a2 + a3);
}

// log(sum exp) from a maximum m and a sum s of 2^(x log2 e - c), c = fl(mu log2 e):
// s = 2^r * sum 2^((x - mu) log2 e) with r = mu log2 e - c (exact by FMA).
__device__ __forceinline__ float finalize_scaled(float m, float s, float mu, float c) {
    if (s != s) return s;
    if (m == __int_as_float(0x7f800000)) return m;
    if (m == __int_as_float(kNegInfF32)) return m;
    const float r = fmaf(mu, kLog2e, -c);
    return m + kLn2 * (lg2(s) - r);
}

// ---------------------------------------------------------------------------
// Reduced-bit exponentials (E16), the 16-bit compute variant of the method
// ("Speeding up Log-Sum-Exp ...", Sec. 4.3, Fig. 5).  Each term's argument is
// formed in f32 exactly as above; two arguments are rounded to bf16 (nearest
// even) and exponentiated by one packed SFU operation, ex2.approx.ftz.bf16x2;
// the two bf16 terms are added into the f32 sum by mixed-precision adds
// (add.rn.f32.bf16, sm_100+).  Half the SFU operations of the f32 path.  bf16
// keeps the f32 exponent range, so terms down to 2^-126 of the maximum still
// count; the error comes from rounding the argument a to 8 significant bits
// (a term is off by a factor 2^(|a| * 2^-8) at most) and from the bf16 result.
// Special values behave as in the f32 path: ex2(-inf) = 0, ex2(+inf) = +inf,
// NaN stays NaN through the conversion, the SFU and the adds.
//
// The packed instruction rounds its bf16 result toward zero (measured: every
// result is the bf16 value at or below 2^a over the whole argument grid), which
// lowers a term by half a bf16 ulp on average, 2^-8 / (2 ln 2) = 0.28 % of its
// value for mantissas spread evenly on a log scale.  Every argument therefore
// carries kE16Bias = -log2(1 - 2^-8 / (2 ln 2)): each term is scaled up by that
// amount before the truncation takes it back off, so terms are unbiased on
// average.  The maximum's own term, 2^kE16Bias = 1.0028, still truncates to
// exactly 1, so one-element and constant rows stay exact.
// ---------------------------------------------------------------------------
constexpr float kE16Bias = 0.0040709119f;

// The E16 argument of element x under shift mu.
__device__ __forceinline__ float e16_arg(float x, float mu) {
    return fmaf(x - mu, kLog2e, kE16Bias);
}

// 2^lo and 2^hi as a bf16 pair (lo in the low half).
__device__ __forceinline__ uint32_t ex2_bf16_pair(float lo, float hi) {
    uint32_t p, e;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p) : "f"(hi), "f"(lo));
    asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(p));
    return e;
}

// acc + lo + hi for a bf16 pair, in f32.
__device__ __forceinline__ float add_bf16_pair(float acc, uint32_t e) {
    float d;
    asm("{\n .reg .b16 lo, hi;\n .reg .f32 t;\n mov.b32 {lo, hi}, %1;\n"
        " add.rn.f32.bf16 t, lo, %2;\n add.rn.f32.bf16 %0, hi, t;\n}\n"
        : "=f"(d)
        : "r"(e), "f"(acc));
    return d;
}

// words_expsum with E16 exponentials: pairs are two f32 words, or the two
// 16-bit halves of one word.
template <int DT, int W>
__device__ __forceinline__ float words_expsum16(const uint32_t (&w)[W], float mu) {
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if constexpr (DT == kF32) {
        static_assert(W % 2 == 0, "f32 words are taken in pairs");
#pragma unroll
        for (int i = 0; i < W / 2; ++i)
            acc[i & 3] = add_bf16_pair(acc[i & 3], ex2_bf16_pair(e16_arg(__uint_as_float(w[2 * i]), mu),
                                                                 e16_arg(__uint_as_float(w[2 * i + 1]), mu)));
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i)
            acc[i & 3] = add_bf16_pair(acc[i & 3], ex2_bf16_pair(e16_arg(word_lo<DT>(w[i]), mu),
                                                                 e16_arg(word_hi<DT>(w[i]), mu)));
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Exp-sum of raw words with f32 (E16 = false) or reduced-bit exponentials.
template <int DT, int W, bool E16>
__device__ __forceinline__ float expsum_words(const uint32_t (&w)[W], float mu) {
    if constexpr (E16) return words_expsum16<DT, W>(w, mu);
    else return words_expsum<DT, W>(w, mu);
}

// Fold a chunk of W raw words into an accumulator.
template <int DT, int W, bool E16 = false>
__device__ __forceinline__ void acc_add_words(Acc& a, float& mu, const uint32_t (&w)[W]) {
    acc_raise(a, mu, words_max<DT, W>(w));
    a.s += expsum_words<DT, W, E16>(w, mu);
}

// Fold a chunk of K converted floats into an accumulator.
template <int K, bool E16 = false>
__device__ __forceinline__ void acc_add_floats(Acc& a, float& mu, const float (&v)[K]) {
    float cm = v[0];
#pragma unroll
    for (int i = 1; i < K; ++i) cm = fmaxf(cm, v[i]);
    acc_raise(a, mu, cm);
    if constexpr (E16) {
        static_assert(K % 2 == 0, "elements are taken in pairs");
        float acc[2] = {0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < K / 2; ++i)
            acc[i & 1] = add_bf16_pair(acc[i & 1], ex2_bf16_pair(e16_arg(v[2 * i], mu),
                                                                 e16_arg(v[2 * i + 1], mu)));
        a.s += acc[0] + acc[1];
    } else {
        float e[K];
#pragma unroll
        for (int i = 0; i < K; ++i) e[i] = ex2((v[i] - mu) * kLog2e);
#pragma unroll
        for (int stride = 1; stride < K; stride *= 2) {
#pragma unroll
            for (int i = 0; i + stride < K; i += 2 * stride) e[i] += e[i + stride];
        }
        a.s += e[0];
    }
}

}  // namespace lse
