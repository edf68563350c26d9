// Element types and per-element operator functors of the broadcast binary
// engine (device side).
//
// Semantics follow "Binary Kernel Design" (onnx-light-cpu), section
// "Operators and traversal" (operator set; Mod opset-28 sign rules; FLOAT16
// and BFLOAT16 computed through float) and section "Compute, scheduling, and
// safety" (validation of integer division, modulo and shifts; one byte per
// BOOL); BatchNormalization, PRelu and Clip follow the 0verkilll/onnx "ops"
// docs (BatchNormalizationOp, PReluOp, ClipOp) and ncnn operators.md
// (batchnorm, bias, clip).
//
// Floating arithmetic uses the round-to-nearest intrinsics (__fadd_rn, ...)
// so that nothing is contracted into an FMA: every step rounds alone, as in
// IEEE-754 binary32.  Half and bfloat16 widen exactly to float, operate in
// float and round once (round to nearest even) on the way out.
#pragma once

#include <cstdint>
#include <cstring>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ebin_launch.h"

namespace ebin {

// One byte per BOOL; any nonzero byte reads as true, results are 0 or 1.
struct Bool8 {
    uint8_t v;
};

constexpr uint32_t kErrDivByZero = 0x1u;
constexpr uint32_t kErrShiftRange = 0x2u;

// ---------------------------------------------------------------- type traits
template <class T> struct Tr;

template <> struct Tr<float> {
    using C = float;
    static constexpr bool kFloat = true;
    __device__ __forceinline__ static float in(float x) { return x; }
    __device__ __forceinline__ static float out(float v) { return v; }
};
template <> struct Tr<__half> {
    using C = float;
    static constexpr bool kFloat = true;
    __device__ __forceinline__ static float in(__half x) { return __half2float(x); }
    __device__ __forceinline__ static __half out(float v) { return __float2half_rn(v); }
};
template <> struct Tr<double> {
    using C = double;
    static constexpr bool kFloat = true;
    __device__ __forceinline__ static double in(double x) { return x; }
    __device__ __forceinline__ static double out(double v) { return v; }
};
template <> struct Tr<__nv_bfloat16> {
    using C = float;
    static constexpr bool kFloat = true;
    __device__ __forceinline__ static float in(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ __forceinline__ static __nv_bfloat16 out(float v) { return __float2bfloat16_rn(v); }
};
template <class I, class U, bool S> struct IntTr {
    using C = I;
    using UT = U;
    static constexpr bool kFloat = false;
    static constexpr bool kSigned = S;
    static constexpr int kBits = 8 * sizeof(I);
    __device__ __forceinline__ static I in(I x) { return x; }
    __device__ __forceinline__ static I out(I v) { return v; }
};
template <> struct Tr<int32_t> : IntTr<int32_t, uint32_t, true> {};
template <> struct Tr<int64_t> : IntTr<int64_t, uint64_t, true> {};
template <> struct Tr<uint8_t> : IntTr<uint8_t, uint8_t, false> {};
template <> struct Tr<uint32_t> : IntTr<uint32_t, uint32_t, false> {};
template <> struct Tr<int8_t> : IntTr<int8_t, uint8_t, true> {};
template <> struct Tr<int16_t> : IntTr<int16_t, uint16_t, true> {};
template <> struct Tr<uint16_t> : IntTr<uint16_t, uint16_t, false> {};
template <> struct Tr<uint64_t> : IntTr<uint64_t, uint64_t, false> {};
template <> struct Tr<Bool8> {
    using C = bool;
    static constexpr bool kFloat = false;
    __device__ __forceinline__ static bool in(Bool8 x) { return x.v != 0; }
};

// binary32 and the 16-bit types computed through it
template <class T> constexpr bool is_float_v = std::is_same_v<T, float> ||
                                               std::is_same_v<T, __half> ||
                                               std::is_same_v<T, __nv_bfloat16>;
// binary64 (DOUBLE), computed natively
template <class T> constexpr bool is_double_v = std::is_same_v<T, double>;
template <class T> constexpr bool is_fp_v = is_float_v<T> || is_double_v<T>;
template <class T> constexpr bool is_int_v = std::is_same_v<T, int32_t> ||
                                             std::is_same_v<T, int64_t> ||
                                             std::is_same_v<T, uint8_t> ||
                                             std::is_same_v<T, uint32_t> ||
                                             std::is_same_v<T, int8_t> ||
                                             std::is_same_v<T, int16_t> ||
                                             std::is_same_v<T, uint16_t> ||
                                             std::is_same_v<T, uint64_t>;
template <class T> constexpr bool is_bool_v = std::is_same_v<T, Bool8>;
template <class T> constexpr bool is_signed_int_v = std::is_same_v<T, int32_t> ||
                                                    std::is_same_v<T, int64_t> ||
                                                    std::is_same_v<T, int8_t> ||
                                                    std::is_same_v<T, int16_t>;
// ONNX Pow's integer base types
template <class T> constexpr bool is_pow_int_v = std::is_same_v<T, int32_t> ||
                                                 std::is_same_v<T, int64_t>;

// Common shape of an operator functor whose B operand is an ordinary
// broadcast tensor of the input type.
template <class T, class O> struct PlainB {
    using In = T;
    using Out = O;
    using BV = T;
    static constexpr bool kPlainB = true;
    __device__ __forceinline__ static BV loadB(const T *B, int64_t off, const OpArgs &) {
        return B[off];
    }
};

// float16 and bfloat16: computed through binary32
template <class T> constexpr bool is_half_like_v = std::is_same_v<T, __half> ||
                                                   std::is_same_v<T, __nv_bfloat16>;

// ---------------------------------------------------------------- 16-bit words
// Groups of 16-bit elements move as 32-bit words, two elements each.
// Two values rounded to a 16-bit type, packed (the first in the low half).
template <class T> __device__ __forceinline__ uint32_t round2(float a, float b);
template <> __device__ __forceinline__ uint32_t round2<__nv_bfloat16>(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    uint32_t w;
    memcpy(&w, &v, 4);
    return w;
}
template <> __device__ __forceinline__ uint32_t round2<__half>(float a, float b) {
    const __half2 v = __floats2half2_rn(a, b);
    uint32_t w;
    memcpy(&w, &v, 4);
    return w;
}

// Two 16-bit values of one 32-bit word (the first in the low half), widened
// exactly to binary32.
template <class T> __device__ __forceinline__ float2 widen2(uint32_t w);
template <> __device__ __forceinline__ float2 widen2<__nv_bfloat16>(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
template <> __device__ __forceinline__ float2 widen2<__half>(uint32_t w) {
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
}

// Mixed-precision operations on the two 16-bit values of a word (PTX
// add.rn.f32.bf16 / .f32.f16 and fma.rn.f32.bf16 / .f32.f16, sm_100 and
// later): each 16-bit operand is widened exactly inside the instruction, which
// rounds once in binary32.  The word's halves are taken as 16-bit registers,
// so no widening instruction is issued.
//   widen_add2(w, c): RN(x + c), RN(x' + c) for the word's values x, x';
//   mul_mixed2(w, v): RN(x y) for the values of the two words, lane by lane,
//     as RN(x y + (-0)): a product of two 16-bit values is exact in binary32
//     (at most 22 significant bits) unless it overflows or underflows, where
//     both forms round the same exact product, and adding -0 changes no value
//     and no zero's sign.
template <class T> struct Mixed16;
template <> struct Mixed16<__nv_bfloat16> {
    __device__ __forceinline__ static float2 add(uint32_t w, float2 c) {
        float lo, hi;
        asm("{\n\t.reg .b16 l, h;\n\t"
            "mov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.bf16 %0, l, %3;\n\t"
            "add.rn.f32.bf16 %1, h, %4;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(w), "f"(c.x), "f"(c.y));
        return make_float2(lo, hi);
    }
    __device__ __forceinline__ static float2 mul(uint32_t w, uint32_t v) {
        float lo, hi;
        asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\t"
            "mov.b32 {xl, xh}, %2;\n\t"
            "mov.b32 {yl, yh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, xl, yl, %4;\n\t"
            "fma.rn.f32.bf16 %1, xh, yh, %4;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(w), "r"(v), "f"(-0.0f));
        return make_float2(lo, hi);
    }
};
template <> struct Mixed16<__half> {
    __device__ __forceinline__ static float2 add(uint32_t w, float2 c) {
        float lo, hi;
        asm("{\n\t.reg .b16 l, h;\n\t"
            "mov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.f16 %0, l, %3;\n\t"
            "add.rn.f32.f16 %1, h, %4;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(w), "f"(c.x), "f"(c.y));
        return make_float2(lo, hi);
    }
    __device__ __forceinline__ static float2 mul(uint32_t w, uint32_t v) {
        float lo, hi;
        asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\t"
            "mov.b32 {xl, xh}, %2;\n\t"
            "mov.b32 {yl, yh}, %3;\n\t"
            "fma.rn.f32.f16 %0, xl, yl, %4;\n\t"
            "fma.rn.f32.f16 %1, xh, yh, %4;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(w), "r"(v), "f"(-0.0f));
        return make_float2(lo, hi);
    }
};
template <class T> __device__ __forceinline__ float2 widen_add2(uint32_t w, float c) {
    return Mixed16<T>::add(w, make_float2(c, c));
}
template <class T> __device__ __forceinline__ float2 mul_mixed2(uint32_t w, uint32_t v) {
    return Mixed16<T>::mul(w, v);
}

// The value in one half of a word, and a 16-bit value's bits.
template <class T> __device__ __forceinline__ T half_of(uint32_t w, bool high) {
    const unsigned short b = (unsigned short)(high ? (w >> 16) : (w & 0xFFFFu));
    T v;
    memcpy(&v, &b, 2);
    return v;
}
template <class T> __device__ __forceinline__ uint32_t bits_of(T v) {
    unsigned short b;
    memcpy(&b, &v, 2);
    return b;
}

// ---------------------------------------------------------------- exact fmod
//
// Truncated remainder r = a - trunc(a/b)*b, exact, for finite a and nonzero
// finite b.  Fast path (|a/b| < 2^23): q = trunc(RN(|a|/|b|)).  Because RN is
// monotone and every integer below 2^24 is representable, q is either
// n = trunc(|a|/|b|) or n + 1.  |a| >= |b| makes |a| a multiple of ulp(|b|),
// so |a| - q|b| is a multiple of ulp(|b|) smaller than |b| in magnitude: it is
// representable and the single rounding of fmaf(-q, |b|, |a|) is exact.  A
// negative result means q was n + 1, and adding |b| back is exact as well.
// Larger quotients, infinities, NaNs and zero divisors go to CUDA's fmodf.
__device__ __forceinline__ float fmod_exact(float a, float b) {
    const float aa = fabsf(a), ab = fabsf(b);
    if (aa < ab) return a;                         // includes a = +-0 (b finite or inf)
    if (!(aa < INFINITY) || !(ab > 0.0f) || !(ab < INFINITY)) return fmodf(a, b);
    const float q = truncf(__fdiv_rn(aa, ab));
    if (q < 8388608.0f) {
        float r = fmaf(-q, ab, aa);
        if (r < 0.0f) r = __fadd_rn(r, ab);
        return copysignf(r, a);                    // a zero result keeps the dividend's sign
    }
    return fmodf(a, b);
}

// Mod with opset-28 rules: fmod=1 truncated; fmod=0 floor remainder where a
// nonzero result with the wrong sign gets b added (one rounded add) and an
// exact zero takes the divisor's sign.
__device__ __forceinline__ float mod_float(float a, float b, int fmod_flag) {
    float r = fmod_exact(a, b);
    if (fmod_flag) return r;
    if (r == 0.0f) return copysignf(0.0f, b);
    if (signbit(r) != signbit(b)) r = __fadd_rn(r, b);
    return r;
}

// ---------------------------------------------------------------- arithmetic
// K_RSUB and K_RDIV are ncnn binaryop's RSUB (B - A) and RDIV (B / A)
// (ncnn operators.md, binaryop, operation types 7 and 8).
enum ArithK { K_ADD = 0, K_SUB = 1, K_MUL = 2, K_DIV = 3, K_RSUB = 4, K_RDIV = 5 };

template <class T, int K> struct OpArith : PlainB<T, T> {
    static constexpr bool kLegal = is_fp_v<T> || is_int_v<T>;
    static constexpr bool kValidates = (K == K_DIV || K == K_RDIV) && is_int_v<T>;
    static constexpr bool kScalarAttr = is_fp_v<T>;        // ncnn binaryop with_scalar
    // Add, Sub, Mul and RSub of float16 / bfloat16 on pairs: two elements
    // from one 32-bit word, each result rounded once in binary32, the two
    // results rounded by one conversion -- the values of apply.  Mul is one
    // mixed-precision multiply-add per element on the 16-bit halves (no
    // widening; bf16 Mul on short general rows 144.8 -> 116.3 us on GB300);
    // Add, Sub and RSub widen both words and take one f32x2 add (x - y is
    // x + (-y)), which measured faster than a mixed-precision add (per-channel
    // bf16 Add 20.7 against 21.0 us).  Division keeps the element form (the
    // IEEE divide).
    static constexpr bool kPack = is_half_like_v<T> && K != K_DIV && K != K_RDIV;
    template <int G>
    __device__ __forceinline__ static void apply_pack(const T *a, const T *b, T *o) {
        constexpr int W = G / 2;
        uint32_t aw[W], bw[W], ow[W];
        memcpy(aw, a, sizeof(aw));
        memcpy(bw, b, sizeof(bw));
#pragma unroll
        for (int k = 0; k < W; ++k) {
            float2 r;
            if constexpr (K == K_MUL) {
                r = mul_mixed2<T>(aw[k], bw[k]);
            } else {
                const float2 x = widen2<T>(aw[k]), y = widen2<T>(bw[k]);
                if constexpr (K == K_ADD) r = __fadd2_rn(x, y);
                else if constexpr (K == K_SUB) r = __fadd2_rn(x, make_float2(-y.x, -y.y));
                else r = __fadd2_rn(y, make_float2(-x.x, -x.y));
            }
            ow[k] = round2<T>(r.x, r.y);
        }
        memcpy(o, ow, sizeof(ow));
    }
    __device__ __forceinline__ static T apply(T a, T b, const OpArgs &, uint32_t &err) {
        if constexpr (K == K_RSUB || K == K_RDIV) {
            // the same operation with the operands exchanged
            return OpArith<T, K == K_RSUB ? K_SUB : K_DIV>::apply(b, a, OpArgs{}, err);
        } else if constexpr (is_double_v<T>) {
            if constexpr (K == K_ADD) return __dadd_rn(a, b);
            else if constexpr (K == K_SUB) return __dsub_rn(a, b);
            else if constexpr (K == K_MUL) return __dmul_rn(a, b);
            else return __ddiv_rn(a, b);
        } else if constexpr (is_float_v<T>) {
            const float x = Tr<T>::in(a), y = Tr<T>::in(b);
            float r;
            if constexpr (K == K_ADD) r = __fadd_rn(x, y);
            else if constexpr (K == K_SUB) r = __fsub_rn(x, y);
            else if constexpr (K == K_MUL) r = __fmul_rn(x, y);
            else r = __fdiv_rn(x, y);
            return Tr<T>::out(r);
        } else {
            using U = typename Tr<T>::UT;
            if constexpr (K == K_ADD) return (T)((U)a + (U)b);
            else if constexpr (K == K_SUB) return (T)((U)a - (U)b);
            else if constexpr (K == K_MUL) return (T)((U)a * (U)b);
            else {
                if (b == 0) { err |= kErrDivByZero; return (T)0; }
                if constexpr (Tr<T>::kSigned) {
                    if (b == (T)-1) return (T)((U)0 - (U)a);    // INT_MIN / -1 wraps
                }
                return (T)(a / b);                               // truncates toward zero
            }
        }
    }
};

// ncnn binaryop MAX / MIN (operators.md, binaryop, operation types 4 and 5),
// read as IEEE 754-2019 maximum / minimum: a NaN operand gives NaN and +0
// counts as larger than -0.  Half and bfloat16 results are one of the two
// widened inputs, so narrowing them back is exact.
template <class T, bool kMax> struct OpMinMax : PlainB<T, T> {
    static constexpr bool kLegal = is_fp_v<T> || is_int_v<T>;
    static constexpr bool kValidates = false;
    static constexpr bool kScalarAttr = is_fp_v<T>;
    __device__ __forceinline__ static T apply(T a, T b, const OpArgs &, uint32_t &) {
        if constexpr (is_fp_v<T>) {
            using C = typename Tr<T>::C;
            const C x = Tr<T>::in(a), y = Tr<T>::in(b);
            C r;
            if (isnan(x) || isnan(y)) r = x + y;                            // a NaN
            else if (x == y) r = (signbit(x) == kMax) ? y : x;             // +0 vs -0
            else r = kMax ? (x > y ? x : y) : (x < y ? x : y);
            return Tr<T>::out(r);
        } else {
            return kMax ? (a > b ? a : b) : (a < b ? a : b);
        }
    }
};

// ncnn binaryop with_scalar: the operator with B replaced by the attribute
// value, rounded to the element type (the same value a 0-d B tensor would
// hold).  No B pointer is read.
template <class Op> struct WithScalar : Op {
    using In = typename Op::In;
    __device__ __forceinline__ static typename Op::BV loadB(const In *, int64_t,
                                                            const OpArgs &p) {
        return Tr<In>::out(p.scalar_b);
    }
};

// A floating divisor that stays the same for many elements (a scalar, or one
// value per row) is prepared once: ab = |b|, rcp = RD(1/ab) and
// lim = RN(2^21 * ab) (exact, or infinity when ab > 2^107, where every finite
// |a| / ab is below 2^21 anyway).  For |a| < lim:
//   p = RD(|a| * rcp) <= |a|/ab and, with two downward roundings of relative
//   size 2^-23, p > |a|/ab - 1/2, so q = trunc(p) is n = trunc(|a|/ab) or n - 1;
//   r0 = fmaf(-q, ab, |a|) and r1 = fmaf(-(q + 1), ab, |a|) (q + 1 exact): for
//   q = n, r0 is the remainder and r1 = r0 - ab < 0; for q = n - 1, r1 is the
//   remainder (>= 0).  Each value that is used is a multiple of ulp(ab) of
//   magnitude at most ab (|a| >= ab makes |a| a multiple of ulp(ab)), hence
//   representable, and each FMA rounds once, so it is exact.  |a| < ab needs no
//   special case (q = 0, r0 = |a|).
// The truncated remainder is then that magnitude with the dividend's sign; the
// floor rule adds b to a nonzero remainder of the other sign (one rounded
// operation) and gives an exact zero the divisor's sign.  Zero, subnormal,
// huge, infinite or NaN divisors, NaN or infinite dividends and quotients of
// 2^21 or more take the exact general path (mod_float) for the whole group.
struct ModPrep {
    float b, ab, rcp, lim;
    bool fast, neg;
};

__device__ __forceinline__ ModPrep mod_prep(float b) {
    ModPrep p;
    p.b = b;
    p.ab = fabsf(b);
    p.fast = p.ab >= 0x1p-125f && p.ab <= 0x1p125f;   // excludes 0, subnormals, inf, NaN
    p.neg = signbit(b);
    p.rcp = __frcp_rd(p.fast ? p.ab : 1.0f);
    p.lim = __fmul_rn(p.ab, 2097152.0f);
    return p;
}

// An int32 divisor shared by many elements is prepared once: d = |b| and
// m0 = trunc(2^32 * rcp_rz(float_ru(d))) <= 2^32 / d (every rounding is toward
// the underestimate; 2^32 itself saturates to 2^32 - 1), within a relative
// 2^-22 plus one unit of 2^32 / d.  For n = |a| <= 2^31:
//   q1 = mulhi(n, m0) <= floor(n/d) and misses it by less than n*2^-22/d + 1.5,
//   so r1 = n - q1*d lies in [0, 2d + 2^9) and fits 32 bits (for d > 2^30 the
//   miss is at most 1 and r1 < 2d <= 2^32);
//   q2 = mulhi(r1, m0) misses floor(r1/d) by at most 1, so r2 = r1 - q2*d lies
//   in [0, 2d), and min(r2, r2 - d) taken unsigned (r2 - d wraps above r2
//   when r2 < d) is n mod d.
// Then the truncated remainder is +-(n mod d) with the dividend's sign, and
// the floor remainder is the magnitude x = n mod d, or d - x when that is
// nonzero and the signs differ, with the divisor's sign.
struct IModPrep {
    int32_t b;
    uint32_t d, nd, m0;
    int32_t sb;     // 0 or -1: the divisor's sign as a mask
    bool zero;
};

__device__ __forceinline__ IModPrep imod_prep(int32_t b) {
    IModPrep p;
    p.b = b;
    p.d = b < 0 ? 0u - (uint32_t)b : (uint32_t)b;
    p.nd = 0u - p.d;
    p.sb = b >> 31;
    p.zero = b == 0;
    const float r = __frcp_rz(__uint2float_ru(p.zero ? 1u : p.d));
    p.m0 = __float2uint_rz(r * 4294967296.0f);
    return p;
}

__device__ __forceinline__ uint32_t umod_prepared(uint32_t n, const IModPrep &p) {
    const uint32_t r1 = n + __umulhi(n, p.m0) * p.nd;
    const uint32_t r2 = r1 + __umulhi(r1, p.m0) * p.nd;
    return umin(r2, r2 + p.nd);
}

// |a| as unsigned; PTX abs.s32 leaves INT_MIN as is, whose bits read 2^31.
__device__ __forceinline__ uint32_t uabs32(int32_t a) {
    int32_t r;
    asm("abs.s32 %0, %1;" : "=r"(r) : "r"(a));
    return (uint32_t)r;
}
// Truncated remainder (fmod=1) of int32 a by the prepared nonzero divisor.
// (The sign flip is done unsigned: (v ^ s) - s negates v when s = -1.)
__device__ __forceinline__ int32_t imod_trunc(int32_t a, const IModPrep &p) {
    const uint32_t sa = (uint32_t)(a >> 31);
    const uint32_t x = umod_prepared(uabs32(a), p);
    return (int32_t)((x ^ sa) - sa);
}
// The floor remainder for a divisor known positive / known negative.
__device__ __forceinline__ int32_t imod_floor_pos(int32_t a, const IModPrep &p) {
    const uint32_t x = umod_prepared(uabs32(a), p);
    return (int32_t)((a < 0 && x != 0u) ? p.d - x : x);
}
__device__ __forceinline__ int32_t imod_floor_neg(int32_t a, const IModPrep &p) {
    const uint32_t x = umod_prepared(uabs32(a), p);
    return (int32_t)((a > 0 && x != 0u) ? x - p.d : 0u - x);
}

template <class T> struct OpMod : PlainB<T, T> {
    static constexpr bool kLegal = is_fp_v<T> || is_int_v<T>;
    static constexpr bool kValidates = is_int_v<T>;
    __device__ __forceinline__ static T apply(T a, T b, const OpArgs &p, uint32_t &err) {
        if constexpr (is_double_v<T>) {
            // binary64: C fmod (exact), then the same floor rule in binary64
            double r = fmod(a, b);
            if (p.fmod) return r;
            if (r == 0.0) return copysign(0.0, b);
            if (signbit(r) != signbit(b)) r = __dadd_rn(r, b);
            return r;
        } else if constexpr (is_float_v<T>) {
            return Tr<T>::out(mod_float(Tr<T>::in(a), Tr<T>::in(b), p.fmod));
        } else {
            if (b == 0) { err |= kErrDivByZero; return (T)0; }
            if constexpr (Tr<T>::kSigned) {
                if (b == (T)-1) return (T)0;
                T r = a % b;                                     // sign of the dividend
                if (!p.fmod && r != 0 && ((r < 0) != (b < 0))) r = (T)(r + b);
                return r;
            } else {
                return (T)(a % b);
            }
        }
    }
    // Mod with a divisor shared by a whole group: floating (see ModPrep) and
    // int32 (see IModPrep)
    static constexpr bool kPrep = is_float_v<T> || std::is_same_v<T, int32_t>;
    // at least two rows per thread in the row kernel (fp32 [4096,4096] vs
    // [4096,1]: 24.1 -> 23.4 us on GB300)
    static constexpr int kMinRows = 2;
    using PB = std::conditional_t<std::is_same_v<T, int32_t>, IModPrep, ModPrep>;
    __device__ __forceinline__ static PB prep(T b) {
        if constexpr (std::is_same_v<T, int32_t>) return imod_prep(b);
        else return mod_prep(Tr<T>::in(b));
    }
    // G elements at once, all taking the fast path without branches, with one
    // uniform branch per group to the general path and one on the divisor's
    // sign and the fmod attribute.
    template <int G, bool SA>
    __device__ __forceinline__ static void apply_prep_group(const T *a, const PB &pb, T *o,
                                                            const OpArgs &p, uint32_t &err) {
        if constexpr (std::is_same_v<T, int32_t>) {
            if (pb.zero) {
                err |= kErrDivByZero;
#pragma unroll
                for (int k = 0; k < G; ++k) o[k] = 0;
                return;
            }
            if (p.fmod) {
#pragma unroll
                for (int k = 0; k < G; ++k) o[k] = imod_trunc(a[SA ? 0 : k], pb);
            } else if (pb.sb == 0) {
#pragma unroll
                for (int k = 0; k < G; ++k) o[k] = imod_floor_pos(a[SA ? 0 : k], pb);
            } else {
#pragma unroll
                for (int k = 0; k < G; ++k) o[k] = imod_floor_neg(a[SA ? 0 : k], pb);
            }
        } else {
            float x[G], r[G];
            bool ok = pb.fast;
#pragma unroll
            for (int k = 0; k < G; ++k) {
                x[k] = Tr<T>::in(a[SA ? 0 : k]);
                const float aa = fabsf(x[k]);
                ok = ok & (aa < pb.lim);
                const float q = truncf(__fmul_rd(aa, pb.rcp));
                const float r0 = fmaf(-q, pb.ab, aa);
                const float r1 = fmaf(-__fadd_rn(q, 1.0f), pb.ab, aa);
                r[k] = r1 < 0.0f ? r0 : r1;
            }
            if (!ok) {
#pragma unroll
                for (int k = 0; k < G; ++k) o[k] = Tr<T>::out(mod_float(x[k], pb.b, p.fmod));
            } else if (p.fmod) {
#pragma unroll
                for (int k = 0; k < G; ++k) o[k] = Tr<T>::out(copysignf(r[k], x[k]));
            } else if (!pb.neg) {
#pragma unroll
                for (int k = 0; k < G; ++k)
                    o[k] = Tr<T>::out((x[k] < 0.0f && r[k] != 0.0f) ? __fsub_rn(pb.ab, r[k]) : r[k]);
            } else {
#pragma unroll
                for (int k = 0; k < G; ++k)
                    o[k] = Tr<T>::out((x[k] > 0.0f && r[k] != 0.0f) ? __fsub_rn(r[k], pb.ab) : -r[k]);
            }
        }
    }
};

// Integer a^e with wrap: square and multiply; a negative e gives
// trunc(1 / a^|e|) (+-1 for a = +-1, else 0) and a = 0 raises DIV_BY_ZERO.
// (e is given as its sign and its magnitude: unsigned 64-bit exponents reach
// 2^64 - 1)
template <class T>
__device__ __forceinline__ T int_pow(T a, bool neg, uint64_t mag, uint32_t &err) {
    using U = typename Tr<T>::UT;
    if (neg) {
        if (a == 0) { err |= kErrDivByZero; return (T)0; }
        if (a == 1) return (T)1;
        if (a == (T)-1) return (mag & 1) ? (T)-1 : (T)1;
        return (T)0;
    }
    U result = 1, base = (U)a;
    uint64_t k = mag;
    while (k) {
        if (k & 1u) result *= base;
        base *= base;
        k >>= 1;
    }
    return (T)result;
}

// Floating a^e: C pow semantics evaluated in binary64, rounded once to
// binary32 (then to a 16-bit type).
template <class T>
__device__ __forceinline__ T float_pow(T a, double e) {
    return Tr<T>::out(__double2float_rn(pow((double)Tr<T>::in(a), e)));
}

template <class T> struct OpPow : PlainB<T, T> {
    static constexpr bool kLegal = is_fp_v<T> || is_pow_int_v<T>;
    static constexpr bool kValidates = is_pow_int_v<T>;
    static constexpr bool kScalarAttr = is_fp_v<T>;        // ncnn binaryop POW with_scalar
    __device__ __forceinline__ static T apply(T a, T b, const OpArgs &, uint32_t &err) {
        if constexpr (is_double_v<T>) return pow(a, b);          // C pow in binary64
        else if constexpr (is_float_v<T>) return float_pow(a, (double)Tr<T>::in(b));
        else return int_pow(a, b < 0, b < 0 ? 0 - (uint64_t)b : (uint64_t)b, err);
    }
};

// Pow with an exponent of another type ("Binary Kernel Design", Compute,
// scheduling, and safety: signatures other than the same-type ones run
// through typed scalar adapters; ONNX Pow takes base T, exponent T1).
//  - floating base: float_pow on the exponent's value as binary64;
//  - integer base, integer exponent: int_pow with the exponent as 64 bits;
//  - integer base, floating exponent: pow in binary64, truncated toward zero,
//    saturated at the base type's bounds, NaN to 0 (no status).
// Only the general (element by element) kernel runs it.
template <class TA, class TB> struct OpPowMixed {
    using In = TA;
    using Out = TA;
    using BV = TB;
    using BIn = TB;                  // B's element type differs from A's
    static constexpr bool kPlainB = false;
    static constexpr bool kLegal = (is_fp_v<TA> || is_pow_int_v<TA>) && !is_bool_v<TB>;
    static constexpr bool kValidates = is_pow_int_v<TA> && !is_fp_v<TB>;
    __device__ __forceinline__ static BV loadB(const TB *B, int64_t off, const OpArgs &) {
        return B[off];
    }
    __device__ __forceinline__ static double as_double(TB e) {
        if constexpr (is_fp_v<TB>) return (double)Tr<TB>::in(e);
        else return (double)e;
    }
    __device__ __forceinline__ static TA apply(TA a, TB b, const OpArgs &, uint32_t &err) {
        if constexpr (is_double_v<TA>) {
            return pow(a, as_double(b));
        } else if constexpr (is_float_v<TA>) {
            return float_pow(a, as_double(b));
        } else if constexpr (!is_fp_v<TB>) {
            if constexpr (is_signed_int_v<TB>)
                return int_pow(a, b < 0, b < 0 ? 0 - (uint64_t)(int64_t)b : (uint64_t)b, err);
            else
                return int_pow(a, false, (uint64_t)b, err);
        } else {
            const double y = pow((double)a, as_double(b));
            constexpr bool k32 = std::is_same_v<TA, int32_t>;
            constexpr TA tmin = k32 ? (TA)INT32_MIN : (TA)INT64_MIN;
            constexpr TA tmax = k32 ? (TA)INT32_MAX : (TA)INT64_MAX;
            if (isnan(y)) return (TA)0;
            if (y >= (double)tmax) return tmax;
            if (y <= (double)tmin) return tmin;
            return (TA)y;                                        // truncates toward zero
        }
    }
};

// ---------------------------------------------------------------- comparisons
enum CmpK { K_EQ = 0, K_LT = 1, K_GT = 2, K_LE = 3, K_GE = 4 };

template <class C, int K> __device__ __forceinline__ bool compare(C x, C y) {
    if constexpr (K == K_EQ) return x == y;
    else if constexpr (K == K_LT) return x < y;
    else if constexpr (K == K_GT) return x > y;
    else if constexpr (K == K_LE) return x <= y;
    else return x >= y;
}


// Two-lane comparison masks (0xFFFF per true lane, NaN compares false).
template <int K, class T2>
__device__ __forceinline__ unsigned cmp_mask2(T2 a, T2 b) {
    if constexpr (K == K_EQ) return __heq2_mask(a, b);
    else if constexpr (K == K_LT) return __hlt2_mask(a, b);
    else if constexpr (K == K_GT) return __hgt2_mask(a, b);
    else if constexpr (K == K_LE) return __hle2_mask(a, b);
    else return __hge2_mask(a, b);
}

template <class T, int K> struct OpCmp : PlainB<T, Bool8> {
    static constexpr bool kLegal = is_fp_v<T> || is_int_v<T> || (K == K_EQ && is_bool_v<T>);
    static constexpr bool kValidates = false;
    // half and bfloat16 compare exactly in their own format, two lanes per
    // instruction; the comparison of the exact float widenings is the same
    static constexpr bool kPack = is_half_like_v<T>;
    __device__ __forceinline__ static Bool8 apply(T a, T b, const OpArgs &, uint32_t &) {
        return Bool8{(uint8_t)(compare<typename Tr<T>::C, K>(Tr<T>::in(a), Tr<T>::in(b)) ? 1 : 0)};
    }
    // G results (G a multiple of 4): two packed compares per four lanes, the
    // lane masks narrowed to one 0/1 byte each.
    template <int G>
    __device__ __forceinline__ static void apply_pack(const T *a, const T *b, Bool8 *o) {
        static_assert(G % 4 == 0, "packs of four");
        using T2 = std::conditional_t<std::is_same_v<T, __half>, __half2, __nv_bfloat162>;
#pragma unroll
        for (int k = 0; k < G; k += 4) {
            T2 a0, a1, b0, b1;
            if constexpr (std::is_same_v<T, __half>) {
                a0 = __halves2half2(a[k], a[k + 1]);
                a1 = __halves2half2(a[k + 2], a[k + 3]);
                b0 = __halves2half2(b[k], b[k + 1]);
                b1 = __halves2half2(b[k + 2], b[k + 3]);
            } else {
                a0 = __halves2bfloat162(a[k], a[k + 1]);
                a1 = __halves2bfloat162(a[k + 2], a[k + 3]);
                b0 = __halves2bfloat162(b[k], b[k + 1]);
                b1 = __halves2bfloat162(b[k + 2], b[k + 3]);
            }
            const unsigned m0 = cmp_mask2<K>(a0, b0), m1 = cmp_mask2<K>(a1, b1);
            const uint32_t w = __byte_perm(m0, m1, 0x6420) & 0x01010101u;
            memcpy(o + k, &w, 4);
        }
    }
};

// ---------------------------------------------------------------- logical / bitwise / shift
enum LogicK { K_AND = 0, K_OR = 1, K_XOR = 2 };

template <class T, int K> struct OpLogic : PlainB<T, Bool8> {
    static constexpr bool kLegal = is_bool_v<T>;
    static constexpr bool kValidates = false;
    __device__ __forceinline__ static Bool8 apply(T a, T b, const OpArgs &, uint32_t &) {
        const bool x = a.v != 0, y = b.v != 0;
        bool r;
        if constexpr (K == K_AND) r = x && y;
        else if constexpr (K == K_OR) r = x || y;
        else r = x != y;
        return Bool8{(uint8_t)(r ? 1 : 0)};
    }
};

template <class T, int K> struct OpBitwise : PlainB<T, T> {
    static constexpr bool kLegal = is_int_v<T>;
    static constexpr bool kValidates = false;
    __device__ __forceinline__ static T apply(T a, T b, const OpArgs &, uint32_t &) {
        if constexpr (K == K_AND) return (T)(a & b);
        else if constexpr (K == K_OR) return (T)(a | b);
        else return (T)(a ^ b);
    }
};

template <class T> struct OpShift : PlainB<T, T> {
    static constexpr bool kLegal = std::is_same_v<T, uint8_t> || std::is_same_v<T, uint16_t> ||
                                   std::is_same_v<T, uint32_t> || std::is_same_v<T, uint64_t>;
    static constexpr bool kValidates = true;
    __device__ __forceinline__ static T apply(T a, T b, const OpArgs &p, uint32_t &err) {
        if constexpr (kLegal) {
            // the count compared in the element's own width; narrow types shift in 32 bits
            using U = std::conditional_t<(sizeof(T) < 4), uint32_t, T>;
            constexpr T w = (T)(8 * sizeof(T));
            if (b >= w) { err |= kErrShiftRange; return (T)0; }
            return p.direction == 0 ? (T)((U)a << (U)b) : (T)((U)a >> (U)b);
        } else {
            return a;
        }
    }
};

// ---------------------------------------------------------------- per-channel operators
// Round-to-nearest arithmetic in the compute type (binary32 or binary64); the
// _rn intrinsics are never contracted into a fused multiply-add.
__device__ __forceinline__ float add_rn(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ double add_rn(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ float sub_rn(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ double sub_rn(double a, double b) { return __dsub_rn(a, b); }
__device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ double mul_rn(double a, double b) { return __dmul_rn(a, b); }
__device__ __forceinline__ float div_rn(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ double div_rn(double a, double b) { return __ddiv_rn(a, b); }
__device__ __forceinline__ float sqrt_rn(float a) { return __fsqrt_rn(a); }
__device__ __forceinline__ double sqrt_rn(double a) { return __dsqrt_rn(a); }

// ---------------------------------------------------------------- prepared exact division
//
// q = RN(t / d) for many t sharing one divisor d, without the IEEE divide: with
// r = RN(1/d) formed once,
//   q0 = RN(t r);  q1 = RN(q0 + RN(t - q0 d) r);  q2 = RN(q1 + RN(t - q1 d) r)
// (every step one rounding; the remainders are FMAs).  Then q2 == RN(t/d)
// whenever d's significand D (an integer in [2^23, 2^24)) is at most
// 2^24 - 5 and no step leaves the normal range.  The argument, scaled to
// d in [1, 2) (powers of two change nothing), u = 2^-24, Q = t/d, and
// eps = d r - 1 with |eps| <= d 2^-25 = D 2^-48 (r within half an ulp):
//  - t r = Q (1 + eps), so |q0 - Q| <= (2u + u^2) |Q|;
//  - q0 + RN(t - q0 d) r = Q + (Q - q0)((1 + e)(1 + eps) - 1), |e| <= u, so
//    it lies within (2u + u^2)^2 |Q| < 2^-22 ulp(Q) of Q, and q1 lies within
//    (1/2 + 2^-22) ulp of Q;
//  - t and q1 d are integer multiples of 2^(eq + ed), the ulps of q1 and d
//    (t ~ q1 d and both significands are normalised), and |t - q1 d| <=
//    (1/2 + 2^-22) D 2^(eq + ed) < 2^24 2^(eq + ed): the second remainder
//    is exact (granularity 2^(eq + ed) >= 2^-149 within the ranges below);
//  - q1 + (t - q1 d) r = Q + (Q - q1) eps, off Q by at most
//    (1/2 + 2^-22) ulp D 2^-48;
//  - Q = T/D-scaled is never a midpoint (a 25-bit odd number times D cannot
//    equal a 24-bit T times a power of two) and lies at least ulp / (2D) from
//    every midpoint (the distance is an integer over 2D, in ulps);
//  - (1/2 + 2^-22) D 2^-48 < 1 / (2D) holds for D <= 2^24 - 5, so rounding
//    Q's neighbour rounds as Q does.
// This is the final-correction scheme of P. Markstein ("Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990), applied twice.
//
// Ranges.  A row takes it when 2^-20 <= d <= 2^20 and D <= 2^24 - 5; an
// element keeps q2 when tlow <= |t| <= thigh = RD(2^99 d).  The upper bound
// keeps |t / d| <= 2^99 and every step finite (and fails for an infinite or NaN
// t).  With |t| >= 2^-100 the remainders' granularity 2^(eq + ed) ~ |t| 2^-46
// stays at or above 2^-149 and every quantity is normal.  For t = +0 the steps
// give q2 = +0 exactly, but t = -0 comes out as +0.  The chains divide
// t = t' - mean with t' and mean binary32 values; when |mean| >= 2^-75, t is +0
// or at least 2^-99 in magnitude (two binary32 values at or above 2^-76 differ
// by a multiple of 2^-99), and never -0, so such rows need no lower test
// (tlow = 0); other rows take tlow = 2^-100 and send their zeros to the IEEE
// divide, as they do tiny, huge, infinite and NaN quotients.
// p + c for two binary32 products p (each already rounded on its own), as a
// fused multiply-add by `one`, which the host sets to exactly 1.0: the
// result is RN(p + c) lane by lane, as an addition.  A paired addition
// written as such was merged with the paired multiply that formed p into one
// fused multiply-add (a few outputs per million one unit off in the last
// place), even with contraction disabled; a multiplier the compiler cannot
// know to be 1 leaves nothing to merge.
__device__ __forceinline__ float2 add2_after_mul(float2 p, float2 c, float one) {
    return __ffma2_rn(p, make_float2(one, one), c);
}

struct DivPrep {
    float r, nd;            // RN(1/d), -d
    float tlow, thigh;      // |t| kept in [tlow, thigh] (thigh = -1: the row is refused)
};

__device__ __forceinline__ DivPrep div_prep(float d, float mean) {
    DivPrep v;
    v.r = __frcp_rn(d);
    v.nd = -d;
    const bool ok = d >= 0x1p-20f && d <= 0x1p20f && (__float_as_uint(d) & 0x7FFFFFu) <= 0x7FFFFBu;
    v.tlow = fabsf(mean) >= 0x1p-75f ? 0.0f : 0x1p-100f;
    v.thigh = ok ? __fmul_rd(d, 0x1p99f) : -1.0f;
    return v;
}

// Two quotients t / d (both lanes one divisor); *ok is cleared when a lane
// falls outside the proven ranges.  LOW: test the lower bound too (rows with
// tlow > 0).
template <bool LOW>
__device__ __forceinline__ float2 div2_prepared(float2 t, const DivPrep &v, bool *ok) {
    const float2 r = make_float2(v.r, v.r), nd = make_float2(v.nd, v.nd);
    const float2 q0 = __fmul2_rn(t, r);
    const float2 q1 = __ffma2_rn(__ffma2_rn(q0, nd, t), r, q0);
    const float2 q2 = __ffma2_rn(__ffma2_rn(q1, nd, t), r, q1);
    const float ax = fabsf(t.x), ay = fabsf(t.y);
    *ok = *ok & (ax <= v.thigh) & (ay <= v.thigh);
    if constexpr (LOW) *ok = *ok & (ax >= v.tlow) & (ay >= v.tlow);
    return q2;
}

// A group of G 16-bit elements whose chain divides by the row's d: pre(x)
// forms two elements' t (x: their binary32 values) exactly as the chain does,
// pre_w(w) the same from the word w that holds them, the quotient is
// div2_prepared's, tail(q) finishes two elements' chains in binary32 (lane by
// lane, as the scalar steps would) and exact(x) is the whole chain with the
// IEEE divide, for the elements outside the proven ranges.  The group moves as 32-bit words, two
// elements each; the rare refused pairs are recomputed in one rolled loop
// (the words rotate through slot 0, so every index stays a constant and the
// arrays stay in registers).
template <class T, int G, bool SA, class Pre, class PreW, class Tail, class Exact>
__device__ __forceinline__ void prepared_group(const T *a, T *o, const DivPrep &v, Pre pre,
                                               PreW pre_w, Tail tail, Exact exact) {
    if constexpr (G % 2 == 0 && !SA) {
        constexpr int W = G / 2;
        uint32_t aw[W], ow[W];
        memcpy(aw, a, sizeof(aw));
        bool ok = true;
        if (v.tlow == 0.0f) {   // uniform per row: the common rows test one bound
#pragma unroll
            for (int k = 0; k < W; ++k) {
                const float2 y = tail(div2_prepared<false>(pre_w(aw[k]), v, &ok));
                ow[k] = round2<T>(y.x, y.y);
            }
        } else {
#pragma unroll
            for (int k = 0; k < W; ++k) {
                const float2 y = tail(div2_prepared<true>(pre_w(aw[k]), v, &ok));
                ow[k] = round2<T>(y.x, y.y);
            }
        }
        if (!ok) {   // rare (zeros, extreme quotients): those elements again, exactly
#pragma unroll 1
            for (int k = 0; k < W; ++k) {
                const uint32_t x = aw[0];
                bool pok = true;
                div2_prepared<true>(pre_w(x), v, &pok);
                uint32_t r = ow[0];
                if (!pok)
                    r = bits_of(exact(half_of<T>(x, false))) |
                        (bits_of(exact(half_of<T>(x, true))) << 16);
#pragma unroll
                for (int i = 0; i + 1 < W; ++i) {
                    aw[i] = aw[i + 1];
                    ow[i] = ow[i + 1];
                }
                aw[W - 1] = x;
                ow[W - 1] = r;
            }
        }
        memcpy(o, ow, sizeof(ow));
    } else {
#pragma unroll
        for (int k = 0; k < G; ++k) {
            const T x = a[SA ? 0 : k];
            bool ok = true;
            const float xf = Tr<T>::in(x);
            const float2 q = div2_prepared<true>(pre(make_float2(xf, xf)), v, &ok);
            o[k] = ok ? Tr<T>::out(tail(q).x) : exact(x);
        }
    }
}

template <class T> struct OpPRelu : PlainB<T, T> {
    static constexpr bool kLegal = is_fp_v<T> || is_pow_int_v<T> ||      // ONNX PRelu T
                                   std::is_same_v<T, uint32_t> || std::is_same_v<T, uint64_t>;
    static constexpr bool kValidates = false;
    __device__ __forceinline__ static T apply(T a, T slope, const OpArgs &, uint32_t &) {
        if constexpr (is_half_like_v<T>) {
            // x >= 0 goes back through the rounding unchanged (-0 included), so
            // both branches round once and pairs of results convert together
            const float x = Tr<T>::in(a);
            return Tr<T>::out(x >= 0.0f ? x : __fmul_rn(Tr<T>::in(slope), x));
        } else if constexpr (is_fp_v<T>) {
            const auto x = Tr<T>::in(a);
            if (x >= 0) return a;                                // keeps -0 and exact bits
            return Tr<T>::out(mul_rn(Tr<T>::in(slope), x));
        } else if constexpr (Tr<T>::kSigned) {
            using U = typename Tr<T>::UT;
            return a >= 0 ? a : (T)((U)slope * (U)a);
        } else {
            return a;                                            // unsigned: never below zero
        }
    }
};

// BiasPRelu (0verkilll/onnx ops, ConvPReluOp: the per-output-channel bias add
// and PReLU fused into one pass, here as an elementwise operator): t = x + bias,
// y = t when t >= 0 else slope * t, steps in the compute type (binary32, or
// binary64 for DOUBLE) rounded once to x's type.  B holds two rows (bias,
// slope) of `plane` elements, read once per row.
template <class C> struct BiasSlope {
    C bias, slope;
};

// P: the parameter block's element type, x's own or binary32 beside a 16-bit
// or binary64 x (a float32 runtime's parameters), widened exactly to C.
template <class T, class P = T> struct OpBiasPRelu {
    using In = T;
    using Out = T;
    using BIn = P;
    using C = typename Tr<T>::C;
    using BV = BiasSlope<C>;
    static constexpr bool kPlainB = false;
    static constexpr bool kLegal = is_fp_v<T> && is_fp_v<P>;
    static constexpr bool kValidates = false;
    __device__ __forceinline__ static BV loadB(const P *B, int64_t off, const OpArgs &p) {
        return BV{(C)Tr<P>::in(B[off]), (C)Tr<P>::in(B[off + p.plane])};
    }
    __device__ __forceinline__ static T apply(T a, const BV &q, const OpArgs &, uint32_t &) {
        const C t = add_rn(Tr<T>::in(a), q.bias);
        return Tr<T>::out(t >= 0 ? t : mul_rn(q.slope, t));
    }
};

// MulAdd (0verkilll/onnx ops, MulAddOp): y = (a * b) + c, a binary32 product
// and sum each rounded on their own (never one FMA) and one rounding to a
// 16-bit type; integers wrap.  A three-input operator (apply3).
template <class T> struct OpMulAdd {
    using In = T;
    using Out = T;
    static constexpr bool kLegal = is_fp_v<T> || is_int_v<T>;
    __device__ __forceinline__ static T apply3(T a, T b, T c) {
        if constexpr (is_fp_v<T>) {
            return Tr<T>::out(add_rn(mul_rn(Tr<T>::in(a), Tr<T>::in(b)), Tr<T>::in(c)));
        } else {
            using U = typename Tr<T>::UT;
            return (T)((U)((U)a * (U)b) + (U)c);
        }
    }
};

// Inference BatchNormalization: y = (x - mean) / sqrt(var + eps) * scale + bias,
// each step rounded in the compute type (binary32, or binary64 for DOUBLE) in
// the order written.  B holds four rows (scale, bias, mean, var) of `plane`
// elements; the per-channel sqrt is formed when the parameters are loaded.
// For float16 and bfloat16 x the per-channel divisor is prepared once (its
// reciprocal) and each quotient is formed by the exact prepared division
// (div_prep / div2_prepared), the IEEE divide only outside its ranges.
template <class C> struct BNParams {
    C scale, bias, mean, d;
    DivPrep v;          // 16-bit outputs: the prepared division's row constants
};

// float16 and bfloat16 outputs (a binary32 chain) divide with the prepared
// exact division, a group of elements at a time
template <class T> constexpr bool prepared_v = is_half_like_v<T>;

// P: the parameter block's element type, as for BiasPRelu.
template <class T, class P = T> struct OpBN {
    using In = T;
    using Out = T;
    using BIn = P;
    using C = typename Tr<T>::C;
    using BV = BNParams<C>;
    // at least four rows per thread in the row kernel (x[8,64,256,256]:
    // 30.9 -> 30.2 us on GB300; six rows 30.4)
    static constexpr int kMinRows = 4;
    static constexpr bool kPlainB = false;
    static constexpr bool kLegal = is_fp_v<T> && is_fp_v<P>;
    static constexpr bool kValidates = false;
    static constexpr bool kGroup = prepared_v<T>;    // apply_group: the prepared division
    __device__ __forceinline__ static BV loadB(const P *B, int64_t off, const OpArgs &p) {
        BV r;
        r.scale = (C)Tr<P>::in(B[off]);
        r.bias = (C)Tr<P>::in(B[off + p.plane]);
        r.mean = (C)Tr<P>::in(B[off + 2 * p.plane]);
        const C var = (C)Tr<P>::in(B[off + 3 * p.plane]);
        r.d = sqrt_rn(add_rn(var, (C)p.eps));
        if constexpr (prepared_v<T>) r.v = div_prep(r.d, r.mean);
        return r;
    }
    __device__ __forceinline__ static T apply(T a, const BV &q, const OpArgs &, uint32_t &) {
        C t = sub_rn(Tr<T>::in(a), q.mean);
        t = div_rn(t, q.d);
        t = mul_rn(t, q.scale);
        return Tr<T>::out(add_rn(t, q.bias));
    }
    // G elements sharing one channel's parameters (16-bit outputs): the same
    // chain with the quotient from the prepared exact division (div_prep).
    template <int G, bool SA>
    __device__ __forceinline__ static void apply_group(const T *a, const BV &q, T *o,
                                                       const OpArgs &p, uint32_t &err) {
        // t = x - mean; t / d prepared; then * scale + bias, each lane's
        // product and sum rounded on their own (add2_after_mul)
        // (x - mean and x + (-mean) are the same IEEE operation)
        prepared_group<T, G, SA>(
            a, o, q.v, [&](float2 x) { return __fadd2_rn(x, make_float2(-q.mean, -q.mean)); },
            [&](uint32_t w) { return widen_add2<T>(w, -q.mean); },
            [&](float2 qd) {
                return add2_after_mul(__fmul2_rn(qd, make_float2(q.scale, q.scale)),
                                      make_float2(q.bias, q.bias), p.one);
            },
            [&](T x) { return apply(x, q, p, err); });
    }
};

// BiasPReluBN: the per-channel chain bias add -> PReLU -> inference
// BatchNormalization in one pass (0verkilll/onnx ops, ConvPReluOp's epilogue
// followed by BatchNormalizationOp): t = x + bias; t = t >= 0 ? t : slope * t;
// y = (t - mean) / sqrt(var + eps) * scale + bn_bias, every step rounded in the
// compute type (binary32, or binary64 for DOUBLE) in the order written, one
// rounding to x's type.  B holds six rows (bias, slope, scale, bn_bias, mean,
// var) of `plane` elements, read once per row with the sqrt formed there.
template <class C> struct ChainParams {
    C bias, slope, scale, bn_bias, mean, d;
    DivPrep v;          // 16-bit outputs: the prepared division's row constants
};

// P: the parameter block's element type, as for BiasPRelu.
template <class T, class P = T> struct OpBiasPReluBN {
    using In = T;
    using Out = T;
    using BIn = P;
    using C = typename Tr<T>::C;
    using BV = ChainParams<C>;
    static constexpr int kMinRows = 4;   // as BatchNormalization (32.6 -> 32.1 us)
    static constexpr bool kPlainB = false;
    static constexpr bool kLegal = is_fp_v<T> && is_fp_v<P>;
    static constexpr bool kValidates = false;
    __device__ __forceinline__ static BV loadB(const P *B, int64_t off, const OpArgs &p) {
        BV r;
        r.bias = (C)Tr<P>::in(B[off]);
        r.slope = (C)Tr<P>::in(B[off + p.plane]);
        r.scale = (C)Tr<P>::in(B[off + 2 * p.plane]);
        r.bn_bias = (C)Tr<P>::in(B[off + 3 * p.plane]);
        r.mean = (C)Tr<P>::in(B[off + 4 * p.plane]);
        r.d = sqrt_rn(add_rn((C)Tr<P>::in(B[off + 5 * p.plane]), (C)p.eps));
        if constexpr (prepared_v<T>) {
            r.v = div_prep(r.d, r.mean);
            // the group form takes PReLU as max(t, slope t): rows whose slope is
            // above 1, infinite or NaN take the exact chain throughout
            if (!(r.slope <= 1.0f && r.slope >= -INFINITY)) r.v.thigh = -1.0f;
        }
        return r;
    }
    __device__ __forceinline__ static T apply(T a, const BV &q, const OpArgs &, uint32_t &) {
        C t = add_rn(Tr<T>::in(a), q.bias);
        if (!(t >= 0)) t = mul_rn(q.slope, t);
        t = div_rn(sub_rn(t, q.mean), q.d);
        return Tr<T>::out(add_rn(mul_rn(t, q.scale), q.bn_bias));
    }
    static constexpr bool kGroup = prepared_v<T>;
    // G elements of one channel (16-bit outputs): the same chain with the
    // quotient from the prepared exact division (div_prep).
    template <int G, bool SA>
    __device__ __forceinline__ static void apply_group(const T *a, const BV &q, T *o,
                                                       const OpArgs &p, uint32_t &err) {
        // The bias add, PReLU and mean subtraction on pairs.  PReLU as
        // max(t1, slope t1): for a finite slope <= 1 this is t1 for t1 > 0 and
        // slope t1 for t1 < 0, as the select; for t1 = +-0 the two may give
        // zeros of other signs, which t1' - mean turns into the same t when
        // mean != 0 (rows with |mean| < 2^-75 send zero t to the exact chain);
        // an infinite t1 makes t infinite, outside the range.  No product
        // feeds an addition here (the max stands between), so nothing can be
        // contracted into a fused multiply-add.
        auto rest = [&](float2 t1) {
            const float2 s1 = __fmul2_rn(t1, make_float2(q.slope, q.slope));
            return __fadd2_rn(make_float2(fmaxf(t1.x, s1.x), fmaxf(t1.y, s1.y)),
                              make_float2(-q.mean, -q.mean));
        };
        prepared_group<T, G, SA>(
            a, o, q.v, [&](float2 x) { return rest(__fadd2_rn(x, make_float2(q.bias, q.bias))); },
            [&](uint32_t w) { return rest(widen_add2<T>(w, q.bias)); },
            [&](float2 qd) {
                return add2_after_mul(__fmul2_rn(qd, make_float2(q.scale, q.scale)),
                                      make_float2(q.bn_bias, q.bn_bias), p.one);
            },
            [&](T x) { return apply(x, q, p, err); });
    }
};

// Clip: y = x, raised to min when below it, then lowered to max when above it.
// B = {min, max}; an absent bound is never applied.  The element offset is
// ignored: the two bounds are shared by every element.
template <class T> struct ClipParams {
    typename Tr<T>::C lo, hi;
};

template <class T> struct OpClip {
    using In = T;
    using Out = T;
    using BV = ClipParams<T>;
    static constexpr bool kPlainB = false;
    static constexpr bool kLegal = is_fp_v<T> || is_int_v<T>;
    static constexpr bool kValidates = false;
    __device__ __forceinline__ static BV loadB(const T *B, int64_t, const OpArgs &p) {
        BV r{};
        if (p.has_min) r.lo = Tr<T>::in(B[0]);
        if (p.has_max) r.hi = Tr<T>::in(B[1]);
        return r;
    }
    __device__ __forceinline__ static T apply(T a, const BV &q, const OpArgs &p, uint32_t &) {
        auto y = Tr<T>::in(a);
        if (p.has_min && y < q.lo) y = q.lo;
        if (p.has_max && y > q.hi) y = q.hi;
        return Tr<T>::out(y);
    }
};

}  // namespace ebin
