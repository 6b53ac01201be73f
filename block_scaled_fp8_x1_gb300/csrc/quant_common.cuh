// quant_common.cuh -- per-group scale and E4M3 encoding used by every quantizer.
//
// Scheme ("Technical summary: Jet-RL", section "Quantization Scheme"; scale formula and
// rounding are this library's stated readings): for a group with amax = max |x|,
//     s = fl32(amax / 448),   code(x) = E4M3_rne_satfinite( fl32(x / s) ),
// and an all-zero group has s = 0 and codes 0x00.
//
// The division is the expensive part at HBM speed: see encode_pair for how the quotient is
// formed from a reciprocal without a divide, exactly.
#pragma once

#include "common.cuh"

namespace fp8rl {

struct GroupScale {
    float s;    // the group's scale
    float r;    // RN(1/s); unused when slow
    bool zero;  // s == 0: every code is 0x00
    bool slow;  // tiny s: always divide
};

// Below this scale the division-free encode's residual could underflow for the elements
// whose code is not a signed zero (|x| >= s * 2^-11), so such groups divide instead.
constexpr float kMinFastScale = 3.3881317890172014e-21f;  // 2^-68

__device__ __forceinline__ bool scale_is_slow(float s) { return s < kMinFastScale; }

// s = fl32(amax / 448).  From amax >= 2^-60 on, by Markstein's correction step with the
// constant reciprocal RN(1/448): q = RN(amax * RN(1/448)), the residual amax - 448 q is
// exact in one FMA, and RN(q + residual * RN(1/448)) is the correctly rounded quotient
// (no intermediate is subnormal there).  Below that, IEEE division.  Every positive BF16
// amax is checked against IEEE division by the exhaustive device test.
__device__ __forceinline__ float scale_of_amax(float amax) {
    constexpr float kR448 = 0x1.24924ap-9f;  // RN(1/448)
    if (amax < 8.673617379884035e-19f)       // 2^-60
        return __fdiv_rn(amax, 448.0f);
    const float q = __fmul_rn(amax, kR448);
    const float e = __fmaf_rn(-q, 448.0f, amax);
    return __fmaf_rn(e, kR448, q);
}

__device__ __forceinline__ GroupScale make_scale(float amax) {
    GroupScale g;
    g.s = scale_of_amax(amax);
    g.zero = (g.s == 0.0f);
    g.slow = scale_is_slow(g.s);  // includes zero, which is handled first
    g.r = g.slow ? 0.0f : __frcp_rn(g.s);
    return g;
}

// Group constants of the branch-free encode.  The encode works on the negated quotient:
// with nr = -RN(1/s), q' = RN(x nr) = -RN(x/s approx), e = RN(x + q' s) is the exact
// residual and d = RN(q' + e nr) = -RN(x/s) exactly (round-to-nearest is symmetric), and
// for x = -0 / +0 it gives +0 / -0.  Converting d and flipping the code's sign bit
// therefore yields code(x/s) with the sign of zero kept, for two codes per bitwise op.
// A zero group (s = 0) has nr = 0 and code mask 0, which clears its codes to 0x00.  Slow
// groups (0 < s < 2^-68) are flagged and re-encoded by division.
struct FastScale {
    float s, nr;       // scale, -RN(1/s)
    uint32_t keep;     // code mask: 0xFFFFFFFF, or 0 for a zero group
    bool slow;
};
__device__ __forceinline__ FastScale fast_scale(float amax) {
    FastScale f;
    f.s = scale_of_amax(amax);
    f.slow = f.s > 0.0f && scale_is_slow(f.s);
    f.nr = (f.s == 0.0f || f.slow) ? 0.0f : -__frcp_rn(f.s);
    f.keep = f.s == 0.0f ? 0u : 0xFFFFFFFFu;
    return f;
}

// Negated quotients of a pair under one group (not slow), converted: the codes of
// -x0/s and -x1/s (bits 0-7 and 8-15); flip_codes() turns them into the codes of x/s.
__device__ __forceinline__ uint32_t encode_pair_neg(float2 x, float s, float nr) {
    const float2 qn = __fmul2_rn(x, make_float2(nr, nr));
    const float2 e = __ffma2_rn(qn, make_float2(s, s), x);
    const float2 d = __ffma2_rn(e, make_float2(nr, nr), qn);
    return e4m3x2(d.x, d.y);
}
// The same for a pair whose two elements belong to different groups (two columns of one
// row under their 128x1 column scales): s = (s0, s1), nr = (nr0, nr1).
__device__ __forceinline__ uint32_t encode_pair_neg2(float2 x, float2 s, float2 nr) {
    const float2 qn = __fmul2_rn(x, nr);
    const float2 e = __ffma2_rn(qn, s, x);
    const float2 d = __ffma2_rn(e, nr, qn);
    return e4m3x2(d.x, d.y);
}
// Four codes (two encode_pair_neg results packed) -> codes of x/s, zero groups cleared.
__device__ __forceinline__ uint32_t flip_codes(uint32_t lo_pair, uint32_t hi_pair, uint32_t keep) {
    return ((lo_pair | (hi_pair << 16)) ^ 0x80808080u) & keep;
}

// Branch-free encode of one pair (for the exhaustive check): codes of x/s in bits 0-15.
__device__ __forceinline__ uint32_t encode_pair_fast(float2 x, float s, float nr, uint32_t keep) {
    return flip_codes(encode_pair_neg(x, s, nr), 0u, keep) & 0xFFFFu;
}

// amax of BF16 values given as raw bits, compared as integers (|x| order equals the
// order of the 15 low bits for finite values).
__device__ __forceinline__ float bf16_bits_amax_to_f32(uint32_t absbits16) {
    return __uint_as_float(absbits16 << 16);
}

// Max of |bf16| over the two halves of each packed word, kept packed (max per half).
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) {
    return __vmaxu2(acc, w & 0x7FFF7FFFu);
}

// Encode two BF16 values (given as binary32) with one group scale; returns the two codes
// packed (x0 in bits 0-7, x1 in bits 8-15).
//
// fl32(x/s) is formed without a divide by Markstein's correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with r = RN(1/s) and q = RN(x*r), the residual e = x - s*q is exact in
// one fused multiply-add and RN(q + e*r) is the correctly rounded quotient.  Both steps run
// on packed FP32x2 pairs.  The sign is copied from x so that -0 keeps its code 0x80.
// Groups with s < 2^-68 take IEEE division: there the residual of an element whose code
// is not a signed zero could fall below the normal range, and the step needs it exact
// (for s >= 2^-68 such elements have |x| >= s * 2^-11, so the residual stays far above
// it; smaller elements encode to a signed zero whatever the last bits).  Every BF16 x
// against every BF16 group maximum is checked against IEEE division by the exhaustive
// device test (fp8rl_debug_encode_check).
__device__ __forceinline__ uint32_t encode_pair(float x0, float x1, const GroupScale& g) {
    if (g.zero) return 0u;
    if (g.slow) return e4m3x2(__fdiv_rn(x0, g.s), __fdiv_rn(x1, g.s));
    const float2 x = make_float2(x0, x1);
    const float2 q = __fmul2_rn(x, make_float2(g.r, g.r));
    const float2 e = __ffma2_rn(q, make_float2(-g.s, -g.s), x);
    const float2 c = __ffma2_rn(e, make_float2(g.r, g.r), q);
    const float c0 = __uint_as_float((__float_as_uint(c.x) & 0x7FFFFFFFu) | (__float_as_uint(x0) & 0x80000000u));
    const float c1 = __uint_as_float((__float_as_uint(c.y) & 0x7FFFFFFFu) | (__float_as_uint(x1) & 0x80000000u));
    return e4m3x2(c0, c1);
}

// Reference: the same codes from the IEEE quotient (used by the exhaustive check only).
__device__ __forceinline__ uint32_t encode_pair_ieee(float x0, float x1, const GroupScale& g) {
    if (g.zero) return 0u;
    return e4m3x2(__fdiv_rn(x0, g.s), __fdiv_rn(x1, g.s));
}

// Unpack a word of two BF16 values.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace fp8rl
