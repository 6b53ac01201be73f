// quant_common.cuh -- per-group scale and E4M3 encoding used by every quantizer.
//
// Scheme ("Technical summary: Jet-RL", section "Quantization Scheme"; scale formula and
// rounding are this library's stated readings): for a group with amax = max |x|,
//     s = fl32(amax / 448),   code(x) = E4M3_rne_satfinite( fl32(x / s) ),
// and an all-zero group has s = 0 and codes 0x00.
//
// The division is the expensive part at HBM speed.  Each element is first encoded from
// q0 = RN(x * RN(1/s)).  q0 and fl32(x/s) each lie within 2^-23 relative of x/s (two
// roundings of relative size 2^-24 for q0, one for the quotient), so they are at most 3
// consecutive binary32 values apart, also across a binade boundary.  E4M3 rounding is
// monotone, so if the codes of |q0| moved 4 values down and 4 values up agree, that code
// is the code of fl32(x/s).  Otherwise (q0 close to an E4M3 rounding midpoint,
// or x = 0) the element is re-encoded from the IEEE quotient __fdiv_rn(x, s).  Groups
// whose scale is subnormal (RN(1/s) could overflow) always take the IEEE path.
#pragma once

#include "common.cuh"

namespace fp8rl {

struct GroupScale {
    float s;    // the group's scale
    float r;    // RN(1/s); unused when slow
    bool zero;  // s == 0: every code is 0x00
    bool slow;  // subnormal s: always divide
};

__device__ __forceinline__ GroupScale make_scale(float amax) {
    GroupScale g;
    g.s = __fdiv_rn(amax, 448.0f);
    g.zero = (g.s == 0.0f);
    g.slow = (g.s < 1.17549435e-38f);  // below FLT_MIN (includes zero, handled first)
    g.r = g.slow ? 0.0f : __frcp_rn(g.s);
    return g;
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

// Encode two binary32 values (exact BF16 values or any finite floats) with one group
// scale; returns the two codes packed (x0 in bits 0-7, x1 in bits 8-15).
__device__ __forceinline__ uint32_t encode_pair(float x0, float x1, const GroupScale& g) {
    if (g.zero) return 0u;
    const float q0 = x0 * g.r;
    const float q1 = x1 * g.r;
    const uint32_t a0 = __float_as_uint(q0) & 0x7FFFFFFFu;
    const uint32_t a1 = __float_as_uint(q1) & 0x7FFFFFFFu;
    const uint32_t lo = e4m3x2(__uint_as_float(a0 - 4u), __uint_as_float(a1 - 4u));
    const uint32_t hi = e4m3x2(__uint_as_float(a0 + 4u), __uint_as_float(a1 + 4u));
    if (!g.slow && lo == hi) {
        const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
        return lo | ((b0 >> 24) & 0x80u) | ((b1 >> 16) & 0x8000u);
    }
    return e4m3x2(__fdiv_rn(x0, g.s), __fdiv_rn(x1, g.s));
}

// Unpack a word of two BF16 values.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace fp8rl
