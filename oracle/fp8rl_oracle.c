/*
 * fp8rl_oracle.c -- plain, slow CPU oracle for the unified-precision FP8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library, its Python
 * binding) may link, load or call this file.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * What it follows: "Technical summary: Jet-RL" (gist.science, paper 2601.14243):
 *   - section "Quantization Scheme": activations are quantized per 1x128 group, weights per
 *     128x128 block, DGrad and WGrad run in FP8 with 1x128 and 128x1 operand quantization;
 *     saved activations are FP8 and produced by the preceding fused operator; gradients
 *     between operators stay BF16.
 *   - section "Core architecture": rollout and training forward share the same quantization
 *     granularity and precision (one quantizer, one GEMM numerics).
 *   - section "Implementation": fused activation (SiLU-mul) and RMSNorm kernels feed the
 *     quantizer.
 * The pages fix no formula.  Readings taken here (each is also listed in the design notes):
 *   R1  FP8 format = OCP E4M3 "FN": bias 7, max 448, no infinities, 0x7F/0xFF = NaN.
 *   R2  scale s = fl32(amax / 448) (IEEE single division); an all-zero group has s = 0 and
 *       all codes 0x00.
 *   R3  code = E4M3 round-to-nearest-even of fl32(x / s), saturating at +-448; the sign of a
 *       value that rounds to zero is kept (0x80 for negative).
 *   R4  block-scaled GEMM: per reduction block kb of 128, P_kb = sum of decoded products
 *       (exact in binary64), y = sum_kb sa*sb*P_kb in binary64, unrounded.
 *   R5  RMSNorm: sum of squares in binary64, ms = fl32(sum/K), rstd = 1/sqrt(ms+eps) in
 *       IEEE single, y = bf16_rne((x*rstd)*gamma) in IEEE single; y is rounded to BF16
 *       before it is quantized.
 *   R6  SiLU-mul: h = bf16_rne(silu(g)*u) evaluated in binary64, g = first I columns.
 *   R7  SiLU-mul backward (the chain rule of R6): with s = 1/(1+exp(-g)),
 *       dg = dh*u*s*(1 + g*(1-s)) and du = dh*g*s in binary64, each rounded to BF16 (the
 *       gradient between operators is BF16); [dg | du] is then quantized as a gradient.
 *   R9  WGrad operand from the saved FP8 activation (the memory-saving variant): the
 *       1x128 codes and scales of X are dequantized back to the BF16 activation,
 *       x^ = bf16_rne(fl32(decode(q) * s)), and x^ is quantized 128x1 (R2, R3) along the
 *       token dimension, as the BF16 path quantizes X itself.
 *   R8  RMSNorm backward (the chain rule of R5 through rstd, the BF16 rounding of y taken
 *       as the identity): with r the forward's rstd and S = sum_k dy_k*gamma_k*x_k,
 *       dx_j = r*gamma_j*dy_j - r^3*x_j*S/K in binary64, rounded to BF16;
 *       dgamma_k = sum_m dy_mk*x_mk*r_m in binary64.
 *   R10 NVFP4, the format the QeRL page names for rollout (the pages fix nothing else, so
 *       the format's public definition): elements are FP4 E2M1 (values 0, 0.5, 1, 1.5, 2,
 *       3, 4, 6 and their negatives), 16 consecutive elements of a row share one E4M3
 *       block scale, and an FP32 second-level scale is applied on top.  Reading: the
 *       second-level scale is per row (per output channel of a weight, per token of an
 *       activation).  For a row with amax a:  g = fl32(a / 2688)  (2688 = 6 * 448);  a
 *       block with amax b gets the E4M3 code sb = E4M3(fl32(b / fl32(6 g))) (R3's
 *       rounding, saturating at 448) and the decode scale d = fl32(decode(sb) * g); each
 *       element gets code E2M1(fl32(x / d)), round to nearest even, saturating at +-6, the
 *       sign kept for values that round to zero.  d = 0 (an all-zero row, or a block too
 *       small for E4M3 against its row) gives codes 0.  x^ = e2m1 * decode(sb) * g.
 *   R11 NVFP4 GEMM: y[m][n] = gx[m] * gw[n] * sum_k e2m1(x_mk) sbx * e2m1(w_nk) sbw in
 *       binary64, unrounded (each product of decoded codes and block scales is exact).
 *
 * Every routine is written as the plain definition: scalar loops, no blocking or fusion.
 * Independent groups are spread over OpenMP threads only to make big inputs finish.
 * Compile with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

static int g_threads = 1;

ORC_API void orc_set_threads(int n) { g_threads = n > 0 ? n : 1; }
ORC_API int orc_get_threads(void) { return g_threads; }
ORC_API int orc_have_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* ---------------------------------------------------------------- BF16 (R5, R6) */

/* BF16 -> binary32 is exact: the BF16 bits are the top half of the binary32 bits. */
ORC_API float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t f32_bits_hi(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Round a finite binary64 value to the nearest BF16, ties to the even significand.
 * Definition: in v's binade the BF16 grid has spacing 2^(e-7); the two grid points that
 * bracket |v| are compared by distance, and a tie goes to the even multiple of the spacing
 * (the one whose last significand bit is 0). */
ORC_API uint16_t orc_f64_to_bf16(double v) {
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int neg = v < 0;
    double a = fabs(v);
    /* BF16 has 8 significant bits; spacing at a is 2^(e-7) for a in [2^e, 2^(e+1)),
       and 2^-133 in the subnormal range (below 2^-126). */
    int e;
    frexp(a, &e);
    e -= 1;
    if (e < -126) e = -126;
    double ulp = ldexp(1.0, e - 7);
    double n = a / ulp; /* exact: scaling by a power of two */
    double lo = floor(n), hi = lo + 1.0;
    double r;
    if (n - lo < hi - n) r = lo;
    else if (n - lo > hi - n) r = hi;
    else r = (fmod(lo, 2.0) == 0.0) ? lo : hi;
    double mag = r * ulp;
    /* mag is exactly a BF16 value (or 2^128 on overflow, which finite inputs here never
       reach); read its bits through binary32, where it is exact. */
    float f = (float)(neg ? -mag : mag);
    return f32_bits_hi(f);
}

ORC_API uint16_t orc_f32_to_bf16(float v) { return orc_f64_to_bf16((double)v); }

/* ---------------------------------------------------------------- E4M3 (R1, R3) */

/* Decode an E4M3 code: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN; there is no infinity. */
ORC_API double orc_e4m3_decode(uint8_t b) {
    int sign = b >> 7;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Encode a finite binary32 value as E4M3: round to nearest, ties to even, saturating at
 * +-448.  Magnitudes below 2^-6 use the subnormal spacing 2^-9; a normal binade [2^e,2^(e+1))
 * has spacing 2^(e-3).  The rounded integer count of spacings is even exactly when the
 * mantissa field is even, so ties-to-even on the count is ties-to-even on the code. */
ORC_API uint8_t orc_e4m3_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    int e;
    if (a < ldexp(1.0, -6)) {
        e = -6;
    } else {
        frexp(a, &e);
        e -= 1;
    }
    double ulp = ldexp(1.0, e - 3);
    double n = a / ulp;
    double lo = floor(n), hi = lo + 1.0;
    double r;
    if (n - lo < hi - n) r = lo;
    else if (n - lo > hi - n) r = hi;
    else r = (fmod(lo, 2.0) == 0.0) ? lo : hi;
    double mag = r * ulp; /* <= 448 because a < 448 and 448 is a grid point */
    if (mag == 0.0) return sign;
    if (mag < ldexp(1.0, -6)) return sign | (uint8_t)(mag / ldexp(1.0, -9));
    int e2;
    frexp(mag, &e2);
    e2 -= 1;
    int m = (int)((mag / ldexp(1.0, e2) - 1.0) * 8.0);
    return sign | (uint8_t)(((e2 + 7) << 3) | m);
}

ORC_API void orc_e4m3_encode_array(const float* v, uint8_t* out, int64_t n) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

/* Encode every binary32 pattern in [first, first+count) (as raw bits). */
ORC_API void orc_e4m3_encode_bits_range(uint32_t first, int64_t count, uint8_t* out) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < count; ++i) {
        uint32_t u = first + (uint32_t)i;
        float f;
        memcpy(&f, &u, sizeof f);
        out[i] = orc_e4m3_encode(f);
    }
}

/* ---------------------------------------------------------------- one quantization group */

/* Quantize n values read from x[i*xs] (binary32, already exact copies of BF16 inputs):
 * amax = max |x|, s = fl32(amax/448), code_i = E4M3(fl32(x_i/s)); s = 0 gives zero codes. */
static void quant_group(const float* x, int64_t n, int64_t xs, uint8_t* q, int64_t qs,
                        float* s_out) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i * xs]);
        if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    *s_out = s;
    for (int64_t i = 0; i < n; ++i) {
        if (s == 0.0f) q[i * qs] = 0x00;
        else q[i * qs] = orc_e4m3_encode(x[i * xs] / s);
    }
}

ORC_API void orc_quant_group_f32(const float* x, int64_t n, uint8_t* q, float* s) {
    quant_group(x, n, 1, q, 1, s);
}

/* ---------------------------------------------------------------- quantizers */

/* 1x128 groups along the columns of a BF16 matrix A[R,C] (row stride lda, C % 128 == 0).
 * Codes q[r*ldq + c]; scales s[(c/128)*R + r]  (reduction-block-major). */
ORC_API void orc_quantize_1x128(const uint16_t* a, int64_t R, int64_t C, int64_t lda,
                                uint8_t* q, int64_t ldq, float* s) {
    int64_t nb = C / 128;
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t r = 0; r < R; ++r) {
        float buf[128];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 128; ++i) buf[i] = orc_bf16_to_f32(a[r * lda + b * 128 + i]);
            quant_group(buf, 128, 1, q + r * ldq + b * 128, 1, &s[b * R + r]);
        }
    }
}

/* 128x1 groups: 128 consecutive rows of one column of X[M,K] (M % 128 == 0).  By definition
 * this is the 1x128 quantization of the transpose: codes qT[k*ldqt + m], scales
 * sT[(m/128)*K + k].  Written literally as transpose-then-quantize. */
ORC_API void orc_quantize_128x1(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                uint8_t* qT, int64_t ldqt, float* sT) {
    int64_t nb = M / 128;
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t k = 0; k < K; ++k) {
        float buf[128];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 128; ++i) buf[i] = orc_bf16_to_f32(x[(b * 128 + i) * ldx + k]);
            quant_group(buf, 128, 1, qT + k * ldqt + b * 128, 1, &sT[b * K + k]);
        }
    }
}

/* 128x128 blocks of a BF16 weight W[N,K] (N, K multiples of 128).  Codes q[n*ldq + k],
 * scales s[(n/128)*(K/128) + k/128].  The transposed copy qT[k*N + n] holds the same codes
 * (a block is one group, so its transpose needs no new scale). */
ORC_API void orc_quantize_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw,
                                  uint8_t* q, int64_t ldq, float* s, uint8_t* qT) {
    int64_t nbn = N / 128, nbk = K / 128;
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t bn = 0; bn < nbn; ++bn) {
        static __thread float buf[128 * 128];
        static __thread uint8_t qb[128 * 128];
        for (int64_t bk = 0; bk < nbk; ++bk) {
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j)
                    buf[i * 128 + j] = orc_bf16_to_f32(w[(bn * 128 + i) * ldw + bk * 128 + j]);
            quant_group(buf, 128 * 128, 1, qb, 1, &s[bn * nbk + bk]);
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    q[(bn * 128 + i) * ldq + bk * 128 + j] = qb[i * 128 + j];
                    if (qT) qT[(bk * 128 + j) * N + bn * 128 + i] = qb[i * 128 + j];
                }
        }
    }
}

/* ---------------------------------------------------------------- RMSNorm (R5) */

/* y[M,K] = bf16_rne((x*rstd)*gamma).  rstd_out (nullable) receives rstd.  If rstd_in is
 * given, its values replace the computed rstd (used to re-check downstream bytes against a
 * device rstd that differs in the last place). */
ORC_API void orc_rmsnorm(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M,
                         int64_t K, uint16_t* y, float* rstd_out, const float* rstd_in) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t m = 0; m < M; ++m) {
        double sum = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = (double)orc_bf16_to_f32(x[m * K + k]);
            sum += v * v;
        }
        float ms = (float)(sum / (double)K);
        float rstd = 1.0f / sqrtf(ms + eps);
        if (rstd_in) rstd = rstd_in[m];
        if (rstd_out) rstd_out[m] = rstd;
        for (int64_t k = 0; k < K; ++k) {
            float xv = orc_bf16_to_f32(x[m * K + k]);
            float g = orc_bf16_to_f32(gamma[k]);
            float t = xv * rstd;
            float yv = t * g;
            y[m * K + k] = orc_f32_to_bf16(yv);
        }
    }
}

/* ---------------------------------------------------------------- SiLU-mul (R6) */

/* Distance test: is the binary64 value v within rel*|v| of a BF16 rounding midpoint? */
static int near_bf16_midpoint(double v, double rel) {
    if (v == 0.0) return 0;
    double a = fabs(v);
    int e;
    frexp(a, &e);
    e -= 1;
    if (e < -126) e = -126;
    double ulp = ldexp(1.0, e - 7);
    double mid = (floor(a / ulp) + 0.5) * ulp;
    return fabs(a - mid) <= rel * a;
}

/* gu[M, 2I] holds g = gu[:, :I] and u = gu[:, I:].  h[M,I] = bf16_rne(silu(g)*u) from a
 * binary64 evaluation, silu(g) = g / (1 + exp(-g)).  alt[M,I] (nullable) receives the other
 * BF16 neighbour where the binary64 value lies within 2^-16 relative of a BF16 midpoint
 * (there a binary32 evaluation may round either way), else a copy of h.  Returns the count
 * of such near-midpoint elements. */
ORC_API int64_t orc_silu_mul(const uint16_t* gu, int64_t M, int64_t I, uint16_t* h,
                             uint16_t* alt) {
    int64_t flagged = 0;
    #pragma omp parallel for schedule(static) num_threads(g_threads) reduction(+ : flagged)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t i = 0; i < I; ++i) {
            double g = (double)orc_bf16_to_f32(gu[m * 2 * I + i]);
            double u = (double)orc_bf16_to_f32(gu[m * 2 * I + I + i]);
            double sg = g / (1.0 + exp(-g));
            double v = sg * u;
            uint16_t hb = orc_f64_to_bf16(v);
            h[m * I + i] = hb;
            if (alt) {
                alt[m * I + i] = hb;
                if (near_bf16_midpoint(v, ldexp(1.0, -16))) {
                    /* the two BF16 neighbours of v, taken in v's binade */
                    double a = fabs(v);
                    int e;
                    frexp(a, &e);
                    e -= 1;
                    if (e < -126) e = -126;
                    double ulp = ldexp(1.0, e - 7);
                    double lo = floor(a / ulp) * ulp, hi = lo + ulp;
                    double hv = fabs((double)orc_bf16_to_f32(hb));
                    double other = (hv == lo) ? hi : lo;
                    alt[m * I + i] = orc_f64_to_bf16(v < 0 ? -other : other);
                    flagged += 1;
                }
            }
        }
    }
    return flagged;
}

/* ---------------------------------------------------------------- requantization (R9) */

/* From the 1x128 codes q[M][K] and scales s[K/128][M] of X: the 128x1 quantization of the
 * dequantized x^ = bf16_rne(fl32(decode(q) * s)), transposed like orc_quantize_128x1:
 * codes qT[k*M + m], scales sT[(m/128)*K + k].  M % 128 == 0, K % 128 == 0. */
ORC_API void orc_requant_128x1(const uint8_t* q, const float* s, int64_t M, int64_t K, uint8_t* qT,
                               float* sT) {
    int64_t nmb = M / 128;
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t k = 0; k < K; ++k) {
        float buf[128];
        for (int64_t mb = 0; mb < nmb; ++mb) {
            for (int i = 0; i < 128; ++i) {
                int64_t m = mb * 128 + i;
                float v = (float)orc_e4m3_decode(q[m * K + k]) * s[(k / 128) * M + m];
                buf[i] = orc_bf16_to_f32(orc_f32_to_bf16(v));
            }
            quant_group(buf, 128, 1, qT + k * M + mb * 128, 1, &sT[mb * K + k]);
        }
    }
}

/* ---------------------------------------------------------------- SiLU-mul backward (R7) */

/* The two BF16 neighbours of v: the one v rounds to is `b`; returns the other. */
static uint16_t other_bf16_neighbour(double v, uint16_t b) {
    double a = fabs(v);
    int e;
    frexp(a, &e);
    e -= 1;
    if (e < -126) e = -126;
    double ulp = ldexp(1.0, e - 7);
    double lo = floor(a / ulp) * ulp, hi = lo + ulp;
    double bv = fabs((double)orc_bf16_to_f32(b));
    double other = (bv == lo) ? hi : lo;
    return orc_f64_to_bf16(v < 0 ? -other : other);
}

/* gu[M, 2I] holds the forward's g = gu[:, :I] and u = gu[:, I:]; dh[M, I] is the gradient
 * of h.  dgu[M, 2I] receives dg in columns [0, I) and du in [I, 2I), each bf16_rne of a
 * binary64 evaluation.  alt[M, 2I] (nullable) receives the other BF16 neighbour where a
 * binary32 evaluation may round either way, else a copy: where the binary64 value lies
 * within 2^-16 of a BF16 midpoint, relative to the size of the terms it is made of (dg =
 * dh*u*s + dh*u*s*g*(1-s) cancels near g = -1.28, where silu' = 0).  Returns the count of
 * such near-midpoint elements. */
ORC_API int64_t orc_silu_mul_bwd(const uint16_t* gu, const uint16_t* dh, int64_t M, int64_t I,
                                 uint16_t* dgu, uint16_t* alt) {
    int64_t flagged = 0;
    #pragma omp parallel for schedule(static) num_threads(g_threads) reduction(+ : flagged)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t i = 0; i < I; ++i) {
            double g = (double)orc_bf16_to_f32(gu[m * 2 * I + i]);
            double u = (double)orc_bf16_to_f32(gu[m * 2 * I + I + i]);
            double d = (double)orc_bf16_to_f32(dh[m * I + i]);
            double sg = 1.0 / (1.0 + exp(-g));
            double dg = d * u * sg * (1.0 + g * (1.0 - sg));
            double du = d * (g * sg);
            double v[2] = {dg, du};
            /* size of the terms, relative to the value: 1 for the product du */
            double cond[2] = {dg != 0.0 ? fabs(d * u * sg) * (1.0 + fabs(g * (1.0 - sg))) / fabs(dg) : 1.0, 1.0};
            int64_t col[2] = {i, I + i};
            for (int h = 0; h < 2; ++h) {
                uint16_t b = orc_f64_to_bf16(v[h]);
                dgu[m * 2 * I + col[h]] = b;
                if (alt) {
                    alt[m * 2 * I + col[h]] = b;
                    if (near_bf16_midpoint(v[h], ldexp(1.0, -16) * cond[h])) {
                        alt[m * 2 * I + col[h]] = other_bf16_neighbour(v[h], b);
                        flagged += 1;
                    }
                }
            }
        }
    }
    return flagged;
}

/* ---------------------------------------------------------------- RMSNorm backward (R8) */

/* x[M,K], gamma[K], rstd[M] (the forward's), dy[M,K] -> dx[M,K] = bf16_rne of the binary64
 * value; mag[M,K] (nullable) receives |r*gamma*dy| + |r^3*x*S/K| (the size of the two terms,
 * for error bounds); dgamma[K] (nullable) receives sum_m dy*x*r in binary64. */
ORC_API void orc_rmsnorm_bwd(const uint16_t* x, const uint16_t* gamma, const float* rstd,
                             const uint16_t* dy, int64_t M, int64_t K, uint16_t* dx,
                             double* mag, double* dgamma) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t m = 0; m < M; ++m) {
        double r = (double)rstd[m];
        double S = 0.0;
        for (int64_t k = 0; k < K; ++k)
            S += (double)orc_bf16_to_f32(dy[m * K + k]) * (double)orc_bf16_to_f32(gamma[k]) *
                 (double)orc_bf16_to_f32(x[m * K + k]);
        for (int64_t k = 0; k < K; ++k) {
            double xv = (double)orc_bf16_to_f32(x[m * K + k]);
            double t1 = r * (double)orc_bf16_to_f32(gamma[k]) * (double)orc_bf16_to_f32(dy[m * K + k]);
            double t2 = r * r * r * xv * S / (double)K;
            dx[m * K + k] = orc_f64_to_bf16(t1 - t2);
            if (mag) mag[m * K + k] = fabs(t1) + fabs(t2);
        }
    }
    if (dgamma) {
        #pragma omp parallel for schedule(static) num_threads(g_threads)
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m)
                acc += (double)orc_bf16_to_f32(dy[m * K + k]) * (double)orc_bf16_to_f32(x[m * K + k]) *
                       (double)rstd[m];
            dgamma[k] = acc;
        }
    }
}

/* ---------------------------------------------------------------- block-scaled GEMM (R4) */

/* One output element of C[r1, r2] = sum over reduction blocks kb of
 *     sa(kb, r1) * sb(kb, r2) * sum_{k in kb} dec(A[r1,k]) * dec(B[r2,k])
 * A is [R1, Kr] codes (row stride lda), B is [R2, Kr] codes (row stride ldb); both hold the
 * reduction dimension contiguously.  Scale indexing:
 *     sa(kb, r1) = sa[kb*sa_kb + r1]
 *     sb(kb, r2) = sb[kb*sb_kb + (r2/sb_rdiv)*sb_r]
 * Forward (B = W, 128x128 blocks):  sb_rdiv = 128, sb_r = Kr/128, sb_kb = 1.
 * DGrad   (B = W^T, same blocks):   sb_rdiv = 128, sb_r = 1,      sb_kb = R2/128.
 * WGrad   (B = X^T, 128x1 groups):  sb_rdiv = 1,   sb_r = 1,      sb_kb = R2.
 * Each block's partial sum is exact in binary64 (codes are multiples of 2^-9 below 448, so
 * a 128-term sum spans fewer than 53 bits); the scale products are exact in binary64. */
static double gemm_elem(const uint8_t* A, int64_t lda, const float* sa, int64_t sa_kb,
                        const uint8_t* B, int64_t ldb, const float* sb, int64_t sb_kb,
                        int64_t sb_r, int64_t sb_rdiv, int64_t Kr, int64_t r1, int64_t r2) {
    double y = 0.0;
    for (int64_t kb = 0; kb < Kr / 128; ++kb) {
        double p = 0.0;
        for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
            p += orc_e4m3_decode(A[r1 * lda + k]) * orc_e4m3_decode(B[r2 * ldb + k]);
        double scale = (double)sa[kb * sa_kb + r1] * (double)sb[kb * sb_kb + (r2 / sb_rdiv) * sb_r];
        y += scale * p;
    }
    return y;
}

/* Full output y[R1, R2] (binary64, unrounded). */
ORC_API void orc_gemm(const uint8_t* A, int64_t lda, const float* sa, int64_t sa_kb,
                      const uint8_t* B, int64_t ldb, const float* sb, int64_t sb_kb,
                      int64_t sb_r, int64_t sb_rdiv, int64_t R1, int64_t R2, int64_t Kr,
                      double* y) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t r1 = 0; r1 < R1; ++r1)
        for (int64_t r2 = 0; r2 < R2; ++r2)
            y[r1 * R2 + r2] = gemm_elem(A, lda, sa, sa_kb, B, ldb, sb, sb_kb, sb_r, sb_rdiv, Kr,
                                        r1, r2);
}

/* Sampled outputs: y[i] = C[r1[i], r2[i]]. */
ORC_API void orc_gemm_sampled(const uint8_t* A, int64_t lda, const float* sa, int64_t sa_kb,
                              const uint8_t* B, int64_t ldb, const float* sb, int64_t sb_kb,
                              int64_t sb_r, int64_t sb_rdiv, int64_t Kr, const int64_t* r1,
                              const int64_t* r2, int64_t n, double* y) {
    #pragma omp parallel for schedule(dynamic, 16) num_threads(g_threads)
    for (int64_t i = 0; i < n; ++i)
        y[i] = gemm_elem(A, lda, sa, sa_kb, B, ldb, sb, sb_kb, sb_r, sb_rdiv, Kr, r1[i], r2[i]);
}

/* ---------------------------------------------------------------- NVFP4 (R10, R11) */

/* Decode an E2M1 code (bits 0-3): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * Exponent field 0 is subnormal (m * 0.5); the format has no infinity and no NaN. */
ORC_API double orc_e2m1_decode(uint8_t c) {
    int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* Encode a finite binary32 value as E2M1: round to nearest, ties to even, saturating at
 * +-6.  Below 2 the grid spacing is 0.5 (the subnormals 0, 0.5 and the binade [1, 2)),
 * [2, 4) has spacing 1 and [4, 8) spacing 2.  As for E4M3, ties to the even count of
 * spacings are ties to the even mantissa bit. */
ORC_API uint8_t orc_e2m1_encode(float v) {
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs((double)v);
    if (a >= 6.0) return sign | 0x7;
    double ulp = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double n = a / ulp;
    double lo = floor(n), hi = lo + 1.0;
    double r;
    if (n - lo < hi - n) r = lo;
    else if (n - lo > hi - n) r = hi;
    else r = (fmod(lo, 2.0) == 0.0) ? lo : hi;
    double mag = r * ulp; /* one of 0, 0.5, 1, 1.5, 2, 3, 4, 6 */
    if (mag < 1.0) return sign | (uint8_t)(mag * 2.0);
    int e;
    frexp(mag, &e);
    e -= 1; /* mag in [2^e, 2^(e+1)) */
    int m = (int)((mag / ldexp(1.0, e) - 1.0) * 2.0);
    return sign | (uint8_t)(((e + 1) << 1) | m);
}

ORC_API void orc_e2m1_encode_array(const float* v, uint8_t* out, int64_t n) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_encode(v[i]);
}

/* Encode every binary32 pattern in [first, first+count) (as raw bits). */
ORC_API void orc_e2m1_encode_bits_range(uint32_t first, int64_t count, uint8_t* out) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < count; ++i) {
        uint32_t u = first + (uint32_t)i;
        float f;
        memcpy(&f, &u, sizeof f);
        out[i] = orc_e2m1_encode(f);
    }
}

/* NVFP4 quantization of the rows of x[M][K] (BF16 bits, row stride ldx), R10.
 * q[M][K/2]: element k of a row in bits 4*(k%2) .. 4*(k%2)+3 of byte k/2;
 * sf[M][K/16]: the E4M3 block scales; g[M]: the per-row FP32 scales. */
ORC_API void orc_quantize_nvfp4(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                                uint8_t* sf, float* g) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t r = 0; r < M; ++r) {
        const uint16_t* row = x + r * ldx;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(orc_bf16_to_f32(row[k]));
            if (a > amax) amax = a;
        }
        float gr = amax / 2688.0f;
        g[r] = gr;
        float g6 = 6.0f * gr;
        for (int64_t b = 0; b < K / 16; ++b) {
            float bmax = 0.0f;
            for (int64_t k = 16 * b; k < 16 * b + 16; ++k) {
                float a = fabsf(orc_bf16_to_f32(row[k]));
                if (a > bmax) bmax = a;
            }
            uint8_t sb = gr > 0.0f ? orc_e4m3_encode(bmax / g6) : 0x00;
            sf[r * (K / 16) + b] = sb;
            float dsb = (float)orc_e4m3_decode(sb);
            float d = dsb * gr;
            for (int64_t k = 16 * b; k < 16 * b + 16; ++k) {
                uint8_t c = d > 0.0f ? orc_e2m1_encode(orc_bf16_to_f32(row[k]) / d) : 0x0;
                uint8_t* byte = q + r * (K / 2) + k / 2;
                if (k % 2 == 0) *byte = c;
                else *byte = (uint8_t)(*byte | (c << 4));
            }
        }
    }
}

/* x^[m][k] of R10 without the per-row scale: e2m1(code) * decode(sb), exact. */
static double nvfp4_elem(const uint8_t* q, const uint8_t* sf, int64_t K, int64_t r, int64_t k) {
    uint8_t byte = q[r * (K / 2) + k / 2];
    uint8_t c = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    return orc_e2m1_decode(c) * orc_e4m3_decode(sf[r * (K / 16) + k / 16]);
}

static double nvfp4_gemm_elem(const uint8_t* qx, const uint8_t* sfx, const float* gx, const uint8_t* qw,
                              const uint8_t* sfw, const float* gw, int64_t K, int64_t m, int64_t n) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += nvfp4_elem(qx, sfx, K, m, k) * nvfp4_elem(qw, sfw, K, n, k);
    return (double)gx[m] * (double)gw[n] * acc;
}

/* y[M][N] of R11 (binary64, unrounded). */
ORC_API void orc_gemm_nvfp4(const uint8_t* qx, const uint8_t* sfx, const float* gx, int64_t M, const uint8_t* qw,
                            const uint8_t* sfw, const float* gw, int64_t N, int64_t K, double* y) {
    #pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) y[m * N + n] = nvfp4_gemm_elem(qx, sfx, gx, qw, sfw, gw, K, m, n);
}

/* Sampled outputs of R11: y[i] = y[m[i]][n[i]]. */
ORC_API void orc_gemm_nvfp4_sampled(const uint8_t* qx, const uint8_t* sfx, const float* gx, const uint8_t* qw,
                                    const uint8_t* sfw, const float* gw, int64_t K, const int64_t* m,
                                    const int64_t* n, int64_t count, double* y) {
    #pragma omp parallel for schedule(dynamic, 16) num_threads(g_threads)
    for (int64_t i = 0; i < count; ++i) y[i] = nvfp4_gemm_elem(qx, sfx, gx, qw, sfw, gw, K, m[i], n[i]);
}
