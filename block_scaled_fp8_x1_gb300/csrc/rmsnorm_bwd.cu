// rmsnorm_bwd.cu -- RMSNorm backward from the forward's saved rstd.
//
// "Technical summary: Jet-RL", section "Quantization Scheme": gradients between operators
// stay BF16.  The forward is y = (x * r) * gamma with r = rstd = 1/sqrt(mean(x^2) + eps)
// (its BF16 rounding passed straight through), so by the chain rule, with
// S = sum_k dy_k * gamma_k * x_k over the row,
//     dx_j     = r * gamma_j * dy_j - r^3 * x_j * S / K          (rounded to BF16)
//     dgamma_k = sum_m dy_mk * x_mk * r_m                          (FP32)
//
// k_rms_bwd: each CTA (one per SM) takes a block of rows; thread t holds columns
// 8t + 8 NT i of a row (16-byte loads), the row's S is reduced over the CTA in a fixed
// order, dx is written as BF16, and the thread's share of dgamma is accumulated over the
// CTA's rows with a compensated (two-sum) FP32 pair.  The per-CTA partials go to a workspace that
// k_rms_bwd_colsum adds in block order, so the result does not depend on timing.
#include "common.cuh"
#include "gemm.h"

namespace fp8rl {

namespace {


__device__ __forceinline__ uint4 ldg_v4(const uint16_t* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// (hi, lo) += v with the exact two-sum, on packed pairs (a - b formed as fma(b, -1, a),
// which is exact).
__device__ __forceinline__ void two_sum_add2(float2& hi, float2& lo, float2 v) {
    const float2 m1 = make_float2(-1.0f, -1.0f);
    const float2 s = __fadd2_rn(hi, v);
    const float2 bp = __ffma2_rn(hi, m1, s);
    const float2 e = __fadd2_rn(__ffma2_rn(__ffma2_rn(bp, m1, s), m1, hi), __ffma2_rn(bp, m1, v));
    hi = s;
    lo = __fadd2_rn(lo, e);
}

// (hi, lo) += v with the exact two-sum.
__device__ __forceinline__ void two_sum_add(float& hi, float& lo, float v) {
    const float s = __fadd_rn(hi, v);
    const float bp = __fsub_rn(s, hi);
    const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(v, bp));
    hi = s;
    lo = __fadd_rn(lo, e);
}

}  // namespace

template <int NCH, int NT>
__global__ void __launch_bounds__(NT, 1) k_rms_bwd(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma,
                                                         const float* __restrict__ rstd, const uint16_t* __restrict__ dy,
                                                         int64_t M, int64_t K, uint16_t* __restrict__ dx,
                                                         float* __restrict__ ws) {
    constexpr int kBwdChunk = 8 * NT;   // columns per pass of the CTA over a row
    __shared__ float s_part[2][NT / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t rows = (M + gridDim.x - 1) / gridDim.x;
    const int64_t m_begin = (int64_t)blockIdx.x * rows;
    const int64_t m_end = m_begin + rows < M ? m_begin + rows : M;

    // every per-element operation below runs on packed pairs (columns 2j, 2j + 1)
    float2 gam[NCH][4];
    bool valid[NCH];
    #pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int64_t c = (int64_t)i * kBwdChunk + 8 * tid;
        valid[i] = c < K;
        const uint4 g = valid[i] ? ldg_v4(gamma + c) : make_uint4(0, 0, 0, 0);
        const uint32_t gv[4] = {g.x, g.y, g.z, g.w};
        #pragma unroll
        for (int j = 0; j < 4; ++j) gam[i][j] = make_float2(lo16(gv[j]), hi16(gv[j]));
    }
    float2 dg_hi[NCH][4], dg_lo[NCH][4];
    #pragma unroll
    for (int i = 0; i < NCH; ++i)
        #pragma unroll
        for (int j = 0; j < 4; ++j) dg_hi[i][j] = dg_lo[i][j] = make_float2(0.0f, 0.0f);

    // the loads of row m + PF run while row m is reduced and written: each thread keeps the
    // raw words of the PF rows ahead in registers (one row at a time leaves the CTA waiting
    // on memory latency at every row's barrier)
    constexpr int PF = 2;
    uint4 ra[PF][NCH], rb[PF][NCH];
    auto load_row = [&](int64_t m, uint4 (&a)[NCH], uint4 (&b)[NCH]) {
        #pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int64_t c = (int64_t)i * kBwdChunk + 8 * tid;
            const bool ok = valid[i] && m < m_end;
            a[i] = ok ? ldg_v4(x + m * K + c) : make_uint4(0, 0, 0, 0);
            b[i] = ok ? ldg_v4(dy + m * K + c) : make_uint4(0, 0, 0, 0);
        }
    };
    #pragma unroll
    for (int f = 0; f < PF; ++f) load_row(m_begin + f, ra[f], rb[f]);
    int par = 0;
    for (int64_t m = m_begin; m < m_end; ++m, par ^= 1) {
        uint4 ca[NCH], cb[NCH];
        #pragma unroll
        for (int i = 0; i < NCH; ++i) {
            ca[i] = ra[0][i];
            cb[i] = rb[0][i];
        }
        #pragma unroll
        for (int f = 0; f + 1 < PF; ++f)
            #pragma unroll
            for (int i = 0; i < NCH; ++i) {
                ra[f][i] = ra[f + 1][i];
                rb[f][i] = rb[f + 1][i];
            }
        load_row(m + PF, ra[PF - 1], rb[PF - 1]);
        float2 xv[NCH][4], dv[NCH][4];
        float2 part2 = make_float2(0.0f, 0.0f);   // even and odd columns, summed in order
        #pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const uint4 a = ca[i];
            const uint4 b = cb[i];
            const uint32_t av[4] = {a.x, a.y, a.z, a.w};
            const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                xv[i][j] = make_float2(lo16(av[j]), hi16(av[j]));
                dv[i][j] = make_float2(lo16(bv[j]), hi16(bv[j]));
                part2 = __ffma2_rn(__fmul2_rn(dv[i][j], gam[i][j]), xv[i][j], part2);
            }
        }
        // S over the row: the thread's two sums, a fixed shuffle tree in each warp, then
        // the warps in order
        float part = __fadd_rn(part2.x, part2.y);
        #pragma unroll
        for (int off = 16; off >= 1; off >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, off));
        if (lane == 0) s_part[par][warp] = part;
        __syncthreads();
        float S = 0.0f;
        #pragma unroll
        for (int w = 0; w < NT / 32; ++w) S = __fadd_rn(S, s_part[par][w]);
        const float r = __ldg(rstd + m);
        const float coef = __fdiv_rn(__fmul_rn(__fmul_rn(__fmul_rn(r, r), r), S), (float)K);
        const float2 r2 = make_float2(r, r), nc2 = make_float2(-coef, -coef);
        #pragma unroll
        for (int i = 0; i < NCH; ++i) {
            if (!valid[i]) continue;
            const int64_t c = (int64_t)i * kBwdChunk + 8 * tid;
            uint32_t o[4];
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                // (r * gamma) * dy - coef * x, each product rounded, then the difference
                const float2 d = __fadd2_rn(__fmul2_rn(__fmul2_rn(r2, gam[i][j]), dv[i][j]), __fmul2_rn(nc2, xv[i][j]));
                o[j] = pack_bf16x2(d.x, d.y);
            }
            *reinterpret_cast<uint4*>(dx + m * K + c) = make_uint4(o[0], o[1], o[2], o[3]);
            if (ws) {
                #pragma unroll
                for (int j = 0; j < 4; ++j) two_sum_add2(dg_hi[i][j], dg_lo[i][j], __fmul2_rn(__fmul2_rn(dv[i][j], xv[i][j]), r2));
            }
        }
    }
    if (ws) {
        #pragma unroll
        for (int i = 0; i < NCH; ++i) {
            if (!valid[i]) continue;
            const int64_t c = (int64_t)i * kBwdChunk + 8 * tid;
            float* dst = ws + (int64_t)blockIdx.x * K + c;
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                dst[2 * j] = __fadd_rn(dg_hi[i][j].x, dg_lo[i][j].x);
                dst[2 * j + 1] = __fadd_rn(dg_hi[i][j].y, dg_lo[i][j].y);
            }
        }
    }
}

// dgamma[k] = sum over the row blocks of their partials, in block order (compensated).
__global__ void __launch_bounds__(256) k_rms_bwd_colsum(const float* __restrict__ ws, int nblocks, int64_t K,
                                                        float* __restrict__ dgamma) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= K) return;
    float hi = 0.0f, lo = 0.0f;
    for (int b = 0; b < nblocks; ++b) two_sum_add(hi, lo, ws[(int64_t)b * K + k]);
    dgamma[k] = __fadd_rn(hi, lo);
}

// Row blocks of the backward: one CTA per SM (its registers fill the SM), at most one per
// row.
int rmsnorm_bwd_blocks(int64_t M, int num_sms) {
    const int64_t b = (int64_t)(num_sms > 0 ? num_sms : 148);
    return (int)(M < b ? (M > 0 ? M : 1) : b);
}

cudaError_t launch_rmsnorm_bwd(const uint16_t* x, const uint16_t* gamma, const float* rstd, const uint16_t* dy,
                               int64_t M, int64_t K, uint16_t* dx, float* dgamma, float* ws, int nblocks,
                               cudaStream_t st) {
    // up to 5120 columns one pass over the row with 8 columns per thread; wider rows take
    // 256 threads and 3-4 passes (measured faster at 8192 columns: 0.169 against 0.182 ms
    // at 16384 rows for 1024 threads, whose 64 registers allow one row of lead)
    float* part = dgamma ? ws : nullptr;
    if (K <= 8 * 512)
        k_rms_bwd<1, 512><<<nblocks, 512, 0, st>>>(x, gamma, rstd, dy, M, K, dx, part);
    else if (K <= 8 * 640)
        k_rms_bwd<1, 640><<<nblocks, 640, 0, st>>>(x, gamma, rstd, dy, M, K, dx, part);
    else if (K <= 3 * 2048)
        k_rms_bwd<3, 256><<<nblocks, 256, 0, st>>>(x, gamma, rstd, dy, M, K, dx, part);
    else if (K <= 4 * 2048)
        k_rms_bwd<4, 256><<<nblocks, 256, 0, st>>>(x, gamma, rstd, dy, M, K, dx, part);
    else
        return cudaErrorInvalidValue;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !dgamma) return e;
    k_rms_bwd_colsum<<<(unsigned)((K + 255) / 256), 256, 0, st>>>(ws, nblocks, K, dgamma);
    return cudaGetLastError();
}

}  // namespace fp8rl
