// nvfp4.cu -- NVFP4 rollout path: the row quantizer and the decode-shaped GEMM on the
// tensor core's FP4 block-scaled MMA (tcgen05.mma kind::mxf4nvf4, scale_vec::4X).
//
// "QeRL" (chatpaper.ai), abstract: rollout runs with NVFP4-quantized weights.  The page
// names the format and nothing more; the format itself is FP4 E2M1 elements with one E4M3
// scale per 16 consecutive elements and an FP32 scale on top.  Readings taken here:
//   * the FP32 scale is per row (per output channel of a weight, per token of an
//     activation):  g = fl32(amax / 2688), 2688 = 6 * 448 (E2M1 max times E4M3 max);
//   * a block of 16 with maximum b gets the E4M3 code sb = E4M3(fl32(b / fl32(6 g))) and
//     the decode scale d = fl32(decode(sb) * g); element x gets E2M1(fl32(x / d)), round
//     to nearest even, saturating at +-6 (d = 0 gives code 0);
//   * Blackwell's FP4 tensor path multiplies FP4 by FP4, so the activation is quantized to
//     NVFP4 too (per call), with the same recipe;
//   * y[m][n] = gx[m] * gw[n] * sum_k x^(m,k) w^(n,k) with x^ = e2m1 * decode(sb): the MMA
//     applies the block scales inside its FP32 accumulation, the epilogue the row scales.
//
// Layouts (all produced by k_quant_nvfp4):
//   q[R][K/2]   packed codes, element k in bits 4(k%2) .. 4(k%2)+3 of byte k/2 (K-major,
//               the tensor core's packed FP4 operand layout);
//   sf          the block scales in the tensor core's scale-factor layout: 512-byte atoms
//               of 128 rows x 4 scales (64 elements of K), atom (row group rg, K-atom ka)
//               at byte 512 (rg * K/64 + ka), inside it row r's scale k at byte
//               16 (r % 32) + 4 ((r % 128) / 32) + k.  Rows past R up to the next multiple
//               of 128 hold zeros.  One K-block of 256 elements of one row group is 2 KB,
//               contiguous, and each atom is one tcgen05.cp.32x128b copy to TMEM;
//   g[R]        the per-row FP32 scales.
#include "cluster.cuh"
#include "common.cuh"
#include "gemm.h"
#include "rollout.h"

namespace fp8rl {

namespace {

// 16-byte read-only load, allocated in L1: the second pass over a row reads it there.
__device__ __forceinline__ uint4 nv_ldg_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two binary32 values -> packed E2M1 pair (lo in bits 0-3, hi in bits 4-7), round to
// nearest even, saturating at +-6 (the PTX .satfinite form).
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r & 0xFFu;
}

// Exact value of an E4M3 code (through the exact E4M3 -> FP16 conversion).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    float v;
    const uint16_t pair = (uint16_t)(code & 0xFFu);
    asm("{\n\t.reg .b32 h;\n\t.reg .f16 a, b;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, %1;\n\t"
        "mov.b32 {a, b}, h;\n\t"
        "cvt.f32.f16 %0, a;\n\t}"
        : "=f"(v)
        : "h"(pair));
    return v;
}

__device__ __forceinline__ size_t sf_offset(int64_t r, int64_t b, int64_t nkb) {
    const int64_t rg = r >> 7, rr = r & 127, ka = b >> 2, k = b & 3;
    return (size_t)((rg * nkb * 4 + ka) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + k);
}

// Codes of 16 consecutive elements (one block) under the decode scale d: 8 bytes.
__device__ __forceinline__ uint2 encode_block(const uint4 (&v)[2], float d) {
    uint32_t out[2] = {0u, 0u};
    if (d > 0.0f) {
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t w[4] = {v[h].x, v[h].y, v[h].z, v[h].w};
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = __fdiv_rn(bf16_bits_to_f32(w[j] & 0xFFFFu), d);
                const float hi = __fdiv_rn(bf16_bits_to_f32(w[j] >> 16), d);
                out[h] |= e2m1x2(lo, hi) << (8 * j);
            }
        }
    }
    return make_uint2(out[0], out[1]);
}

}  // namespace

// CTA (r, c) of 128 threads: row r, blocks of 16 [c * kQuantChunk, (c+1) * kQuantChunk)
// (rows past R, up to the next multiple of 128, only zero their scale factors).  Pass 1:
// the whole row's maximum (BF16 bit maxima, exact) -> g, the same in every chunk's CTA.
// Pass 2: per block of 16 of the chunk, its maximum, sb, d and the 16 codes, one block per
// thread.  Chunking keeps a long row's divisions on many SMs.
constexpr int kQuantChunk = 128;   // blocks of 16 per CTA

__global__ void __launch_bounds__(128) k_quant_nvfp4(const uint16_t* __restrict__ x, int64_t R, int64_t K,
                                                     int64_t ldx, uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                     float* __restrict__ g) {
    // a GEMM launched as this grid's programmatic dependent may start streaming its weights
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t nb = K / 16, nkb = K / 256;
    const int64_t b_lo = (int64_t)blockIdx.y * kQuantChunk;
    const int64_t b_hi = b_lo + kQuantChunk < nb ? b_lo + kQuantChunk : nb;
    if (r >= R) {
        for (int64_t b = b_lo + tid; b < b_hi; b += 128) sf[sf_offset(r, b, nkb)] = 0;
        return;
    }
    const uint16_t* row = x + r * ldx;
    uint32_t m2 = 0;
    for (int64_t c = (int64_t)tid * 8; c < K; c += 128 * 8) {
        const uint4 v = nv_ldg_v4(row + c);
        m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                   __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    #pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    __shared__ uint32_t s_max[4];
    if ((tid & 31) == 0) s_max[tid >> 5] = m;
    __syncthreads();
    m = max(max(s_max[0], s_max[1]), max(s_max[2], s_max[3]));
    const float gr = __fdiv_rn(bf16_bits_to_f32(m), 2688.0f);
    if (tid == 0 && blockIdx.y == 0) g[r] = gr;
    const float g6 = __fmul_rn(6.0f, gr);
    for (int64_t b = b_lo + tid; b < b_hi; b += 128) {
        uint4 v[2];
        v[0] = nv_ldg_v4(row + 16 * b);
        v[1] = nv_ldg_v4(row + 16 * b + 8);
        uint32_t bm2 = 0;
        #pragma unroll
        for (int h = 0; h < 2; ++h)
            bm2 = __vmaxu2(bm2, __vmaxu2(__vmaxu2(v[h].x & 0x7FFF7FFFu, v[h].y & 0x7FFF7FFFu),
                                         __vmaxu2(v[h].z & 0x7FFF7FFFu, v[h].w & 0x7FFF7FFFu)));
        const float bmax = bf16_bits_to_f32(max(bm2 & 0xFFFFu, bm2 >> 16));
        const uint32_t sb = gr > 0.0f ? (uint32_t)(e4m3x2(__fdiv_rn(bmax, g6), 0.0f) & 0xFFu) : 0u;
        const float d = __fmul_rn(e4m3_value(sb), gr);
        const uint2 c = encode_block(v, d);
        *reinterpret_cast<uint2*>(q + r * (K / 2) + 8 * b) = c;
        sf[sf_offset(r, b, nkb)] = (uint8_t)sb;
    }
}

__global__ void k_debug_e2m1(const float* __restrict__ in, uint8_t* __restrict__ out, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)(e2m1x2(in[i], 0.0f) & 0xFu);
}

// ------------------------------------------------------------------------------------
// Decode GEMM, weights on the MMA's M side (A = 128 weight rows, B = the MP-token
// activation tile, N = MP), one K-block = 256 FP4 elements = 128 bytes per row.
//   * The block scales of both operands travel with the codes (bulk copies of their 2 KB
//     K-block pieces) and reach TMEM by tcgen05.cp, one 32x128b copy (replicated to the
//     four lane quarters) per 512-byte atom, into the stage's scale-factor columns; four
//     MMAs of K = 64 each take their 4 columns of A and B scales.  The scale columns of a
//     stage are rewritten only after the stage's MMAs completed (the stage's empty barrier).
//   * The block scales are applied inside the MMA, so the accumulator runs over the whole
//     reduction and the epilogue reads TMEM once per tile: y = acc * gx[m] * gw[n].
//   * Split-K over a cluster of S CTAs for narrow weights, reduced through distributed
//     shared memory in rank order, as the FP8 decode GEMM does.
// Roles (320 threads): warp 0 copies, warp 1 issues tcgen05 (one elected lane), warps 2-9
// read the accumulator (warp w reads TMEM lane quarter w % 4, half of the token columns).
// Every wait is bounded.
// ------------------------------------------------------------------------------------
namespace {

template <int MP>
struct Nvf4Cfg {
    static constexpr int NG = MP > 128 ? 2 : 1;             // 128-row scale groups of the tokens
    static constexpr int W_BYTES = 128 * 128;
    static constexpr int X_BYTES = MP * 128;
    static constexpr int SFW_BYTES = 2048;
    static constexpr int SFX_BYTES = 2048 * NG;
    static constexpr int STAGES = MP <= 64 ? 6 : (MP <= 128 ? 5 : 4);
    static constexpr int NACC = MP <= 128 ? 2 : 1;          // accumulators of MP columns
    static constexpr int SF_COL0 = NACC * MP;
    static constexpr int SF_COLS = 16 + 16 * NG;             // per stage: A scales, then B scales
    static_assert(SF_COL0 + STAGES * SF_COLS <= 512, "TMEM columns");
    static constexpr size_t STAGE_BYTES = (size_t)STAGES * (W_BYTES + X_BYTES + SFW_BYTES + SFX_BYTES);
    static constexpr size_t RED_BYTES = (size_t)MP * 128 * 4;   // [token][weight row] FP32
    static_assert(RED_BYTES <= STAGE_BYTES, "the reduction buffer reuses the stage ring");
    static constexpr int NBARS = 2 * STAGES + 2 * NACC + 1;
    static constexpr size_t BYTES = 1024 + STAGE_BYTES + (size_t)NBARS * 8 + 16;
};

// Instruction descriptor, kind::mxf4nvf4 with block scaling: bits 7-9 / 10-11 A / B format
// (1 = E2M1), 15 / 16 K-major (0), 17-22 N >> 3, 23 scale format (0 = UE4M3), 24-28 M >> 4;
// scale-factor IDs (bits 4-5, 29-30) 0, as scale_vec::4X uses all four bytes of a column.
__host__ __device__ constexpr uint32_t idesc_nvf4(uint32_t m, uint32_t n) {
    return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Shared-memory descriptor of one scale-factor atom as tcgen05.cp reads it: 32 rows of 16
// bytes, no swizzle, K-major core matrices of 8 rows x 16 bytes stored contiguously
// (stride between core matrices along the rows 128 bytes; one core matrix along K).
__device__ __forceinline__ uint64_t sdesc_sf_atom(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);
    d |= (uint64_t)(128 >> 4) << 16;
    d |= (uint64_t)(128 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

__device__ __forceinline__ void tmem_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with E2M1 operands and UE4M3 block scales from TMEM.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

}  // namespace

// Grid: with a cluster of S > 1 CTAs, one cluster per 128-row weight tile (CTA r streams
// K-blocks [r nkb / S, (r+1) nkb / S) and reduces token slice r); with S = 1, persistent
// CTAs over tiles blockIdx.x, +gridDim.x, ..., storing from registers.
template <int MP>
__global__ void __launch_bounds__(320, 1)
    k_gemm_nvf4(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const Nvf4Params p) {
    using C = Nvf4Cfg<MP>;
    constexpr int STAGES = C::STAGES, NACC = C::NACC, NG = C::NG;
    constexpr uint32_t IDESC = idesc_nvf4(128, MP);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sW = smem;
    uint8_t* sX = sW + STAGES * C::W_BYTES;
    uint8_t* sSFW = sX + STAGES * C::X_BYTES;
    uint8_t* sSFX = sSFW + STAGES * C::SFW_BYTES;
    float* red = reinterpret_cast<float*>(smem);                  // after the last MMA
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGE_BYTES);
    uint64_t* full_bar = bars;                   // [STAGES] copies -> MMA
    uint64_t* empty_bar = bars + STAGES;         // [STAGES] MMA -> copies
    uint64_t* tfull_bar = bars + 2 * STAGES;     // [NACC] MMA -> epilogue
    uint64_t* tempty_bar = tfull_bar + NACC;     // [NACC] epilogue -> MMA
    uint64_t* drain_bar = tempty_bar + NACC;     // [1] MMA completion at exit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = (int)cluster_nctarank();
    const int rank = (int)cluster_ctarank();
    const int tile0 = (int)cluster_idx();
    const int tstep = (int)cluster_count();
    const int tiles = p.tiles;
    const int kb0 = (int)(((int64_t)rank * p.nkb) / S);
    const int kb1 = (int)(((int64_t)(rank + 1) * p.nkb) / S);
    const int nk = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), 8);
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ copies
        const uint64_t pol_w = l2_policy_evict_first();   // each weight byte is read once
        const uint64_t pol_x = l2_policy_evict_last();    // every tile reads the activation
        constexpr uint32_t TX = C::W_BYTES + C::X_BYTES + C::SFW_BYTES + C::SFX_BYTES;
        // the weights do not depend on the kernel that produced the activation: the first
        // stages' weight codes and scales are requested before waiting for that kernel
        const uint32_t n_it = tile0 < tiles ? (uint32_t)((tiles - tile0 + tstep - 1) / tstep) * (uint32_t)nk : 0u;
        const uint32_t n_pre = n_it < (uint32_t)STAGES ? n_it : (uint32_t)STAGES;
        if (elect_one_sync()) {
            for (uint32_t j = 0; j < n_pre; ++j) {
                const int tile = tile0 + (int)(j / (uint32_t)nk) * tstep;
                const int kb = kb0 + (int)(j % (uint32_t)nk);
                const uint32_t fb = smem_u32(&full_bar[j]);
                mbar_arrive_expect_tx(fb, TX);
                tma_load_2d(smem_u32(sW + j * C::W_BYTES), &tmW, fb, kb * 128, tile * 128, pol_w);
                bulk_load_1d(smem_u32(sSFW + j * C::SFW_BYTES), p.sfw + ((int64_t)tile * p.nkb + kb) * 2048, 2048, fb);
            }
        }
        __syncwarp();
        asm volatile("griddepcontrol.wait;" ::: "memory");
        uint32_t it = 0;
        for (int tile = tile0; ok && tile < tiles; tile += tstep) {
            for (int i = 0; i < nk; ++i, ++it) {
                const int kb = kb0 + i;
                const uint32_t s = it % STAGES;
                const uint32_t fb = smem_u32(&full_bar[s]);
                if (it >= n_pre &&
                    !mbar_wait(smem_u32(&empty_bar[s]), ((it / STAGES) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one_sync()) {
                    if (it >= n_pre) {
                        mbar_arrive_expect_tx(fb, TX);
                        tma_load_2d(smem_u32(sW + s * C::W_BYTES), &tmW, fb, kb * 128, tile * 128, pol_w);
                        bulk_load_1d(smem_u32(sSFW + s * C::SFW_BYTES), p.sfw + ((int64_t)tile * p.nkb + kb) * 2048,
                                     2048, fb);
                    }
                    tma_load_2d(smem_u32(sX + s * C::X_BYTES), &tmX, fb, kb * 128, 0, pol_x);
                    #pragma unroll
                    for (int gi = 0; gi < NG; ++gi)
                        bulk_load_1d(smem_u32(sSFX + s * C::SFX_BYTES + gi * 2048),
                                     p.sfx + ((int64_t)gi * p.nkb + kb) * 2048, 2048, fb);
                }
                __syncwarp();
            }
        }
        // Every issued copy lands before the stage memory is reused or freed.  The loop
        // only stops at an item past the prefetched ones (the empty waits start there), so
        // every prefetched item also got its activation copies and its barrier completes.
        volatile int no_abort = 0;
        const uint32_t n_out = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
        for (uint32_t j = it - n_out; j < it; ++j)
            mbar_wait(smem_u32(&full_bar[j % STAGES]), (j / STAGES) & 1, p.timeout_ns, &no_abort);
    } else if (warp == 1) {
        // ------------------------------------------------------------ tcgen05 issuer
        const uint32_t w_base = smem_u32(sW), x_base = smem_u32(sX);
        const uint32_t sfw_base = smem_u32(sSFW), sfx_base = smem_u32(sSFX);
        uint32_t it = 0, lt = 0;
        for (int tile = tile0; ok && tile < tiles; tile += tstep, ++lt) {
            const uint32_t a = lt % NACC;
            if (!mbar_wait(smem_u32(&tempty_bar[a]), ((lt / NACC) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + a * MP;
            for (int i = 0; i < nk; ++i, ++it) {
                const uint32_t s = it % STAGES;
                if (!mbar_wait(smem_u32(&full_bar[s]), (it / STAGES) & 1, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sfa = tmem_base + C::SF_COL0 + s * C::SF_COLS;
                const uint32_t sfb = sfa + 16;
                const uint64_t da = sdesc_kmajor_sw128(w_base + s * C::W_BYTES);
                const uint64_t db = sdesc_kmajor_sw128(x_base + s * C::X_BYTES);
                if (elect_one_sync()) {
                    #pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tmem_cp_sf_atom(sfa + 4 * j, sdesc_sf_atom(sfw_base + s * C::SFW_BYTES + 512 * j));
                    #pragma unroll
                    for (int gi = 0; gi < NG; ++gi)
                        #pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tmem_cp_sf_atom(sfb + 4 * (NG * j + gi),
                                            sdesc_sf_atom(sfx_base + s * C::SFX_BYTES + gi * 2048 + 512 * j));
                    #pragma unroll
                    for (int k = 0; k < 4; ++k)   // 32-byte (64-element) steps inside the 128-byte rows
                        mma_nvf4(d, da + 2 * k, db + 2 * k, IDESC, sfa + 4 * k, sfb + 4 * NG * k,
                                 (i > 0 || k > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&empty_bar[s]));
                    if (i == nk - 1) mma_commit(smem_u32(&tfull_bar[a]));
                }
                __syncwarp();
            }
        }
        if (elect_one_sync()) mma_commit(smem_u32(drain_bar));
        __syncwarp();
        volatile int no_abort = 0;
        mbar_wait(smem_u32(drain_bar), 0, p.timeout_ns, &no_abort);
    } else {
        // ------------------------------------------------------------ accumulator readers
        // two warps per TMEM lane quadrant, each MP/2 token columns: the whole share is
        // loaded first and the accumulator handed back before any arithmetic or store
        constexpr int CH = MP / 2, LW = CH >= 32 ? 32 : 16, NL = CH / LW;
        const int quad = warp & 3;
        const int col0 = ((warp - 2) >> 2) * CH;
        const int row = quad * 32 + lane;               // weight row within the tile
        const uint32_t tl = tmem_base + ((uint32_t)(quad * 32) << 16) + col0;
        uint32_t lt = 0;
        for (int tile = tile0; ok && tile < tiles; tile += tstep, ++lt) {
            const uint32_t a = lt % NACC;
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[a]), (lt / NACC) & 1, p.timeout_ns, abort_flag));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[NL][LW];
            #pragma unroll
            for (int h = 0; h < NL; ++h) tmem_ld_cols(tl + a * MP + h * LW, v[h]);
            #pragma unroll
            for (int h = 0; h < NL; ++h) tmem_ld_wait(v[h]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[a]));
            const int n = tile * 128 + row;
            if (S == 1) {
                const float gwn = p.gw[n];
                uint16_t* yt = p.y + n;
                #pragma unroll
                for (int h = 0; h < NL; ++h)
                    #pragma unroll
                    for (int j = 0; j < LW; ++j) {
                        const int t = col0 + h * LW + j;
                        if (t < p.M) {
                            const float yv = __fmul_rn(__fmul_rn(__uint_as_float(v[h][j]), __ldg(p.gx + t)), gwn);
                            yt[(int64_t)t * p.ldy] = (uint16_t)(pack_bf16x2(yv, 0.0f) & 0xFFFFu);
                        }
                    }
            } else {
                // one tile per cluster: the last commit covered every MMA of this CTA, and
                // every copy was consumed by one, so the stage ring is free
                #pragma unroll
                for (int h = 0; h < NL; ++h)
                    #pragma unroll
                    for (int j = 0; j < LW; ++j) red[(col0 + h * LW + j) * 128 + row] = __uint_as_float(v[h][j]);
            }
        }
    }

    // ---- cluster reduction: CTA r adds token slice r of every CTA's partial sums in rank
    // order, then applies the row scales
    __syncwarp();
    tc_fence_before();
    if (S > 1) {
        cluster_sync_all();
        if (warp >= 2 && *abort_flag == 0 && tile0 < tiles) {
            const int et = threadIdx.x - 64;                      // 0..255
            const int n4 = p.M * 32;                              // float4s of valid tokens
            const int per = (n4 + S - 1) / S;
            const int e_end = min(n4, (rank + 1) * per);
            const uint32_t red_local = smem_u32(red);
            const int n0 = tile0 * 128;
            for (int e = rank * per + et; e < e_end; e += 256) {
                const int tok = e >> 5;
                const int r4 = (e & 31) * 4;
                const uint32_t off = (uint32_t)(tok * 128 + r4) * 4u;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int j = 0; j < S; ++j) {
                    const float4 w = ld_dsmem_v4(mapa_shared(red_local + off, (uint32_t)j));
                    v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
                }
                const float gxt = __ldg(p.gx + tok);
                const float4 gw4 = *reinterpret_cast<const float4*>(p.gw + n0 + r4);
                uint2 o;
                o.x = pack_bf16x2(__fmul_rn(__fmul_rn(v.x, gxt), gw4.x), __fmul_rn(__fmul_rn(v.y, gxt), gw4.y));
                o.y = pack_bf16x2(__fmul_rn(__fmul_rn(v.z, gxt), gw4.z), __fmul_rn(__fmul_rn(v.w, gxt), gw4.w));
                *reinterpret_cast<uint2*>(p.y + (int64_t)tok * p.ldy + n0 + r4) = o;
            }
        }
        cluster_sync_all();   // no CTA leaves while another still reads its shared memory
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

namespace {

int nvf4_mp(int M) { return M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256)); }

template <int MP>
cudaError_t launch_nvf4_t(const CUtensorMap& tw, const CUtensorMap& tx, const Nvf4Params& p, int grid_clusters,
                          int splits, bool pdl, cudaStream_t st) {
    auto kern = k_gemm_nvf4<MP>;
    constexpr size_t smem = Nvf4Cfg<MP>::BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(grid_clusters * splits), 1, 1);
    cfg.blockDim = dim3(320, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)splits;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, tw, tx, p);
}

template <int MP>
int nvf4_max_clusters_t(int splits) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)splits * 64, 1, 1);
    cfg.blockDim = dim3(320, 1, 1);
    cfg.dynamicSmemBytes = Nvf4Cfg<MP>::BYTES;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)splits;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaFuncSetAttribute(k_gemm_nvf4<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Nvf4Cfg<MP>::BYTES);
    int n = 0;
    return cudaOccupancyMaxActiveClusters(&n, k_gemm_nvf4<MP>, &cfg) == cudaSuccess ? n : 0;
}

}  // namespace

int nvf4_token_tile(int M) { return nvf4_mp(M); }

int nvf4_max_clusters(int M, int splits) {
    switch (nvf4_mp(M)) {
        case 32: return nvf4_max_clusters_t<32>(splits);
        case 64: return nvf4_max_clusters_t<64>(splits);
        case 128: return nvf4_max_clusters_t<128>(splits);
        default: return nvf4_max_clusters_t<256>(splits);
    }
}

cudaError_t launch_gemm_nvf4(const CUtensorMap& tw, const CUtensorMap& tx, const Nvf4Params& p, int grid_clusters,
                             int splits, bool pdl, cudaStream_t st) {
    if (splits > 1 && grid_clusters != p.tiles) return cudaErrorInvalidValue;   // one tile per cluster
    switch (nvf4_mp(p.M)) {
        case 32: return launch_nvf4_t<32>(tw, tx, p, grid_clusters, splits, pdl, st);
        case 64: return launch_nvf4_t<64>(tw, tx, p, grid_clusters, splits, pdl, st);
        case 128: return launch_nvf4_t<128>(tw, tx, p, grid_clusters, splits, pdl, st);
        default: return launch_nvf4_t<256>(tw, tx, p, grid_clusters, splits, pdl, st);
    }
}

cudaError_t launch_quant_nvfp4(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q, uint8_t* sf,
                               float* g, cudaStream_t st) {
    const int64_t rows = (R + 127) / 128 * 128;
    const int64_t chunks = (K / 16 + kQuantChunk - 1) / kQuantChunk;
    k_quant_nvfp4<<<dim3((unsigned)rows, (unsigned)chunks), 128, 0, st>>>(x, R, K, ldx, q, sf, g);
    return cudaGetLastError();
}

cudaError_t launch_debug_e2m1(const float* in, uint8_t* out, int64_t n, cudaStream_t st) {
    const int64_t blocks = std::max<int64_t>(std::min<int64_t>((n + 255) / 256, 4096), 1);
    k_debug_e2m1<<<(unsigned)blocks, 256, 0, st>>>(in, out, n);
    return cudaGetLastError();
}

// Reads and clears this translation unit's device status word (the GEMM's bounded waits
// record their timeouts in it).  The caller has synchronized the stream.
fp8rl_status read_and_clear_nvf4_status() {
    unsigned int v = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return FP8RL_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) return FP8RL_ERR_CUDA;
    return static_cast<fp8rl_status>(v);
}

}  // namespace fp8rl
