// quantize.cu -- BF16 -> E4M3 quantizers (1x128, 128x1 transposed, 128x128 blocks) and
// the fused RMSNorm / SiLU-mul producers that feed them.
//
// "Technical summary: Jet-RL", section "Quantization Scheme": activations 1x128 per group,
// weights 128x128 per block, WGrad operands additionally 128x1; activations saved for the
// backward pass are FP8 and produced by the preceding fused operator.  Section
// "Implementation": quantization, transposition and fused activation / RMSNorm kernels.
//
// All quantizers are HBM-bound.  The panel kernels read a 128-row x 128-column BF16
// sub-tile once and emit both the 1x128 (row-group) codes, straight from registers, and
// the transposed 128x1 (column-group) codes, through a shared-memory tile that leaves in
// 128-byte rows.  Thread layout in a 256-thread CTA: warp w, lane l
// owns rows 16w + 8*(l/16) + [0,8) and columns 8*(l%16) + [0,8) of the sub-tile, so each
// warp-wide load reads two full 256-byte rows, a row group is reduced over 16 lanes and a
// column group over the two half-warps and the 8 warps.
#include <cooperative_groups.h>

#include <algorithm>

#include "gemm.h"
#include "quant_common.cuh"

namespace cg = cooperative_groups;

namespace fp8rl {

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_v2(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void stg_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// ------------------------------------------------------------------------------------
// 1x128 quantization of rows, any M.  16 threads per group (8 BF16 each), groups ordered
// block-major (g = kb*M + m) so that the scale stores of neighbouring groups coalesce.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_quant_1x128(const uint16_t* __restrict__ x, int64_t M,
                                                     int64_t K, int64_t ldx,
                                                     uint8_t* __restrict__ q,
                                                     float* __restrict__ s) {
    // a grid launched as this one's dependent may start its own prologue now (it waits for
    // this grid's completion before it reads q or s)
    asm volatile("griddepcontrol.launch_dependents;");
    const int sub = threadIdx.x & 15;
    const int half = (threadIdx.x >> 4) & 1;
    const int warp = threadIdx.x >> 5;
    const int64_t ngroups = M * (K / 128);
    const int64_t step = (int64_t)gridDim.x * 16;
    // warp-uniform loop: both half-warps always execute the shuffles together
    for (int64_t base = (int64_t)blockIdx.x * 16 + warp * 2; base < ngroups; base += step) {
        const int64_t g = base + half;
        const bool valid = g < ngroups;
        const int64_t kb = valid ? g / M : 0;
        const int64_t m = valid ? g - kb * M : 0;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (valid) v = ldg_nc_v4(x + m * ldx + kb * 128 + sub * 8);
        uint32_t mx = absmax2(absmax2(absmax2(absmax2(0u, v.x), v.y), v.z), v.w);
        mx = max(mx & 0xFFFFu, mx >> 16);
        #pragma unroll
        for (int off = 8; off >= 1; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const GroupScale gs = make_scale(bf16_bits_amax_to_f32(mx));
        const uint32_t c0 = encode_pair(bf16_lo(v.x), bf16_hi(v.x), gs);
        const uint32_t c1 = encode_pair(bf16_lo(v.y), bf16_hi(v.y), gs);
        const uint32_t c2 = encode_pair(bf16_lo(v.z), bf16_hi(v.z), gs);
        const uint32_t c3 = encode_pair(bf16_lo(v.w), bf16_hi(v.w), gs);
        if (valid) {
            stg_v2(q + m * K + kb * 128 + sub * 8, c0 | (c1 << 16), c2 | (c3 << 16));
            if (sub == 0) s[kb * M + m] = gs.s;
        }
    }
}

// ------------------------------------------------------------------------------------
// Panel kernel: 128-row panels, 128-column sub-tiles, optional fused producer.
// ------------------------------------------------------------------------------------
// PRO_RMSNORM computes the rows' rstd itself (a cluster of CTAs per panel, two passes);
// PRO_RMSNORM_G reads rstd computed beforehand by k_rms_rstd.
// PRO_SILU_BWD quantizes the gradient of the gate_up output, [dg | du], from the forward's
// gate / up tiles and the gradient of h (a second tensor map).  PRO_DEQUANT rebuilds the
// BF16 activation from its saved 1x128 codes and row scales (the stage holds a 128x128
// code tile and the tile's 128 row scales) for the 128x1 WGrad operand.
enum Prologue : int { PRO_COPY = 0, PRO_SILU = 1, PRO_RMSNORM = 2, PRO_RMSNORM_G = 3, PRO_SILU_BWD = 5,
                      PRO_DEQUANT = 6 };

struct PanelArgs {
    const uint16_t* x;      // COPY / RMSNORM: x[M][ldx];  SILU: gu[M][ldx], ldx = 2*K;
                            // SILU_BWD: gu[M][ldx], ldx = K (K = 2I quantized columns)
    const uint16_t* x2;     // SILU_BWD: dh[M][K/2]
    const float* xs;        // DEQUANT: the codes' scales xs[K/128][M] (x holds the codes)
    int64_t ldx;
    const uint16_t* gamma;  // RMSNORM: gamma[K]
    float eps;
    float* rstd_out;        // RMSNORM: rstd[M] (nullable)
    int64_t M, K;           // K = number of quantized columns (I for SiLU-mul)
    uint8_t* q;             // 1x128 codes q[M][K]
    float* s;               // scales s[K/128][M]
    uint8_t* qT;            // 128x1 codes, transposed: qT[K][M]
    float* sT;              // scales sT[M/128][K]
    int tiles_per_cta;      // RMSNorm: 128-column sub-tiles handled by one CTA of a panel's cluster
    uint64_t timeout_ns;    // bound of every wait on a TMA copy
};

// Accurate sum of squares: binary32 pairs (hi, lo) updated with the exact two-sum, so
// that a row's total is known to about 2^-44 relative before it is rounded to binary32.
struct F2 {
    float hi, lo;
};
__device__ __forceinline__ F2 two_sum_acc(F2 a, float v) {
    const float s = __fadd_rn(a.hi, v);
    const float bp = __fsub_rn(s, a.hi);
    const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bp)), __fsub_rn(v, bp));
    return F2{s, __fadd_rn(a.lo, e)};
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    F2 r = two_sum_acc(F2{a.hi, __fadd_rn(a.lo, b.lo)}, b.hi);
    // renormalise so that |lo| stays below half an ulp of hi
    const float s = __fadd_rn(r.hi, r.lo);
    const float e = __fsub_rn(r.lo, __fsub_rn(s, r.hi));
    return F2{s, e};
}

// One thread's 8 rows x 8 columns of the staged tile -> BF16 words of y (the value that is
// quantized): x itself, bf16((x*rstd)*gamma), or bf16(silu(g)*u).  The stage holds the
// 128x128 BF16 tile row-major (256 bytes per row); SiLU-mul stages the up tile after it.
template <int PRO>
__device__ __forceinline__ void rows_from_smem(const uint8_t* stage, const PanelArgs& a, int64_t k0,
                                               int R0, int C0, const float* s_rstd, const float (&rg)[8],
                                               uint32_t (&w)[8][4]) {
    float2 gam[4];   // gamma of columns (2j, 2j+1)
    if (PRO == PRO_RMSNORM || PRO == PRO_RMSNORM_G) {
        const uint4 gv = ldg_nc_v4(a.gamma + k0 + C0);
        gam[0] = make_float2(bf16_lo(gv.x), bf16_hi(gv.x));
        gam[1] = make_float2(bf16_lo(gv.y), bf16_hi(gv.y));
        gam[2] = make_float2(bf16_lo(gv.z), bf16_hi(gv.z));
        gam[3] = make_float2(bf16_lo(gv.w), bf16_hi(gv.w));
    }
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (PRO == PRO_DEQUANT) {
            // x^ = bf16(fl32(decode(code) * s_row)).  The hardware conversion decodes two
            // codes into two FP16 values, exactly (every finite E4M3 value, subnormals
            // included, is an FP16 value), and FP16 -> FP32 is exact.
            const uint2 c8 = *reinterpret_cast<const uint2*>(stage + (R0 + i) * 128 + C0);
            const float sr = *reinterpret_cast<const float*>(stage + 128 * 128 + 4 * (R0 + i));
            const uint32_t cw[2] = {c8.x, c8.y};
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint16_t pair = (uint16_t)(cw[j >> 1] >> (16 * (j & 1)));   // codes 2j (low), 2j + 1
                float d0, d1;
                asm("{\n\t.reg .b32 h;\n\t.reg .f16 a, b;\n\t"
                    "cvt.rn.f16x2.e4m3x2 h, %2;\n\t"
                    "mov.b32 {a, b}, h;\n\t"
                    "cvt.f32.f16 %0, a;\n\t"
                    "cvt.f32.f16 %1, b;\n\t}"
                    : "=f"(d0), "=f"(d1)
                    : "h"(pair));
                const float2 y = __fmul2_rn(make_float2(d0, d1), make_float2(sr, sr));
                w[i][j] = pack_bf16x2(y.x, y.y);
            }
            continue;
        }
        const uint4 v = *reinterpret_cast<const uint4*>(stage + (R0 + i) * 256 + C0 * 2);
        const uint32_t xv[4] = {v.x, v.y, v.z, v.w};
        if (PRO == PRO_COPY) {
            #pragma unroll
            for (int j = 0; j < 4; ++j) w[i][j] = xv[j];
        } else if (PRO == PRO_RMSNORM || PRO == PRO_RMSNORM_G) {
            const float r = (PRO == PRO_RMSNORM_G) ? rg[i] : s_rstd[R0 + i];
            // (x * rstd) * gamma, each product rounded, on packed pairs
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 y = __fmul2_rn(__fmul2_rn(make_float2(bf16_lo(xv[j]), bf16_hi(xv[j])), make_float2(r, r)), gam[j]);
                w[i][j] = pack_bf16x2(y.x, y.y);
            }
        } else {  // SILU: h = bf16(silu(g) * u), silu(g) = g / (1 + exp(-g))
            const uint4 u = *reinterpret_cast<const uint4*>(stage + 128 * 256 + (R0 + i) * 256 + C0 * 2);
            const uint32_t uv[4] = {u.x, u.y, u.z, u.w};
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float g0 = bf16_lo(xv[j]), g1 = bf16_hi(xv[j]);
                const float u0 = bf16_lo(uv[j]), u1 = bf16_hi(uv[j]);
                const float h0 = __fmul_rn(__fdividef(g0, 1.0f + __expf(-g0)), u0);
                const float h1 = __fmul_rn(__fdividef(g1, 1.0f + __expf(-g1)), u1);
                w[i][j] = pack_bf16x2(h0, h1);
            }
        }
    }
}

// SiLU-mul backward from the staged gate, up and dh tiles (256-byte rows each, in that
// order), for this thread's 8 rows x 8 columns: dg = dh*u*s*(1 + g*(1 - s)) into w and
// du = dh*g*s as BF16 over the up tile, where this thread alone reads it again; the
// sigmoid s = 1/(1 + exp(-g)) is evaluated once for both.
__device__ __forceinline__ void silu_bwd_pair_from_smem(uint8_t* stage, int R0, int C0, uint32_t (&w)[8][4]) {
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 gv = *reinterpret_cast<const uint4*>(stage + (R0 + i) * 256 + C0 * 2);
        uint4* up = reinterpret_cast<uint4*>(stage + 128 * 256 + (R0 + i) * 256 + C0 * 2);
        const uint4 u = *up;
        const uint4 d = *reinterpret_cast<const uint4*>(stage + 2 * 128 * 256 + (R0 + i) * 256 + C0 * 2);
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
        const uint32_t uv[4] = {u.x, u.y, u.z, u.w};
        const uint32_t dv[4] = {d.x, d.y, d.z, d.w};
        uint32_t du[4];
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            float og[2], ou[2];
            #pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float g = e ? bf16_hi(gw[j]) : bf16_lo(gw[j]);
                const float uu = e ? bf16_hi(uv[j]) : bf16_lo(uv[j]);
                const float dd = e ? bf16_hi(dv[j]) : bf16_lo(dv[j]);
                const float sg = __fdividef(1.0f, 1.0f + __expf(-g));
                og[e] = __fmul_rn(__fmul_rn(__fmul_rn(dd, uu), sg), __fmaf_rn(g, __fsub_rn(1.0f, sg), 1.0f));
                ou[e] = __fmul_rn(dd, __fmul_rn(g, sg));
            }
            w[i][j] = pack_bf16x2(og[0], og[1]);
            du[j] = pack_bf16x2(ou[0], ou[1]);
        }
        *up = make_uint4(du[0], du[1], du[2], du[3]);
    }
    // the stage is refilled by TMA after these generic writes
    fence_proxy_async_smem();
}

// BF16 unpacking that the compiler may not merge with the plain one: the column codes
// unpack again instead of keeping all 64 unpacked values live from the row codes.
__device__ __forceinline__ float bf16_lo_v(uint32_t w) {
    uint32_t r;
    asm volatile("shl.b32 %0, %1, 16;" : "=r"(r) : "r"(w));
    return __uint_as_float(r);
}
__device__ __forceinline__ float bf16_hi_v(uint32_t w) {
    uint32_t r;
    asm volatile("and.b32 %0, %1, 0xFFFF0000;" : "=r"(r) : "r"(w));
    return __uint_as_float(r);
}

// Codes of four pairs of one group whose scale is too small for the division-free encode
// (0 < s < 2^-68): IEEE division.  Out of line: it runs only for such groups.
__device__ __noinline__ uint4 encode4_slow(float2 x0, float2 x1, float2 x2, float2 x3, float s) {
    return make_uint4(e4m3x2(__fdiv_rn(x0.x, s), __fdiv_rn(x0.y, s)), e4m3x2(__fdiv_rn(x1.x, s), __fdiv_rn(x1.y, s)),
                      e4m3x2(__fdiv_rn(x2.x, s), __fdiv_rn(x2.y, s)), e4m3x2(__fdiv_rn(x3.x, s), __fdiv_rn(x3.y, s)));
}

// rstd of every row for PRO_RMSNORM_G: one warp per row.  The squares are summed in
// binary32 pairs with the exact two-sum (lane-strided 16-byte chunks, then a fixed
// shuffle tree), so the total is known to about 2^-44 relative; then
// rstd = 1 / sqrt(fl32(sum / K) + eps) in IEEE single precision.
__global__ void __launch_bounds__(256) k_rms_rstd(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                  float eps, float* __restrict__ rstd) {
    const int lane = threadIdx.x & 31;
    const int64_t m = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (m >= M) return;
    const uint16_t* row = x + m * K;
    F2 acc = F2{0.0f, 0.0f};
    #pragma unroll 4
    for (int64_t c = (int64_t)lane * 8; c < K; c += 256) {
        const uint4 v = ldg_nc_v4(row + c);
        const uint32_t xv[4] = {v.x, v.y, v.z, v.w};
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float x0 = bf16_lo(xv[j]), x1 = bf16_hi(xv[j]);
            acc = two_sum_acc(acc, __fmul_rn(x0, x0));
            acc = two_sum_acc(acc, __fmul_rn(x1, x1));
        }
    }
    #pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        F2 o;
        o.hi = __shfl_xor_sync(0xffffffffu, acc.hi, off);
        o.lo = __shfl_xor_sync(0xffffffffu, acc.lo, off);
        acc = f2_add(acc, o);
    }
    if (lane == 0) {
        const double sum = (double)acc.hi + (double)acc.lo;
        const float ms = __double2float_rn(sum / (double)K);
        rstd[m] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    }
}

// Input stages of the TMA ring (each a 128x128 BF16 tile; SiLU-mul stages gate and up).
template <int PRO, bool COLQ>
struct PanelStages {
    static constexpr int NIN = (PRO == PRO_SILU) ? 2 : (PRO == PRO_SILU_BWD ? 3 : 1);
    // DEQUANT: a 128x128 code tile and its 128 row scales
    static constexpr int STAGE_BYTES = PRO == PRO_DEQUANT ? 128 * 128 + 128 * 4 : NIN * 128 * 128 * 2;
    // SiLU-mul stages 64 KB per tile: one stage lets two CTAs share an SM, which hides the
    // copy latency better than three stages in one CTA (0.186 vs 0.242 ms at 8192x14336).
    // The 128x1 codes pass through two 16 KB shared-memory tiles (COLQ), which leaves room
    // for two input stages of 32 KB at two CTAs per SM.
    static constexpr int STAGES = (PRO == PRO_SILU || PRO == PRO_SILU_BWD) ? 1 : (COLQ && PRO != PRO_DEQUANT ? 2 : 3);
    static constexpr int COLQ_OFF = ((STAGES * STAGE_BYTES + 127) / 128) * 128;
    // (SiLU-mul backward stages its 128x1 codes in the stage's gate tile, dead after its
    // prologue: no separate staging tiles)
    static constexpr size_t SMEM = (size_t)COLQ_OFF + (COLQ && PRO != PRO_SILU_BWD ? 2 * 128 * 128 : 0) + 128;
};

// A CTA works through a sequence of 128x128 tiles (see tile_at below).
// Thread 0 streams the tiles through a ring of TMA stages in shared memory; all threads
// pull a tile into registers, and once everyone has it (the first barrier of the tile)
// thread 0 refills that stage, so copies of the next tiles overlap the current one's math.
// RMSNorm streams the CTA's tiles twice: pass 1 sums squares, pass 2 quantizes.
// The 128x1 codes of a tile leave through shared memory (two staging tiles of their own;
// the SiLU-mul backward uses its stage's gate tile, dead after its prologue): each thread
// writes its 8 columns x 8 rows of codes there, and after a CTA barrier the tile goes out
// as 16-byte pieces, 8 lanes per 128-byte row of qT, instead of 16 scattered 8-byte pieces
// per warp store.  A SiLU-mul backward item is one source column block, which yields its
// dg and its du tile from one evaluation of the sigmoid.
template <int PRO, bool ROW_OUT, bool COL_OUT>
__global__ void __launch_bounds__(256, 2) k_quant_panel(const __grid_constant__ CUtensorMap tmx,
                                                     const __grid_constant__ CUtensorMap tmy,
                                                     const PanelArgs a) {
    constexpr bool COLQ = COL_OUT;
    using PS = PanelStages<PRO, COLQ>;
    constexpr int STAGES = PS::STAGES;
    extern __shared__ uint8_t q_smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q_smem_raw) + 127) & ~uintptr_t(127));
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ int abort_flag;
    __shared__ __align__(16) uint32_t s_colmax[8][64];  // per-warp column maxima (BF16 bits, pairs)
    __shared__ __align__(16) float s_rstd[128];
    __shared__ __align__(16) F2 s_part[128];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = lane >> 4, cl = lane & 15;
    const int R0 = 16 * warp + 8 * half, C0 = 8 * cl;
    const int64_t ntiles = a.K / 128;
    // Tile sequence of this CTA.  RMSNorm: tiles [t_begin, t_end) of panel blockIdx.y, its
    // share of the panel's cluster (streamed twice).  Otherwise persistent: every
    // gridDim.x-th (panel, tile) pair from blockIdx.x, so the TMA ring runs across tiles
    // and panels without a cold start per CTA.
    constexpr bool PERSIST = PRO != PRO_RMSNORM;
    const int64_t rms_panel = blockIdx.y;
    const int64_t rms_m0 = rms_panel * 128;
    const int64_t all_tiles = ((a.M + 127) / 128) * (PRO == PRO_SILU_BWD ? ntiles / 2 : ntiles);   // items
    const int64_t t_begin = PERSIST ? 0 : (int64_t)blockIdx.x * a.tiles_per_cta;
    const int64_t t_end = (t_begin + a.tiles_per_cta < ntiles) ? t_begin + a.tiles_per_cta : ntiles;
    const int n = PERSIST ? (int)((all_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x) : (int)(t_end - t_begin);
    const int total = (PRO == PRO_RMSNORM) ? 2 * n : n;   // items streamed through the ring
    auto tile_at = [&](int it, int64_t& pnl, int64_t& tt) {
        if (PERSIST) {
            // SiLU-mul backward: an item is a source column block, which gives both its dg
            // and its du tile
            const int64_t per = PRO == PRO_SILU_BWD ? ntiles / 2 : ntiles;
            const int64_t id = blockIdx.x + (int64_t)(it % n) * gridDim.x;
            pnl = id / per;
            tt = id - pnl * per;
        } else {
            pnl = rms_panel;
            tt = t_begin + it % n;
        }
    };

    if (tid == 0) {
        for (int st = 0; st < STAGES; ++st) mbar_init(smem_u32(&full_bar[st]), 1);
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmx);
        if (PRO == PRO_SILU_BWD) tma_prefetch_desc(&tmy);
    }
    __syncthreads();
    // part: 0 every tile of the item; SiLU-mul backward also 1 (the barrier's arrival and
    // the up and dh tiles) and 2 (the gate tile), issued at different times
    auto issue = [&](int item, int part = 0) {
        const int st = item % STAGES;
        int64_t pnl, tt;
        tile_at(item, pnl, tt);
        const int64_t k0 = tt * 128, m0 = pnl * 128;
        const uint32_t bar = smem_u32(&full_bar[st]);
        uint8_t* dst = stages + st * PS::STAGE_BYTES;
        if (part != 2) mbar_arrive_expect_tx(bar, PS::STAGE_BYTES);
        if (PRO == PRO_DEQUANT) {
            // the code tile and the 128 row scales of its column block (one bulk copy:
            // 512 bytes at a 16-byte-aligned offset, since M is a multiple of 128)
            tma_load_2d(smem_u32(dst), &tmx, bar, (int)k0, (int)m0, 0);
            bulk_load_1d(smem_u32(dst + 128 * 128), a.xs + tt * a.M + m0, 128 * 4, bar);
        } else if (PRO == PRO_SILU_BWD) {
            // output column tile k0 is dg (k0 < I) or du (k0 >= I) of source column block j0:
            // the gate tile, the up tile and the tile of dh of that block
            const int64_t half_k = a.K / 2;
            const int64_t j0 = k0 < half_k ? k0 : k0 - half_k;
            if (part != 1) tma_load_2d(smem_u32(dst), &tmx, bar, (int)j0, (int)m0, 0);
            if (part != 2) {
                tma_load_2d(smem_u32(dst + 128 * 128 * 2), &tmx, bar, (int)(half_k + j0), (int)m0, 0);
                tma_load_2d(smem_u32(dst + 2 * 128 * 128 * 2), &tmy, bar, (int)j0, (int)m0, 0);
            }
        } else {
            tma_load_2d(smem_u32(dst), &tmx, bar, (int)k0, (int)m0, 0);
            if (PRO == PRO_SILU) tma_load_2d(smem_u32(dst + 128 * 128 * 2), &tmx, bar, (int)(a.K + k0), (int)m0, 0);
        }
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < STAGES && issued < total; ++issued) issue(issued);
    // every thread waits for item `it`; the decision to stop is made block-wide
    auto wait_item = [&](int it) -> bool {
        const bool got = mbar_wait(smem_u32(&full_bar[it % STAGES]), (it / STAGES) & 1, a.timeout_ns, &abort_flag);
        return !__syncthreads_or(got ? 0 : 1);
    };
    bool ok = true;
    int item = 0;

    if (PRO == PRO_RMSNORM) {
        // Pass 1: this CTA's share of every row's sum of squares.
        F2 acc[8];
        #pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = F2{0.0f, 0.0f};
        for (; ok && item < n; ++item) {
            ok = wait_item(item);
            if (!ok) break;
            const uint8_t* stage = stages + (item % STAGES) * PS::STAGE_BYTES;
            uint4 v[8];
            #pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = *reinterpret_cast<const uint4*>(stage + (R0 + i) * 256 + C0 * 2);
            __syncthreads();                              // stage consumed: refill it
            if (tid == 0 && issued < total) issue(issued++);
            #pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t xv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                #pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x0 = bf16_lo(xv[j]), x1 = bf16_hi(xv[j]);
                    acc[i] = two_sum_acc(acc[i], __fmul_rn(x0, x0));
                    acc[i] = two_sum_acc(acc[i], __fmul_rn(x1, x1));
                }
            }
        }
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            #pragma unroll
            for (int off = 8; off >= 1; off >>= 1) {
                F2 o;
                o.hi = __shfl_xor_sync(0xffffffffu, acc[i].hi, off);
                o.lo = __shfl_xor_sync(0xffffffffu, acc[i].lo, off);
                acc[i] = f2_add(acc[i], o);
            }
        }
        if (cl == 0) {
            #pragma unroll
            for (int i = 0; i < 8; ++i) s_part[R0 + i] = acc[i];
        }
        // Every CTA of the cluster reaches both cluster barriers, also after an abort.
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (tid < 128) {
            const unsigned nranks = cluster.num_blocks();
            F2 tot = F2{0.0f, 0.0f};
            for (unsigned rk = 0; rk < nranks; ++rk) {
                const F2* peer = cluster.map_shared_rank(s_part, rk);
                tot = f2_add(tot, peer[tid]);
            }
            const double sum = (double)tot.hi + (double)tot.lo;
            const float ms = __double2float_rn(sum / (double)a.K);
            const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
            s_rstd[tid] = rstd;
            const int64_t m = rms_m0 + tid;
            if (ok && a.rstd_out && cluster.block_rank() == 0 && m < a.M) a.rstd_out[m] = rstd;
        }
        __syncthreads();
    }

    for (; ok && item < total; ++item) {
        ok = wait_item(item);
        if (!ok) break;
        int64_t panel, t;
        tile_at(item, panel, t);
        const int64_t m0 = panel * 128;
        uint8_t* const stage = stages + (item % STAGES) * PS::STAGE_BYTES;
        // Quantize one output tile, column block tt, from this thread's BF16 words w (8 rows
        // x 8 columns), its 128x1 codes staged at colq.  After the first barrier the stage
        // is refilled (refill 1), has its up and dh tiles requested (refill 2), or neither.
        auto quantize_tile = [&](uint32_t (&w)[8][4], const int64_t tt, const uint32_t colq, const int refill) {
            const int64_t k0 = tt * 128;
            const int64_t t = tt;
            // group maxima (exact BF16 values) on the packed words with the sign bits cleared
            // rows over the 16 lanes of the half-warp, columns over this warp's
            // 16 rows here and over the 8 warps through shared memory
            auto wa = [&](int i, int j) { return w[i][j] & 0x7FFF7FFFu; };
            uint32_t pm[4];   // rows (2k, 2k+1) of this half, as BF16 bits
            if (ROW_OUT) {
                #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t m2[2];
                    #pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        uint32_t v = __vmaxu2(wa(2 * k + e, 0), wa(2 * k + e, 1));
                        v = __vmaxu2(v, __vmaxu2(wa(2 * k + e, 2), wa(2 * k + e, 3)));
                        m2[e] = v;
                    }
                    // per row: max of its two halves; rows 2k (low) and 2k+1 (high) in one word
                    pm[k] = __vmaxu2(__byte_perm(m2[0], m2[1], 0x5410), __byte_perm(m2[0], m2[1], 0x7632));
                }
                #pragma unroll
                for (int off = 8; off >= 1; off >>= 1)
                    #pragma unroll
                    for (int k = 0; k < 4; ++k) pm[k] = __vmaxu2(pm[k], __shfl_xor_sync(0xffffffffu, pm[k], off));
            }
            if (COL_OUT) {
                uint32_t cm[4];
                #pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t c = __vmaxu2(__vmaxu2(wa(0, j), wa(1, j)), __vmaxu2(wa(2, j), wa(3, j)));
                    c = __vmaxu2(c, __vmaxu2(__vmaxu2(wa(4, j), wa(5, j)), __vmaxu2(wa(6, j), wa(7, j))));
                    cm[j] = __vmaxu2(c, __shfl_xor_sync(0xffffffffu, c, 16));
                }
                // half h keeps the pair words 4cl + 2h, +1 (its own four columns) at word 32h + 2cl
                *reinterpret_cast<uint2*>(&s_colmax[warp][32 * half + 2 * cl]) = half ? make_uint2(cm[2], cm[3]) : make_uint2(cm[0], cm[1]);
            }
            // values are unpacked where they are encoded: holding the 64 unpacked floats would
            // double the registers and halve the CTAs per SM
            auto xrow = [&](int i, int j) { return make_float2(bf16_lo(w[i][j]), bf16_hi(w[i][j])); };
            __syncthreads();                                  // stage consumed, column maxima published
            if (tid == 0 && issued < total) {
                if (refill == 1) issue(issued++);
                else if (refill == 2) issue(issued, 1);
            }

            // row scales: lane cl computes the scale of row (cl & 7) of its half; every lane
            // takes the scales of its 8 rows from those lanes
            FastScale fs = {};
            if (ROW_OUT) {
                const int ri = cl & 7;
                const uint32_t pw = (ri >> 1) == 0 ? pm[0] : (ri >> 1) == 1 ? pm[1] : (ri >> 1) == 2 ? pm[2] : pm[3];
                fs = fast_scale(bf16_bits_amax_to_f32((ri & 1) ? (pw >> 16) : (pw & 0xFFFFu)));
                if (cl < 8 && m0 + R0 + ri < a.M) a.s[t * a.M + m0 + R0 + ri] = fs.s;
            }
            // column scales: this half computes those of columns C0 + 4*half + {0..3} (from the
            // 8 warps' maxima) and swaps them with the other half for the remaining four
            float cs[8], cr[8];
            if (COL_OUT) {
                uint32_t mx0 = 0, mx1 = 0;
                #pragma unroll
                for (int ww = 0; ww < 8; ++ww) {
                    const uint2 v = *reinterpret_cast<const uint2*>(&s_colmax[ww][32 * half + 2 * cl]);
                    mx0 = __vmaxu2(mx0, v.x);
                    mx1 = __vmaxu2(mx1, v.y);
                }
                const uint32_t mb[4] = {mx0 & 0xFFFFu, mx0 >> 16, mx1 & 0xFFFFu, mx1 >> 16};
                float os[4], orr[4];
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const FastScale f = fast_scale(bf16_bits_amax_to_f32(mb[e]));
                    os[e] = f.s;
                    orr[e] = f.nr;
                }
                if (warp == 0)
                    *reinterpret_cast<float4*>(a.sT + panel * a.K + k0 + C0 + 4 * half) = make_float4(os[0], os[1], os[2], os[3]);
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float ts = __shfl_xor_sync(0xffffffffu, os[e], 16);
                    const float tr = __shfl_xor_sync(0xffffffffu, orr[e], 16);
                    cs[e] = half ? ts : os[e];
                    cr[e] = half ? tr : orr[e];
                    cs[4 + e] = half ? os[e] : ts;
                    cr[4 + e] = half ? orr[e] : tr;
                }
            }
            // the 8 codes of column C0 + cc, rows R0 .. R0 + 7: into the qT staging tile, or
            // straight to qT
            auto col_store = [&](int cc, uint32_t lo, uint32_t hi) {
                if (COLQ) {
                    // row c = C0 + cc of the staging tile holds its 8-byte pieces r8 = R0 / 8 at
                    // slot r8 ^ (2 (c/8 mod 8) + c/64): the 16 lanes of each half-warp store to 16
                    // different slots, so a store takes the minimum two wavefronts
                    const uint32_t slot = (uint32_t)((R0 >> 3) ^ (2 * (cl & 7) + (cl >> 3)));
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(colq + (uint32_t)(C0 + cc) * 128u + slot * 8u),
                                 "r"(lo), "r"(hi)
                                 : "memory");
                } else {
                    stg_v2(a.qT + (k0 + C0 + cc) * a.M + m0 + R0, lo, hi);
                }
            };
            // 1x128 codes, one row at a time, any scale
            auto row_codes = [&]() {
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int src = (lane & 16) | i;
                    const float si = __shfl_sync(0xffffffffu, fs.s, src);
                    const float nri = __shfl_sync(0xffffffffu, fs.nr, src);
                    const uint32_t keep = si == 0.0f ? 0u : 0xFFFFFFFFu;
                    uint32_t c[4];
                    #pragma unroll
                    for (int j = 0; j < 4; ++j) c[j] = encode_pair_neg(xrow(i, j), si, nri);
                    uint32_t lo = flip_codes(c[0], c[1], keep), hi = flip_codes(c[2], c[3], keep);
                    if (si > 0.0f && scale_is_slow(si)) {
                        const uint4 v = encode4_slow(xrow(i, 0), xrow(i, 1), xrow(i, 2), xrow(i, 3), si);
                        lo = v.x | (v.y << 16);
                        hi = v.z | (v.w << 16);
                    }
                    const int64_t m = m0 + R0 + i;
                    if (m < a.M) stg_v2(a.q + m * a.K + k0 + C0, lo, hi);
                }
            };
            // 128x1 codes, one column at a time (vertically adjacent pairs), any scale
            auto col_codes = [&]() {
                #pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const int j = cc >> 1;
                    const uint32_t keep = cs[cc] == 0.0f ? 0u : 0xFFFFFFFFu;
                    float2 x[4];
                    #pragma unroll
                    for (int k = 0; k < 4; ++k)
                        x[k] = (cc & 1) ? make_float2(bf16_hi_v(w[2 * k][j]), bf16_hi_v(w[2 * k + 1][j]))
                                        : make_float2(bf16_lo_v(w[2 * k][j]), bf16_lo_v(w[2 * k + 1][j]));
                    uint32_t c[4];
                    #pragma unroll
                    for (int k = 0; k < 4; ++k) c[k] = encode_pair_neg(x[k], cs[cc], cr[cc]);
                    uint32_t lo = flip_codes(c[0], c[1], keep), hi = flip_codes(c[2], c[3], keep);
                    if (cs[cc] > 0.0f && scale_is_slow(cs[cc])) {
                        const uint4 v = encode4_slow(x[0], x[1], x[2], x[3], cs[cc]);
                        lo = v.x | (v.y << 16);
                        hi = v.z | (v.w << 16);
                    }
                    col_store(cc, lo, hi);
                }
            };
            if (ROW_OUT && COL_OUT) {
                bool slow = fs.slow;
                #pragma unroll
                for (int cc = 0; cc < 8; ++cc) slow = slow || (cs[cc] > 0.0f && scale_is_slow(cs[cc]));
                if (__any_sync(0xffffffffu, slow)) {
                    row_codes();
                    col_codes();
                } else {
                    // No group of this warp needs a division: both directions from one unpack
                    // of each BF16 pair (columns 2j, 2j+1 of a row), the row code pair under the
                    // row's scale and the column code pair under the two columns' scales.  The
                    // column pairs of rows 2k and 2k+1 are packed as P[j][k] = bytes (r2k c2j,
                    // r2k c2j+1, r2k+1 c2j, r2k+1 c2j+1); byte permutes then give each column's
                    // 8 codes in row order.
                    float2 csp[4], crp[4];
                    #pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        csp[j] = make_float2(cs[2 * j], cs[2 * j + 1]);
                        crp[j] = make_float2(cr[2 * j], cr[2 * j + 1]);
                    }
                    uint32_t P[4][4], ev[4];
                    #pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int src = (lane & 16) | i;
                        const float si = __shfl_sync(0xffffffffu, fs.s, src);
                        const float nri = __shfl_sync(0xffffffffu, fs.nr, src);
                        const uint32_t keep = si == 0.0f ? 0u : 0xFFFFFFFFu;
                        uint32_t rc[4];
                        #pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float2 x = xrow(i, j);
                            rc[j] = encode_pair_neg(x, si, nri);
                            const uint32_t c = encode_pair_neg2(x, csp[j], crp[j]);
                            if (i & 1) P[j][i >> 1] = ev[j] | (c << 16);
                            else ev[j] = c;
                        }
                        const int64_t m = m0 + R0 + i;
                        if (m < a.M) stg_v2(a.q + m * a.K + k0 + C0, flip_codes(rc[0], rc[1], keep), flip_codes(rc[2], rc[3], keep));
                    }
                    #pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        #pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int cc = 2 * j + e;
                            const uint32_t keep = cs[cc] == 0.0f ? 0u : 0xFFFFFFFFu;
                            const uint32_t sel = e ? 0x7531u : 0x6420u;
                            col_store(cc, (__byte_perm(P[j][0], P[j][1], sel) ^ 0x80808080u) & keep,
                                      (__byte_perm(P[j][2], P[j][3], sel) ^ 0x80808080u) & keep);
                        }
                    }
                }
            } else if (ROW_OUT) {
                row_codes();
            } else if (COL_OUT) {
                col_codes();
            }
            if (COLQ) {
                __syncthreads();
                {
                    // thread tid copies the 16-byte pieces id = tid + 256 i: row c = id / 8 of
                    // the staging tile, bytes 16k .. 16k + 15 (k = id % 8), i.e. its slots 2k and
                    // 2k + 1, which sit together at chunk k ^ (c/8 mod 8); 8 lanes write one
                    // 128-byte row of qT
                    #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int id = tid + 256 * i, c = id >> 3, k = id & 7;
                        uint4 v;
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                     : "r"(colq + (uint32_t)c * 128u + (uint32_t)((k ^ ((c >> 3) & 7)) * 16)));
                        // rows c with c / 8 >= 8 hold the pair (2k, 2k+1) in swapped order
                        if ((c >> 6) & 1) stg_v4(a.qT + (k0 + c) * a.M + m0 + 16 * k, v.z, v.w, v.x, v.y);
                        else stg_v4(a.qT + (k0 + c) * a.M + m0 + 16 * k, v.x, v.y, v.z, v.w);
                    }
                }
            }
        };
        uint32_t w[8][4];
        if constexpr (PRO == PRO_SILU_BWD) {
            // source column block t gives two output tiles: dg (block t) from the
            // registers, then du (block ntiles/2 + t) from the stage's up slot, where the
            // prologue left it; the sigmoid is evaluated once for both
            // The gate tile is dead after the prologue: its two halves stage the two tiles'
            // 128x1 codes, and the next item's gate tile is requested once they have left
            // (its up and dh tiles after the du tile has been read back).
            silu_bwd_pair_from_smem(stage, R0, C0, w);
            quantize_tile(w, t, smem_u32(stage), 0);
            const float rg0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            rows_from_smem<PRO_COPY>(stage + 128 * 256, a, 0, R0, C0, nullptr, rg0, w);
            quantize_tile(w, ntiles / 2 + t, smem_u32(stage) + 128u * 128u, COL_OUT ? 2 : 1);
            if (COL_OUT) {
                fence_proxy_async_smem();   // the staged codes are overwritten by TMA next
                __syncthreads();
                if (tid == 0 && issued < total) issue(issued++, 2);
            }
        } else {
            float rg[8];
            #pragma unroll
            for (int i = 0; i < 8; ++i)   // rows past M (TMA zero fill) are never stored
                rg[i] = (PRO == PRO_RMSNORM_G && m0 + R0 + i < a.M) ? __ldg(a.rstd_out + m0 + R0 + i) : 0.0f;
            rows_from_smem<PRO>(stage, a, t * 128, R0, C0, s_rstd, rg, w);
            // this tile's qT staging buffer (two, alternating: the next tile's barrier orders
            // this tile's reads before the writes of the tile after)
            quantize_tile(w, t, smem_u32(stages + PS::COLQ_OFF) + (uint32_t)(item & 1) * (128u * 128u), 1);
        }
    }
    if (tid == 0) {
        // after an abort: let every issued copy land before the CTA exits
        for (int j = item; j < issued; ++j) {
            volatile int no_abort = 0;
            mbar_wait(smem_u32(&full_bar[j % STAGES]), (j / STAGES) & 1, a.timeout_ns, &no_abort);
        }
    }
    if (PRO == PRO_RMSNORM) {
        // Keep this CTA's partial sums alive until every peer has read them.
        cg::this_cluster().sync();
    }
}

// ------------------------------------------------------------------------------------
// 128x128 weight blocks (+ optional transposed copy with the same scale).
// Persistent: each CTA takes every gridDim.x-th block.  Thread 0 streams the blocks through
// a ring of TMA stages (one 128x128 BF16 tile each); all threads pull their 8x8 sub-block
// into registers, and once everyone has it (the barrier that also publishes the warps'
// maxima) thread 0 refills that stage, so the copies of the next blocks overlap this
// block's encode and stores.
// ------------------------------------------------------------------------------------
struct W128Args {
    int64_t N, K;
    uint8_t* q;
    float* s;
    uint8_t* qT;
    uint64_t timeout_ns;
};
constexpr int kW128Stages = 2;
constexpr int kW128StageBytes = 128 * 128 * 2;
// + two 16 KB staging tiles for the W^T codes, + alignment slack
constexpr size_t kW128Smem = (size_t)kW128Stages * kW128StageBytes + 2 * 128 * 128 + 128;

__global__ void __launch_bounds__(256, 2) k_quant_128x128(const __grid_constant__ CUtensorMap tmw,
                                                          const W128Args a) {
    extern __shared__ uint8_t w_smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(w_smem_raw) + 127) & ~uintptr_t(127));
    __shared__ __align__(8) uint64_t full_bar[kW128Stages];
    __shared__ int abort_flag;
    __shared__ uint32_t s_wmax[2][8];   // per-warp maxima, double-buffered across blocks
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = lane >> 4, cl = lane & 15;
    const int R0 = 16 * warp + 8 * half, C0 = 8 * cl;
    const int64_t nbk = a.K / 128;
    const int64_t blocks = (a.N / 128) * nbk;
    const int n = (int)((blocks - blockIdx.x + gridDim.x - 1) / gridDim.x);   // blocks of this CTA

    if (tid == 0) {
        for (int st = 0; st < kW128Stages; ++st) mbar_init(smem_u32(&full_bar[st]), 1);
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmw);
    }
    __syncthreads();
    auto issue = [&](int item) {
        const int st = item % kW128Stages;
        const int64_t id = blockIdx.x + (int64_t)item * gridDim.x;
        const int64_t bn = id / nbk, bk = id - bn * nbk;
        const uint32_t bar = smem_u32(&full_bar[st]);
        mbar_arrive_expect_tx(bar, kW128StageBytes);
        tma_load_2d(smem_u32(stages + st * kW128StageBytes), &tmw, bar, (int)(bk * 128), (int)(bn * 128), 0);
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < kW128Stages && issued < n; ++issued) issue(issued);

    int done = n;   // blocks processed (fewer only after a wait gave up)
    for (int item = 0; item < n; ++item) {
        // every thread waits for the block; the decision to stop is made block-wide
        const bool got = mbar_wait(smem_u32(&full_bar[item % kW128Stages]), (item / kW128Stages) & 1,
                                   a.timeout_ns, &abort_flag);
        if (__syncthreads_or(got ? 0 : 1)) {
            done = item;
            break;
        }
        const int64_t id = blockIdx.x + (int64_t)item * gridDim.x;
        const int64_t bn = id / nbk, bk = id - bn * nbk;
        const int64_t n0 = bn * 128, k0 = bk * 128;
        const uint8_t* stage = stages + (item % kW128Stages) * kW128StageBytes;

        uint32_t w[8][4];
        uint32_t mx = 0;
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(stage + (R0 + i) * 256 + C0 * 2);
            w[i][0] = v.x; w[i][1] = v.y; w[i][2] = v.z; w[i][3] = v.w;
            #pragma unroll
            for (int j = 0; j < 4; ++j) mx = absmax2(mx, w[i][j]);
        }
        mx = max(mx & 0xFFFFu, mx >> 16);
        #pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) s_wmax[item & 1][warp] = mx;
        __syncthreads();                              // stage consumed, maxima published
        if (tid == 0 && issued < n) issue(issued++);
        uint32_t m = 0;
        #pragma unroll
        for (int i = 0; i < 8; ++i) m = max(m, s_wmax[item & 1][i]);
        const FastScale f = fast_scale(bf16_bits_amax_to_f32(m));
        if (tid == 0) a.s[bn * nbk + bk] = f.s;
        const int64_t N = a.N, K = a.K;
        uint8_t* const q = a.q;
        uint8_t* const qT = a.qT;
        // codes of the 8x8 block, row-major: rc[i] = row i, columns 0-3 | 4-7
        uint32_t rc[8][2];
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t c[4];
            #pragma unroll
            for (int j = 0; j < 4; ++j) c[j] = encode_pair_neg(make_float2(bf16_lo(w[i][j]), bf16_hi(w[i][j])), f.s, f.nr);
            rc[i][0] = flip_codes(c[0], c[1], f.keep);
            rc[i][1] = flip_codes(c[2], c[3], f.keep);
        }
        if (f.slow) {   // tiny block scale: divide (whole CTA, rare)
            #pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 v = encode4_slow(make_float2(bf16_lo(w[i][0]), bf16_hi(w[i][0])),
                                             make_float2(bf16_lo(w[i][1]), bf16_hi(w[i][1])),
                                             make_float2(bf16_lo(w[i][2]), bf16_hi(w[i][2])),
                                             make_float2(bf16_lo(w[i][3]), bf16_hi(w[i][3])), f.s);
                rc[i][0] = v.x | (v.y << 16);
                rc[i][1] = v.z | (v.w << 16);
            }
        }
        // 16-byte stores: lanes cl and cl^1 hold the two 8-byte halves of a 16-byte row
        // piece.  For each row pair the even lane stores the even row and the odd lane the
        // odd one, each after swapping the other row's half with its partner.
        const bool odd = cl & 1;
        #pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
            const uint32_t g0 = __shfl_xor_sync(0xffffffffu, odd ? rc[2 * pr][0] : rc[2 * pr + 1][0], 1);
            const uint32_t g1 = __shfl_xor_sync(0xffffffffu, odd ? rc[2 * pr][1] : rc[2 * pr + 1][1], 1);
            const uint32_t o0 = odd ? rc[2 * pr + 1][0] : rc[2 * pr][0];
            const uint32_t o1 = odd ? rc[2 * pr + 1][1] : rc[2 * pr][1];
            const int i = 2 * pr + (odd ? 1 : 0);
            if (odd) stg_v4(q + (n0 + R0 + i) * K + k0 + C0 - 8, g0, g1, o0, o1);
            else     stg_v4(q + (n0 + R0 + i) * K + k0 + C0, o0, o1, g0, g1);
        }
        if (qT) {
            // transposed codes: four 4x4 byte transposes (rows 0-3 | 4-7 x columns 0-3 | 4-7)
            uint32_t ct[8][2];   // ct[j] = column j, rows 0-3 | 4-7
            #pragma unroll
            for (int rh = 0; rh < 2; ++rh)
                #pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const uint32_t a0 = rc[4 * rh + 0][ch], a1 = rc[4 * rh + 1][ch];
                    const uint32_t a2 = rc[4 * rh + 2][ch], a3 = rc[4 * rh + 3][ch];
                    const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);
                    const uint32_t t2 = __byte_perm(a2, a3, 0x5140), t3 = __byte_perm(a2, a3, 0x7362);
                    ct[4 * ch + 0][rh] = __byte_perm(t0, t2, 0x5410);
                    ct[4 * ch + 1][rh] = __byte_perm(t0, t2, 0x7632);
                    ct[4 * ch + 2][rh] = __byte_perm(t1, t3, 0x5410);
                    ct[4 * ch + 3][rh] = __byte_perm(t1, t3, 0x7632);
                }
            // The W^T codes go out through a shared-memory tile, as in the panel
            // quantizers: row c = C0 + j of the tile holds its 8-byte pieces r8 = R0 / 8 at
            // slot r8 ^ (2 (c/8 mod 8) + c/64), so a warp store takes two wavefronts; after
            // a CTA barrier the tile leaves as 16-byte pieces, 8 lanes per 128-byte W^T row.
            const uint32_t colq = smem_u32(stages + kW128Stages * kW128StageBytes) + (uint32_t)(item & 1) * (128u * 128u);
            const uint32_t slot = (uint32_t)((R0 >> 3) ^ (2 * (cl & 7) + (cl >> 3)));
            #pragma unroll
            for (int j = 0; j < 8; ++j)
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(colq + (uint32_t)(C0 + j) * 128u + slot * 8u),
                             "r"(ct[j][0]), "r"(ct[j][1])
                             : "memory");
            __syncthreads();
            #pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int id = tid + 256 * i, c = id >> 3, k = id & 7;
                uint4 v;
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                             : "r"(colq + (uint32_t)c * 128u + (uint32_t)((k ^ ((c >> 3) & 7)) * 16)));
                // rows c with c / 8 >= 8 hold the pair (2k, 2k+1) in swapped order
                if ((c >> 6) & 1) stg_v4(qT + (k0 + c) * N + n0 + 16 * k, v.z, v.w, v.x, v.y);
                else stg_v4(qT + (k0 + c) * N + n0 + 16 * k, v.x, v.y, v.z, v.w);
            }
        }
    }
    // After a wait gave up: the copies already issued land before the CTA exits.
    if (tid == 0 && done < issued) {
        volatile int no_abort = 0;
        for (int j = done; j < issued; ++j)
            mbar_wait(smem_u32(&full_bar[j % kW128Stages]), (j / kW128Stages) & 1, a.timeout_ns, &no_abort);
    }
}

// ------------------------------------------------------------------------------------
// Diagnostic: the production scale (amax / 448 by correction step) and both production
// encodes (the branching one and the branch-free one with its zero-group sign mask)
// against IEEE division, for every BF16 group maximum in [amax_lo, amax_hi) and every BF16
// x with |x| <= amax (both signs, and both zeros).  Counts mismatches; records the first
// one found (x bits 0xFFFF: the scale itself).
// ------------------------------------------------------------------------------------
__global__ void k_debug_encode_check(uint32_t amax_lo, uint32_t amax_hi,
                                     unsigned long long* mismatches, uint32_t* first_bad) {
    unsigned long long bad = 0;
    for (uint32_t ab = amax_lo + blockIdx.x; ab < amax_hi; ab += gridDim.x) {
        const float amax = bf16_bits_amax_to_f32(ab);
        // reference: IEEE division for the scale and for every quotient
        GroupScale ref;
        ref.s = __fdiv_rn(amax, 448.0f);
        ref.zero = (ref.s == 0.0f);
        ref.slow = true;
        ref.r = 0.0f;
        const GroupScale g = make_scale(amax);
        const FastScale f = fast_scale(amax);
        if (threadIdx.x == 0 && (g.s != ref.s || f.s != ref.s || (!f.slow && f.s != 0.0f && -f.nr != __frcp_rn(f.s)))) {
            ++bad;   // the scale itself (reported with x bits 0xFFFF)
            atomicCAS(first_bad, 0xFFFFFFFFu, (ab << 16) | 0xFFFFu);
        }
        // x magnitudes 0 .. ab, both signs: 2*(ab+1) values, two per encode
        for (uint32_t i = threadIdx.x; i <= ab; i += blockDim.x) {
            const float xp = __uint_as_float(i << 16);
            const float xn = __uint_as_float((i | 0x8000u) << 16);
            const uint32_t want = encode_pair_ieee(xp, xn, ref);
            const uint32_t a = encode_pair(xp, xn, g);
            const uint32_t b = f.slow ? encode_pair_ieee(xp, xn, ref)
                                      : encode_pair_fast(make_float2(xp, xn), f.s, f.nr, f.keep);
            if (a != want || b != want) {
                ++bad;
                atomicCAS(first_bad, 0xFFFFFFFFu, (ab << 16) | i);
            }
        }
    }
    if (bad) atomicAdd(mismatches, bad);
}

cudaError_t launch_debug_encode_check(uint32_t amax_lo, uint32_t amax_hi,
                                      unsigned long long* mismatches, uint32_t* first_bad,
                                      cudaStream_t st) {
    k_debug_encode_check<<<2048, 256, 0, st>>>(amax_lo, amax_hi, mismatches, first_bad);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// Diagnostic: the raw device encoder over an array.
// ------------------------------------------------------------------------------------
__global__ void k_debug_e4m3(const float* __restrict__ in, uint8_t* __restrict__ out, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)(e4m3x2(in[i], 0.0f) & 0xFFu);
}

// ------------------------------------------------------------------------------------
// Host-side launchers (argument checks are done by the C ABI layer).
// ------------------------------------------------------------------------------------
cudaError_t launch_quant_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                               float* s, int num_sms, cudaStream_t st) {
    const int64_t ngroups = M * (K / 128);
    const int64_t blocks_needed = (ngroups + 15) / 16;
    const int64_t blocks = std::min<int64_t>(blocks_needed, (int64_t)num_sms * 16);
    k_quant_1x128<<<(unsigned)blocks, 256, 0, st>>>(x, M, K, ldx, q, s);
    return cudaGetLastError();
}

// 2-D tensor map of a BF16 matrix [rows][cols] (row stride ld elements), 128x128 boxes.
static cudaError_t tmap_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {128u, 128u};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D tensor map of a code matrix [rows][cols] bytes (rows contiguous), 128x128 boxes.
static cudaError_t tmap_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {128u, 128u};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int PRO, bool ROW_OUT, bool COL_OUT>
static cudaError_t launch_panel_t(const PanelArgs& a, int64_t in_cols, int cluster, cudaStream_t st) {
    CUtensorMap tm, tm2;
    cudaError_t e = PRO == PRO_DEQUANT ? tmap_u8(&tm, a.x, a.M, in_cols) : tmap_bf16(&tm, a.x, a.M, in_cols, a.ldx);
    if (e != cudaSuccess) return e;
    if (PRO == PRO_SILU_BWD) {
        e = tmap_bf16(&tm2, a.x2, a.M, a.K / 2, a.K / 2);
        if (e != cudaSuccess) return e;
    } else {
        tm2 = tm;   // unused
    }
    auto kern = k_quant_panel<PRO, ROW_OUT, COL_OUT>;
    constexpr size_t smem = PanelStages<PRO, COL_OUT>::SMEM;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = a.K / 128;
    cudaLaunchConfig_t cfg = {};
    if (PRO == PRO_RMSNORM) {
        cfg.gridDim = dim3((unsigned)((ntiles + a.tiles_per_cta - 1) / a.tiles_per_cta),
                           (unsigned)((a.M + 127) / 128), 1);
    } else {
        // persistent: as many CTAs as fit on the GPU at once, at most one per tile
        static const int resident = [&] {
            int dev = 0, sms = 0, per_sm = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem);
            return std::max(1, sms * std::max(1, per_sm));
        }();
        const int64_t all_tiles = ((a.M + 127) / 128) * (PRO == PRO_SILU_BWD ? ntiles / 2 : ntiles);   // items
        cfg.gridDim = dim3((unsigned)std::min<int64_t>(all_tiles, resident), 1, 1);
    }
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (cluster > 0) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, tm, tm2, a);
}

// Column tiles per CTA for the streaming kernels: enough to keep the TMA ring busy.

// quantize 1x128 with the transposed 128x1 output (dual), or 128x1 alone
cudaError_t launch_quant_dual(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                              float* s, uint8_t* qT, float* sT, uint64_t timeout_ns, cudaStream_t st) {
    PanelArgs a = {};
    a.x = x; a.ldx = ldx; a.M = M; a.K = K; a.q = q; a.s = s; a.qT = qT; a.sT = sT;
    a.timeout_ns = timeout_ns;
    if (q) return launch_panel_t<PRO_COPY, true, true>(a, K, 0, st);
    return launch_panel_t<PRO_COPY, false, true>(a, K, 0, st);
}

cudaError_t launch_silu_mul_quant(const uint16_t* gu, int64_t M, int64_t I, uint8_t* q, float* s,
                                  uint8_t* qT, float* sT, uint64_t timeout_ns, cudaStream_t st) {
    PanelArgs a = {};
    a.x = gu; a.ldx = 2 * I; a.M = M; a.K = I; a.q = q; a.s = s; a.qT = qT; a.sT = sT;
    a.timeout_ns = timeout_ns;
    if (qT) return launch_panel_t<PRO_SILU, true, true>(a, 2 * I, 0, st);
    return launch_panel_t<PRO_SILU, true, false>(a, 2 * I, 0, st);
}

// SiLU-mul backward -> dual quantization of the gate_up output's gradient [dg | du]
cudaError_t launch_silu_mul_bwd_quant(const uint16_t* gu, const uint16_t* dh, int64_t M, int64_t I, uint8_t* q,
                                      float* s, uint8_t* qT, float* sT, uint64_t timeout_ns, cudaStream_t st) {
    PanelArgs a = {};
    a.x = gu; a.ldx = 2 * I; a.x2 = dh; a.M = M; a.K = 2 * I; a.q = q; a.s = s; a.qT = qT; a.sT = sT;
    a.timeout_ns = timeout_ns;
    if (qT) return launch_panel_t<PRO_SILU_BWD, true, true>(a, 2 * I, 0, st);
    return launch_panel_t<PRO_SILU_BWD, true, false>(a, 2 * I, 0, st);
}

// 128x1 WGrad operand rebuilt from the saved 1x128 codes and scales of X
cudaError_t launch_requant_128x1(const uint8_t* q, const float* s, int64_t M, int64_t K, uint8_t* qT, float* sT,
                                 uint64_t timeout_ns, cudaStream_t st) {
    PanelArgs a = {};
    a.x = reinterpret_cast<const uint16_t*>(q); a.ldx = K; a.xs = s; a.M = M; a.K = K; a.qT = qT; a.sT = sT;
    a.timeout_ns = timeout_ns;
    return launch_panel_t<PRO_DEQUANT, false, true>(a, K, 0, st);
}

// Number of CTAs that split one 128-row panel of an RMSNorm along K: the largest divisor
// of K/128 that is at most 8 (a portable cluster size).
int rmsnorm_cluster_size(int64_t K) {
    const int64_t nt = K / 128;
    for (int c = 8; c >= 1; --c)
        if (nt % c == 0) return c;
    return 1;
}

cudaError_t launch_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M,
                                 int64_t K, uint8_t* q, float* s, uint8_t* qT, float* sT,
                                 float* rstd, uint64_t timeout_ns, cudaStream_t st) {
    PanelArgs a = {};
    a.x = x; a.ldx = K; a.gamma = gamma; a.eps = eps; a.rstd_out = rstd;
    a.M = M; a.K = K; a.q = q; a.s = s; a.qT = qT; a.sT = sT;
    a.timeout_ns = timeout_ns;
    if (rstd) {
        // rstd into the caller's buffer first, then the persistent quantizer reads it
        k_rms_rstd<<<(unsigned)((M + 7) / 8), 256, 0, st>>>(x, M, K, eps, rstd);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (qT) return launch_panel_t<PRO_RMSNORM_G, true, true>(a, K, 0, st);
        return launch_panel_t<PRO_RMSNORM_G, true, false>(a, K, 0, st);
    }
    // no rstd buffer (the library allocates none): the cluster kernel computes rstd in
    // shared memory
    const int c = rmsnorm_cluster_size(K);
    a.tiles_per_cta = (int)((K / 128) / c);
    if (qT) return launch_panel_t<PRO_RMSNORM, true, true>(a, K, c, st);
    return launch_panel_t<PRO_RMSNORM, true, false>(a, K, c, st);
}

cudaError_t launch_quant_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                 float* s, uint8_t* qT, uint64_t timeout_ns, cudaStream_t st) {
    CUtensorMap tm;
    cudaError_t e = tmap_bf16(&tm, w, N, K, ldw);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_quant_128x128, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kW128Smem);
    if (e != cudaSuccess) return e;
    // persistent: as many CTAs as fit on the GPU at once, at most one per block
    static const int resident = [] {
        int dev = 0, sms = 0, per_sm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_quant_128x128, 256, kW128Smem);
        return std::max(1, sms * std::max(1, per_sm));
    }();
    const int64_t blocks = (N / 128) * (K / 128);
    W128Args a = {N, K, q, s, qT, timeout_ns};
    k_quant_128x128<<<(unsigned)std::min<int64_t>(blocks, resident), 256, kW128Smem, st>>>(tm, a);
    return cudaGetLastError();
}

// This translation unit's copy of the device status word (its TMA waits write it).
fp8rl_status read_and_clear_quant_status() {
    unsigned int v = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return FP8RL_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
        return FP8RL_ERR_CUDA;
    return static_cast<fp8rl_status>(v);
}

cudaError_t launch_debug_e4m3(const float* in, uint8_t* out, int64_t n, cudaStream_t st) {
    const int64_t blocks = std::max<int64_t>(std::min<int64_t>((n + 255) / 256, 4096), 1);
    k_debug_e4m3<<<(unsigned)blocks, 256, 0, st>>>(in, out, n);
    return cudaGetLastError();
}

}  // namespace fp8rl
