// gemm.cu -- host side of the one-SM block-scaled FP8 GEMM (the kernel is in
// gemm_tiled.cuh), the split-K reduction of the decode-shaped form, and the device status
// word of this translation unit.
//
// "Technical summary: Jet-RL", section "Quantization Scheme": the linear layers' GEMMs
// (forward, DGrad, WGrad) run in FP8 on operands quantized per 1x128 group (activations,
// gradients), per 128x128 block (weights) and, for WGrad, per 128x1 group.
#include "gemm_tiled.cuh"

#include <algorithm>

namespace fp8rl {

// ------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------

// Tile order of the persistent GEMMs (raster_tile in gemm.h).  The tiles running at once
// advance through the reduction at about the same pace, so within a wave each operand tile
// is fetched from HBM about once.  Across waves, a group's panel of the grouped operand
// (its rows or columns across the whole reduction) is re-used from L2 when it is held to
// kRasterPanelBytes, and the other operand is read once per group: of the two
// orientations, the one with the fewest HBM reads of A and B together.  When even one
// row unit and one column tile are a sizeable share of that budget (a long reduction),
// no panel survives from one wave to the next and square waves (sqrt(wave) row units per
// group) read the fewest tiles per wave.  (Groups spanning all of an 84 MB operand, kept
// in L2 with evict-last hints while the other streamed with evict-first, measured 2.3 to
// 10 times the DRAM reads of these choices on GB300.)
constexpr int64_t kRasterPanelBytes = 48ll << 20;

void choose_raster(int64_t m_units, int64_t n_units, int64_t a_unit_bytes, int64_t b_unit_bytes, int wave,
                   int* group, int* raster_n) {
    m_units = std::max<int64_t>(m_units, 1);
    n_units = std::max<int64_t>(n_units, 1);
    if (std::min(a_unit_bytes, b_unit_bytes) > kRasterPanelBytes / 8) {
        int g = 1;
        while ((g + 1) * (g + 1) <= std::max(wave, 1)) ++g;
        *raster_n = 0;
        *group = (int)std::min<int64_t>(g, m_units);
        return;
    }
    const int64_t gm = std::min(m_units, std::max<int64_t>(1, kRasterPanelBytes / std::max<int64_t>(a_unit_bytes, 1)));
    const int64_t gn = std::min(n_units, std::max<int64_t>(1, kRasterPanelBytes / std::max<int64_t>(b_unit_bytes, 1)));
    const double a = (double)m_units * (double)a_unit_bytes, b = (double)n_units * (double)b_unit_bytes;
    const double reads_m = a + b * (double)((m_units + gm - 1) / gm);   // B once per row group
    const double reads_n = b + a * (double)((n_units + gn - 1) / gn);   // A once per column group
    *raster_n = reads_n < reads_m ? 1 : 0;
    *group = (int)(*raster_n ? gn : gm);
}


template <int BN, int SD, int B_MODE, int STAGES, bool SPLITK>
static cudaError_t launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                            const CUtensorMap& tsb, const CUtensorMap& tc, const GemmParams& p, int grid,
                            cudaStream_t st) {
    auto kern = k_gemm_bs<BN, SD, B_MODE, STAGES, SPLITK, 1, PlainOps>;
    constexpr size_t smem = GemmSmem<BN, STAGES, B_MODE, SD, SPLITK>::BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, gemm_threads(B_MODE), smem, st>>>(ta, tb, tsa, tsb, tc, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_tiled(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap* tsa,
                              const CUtensorMap* tsb, const CUtensorMap& tc, const GemmParams& p, int b_mode,
                              int bn, int grid, cudaStream_t st) {
    if (b_mode == SCALE_ROW) {
        // WGrad: both operands come from 128x1 quantization, every scale array is TMA-able
        if (!tsa || !tsb) return cudaErrorInvalidValue;
        if (bn == 128) return launch_t<128, SD_TMA, SCALE_ROW, 5, false>(ta, tb, *tsa, *tsb, tc, p, grid, st);
        return launch_t<256, SD_TMA, SCALE_ROW, 3, false>(ta, tb, *tsa, *tsb, tc, p, grid, st);
    }
    if (tsa && tsb) {
        if (bn == 128) return launch_t<128, SD_TMA, SCALE_BLOCK, 6, false>(ta, tb, *tsa, *tsb, tc, p, grid, st);
        return launch_t<256, SD_TMA, SCALE_BLOCK, 4, false>(ta, tb, *tsa, *tsb, tc, p, grid, st);
    }
    if (bn != 256) return cudaErrorInvalidValue;
    return launch_t<256, SD_THREAD, SCALE_BLOCK, 4, false>(ta, tb, tb, tb, tc, p, grid, st);
}

// Split-K reduction of the decode form: each output tile's FP32 slices summed in slice
// order (deterministic: the same order whatever the timing), rounded to BF16.  One CTA of
// 128 threads per (tile, 16-column chunk), thread t on row t of the tile, so the whole GPU
// shares the reduction instead of one CTA per tile.
constexpr int kSplitBN = 256;
__global__ void __launch_bounds__(128) k_splitk_reduce(const GemmParams p) {
    constexpr int CH = kSplitBN / 16;   // chunks per tile
    const int tile = blockIdx.x / CH, chunk = blockIdx.x - tile * CH;
    const WorkItem w = work_item<1>(p, tile * p.splits);
    const int64_t r1 = (int64_t)w.mt * 128 + threadIdx.x;
    const int64_t c0 = (int64_t)w.nt * kSplitBN + chunk * 16;
    if (r1 >= p.R1 || c0 >= p.R2) return;
    const float4* src = reinterpret_cast<const float4*>(p.ws) + (int64_t)tile * p.splits * (kSplitBN * 32) +
                        (int64_t)chunk * 4 * 128 + threadIdx.x;
    float4 sum[4];
    #pragma unroll
    for (int j = 0; j < 4; ++j) sum[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    int sp = 0;
    #pragma unroll 1
    for (; sp + 4 <= p.splits; sp += 4) {   // four slices' loads in flight
        float4 v[4][4];
        #pragma unroll
        for (int q = 0; q < 4; ++q)
            #pragma unroll
            for (int j = 0; j < 4; ++j) v[q][j] = __ldcg(src + (int64_t)(sp + q) * (kSplitBN * 32) + j * 128);
        #pragma unroll
        for (int q = 0; q < 4; ++q)
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                sum[j].x += v[q][j].x; sum[j].y += v[q][j].y;
                sum[j].z += v[q][j].z; sum[j].w += v[q][j].w;
            }
    }
    #pragma unroll 1
    for (; sp < p.splits; ++sp) {
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 v = __ldcg(src + (int64_t)sp * (kSplitBN * 32) + j * 128);
            sum[j].x += v.x; sum[j].y += v.y; sum[j].z += v.z; sum[j].w += v.w;
        }
    }
    // A slice whose bounded wait ran out stored no partial sums, so its slot may hold
    // another call's: once a timeout is on record (until fp8rl_check_status clears it)
    // the result is NaN rather than plausible but wrong values.
    if (*reinterpret_cast<volatile unsigned int*>(&g_device_status) == FP8RL_ERR_DEVICE_TIMEOUT) {
        const float qnan = __uint_as_float(0x7FC00000u);
        #pragma unroll
        for (int j = 0; j < 4; ++j) sum[j] = make_float4(qnan, qnan, qnan, qnan);
    }
    uint4 o0, o1;
    o0.x = pack_bf16x2(sum[0].x, sum[0].y); o0.y = pack_bf16x2(sum[0].z, sum[0].w);
    o0.z = pack_bf16x2(sum[1].x, sum[1].y); o0.w = pack_bf16x2(sum[1].z, sum[1].w);
    o1.x = pack_bf16x2(sum[2].x, sum[2].y); o1.y = pack_bf16x2(sum[2].z, sum[2].w);
    o1.z = pack_bf16x2(sum[3].x, sum[3].y); o1.w = pack_bf16x2(sum[3].z, sum[3].w);
    uint16_t* dst = p.c + r1 * p.ldc + c0;
    *reinterpret_cast<uint4*>(dst) = o0;
    *reinterpret_cast<uint4*>(dst + 8) = o1;
}

cudaError_t launch_gemm_splitk(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap* tsa,
                               const CUtensorMap* tsb, const GemmParams& p, int grid, cudaStream_t st) {
    // (the split-K form stores no BF16 boxes: tb stands in for the output map)
    cudaError_t e = (tsa && tsb) ? launch_t<kSplitBN, SD_TMA, SCALE_BLOCK, 4, true>(ta, tb, *tsa, *tsb, tb, p, grid, st)
                                 : launch_t<kSplitBN, SD_THREAD, SCALE_BLOCK, 4, true>(ta, tb, tb, tb, tb, p, grid, st);
    if (e != cudaSuccess || p.splits <= 1) return e;
    k_splitk_reduce<<<p.m_tiles * p.n_tiles * (kSplitBN / 16), 128, 0, st>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// Diagnostic: one CTA waits on an mbarrier nothing completes, with the bounded wait.
// ------------------------------------------------------------------------------------
__global__ void k_debug_wait_timeout(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, timeout_ns, &abort_flag);
}

cudaError_t launch_debug_wait_timeout(uint64_t timeout_ns, cudaStream_t st) {
    k_debug_wait_timeout<<<1, 32, 0, st>>>(timeout_ns);
    return cudaGetLastError();
}

fp8rl_status read_and_clear_device_status(cudaStream_t st) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return FP8RL_ERR_CUDA;
    unsigned int v = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return FP8RL_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
        return FP8RL_ERR_CUDA;
    return static_cast<fp8rl_status>(v);
}

}  // namespace fp8rl
