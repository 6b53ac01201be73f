// gemm.cu -- block-scaled FP8 GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// "Technical summary: Jet-RL", section "Quantization Scheme": the linear layers' GEMMs
// (forward, DGrad, WGrad) run in FP8 on operands quantized per 1x128 group (activations,
// gradients), per 128x128 block (weights) and, for WGrad, per 128x1 group.  Section "Core
// architecture": rollout uses the same numerics as the training forward pass, so the
// decode-shaped kernel below computes exactly the same sums as the tiled one.
//
// Computes  C[r1, r2] = sum_kb  fa(kb, r1) * fb(kb, r2) * P_kb[r1, r2],
//           P_kb = sum_{k in block kb} A[r1, k] * B[r2, k]      (E4M3 x E4M3, FP32)
// with A [R1, Kr] and B [R2, Kr] stored K-major (reduction dimension contiguous).
//
// Structure (one CTA of 320 threads per SM, persistent over work items):
//   warp 0      TMA producer: 128x128 A tile and BNx128 B tile per K-block into a
//               STAGES-deep shared-memory ring (128-byte swizzle).
//   warp 1      allocates TMEM and issues, per K-block, four tcgen05.mma (K = 32 each)
//               into one of two TMEM partial-sum buffers (fresh accumulate per block).
//   warps 2-9   epilogue: per K-block, load the 128 x BN FP32 partial from TMEM, release
//               the buffer, and promote it into FP32 registers with the block's scales
//               ("per-block scale promotion"); finally round to BF16 and store, or, in
//               the split-K form, store FP32 partials and let the last CTA of a tile sum
//               them in split order (deterministic, no spin-wait).
// Every mbarrier wait is bounded; on timeout the CTA records FP8RL_ERR_DEVICE_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "gemm.h"

namespace fp8rl {

// ------------------------------------------------------------------------------------
// Work decomposition shared by all roles.
// ------------------------------------------------------------------------------------
struct WorkItem {
    int mt;        // tile index along R1 (128 rows)
    int nt;        // tile index along R2 (BN columns)
    int kb_begin;  // first reduction block
    int kb_end;    // one past the last
    int tile;      // split-K: output tile id (counter index)
    int split;     // split-K: slice index
};

__device__ __forceinline__ WorkItem work_item(const GemmParams& p, int item) {
    WorkItem w;
    if (p.splits <= 0) {
        // tiled: grouped order, GROUP m-tiles share each sweep over the n-tiles
        constexpr int GROUP = 16;
        const int per_group = GROUP * p.n_tiles;
        const int g = item / per_group;
        const int first_m = g * GROUP;
        const int gm = min(GROUP, p.m_tiles - first_m);
        const int r = item - g * per_group;
        w.mt = first_m + r % gm;
        w.nt = r / gm;
        w.kb_begin = 0;
        w.kb_end = p.nkb;
        w.tile = 0;
        w.split = 0;
    } else {
        w.tile = item / p.splits;
        w.split = item - w.tile * p.splits;
        w.mt = w.tile;
        w.nt = 0;
        w.kb_begin = (int)(((int64_t)w.split * p.nkb) / p.splits);
        w.kb_end = (int)(((int64_t)(w.split + 1) * p.nkb) / p.splits);
    }
    return w;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int BN>
struct GemmSmem {
    static constexpr int A_BYTES = 128 * 128;
    static constexpr int B_BYTES = BN * 128;
};

constexpr int kGemmThreads = 320;

template <int BN, int A_MODE, int B_MODE, int STAGES, bool DECODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_bs(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const GemmParams p) {
    constexpr int A_BYTES = GemmSmem<BN>::A_BYTES;
    constexpr int B_BYTES = GemmSmem<BN>::B_BYTES;
    constexpr int HALF = BN / 2;      // columns per epilogue thread
    constexpr int NCH = HALF / 16;    // 16-column TMEM loads per K-block
    constexpr uint32_t TMEM_COLS = 2 * BN;
    constexpr uint32_t IDESC = idesc_e4m3_f32(128, BN);
    static_assert(HALF % 32 == 0, "BN must be a multiple of 64");
    static_assert(kGemmThreads == 320, "2 role warps + 8 epilogue warps");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
    uint64_t* full_bar = bars;                 // [STAGES] TMA -> MMA
    uint64_t* empty_bar = bars + STAGES;       // [STAGES] MMA -> TMA
    uint64_t* tfull_bar = bars + 2 * STAGES;   // [2] MMA -> epilogue
    uint64_t* tempty_bar = tfull_bar + 2;      // [2] epilogue -> MMA
    uint64_t* drain_bar = tempty_bar + 2;      // [1] MMA completion at exit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* last_flag = reinterpret_cast<int*>(tmem_slot + 2);
    // [8 warps][HALF] column scales, 16-byte aligned for vector reads
    float* bvec = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~uintptr_t(15));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&tfull_bar[t]), 1);
            mbar_init(smem_u32(&tempty_bar[t]), 8);
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_a = (p.splits > 0) ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_b = l2_policy_evict_last();
            uint32_t it = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x) {
                const WorkItem w = work_item(p, item);
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[s]);
                    mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
                    tma_load_2d(smem_u32(sA + s * A_BYTES), &tmA, fb, kb * 128, w.mt * 128, pol_a);
                    tma_load_2d(smem_u32(sB + s * B_BYTES), &tmB, fb, kb * 128, w.nt * BN, pol_b);
                }
            }
            // Drain: every issued copy must land before the CTA can exit.
            const uint32_t n_out = it < STAGES ? it : STAGES;
            for (uint32_t j = it - n_out; j < it; ++j) {
                volatile int no_abort = 0;
                mbar_wait(smem_u32(&full_bar[j % STAGES]), (j / STAGES) & 1, p.timeout_ns, &no_abort);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, acc_it = 0;
            bool ok = true;
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
            for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x) {
                const WorkItem w = work_item(p, item);
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it, ++acc_it) {
                    const uint32_t ts = acc_it & 1;
                    const uint32_t tph = (acc_it >> 1) & 1;
                    if (!mbar_wait(smem_u32(&tempty_bar[ts]), tph ^ 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t s = it % STAGES;
                    if (!mbar_wait(smem_u32(&full_bar[s]), (it / STAGES) & 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + ts * BN;
                    const uint64_t da = sdesc_kmajor_sw128(a_base + s * A_BYTES);
                    const uint64_t db = sdesc_kmajor_sw128(b_base + s * B_BYTES);
                    #pragma unroll
                    for (int k = 0; k < 4; ++k)  // 32-byte steps inside the 128-byte row
                        mma_f8(d, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                    mma_commit(smem_u32(&empty_bar[s]));
                    mma_commit(smem_u32(&tfull_bar[ts]));
                }
            }
            // All MMAs issued by this thread complete before TMEM is freed.
            mma_commit(smem_u32(drain_bar));
            volatile int no_abort = 0;
            mbar_wait(smem_u32(drain_bar), 0, p.timeout_ns, &no_abort);
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        // After an abort every warp keeps walking the same items and blocks (no waits, no
        // TMEM loads) so that all of them reach the same named barriers.
        const int ew = warp - 2;            // 0..7
        const int quad = warp & 3;          // TMEM lane quadrant this warp may access
        const int col_base = (ew >> 2) * HALF;
        const int row_local = quad * 32 + lane;
        const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
        float* my_bvec = bvec + ew * HALF;
        uint32_t acc_it = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
            const WorkItem w = work_item(p, item);
            const int64_t r1 = (int64_t)w.mt * 128 + row_local;
            const int64_t r1c = r1 < p.R1 ? r1 : p.R1 - 1;
            const int64_t n0 = (int64_t)w.nt * BN + col_base;  // first column of this thread
            float acc[HALF];
            #pragma unroll
            for (int c = 0; c < HALF; ++c) acc[c] = 0.0f;

            for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++acc_it) {
                if (!ok) continue;
                // scales of this K-block
                float fa;
                if (A_MODE == SCALE_ROW) fa = __ldg(p.sa + (int64_t)kb * p.sa_kb + r1c);
                else fa = __ldg(p.sa + (int64_t)w.mt * p.sa_r + (int64_t)kb * p.sa_kb);
                float fb_uniform = 1.0f;
                if (B_MODE == SCALE_BLOCK) {
                    const int64_t nb = n0 < p.R2 ? n0 / 128 : 0;
                    fb_uniform = __ldg(p.sb + nb * p.sb_r + (int64_t)kb * p.sb_kb);
                } else {
                    // this warp's HALF column scales -> its own shared slice
                    __syncwarp();
                    #pragma unroll
                    for (int c = lane; c < HALF; c += 32)
                        my_bvec[c] = (n0 + c < p.R2) ? __ldg(p.sb + (int64_t)kb * p.sb_kb + n0 + c) : 0.0f;
                    __syncwarp();
                }
                const uint32_t ts = acc_it & 1;
                const uint32_t tph = (acc_it >> 1) & 1;
                const bool got = mbar_wait(smem_u32(&tfull_bar[ts]), tph, p.timeout_ns, abort_flag);
                ok = __all_sync(0xffffffffu, got);
                if (!ok) continue;
                tc_fence_after();
                const float f = fa * fb_uniform;
                #pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tmem_base + t_lane + ts * BN + col_base + ch * 16, r);
                    tmem_ld_wait();
                    if (ch == NCH - 1) {
                        // partial fully in registers: hand the TMEM buffer back
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[ts]));
                    }
                    if (B_MODE == SCALE_BLOCK) {
                        #pragma unroll
                        for (int j = 0; j < 16; ++j)
                            acc[ch * 16 + j] = fmaf(__uint_as_float(r[j]), f, acc[ch * 16 + j]);
                    } else {
                        #pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            const float4 sbv = *reinterpret_cast<const float4*>(my_bvec + ch * 16 + j);
                            acc[ch * 16 + j + 0] = fmaf(__uint_as_float(r[j + 0]), fa * sbv.x, acc[ch * 16 + j + 0]);
                            acc[ch * 16 + j + 1] = fmaf(__uint_as_float(r[j + 1]), fa * sbv.y, acc[ch * 16 + j + 1]);
                            acc[ch * 16 + j + 2] = fmaf(__uint_as_float(r[j + 2]), fa * sbv.z, acc[ch * 16 + j + 2]);
                            acc[ch * 16 + j + 3] = fmaf(__uint_as_float(r[j + 3]), fa * sbv.w, acc[ch * 16 + j + 3]);
                        }
                    }
                }
            }

            if (!DECODE) {
                // ---- tiled: BF16 row segment of this thread
                if (ok && r1 < p.R1 && n0 < p.R2) {
                    uint16_t* dst = p.c + r1 * p.ldc + n0;
                    #pragma unroll
                    for (int c = 0; c < HALF; c += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(acc[c + 0], acc[c + 1]);
                        v.y = pack_bf16x2(acc[c + 2], acc[c + 3]);
                        v.z = pack_bf16x2(acc[c + 4], acc[c + 5]);
                        v.w = pack_bf16x2(acc[c + 6], acc[c + 7]);
                        *reinterpret_cast<uint4*>(dst + c) = v;
                    }
                }
            } else if (p.splits == 1) {
                // ---- decode, no split: transposed BF16 store C[r2][r1]
                if (ok && r1 < p.R1) {
                    #pragma unroll
                    for (int c = 0; c < HALF; ++c)
                        if (n0 + c < p.R2) p.c[(n0 + c) * p.ldc + r1] = (uint16_t)(pack_bf16x2(acc[c], 0.0f) & 0xFFFFu);
                }
            } else {
                // ---- decode, split-K: FP32 partial, then the last CTA of the tile reduces
                float* part = p.ws + ((int64_t)w.tile * p.splits + w.split) * (int64_t)(BN * 128);
                #pragma unroll
                for (int c = 0; c < HALF; ++c) __stcg(part + (int64_t)(col_base + c) * 128 + row_local, acc[c]);
                __threadfence();
                named_bar_sync(1, 256);
                if (ew == 0 && lane == 0) {
                    const unsigned prev = atomicAdd(p.counters + w.tile, 1u);
                    *last_flag = (prev == (unsigned)p.splits - 1) ? 1 : 0;
                }
                named_bar_sync(1, 256);
                if (*last_flag) {
                    __threadfence();
                    const float* tile_ws = p.ws + (int64_t)w.tile * p.splits * (int64_t)(BN * 128);
                    for (int c = 0; c < HALF; ++c) {
                        const int64_t col = col_base + c;
                        float sum = 0.0f;
                        for (int sp = 0; sp < p.splits; ++sp)
                            sum += __ldcg(tile_ws + (int64_t)sp * (BN * 128) + col * 128 + row_local);
                        if (r1 < p.R1 && col < p.R2)
                            p.c[col * p.ldc + r1] = (uint16_t)(pack_bf16x2(sum, 0.0f) & 0xFFFFu);
                    }
                    named_bar_sync(1, 256);
                    if (ew == 0 && lane == 0) {
                        p.counters[w.tile] = 0u;  // leave the counter ready for the next call
                        *last_flag = 0;
                    }
                }
                named_bar_sync(1, 256);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------
template <int BN, int STAGES>
constexpr size_t gemm_smem_bytes() {
    return 1024 + (size_t)STAGES * (GemmSmem<BN>::A_BYTES + GemmSmem<BN>::B_BYTES) +
           (2 * STAGES + 5) * 8 + 16 + 16 + 8 * (BN / 2) * 4 + 64;
}

template <int BN, int A_MODE, int B_MODE, int STAGES, bool DECODE>
static cudaError_t launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                            int grid, cudaStream_t st) {
    auto kern = k_gemm_bs<BN, A_MODE, B_MODE, STAGES, DECODE>;
    constexpr size_t smem = gemm_smem_bytes<BN, STAGES>();
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kGemmThreads, smem, st>>>(ta, tb, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_tiled(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                              int b_mode, int grid, cudaStream_t st) {
    if (b_mode == SCALE_BLOCK) return launch_t<256, SCALE_ROW, SCALE_BLOCK, 4, false>(ta, tb, p, grid, st);
    return launch_t<256, SCALE_ROW, SCALE_ROW, 4, false>(ta, tb, p, grid, st);
}

cudaError_t launch_gemm_splitk(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                               int bn, int grid, cudaStream_t st) {
    if (bn == 64) return launch_t<64, SCALE_BLOCK, SCALE_ROW, 8, true>(ta, tb, p, grid, st);
    if (bn == 128) return launch_t<128, SCALE_BLOCK, SCALE_ROW, 6, true>(ta, tb, p, grid, st);
    return launch_t<256, SCALE_BLOCK, SCALE_ROW, 4, true>(ta, tb, p, grid, st);
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
