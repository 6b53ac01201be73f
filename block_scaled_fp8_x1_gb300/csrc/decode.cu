// decode.cu -- decode-shaped forward GEMM for rollout (small M), weights on the MMA's M side.
//
// "Technical summary: Jet-RL", section "Core architecture": the rollout graph is a
// sub-graph of the training forward graph with the same quantization granularity and
// precision, so rollout's linear layers compute exactly the block-scaled sums of the
// training kernels (1x128 activations, 128x128 weight blocks, FP32 promotion per K-block):
//     Y[m, n] = sum_kb sx(kb, m) * sw(n/128, kb) * sum_{k in kb} X[m, k] W[n, k].
// Section "Problem definition": rollout dominates RL time at long generations, and at
// decode sizes (M = 64..256 tokens) the weight stream from HBM is the bound.
//
// Work split (one output tile = 128 weight rows x all M tokens):
//   * Swap of operands: A = the 128x128 weight tile (MMA M = 128), B = the activation tile
//     of M tokens (MMA N = MP, the tokens padded to 32/64/128/256 by TMA zero fill), so
//     every weight byte crosses HBM once and no MMA row is padding.
//   * Split-K over a cluster of S CTAs (S = 1..8): CTA r of the cluster streams K-blocks
//     [r*nkb/S, (r+1)*nkb/S) of the tile's weights.  Each CTA keeps its promoted FP32
//     partial sums in registers, parks them in its shared memory, and after a cluster
//     barrier CTA r adds every CTA's part of slice r through distributed shared memory,
//     in rank order (the result does not depend on timing), and writes BF16.  No
//     workspace, no second kernel.
// Roles (384 threads): warp 0 copies (weights and activation tiles by TMA; each K-block's
// per-token scales and the weight block's scale by cp.async into a scale ring); warp 1
// issues the MMAs (one elected lane) into one of NB TMEM buffers per K-block; warp 2
// multiplies each K-block's token scales by the weight block's scale once for everyone;
// warps 4-11 promote each K-block's partial into FP32 registers (two warps per TMEM lane
// quadrant, each half of the tokens), then store or run the cluster reduction.  Every mbarrier wait is bounded (FP8RL_ERR_DEVICE_TIMEOUT).
#include "cluster.cuh"
#include "common.cuh"
#include "gemm.h"

namespace fp8rl {

namespace {

template <int MP>
struct DecodeCfg {
    static constexpr int W_BYTES = 128 * 128;        // weight tile of one K-block
    static constexpr int X_BYTES = MP * 128;         // activation tile of one K-block
    static constexpr int STAGES = MP <= 64 ? 8 : (MP <= 128 ? 6 : 4);
    static constexpr int NB = (512 / MP) < 8 ? (512 / MP) : 8;   // TMEM buffers of MP columns
    static constexpr int NSC = 8;                    // scale-ring slots
    static constexpr int SLOT = MP + 4;              // floats: the tokens' scales, the weight block's
    static constexpr int CPT = MP / 2;               // token columns per epilogue thread
    static constexpr int LW = CPT >= 32 ? 32 : 16;   // columns per TMEM load
    static constexpr size_t STAGE_BYTES = (size_t)STAGES * (W_BYTES + X_BYTES);
    static constexpr size_t RED_BYTES = (size_t)MP * 128 * 4;   // [token][weight row] FP32
    static_assert(RED_BYTES <= STAGE_BYTES, "the reduction buffer reuses the stage ring");
    static constexpr int NBARS = 2 * STAGES + 2 * NB + 3 * NSC + 1;
    static constexpr size_t BYTES = 1024 + STAGE_BYTES + (size_t)NSC * (SLOT + MP) * 4 + NBARS * 8 + 16;
};

}  // namespace

// Grid: with a cluster of S > 1 CTAs, one cluster per weight tile (CTA r takes reduction
// slice r); with S = 1, persistent CTAs that each walk tiles blockIdx.x, +gridDim.x, ...
// with one continuous copy / MMA / epilogue pipeline, storing straight from registers.
template <int MP>
__global__ void __launch_bounds__(384, 1)
    k_decode(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
             const DecodeParams p) {
    using C = DecodeCfg<MP>;
    constexpr int STAGES = C::STAGES, NB = C::NB, NSC = C::NSC, CPT = C::CPT, LW = C::LW, SLOT = C::SLOT;
    constexpr uint32_t IDESC = idesc_e4m3_f32(128, MP);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sW = smem;
    uint8_t* sX = smem + STAGES * C::W_BYTES;
    float* red = reinterpret_cast<float*>(smem);                               // after the last K-block
    float* sc_ring = reinterpret_cast<float*>(smem + C::STAGE_BYTES);          // [NSC][SLOT] copied scales
    float* comb = sc_ring + NSC * SLOT;                                        // [NSC][MP] combined scales
    uint64_t* bars = reinterpret_cast<uint64_t*>(comb + NSC * MP);
    uint64_t* full_bar = bars;                  // [STAGES] tile copies -> MMA
    uint64_t* empty_bar = bars + STAGES;        // [STAGES] MMA -> copies
    uint64_t* tfull_bar = bars + 2 * STAGES;    // [NB] MMA -> epilogue
    uint64_t* tempty_bar = tfull_bar + NB;      // [NB] epilogue -> MMA
    uint64_t* sfull_bar = tempty_bar + NB;      // [NSC] scale copies landed -> combiner
    uint64_t* cfull_bar = sfull_bar + NSC;      // [NSC] combined scales -> epilogue
    uint64_t* sempty_bar = cfull_bar + NSC;     // [NSC] epilogue -> scale copies
    uint64_t* drain_bar = sempty_bar + NSC;     // [1] MMA completion at exit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = (int)cluster_nctarank();
    const int rank = (int)cluster_ctarank();
    const int tile0 = (int)cluster_idx();       // first 128-row weight tile of this CTA
    const int tstep = (int)cluster_count();
    const int tiles = p.tiles;
    const int kb0 = (int)(((int64_t)rank * p.nkb) / S);
    const int kb1 = (int)(((int64_t)(rank + 1) * p.nkb) / S);
    const int nk = kb1 - kb0;                   // K-blocks per tile of this CTA (>= 1)

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int t = 0; t < NB; ++t) {
            mbar_init(smem_u32(&tfull_bar[t]), 1);
            mbar_init(smem_u32(&tempty_bar[t]), 8);
        }
        for (int t = 0; t < NSC; ++t) {
            mbar_init(smem_u32(&sfull_bar[t]), 32);   // one cp.async arrival per copy lane
            mbar_init(smem_u32(&cfull_bar[t]), 1);
            mbar_init(smem_u32(&sempty_bar[t]), 8);
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

    if (warp < 4) {
        warpgroup_reg_dealloc<56>();
        if (warp == 0) {
            // ------------------------------------------------------------ copies
            const uint64_t pol_w = l2_policy_evict_first();   // each weight byte is read once
            const uint64_t pol_x = l2_policy_evict_last();    // every tile reads the activation
            constexpr uint32_t TX = C::W_BYTES + C::X_BYTES;
            // The weights do not depend on the kernel that produces the activation: the
            // first stages' weight tiles are requested before waiting for that kernel
            // (a no-op when this grid was not launched as its dependent).
            const uint32_t n_it = tile0 < tiles ? (uint32_t)((tiles - tile0 + tstep - 1) / tstep) * (uint32_t)nk : 0u;
            const uint32_t n_pre = n_it < (uint32_t)STAGES ? n_it : (uint32_t)STAGES;
            if (elect_one_sync()) {
                for (uint32_t j = 0; j < n_pre; ++j) {
                    const int tile = tile0 + (int)(j / (uint32_t)nk) * tstep;
                    const int kb = kb0 + (int)(j % (uint32_t)nk);
                    mbar_arrive_expect_tx(smem_u32(&full_bar[j]), TX);
                    tma_load_2d(smem_u32(sW + j * C::W_BYTES), &tmW, smem_u32(&full_bar[j]), kb * 128, tile * 128, pol_w);
                }
            }
            __syncwarp();
            asm volatile("griddepcontrol.wait;" ::: "memory");
            uint32_t it = 0;
            for (int tile = tile0; ok && tile < tiles; tile += tstep) {
                const float* swt = p.sw + (int64_t)tile * p.sw_r;
                for (int i = 0; i < nk; ++i, ++it) {
                    const int kb = kb0 + i;
                    const uint32_t s = it % STAGES;
                    if (it >= n_pre &&
                        !mbar_wait(smem_u32(&empty_bar[s]), ((it / STAGES) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (elect_one_sync()) {
                        if (it >= n_pre) {
                            mbar_arrive_expect_tx(smem_u32(&full_bar[s]), TX);
                            tma_load_2d(smem_u32(sW + s * C::W_BYTES), &tmW, smem_u32(&full_bar[s]), kb * 128, tile * 128, pol_w);
                        }
                        tma_load_2d(smem_u32(sX + s * C::X_BYTES), &tmX, smem_u32(&full_bar[s]), kb * 128, 0, pol_x);
                    }
                    __syncwarp();
                    // this K-block's scales: sx(kb, m) of every token (zero past M) and
                    // sw(tile, kb), by asynchronous copies whose landing completes the slot's
                    // barrier, so the tile copies never wait for a load
                    const uint32_t ss = it % NSC;
                    if (!mbar_wait(smem_u32(&sempty_bar[ss]), ((it / NSC) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t slot = smem_u32(sc_ring + ss * SLOT);
                    const float* sxk = p.sx + (int64_t)kb * p.sx_kb;
                    #pragma unroll
                    for (int c = lane; c < MP; c += 32) {
                        const bool v = c < p.M;
                        cp_async_4(slot + 4u * (uint32_t)c, v ? sxk + c : sxk, v ? 4u : 0u);
                    }
                    if (lane == 0) cp_async_4(slot + 4u * MP, swt + kb, 4u);
                    cp_async_arrive(smem_u32(&sfull_bar[ss]));
                }
            }
            // Drain: every issued copy lands before the stage memory is reused or freed.
            cp_async_wait_all();
            volatile int no_abort = 0;
            const uint32_t n_out = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
            for (uint32_t j = it - n_out; j < it; ++j)
                mbar_wait(smem_u32(&full_bar[j % STAGES]), (j / STAGES) & 1, p.timeout_ns, &no_abort);
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            const uint32_t w_base = smem_u32(sW), x_base = smem_u32(sX);
            uint32_t it = 0;
            for (int tile = tile0; ok && tile < tiles; tile += tstep) {
                for (int i = 0; i < nk; ++i, ++it) {
                    const uint32_t ts = it % NB;
                    const uint32_t s = it % STAGES;
                    if (!mbar_wait(smem_u32(&tempty_bar[ts]), ((it / NB) & 1) ^ 1, p.timeout_ns, abort_flag) ||
                        !mbar_wait(smem_u32(&full_bar[s]), (it / STAGES) & 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + ts * MP;
                    const uint64_t da = sdesc_kmajor_sw128(w_base + s * C::W_BYTES);
                    const uint64_t db = sdesc_kmajor_sw128(x_base + s * C::X_BYTES);
                    if (elect_one_sync()) {
                        #pragma unroll
                        for (int k = 0; k < 4; ++k)   // 32-byte steps inside the 128-byte rows
                            mma_f8(d, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                        mma_commit(smem_u32(&empty_bar[s]));
                        mma_commit(smem_u32(&tfull_bar[ts]));
                    }
                    __syncwarp();
                }
            }
            if (elect_one_sync()) mma_commit(smem_u32(drain_bar));
            __syncwarp();
            volatile int no_abort = 0;
            mbar_wait(smem_u32(drain_bar), 0, p.timeout_ns, &no_abort);
        } else if (warp == 2) {
            // ------------------------------------------------------------ scale combiner
            // per K-block, once for all epilogue threads: comb[m] = sx(kb, m) * sw(tile, kb)
            uint32_t it = 0;
            for (int tile = tile0; ok && tile < tiles; tile += tstep) {
                for (int i = 0; i < nk; ++i, ++it) {
                    const uint32_t ss = it % NSC;
                    if (!mbar_wait(smem_u32(&sfull_bar[ss]), (it / NSC) & 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const float* src = sc_ring + ss * SLOT;
                    const float fw = src[MP];
                    #pragma unroll
                    for (int c = lane; c < MP; c += 32) comb[ss * MP + c] = src[c] * fw;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&cfull_bar[ss]));
                }
            }
        }
    } else {
        warpgroup_reg_alloc<224>();
        // ------------------------------------------------------------ epilogue warps
        const int quad = warp & 3;                    // TMEM lane quadrant of this warp
        const int col0 = ((warp - 4) >> 2) * CPT;     // first token column of this thread
        const int row = quad * 32 + lane;             // weight row within the tile
        const uint32_t tb_lane = tmem_base + ((uint32_t)(quad * 32) << 16) + col0;
        uint32_t it = 0;
        for (int tile = tile0; ok && tile < tiles; tile += tstep) {
            float2 acc[CPT / 2];
            #pragma unroll
            for (int c = 0; c < CPT / 2; ++c) acc[c] = make_float2(0.0f, 0.0f);
            for (int i = 0; i < nk; ++i, ++it) {
                const uint32_t ts = it % NB, ss = it % NSC;
                bool got = mbar_wait(smem_u32(&cfull_bar[ss]), (it / NSC) & 1, p.timeout_ns, abort_flag);
                got = got && mbar_wait(smem_u32(&tfull_bar[ts]), (it / NB) & 1, p.timeout_ns, abort_flag);
                ok = __all_sync(0xffffffffu, got);
                if (!ok) break;
                tc_fence_after();
                const float* sc = comb + ss * MP + col0;
                const uint32_t tb = tb_lane + ts * MP;
                if constexpr (CPT <= 64) {
                    // the whole partial of this thread at once, then hand the buffer back
                    uint32_t r[CPT / LW][LW];
                    #pragma unroll
                    for (int h = 0; h < CPT / LW; ++h) tmem_ld_cols(tb + h * LW, r[h]);
                    #pragma unroll
                    for (int h = 0; h < CPT / LW; ++h) tmem_ld_wait(r[h]);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[ts]));
                    #pragma unroll
                    for (int h = 0; h < CPT / LW; ++h)
                        #pragma unroll
                        for (int j = 0; j < LW; j += 4) {
                            const float4 f = *reinterpret_cast<const float4*>(sc + h * LW + j);
                            const int a = (h * LW + j) / 2;
                            acc[a] = __ffma2_rn(make_float2(__uint_as_float(r[h][j]), __uint_as_float(r[h][j + 1])),
                                                make_float2(f.x, f.y), acc[a]);
                            acc[a + 1] = __ffma2_rn(make_float2(__uint_as_float(r[h][j + 2]), __uint_as_float(r[h][j + 3])),
                                                    make_float2(f.z, f.w), acc[a + 1]);
                        }
                } else {
                    // 128 columns: one 32-column load at a time, the buffer handed back after the last
                    #pragma unroll
                    for (int h = 0; h < CPT / LW; ++h) {
                        uint32_t r[LW];
                        tmem_ld_cols(tb + h * LW, r);
                        tmem_ld_wait(r);
                        if (h == CPT / LW - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[ts]));
                        }
                        #pragma unroll
                        for (int j = 0; j < LW; j += 4) {
                            const float4 f = *reinterpret_cast<const float4*>(sc + h * LW + j);
                            const int a = (h * LW + j) / 2;
                            acc[a] = __ffma2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                                                make_float2(f.x, f.y), acc[a]);
                            acc[a + 1] = __ffma2_rn(make_float2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])),
                                                    make_float2(f.z, f.w), acc[a + 1]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sempty_bar[ss]));
            }
            if (!ok) break;
            if (S == 1) {
                // the whole reduction is here: BF16 straight from registers, token by token
                // (a warp's 32 rows of one token are 64 contiguous bytes)
                uint16_t* yt = p.y + tile * 128 + row;
                #pragma unroll
                for (int c = 0; c < CPT / 2; ++c) {
                    const int t0 = col0 + 2 * c;
                    const uint32_t pk = pack_bf16x2(acc[c].x, acc[c].y);
                    if (t0 < p.M) yt[(int64_t)t0 * p.ldy] = (uint16_t)(pk & 0xFFFFu);
                    if (t0 + 1 < p.M) yt[(int64_t)(t0 + 1) * p.ldy] = (uint16_t)(pk >> 16);
                }
            } else {
                // one tile per cluster: every MMA of this CTA has completed (this warp waited
                // for the last K-block's buffer, and a commit covers all earlier MMAs), and
                // every tile copy was consumed by one, so the stage ring is free: park this
                // CTA's partial sums as red[token][weight row]
                #pragma unroll
                for (int c = 0; c < CPT / 2; ++c) {
                    red[(col0 + 2 * c) * 128 + row] = acc[c].x;
                    red[(col0 + 2 * c + 1) * 128 + row] = acc[c].y;
                }
            }
        }
    }

    // ---- cluster reduction: CTA r adds slice r of every CTA's partial sums in rank order
    __syncwarp();
    tc_fence_before();
    if (S > 1) {
        cluster_sync_all();
        if (warp >= 4 && *abort_flag == 0 && tile0 < tiles) {
            const int et = threadIdx.x - 128;                     // 0..255
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
                uint2 o;
                o.x = pack_bf16x2(v.x, v.y);
                o.y = pack_bf16x2(v.z, v.w);
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

template <int MP>
static cudaError_t launch_decode_t(const CUtensorMap& tw, const CUtensorMap& tx, const DecodeParams& p,
                                   int grid_clusters, int splits, bool pdl, cudaStream_t st) {
    auto kern = k_decode<MP>;
    constexpr size_t smem = DecodeCfg<MP>::BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(grid_clusters * splits), 1, 1);
    cfg.blockDim = dim3(384, 1, 1);
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

int decode_mp(int M) { return M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256)); }

// Clusters of `splits` CTAs of this kernel that fit on the device at once (0 on error).
int decode_max_clusters(int M, int splits) {
    const int mp = decode_mp(M);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)splits * 64, 1, 1);
    cfg.blockDim = dim3(384, 1, 1);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)splits;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e;
    switch (mp) {
        case 32: cfg.dynamicSmemBytes = DecodeCfg<32>::BYTES;
            cudaFuncSetAttribute(k_decode<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DecodeCfg<32>::BYTES);
            e = cudaOccupancyMaxActiveClusters(&n, k_decode<32>, &cfg); break;
        case 64: cfg.dynamicSmemBytes = DecodeCfg<64>::BYTES;
            cudaFuncSetAttribute(k_decode<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DecodeCfg<64>::BYTES);
            e = cudaOccupancyMaxActiveClusters(&n, k_decode<64>, &cfg); break;
        case 128: cfg.dynamicSmemBytes = DecodeCfg<128>::BYTES;
            cudaFuncSetAttribute(k_decode<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DecodeCfg<128>::BYTES);
            e = cudaOccupancyMaxActiveClusters(&n, k_decode<128>, &cfg); break;
        default: cfg.dynamicSmemBytes = DecodeCfg<256>::BYTES;
            cudaFuncSetAttribute(k_decode<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DecodeCfg<256>::BYTES);
            e = cudaOccupancyMaxActiveClusters(&n, k_decode<256>, &cfg); break;
    }
    return e == cudaSuccess ? n : 0;
}

cudaError_t launch_decode(const CUtensorMap& tw, const CUtensorMap& tx, const DecodeParams& p, int grid_clusters,
                          int splits, bool pdl, cudaStream_t st) {
    if (splits > 1 && grid_clusters != p.tiles) return cudaErrorInvalidValue;   // one tile per cluster
    switch (decode_mp(p.M)) {
        case 32: return launch_decode_t<32>(tw, tx, p, grid_clusters, splits, pdl, st);
        case 64: return launch_decode_t<64>(tw, tx, p, grid_clusters, splits, pdl, st);
        case 128: return launch_decode_t<128>(tw, tx, p, grid_clusters, splits, pdl, st);
        default: return launch_decode_t<256>(tw, tx, p, grid_clusters, splits, pdl, st);
    }
}

// Reads and clears this translation unit's device status word (the decode kernel's
// bounded waits record their timeouts in it).  The caller has synchronized the stream.
fp8rl_status read_and_clear_decode_status() {
    unsigned int v = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return FP8RL_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) return FP8RL_ERR_CUDA;
    return static_cast<fp8rl_status>(v);
}

}  // namespace fp8rl
