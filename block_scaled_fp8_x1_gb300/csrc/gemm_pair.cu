// gemm_pair.cu -- block-scaled FP8 GEMM on pairs of SMs (tcgen05 cta_group::2).
//
// "Technical summary: Jet-RL", section "Quantization Scheme": the forward, DGrad and
// WGrad GEMMs run in FP8 on operands quantized per 1x128 group (activations, gradients),
// per 128x128 block (weights) and, for WGrad, per 128x1 group; each 128-long reduction
// block's FP32 partial sum is promoted into an FP32 accumulator with the product of the
// two operands' scales for that block.
//
// Computes  C[r1, r2] = sum_kb  fa(kb, r1) * fb(kb, r2) * P_kb[r1, r2],
//           P_kb = sum_{k in block kb} A[r1, k] * B[r2, k]      (E4M3 x E4M3, FP32)
// with A [R1, Kr] and B [R2, Kr] K-major, the same contract as the one-SM kernel in
// gemm.cu.
//
// Why pairs.  The tensor pipe reads the operands of every MMA from shared memory, and a
// 128 x 256 tile on one SM moves 48 KB of A and B through it per K-block (written by TMA,
// read by the MMAs).  A cluster of two CTAs computes a 256 x PN tile with M = 256 MMAs
// (cta_group::2): each CTA holds 128 rows of A and half of B's PN rows, and the MMA
// reads B's halves from both CTAs, so with PN = 256 each SM moves 32 KB per K-block for
// the same 128 x 256 partial sum in its TMEM (two 256-column buffers).  PN = 128 keeps
// four 128-column buffers in flight instead, at the one-SM tile's traffic per FLOP.
//
// Roles (per CTA; both CTAs of a pair run all roles except the MMA issuer):
//   warp 0  TMA copies (the warp walks the loop, one elected lane issues).  Per K-block
//           this CTA's 128x128 tile of A and PN/2 x 128 half of B into a STAGES-deep
//           ring; both CTAs' copies complete on the leader's (rank 0) stage barrier.  Per
//           scale group, this CTA's row scales of A and the tile's scales of B into a
//           local scale ring.
//   warp 1  allocates the pair's TMEM (512 columns in each CTA); in the leader, one
//           elected lane issues four M256 x N(PN) x K32 MMAs per K-block into one of
//           512/PN buffers and commits to both CTAs' barriers (stage empty, buffer full).
//   warps 4.. epilogue: per K-block, load this CTA's 128 x PN partial from TMEM, hand the
//           buffer back to the leader, promote it with the block's scales into FP32
//           registers (WGrad: 16x256b fragments, each 16-row x 32-column part promoted
//           while the next part's load is in flight); at the end of a tile round to BF16
//           and store 32 x 32 boxes with TMA, double-buffered per warp.
// Every mbarrier wait is bounded; on timeout the waiting role records
// FP8RL_ERR_DEVICE_TIMEOUT and the CTA stops waiting, drains its MMAs and frees TMEM.
#include "common.cuh"
#include "gemm.h"

namespace fp8rl {

namespace {

// A pair tile is 256 rows x PN columns (PN = 128 or 256); each CTA's TMEM holds 512/PN
// partial-sum buffers of PN columns.
__host__ __device__ constexpr int pair_bufs(int pn) { return 512 / pn; }

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Pair tiles (pair-rows of 256 rows of C x column tiles) in the grouped order of
// raster_tile, so the clusters running at the same time reuse A and B through L2.
struct PairTile {
    int mp;   // pair-row tile (256 rows)
    int nt;   // column tile (PN columns)
};

__device__ __forceinline__ PairTile pair_tile(const GemmParams& p, int m_pairs, int item) {
    PairTile t;
    raster_tile(item, m_pairs, p.n_tiles, p.group, p.raster_n, &t.mp, &t.nt);
    return t;
}

// Register split: warpgroup 0 (copies, MMA, two idle warps) keeps few registers, the
// epilogue warpgroups take the rest of what the CTA is launched with.
__host__ __device__ constexpr int pair_threads(int epi) { return 128 + 32 * epi; }
__host__ __device__ constexpr int pair_launch_regs(int epi) { return epi == 16 ? 96 : 168; }
__host__ __device__ constexpr uint32_t pair_reg_lo(int epi) { return epi == 16 ? 32 : 56; }
__host__ __device__ constexpr uint32_t pair_reg_hi(int epi) { return epi == 16 ? 112 : 224; }
static_assert(128 * pair_reg_lo(8) + 256 * pair_reg_hi(8) <= pair_threads(8) * pair_launch_regs(8), "split");
static_assert(128 * pair_reg_lo(16) + 512 * pair_reg_hi(16) <= pair_threads(16) * pair_launch_regs(16), "split");

// Shared-memory plan of one CTA of the pair.
// BF16 output staging: each epilogue warp owns this many 2 KB boxes (32 x 32 BF16) and
// cycles through them, so one box's TMA store overlaps the filling of the next.
__host__ __device__ constexpr int pair_boxes(int epi) { return epi == 16 ? 1 : 2; }

template <int B_MODE, int EPI, int STAGES, int PN>
struct PairSmem {
    static constexpr int A_BYTES = 128 * 128;            // this CTA's 128 rows of A, one K-block
    static constexpr int B_BYTES = (PN / 2) * 128;       // this CTA's half of B's rows
    static constexpr int SG = scale_group(B_MODE, false);
    static constexpr int NS = (B_MODE == SCALE_ROW) ? 8 : 4;   // scale-ring slots (groups)
    static constexpr int SLOT_A = 128 * SG;                    // floats
    // B's scales: PN row scales per K-block, or a box of at most 16 block scales
    // (padded so that every TMA destination starts on a 128-byte boundary)
    static constexpr int SLOT_B = (B_MODE == SCALE_ROW) ? PN * SG : 32;
    static constexpr int SLOT = SLOT_A + SLOT_B;
    static_assert((SLOT_A * 4) % 128 == 0 && (SLOT * 4) % 128 == 0, "TMA destinations 128-byte aligned");
    static constexpr int RING_BYTES = NS * SLOT * 4;
    static constexpr int STAGE_C_BYTES = EPI * pair_boxes(EPI) * 2048;   // [warp][box][32x32 BF16]
    static constexpr int NBARS = 2 * STAGES + 2 * pair_bufs(PN) + 2 * NS + 1;
    static constexpr size_t BYTES = 1024 + (size_t)STAGES * (A_BYTES + B_BYTES) + STAGE_C_BYTES + RING_BYTES +
                                    NBARS * 8 + 16;
};

template <int B_MODE, int EPI, int STAGES, int PN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(EPI), 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    using S = PairSmem<B_MODE, EPI, STAGES, PN>;
    constexpr int kPairN = PN;
    constexpr int kPairBufs = pair_bufs(PN);
    constexpr int COLS = kPairN / (EPI / 4);        // columns per epilogue thread: 32 .. 128
    // TMEM loads of 32 columns, LPW of them per wait: the partial and the accumulators of
    // one thread stay within its registers
    constexpr int LPW = EPI == 16 ? 1 : 2;
    constexpr int NG = COLS / (32 * LPW);
    constexpr int NS = S::NS;
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t IDESC = idesc_e4m3_f32(256, kPairN);
    static_assert(COLS % 32 == 0, "whole 32-column TMEM loads");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * S::A_BYTES;
    uint8_t* stage_c = sB + STAGES * S::B_BYTES;                          // [warp][box][2 KB]
    float* ring = reinterpret_cast<float*>(stage_c + S::STAGE_C_BYTES);   // [NS][SLOT]
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ring) + S::RING_BYTES);
    uint64_t* full_bar = bars;                       // [STAGES] copies of both CTAs -> MMA (leader's)
    uint64_t* empty_bar = bars + STAGES;             // [STAGES] MMA -> copies (each CTA's own)
    uint64_t* tfull_bar = bars + 2 * STAGES;         // [bufs] MMA -> epilogue (each CTA's own)
    uint64_t* tempty_bar = tfull_bar + kPairBufs;    // [bufs] both epilogues -> MMA (leader's)
    uint64_t* sfull_bar = tempty_bar + kPairBufs;    // [NS] scale copies -> epilogue
    uint64_t* sempty_bar = sfull_bar + NS;           // [NS] epilogue -> scale copies
    uint64_t* drain_bar = sempty_bar + NS;           // [1] MMA completion at exit (leader)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cid = (int)cluster_id_x();
    const int ncl = (int)num_clusters_x();
    const int m_pairs = (p.m_tiles + 1) / 2;
    const int num_items = m_pairs * p.n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int t = 0; t < kPairBufs; ++t) {
            mbar_init(smem_u32(&tfull_bar[t]), 1);
            mbar_init(smem_u32(&tempty_bar[t]), 2 * EPI);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&sfull_bar[s]), 1);
            mbar_init(smem_u32(&sempty_bar[s]), EPI);
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 4) {
        warpgroup_reg_dealloc<pair_reg_lo(EPI)>();
        if (warp == 0) {
            // ------------------------------------------------------------ copies
            // (the whole warp walks the loop and waits; one elected lane issues, so the
            // coordinates and addresses stay warp-uniform)
            const uint64_t pol = l2_policy_evict_last();
            const int sgrp = p.nkb < S::SG ? p.nkb : S::SG;
            const uint32_t full0 = mapa_shared(smem_u32(full_bar), 0);   // the leader's
            uint32_t it = 0, s_issued = 0;
            bool ok = true;
            for (int item = cid; ok && item < num_items; item += ncl) {
                const PairTile t = pair_tile(p, m_pairs, item);
                const int m0 = t.mp * 256 + (int)rank * 128;            // this CTA's rows of A
                const int n0 = t.nt * kPairN;                           // the tile's first column
                const int nb = n0 + (int)rank * (kPairN / 2);           // this CTA's rows of B
                for (int kb = 0; kb < p.nkb; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    if (!mbar_wait(smem_u32(&empty_bar[s]), ((it / STAGES) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    // first K-block of a scale group: this CTA's row scales of A and the
                    // tile's scales of B for the whole group go into the next scale slot
                    const bool g_first = kb % S::SG == 0;
                    const uint32_t ss = s_issued % NS;
                    if (g_first && !mbar_wait(smem_u32(&sempty_bar[ss]), ((s_issued / NS) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (elect_one_sync()) {
                        if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[s]), 2 * (S::A_BYTES + S::B_BYTES));
                        tma_load_2d_pair(smem_u32(sA + s * S::A_BYTES), &tmA, full0 + 8 * s, kb * 128, m0, pol);
                        tma_load_2d_pair(smem_u32(sB + s * S::B_BYTES), &tmB, full0 + 8 * s, kb * 128, nb, pol);
                        if (g_first) {
                            const uint32_t sb = smem_u32(&sfull_bar[ss]);
                            float* slot = ring + ss * S::SLOT;
                            const uint32_t a_bytes = 128u * 4u * (uint32_t)sgrp;
                            if (B_MODE == SCALE_ROW) {
                                mbar_arrive_expect_tx(sb, a_bytes + (uint32_t)kPairN * 4u * (uint32_t)sgrp);
                                tma_load_2d(smem_u32(slot + S::SLOT_A), &tmSB, sb, n0, kb, pol);
                            } else if (p.sb_kb == 1) {
                                // block scales stored [column block][K-block]: 4 K-blocks of the
                                // tile's PN/128 column blocks (x, a K-block index, is a multiple of 4)
                                mbar_arrive_expect_tx(sb, a_bytes + 16u * (kPairN / 128));
                                tma_load_2d(smem_u32(slot + S::SLOT_A), &tmSB, sb, kb, n0 >> 7, pol);
                            } else {
                                // block scales stored [K-block][column block]: 4 column blocks
                                // from a 4-aligned one, for each K-block of the group
                                mbar_arrive_expect_tx(sb, a_bytes + 16u * (uint32_t)sgrp);
                                tma_load_2d(smem_u32(slot + S::SLOT_A), &tmSB, sb, (n0 >> 7) & ~3, kb, pol);
                            }
                            tma_load_2d(smem_u32(slot), &tmSA, sb, m0, kb, pol);
                        }
                    }
                    __syncwarp();
                    if (g_first) ++s_issued;
                }
            }
            // Drain: the copies issued here land before the CTA can exit.  The leader's
            // stage barriers count both CTAs' bytes; the local scale barriers this CTA's.
            volatile int no_abort = 0;
            if (leader) {
                const uint32_t n_out = it < STAGES ? it : STAGES;
                for (uint32_t j = it - n_out; j < it; ++j)
                    mbar_wait(smem_u32(&full_bar[j % STAGES]), (j / STAGES) & 1, p.timeout_ns, &no_abort);
            }
            const uint32_t s_out = s_issued < NS ? s_issued : NS;
            for (uint32_t j = s_issued - s_out; j < s_issued; ++j)
                mbar_wait(smem_u32(&sfull_bar[j % NS]), (j / NS) & 1, p.timeout_ns, &no_abort);
        } else if (warp == 1 && leader) {
            // ------------------------------------------------------------ MMA issuer
            // (warp-wide loop, one elected lane issues the pair's MMAs and commits)
            uint32_t it = 0;
            bool ok = true;
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
            for (int item = cid; ok && item < num_items; item += ncl) {
                for (int kb = 0; kb < p.nkb; ++kb, ++it) {
                    const uint32_t ts = it % kPairBufs;
                    if (!mbar_wait(smem_u32(&tempty_bar[ts]), ((it / kPairBufs) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t s = it % STAGES;
                    if (!mbar_wait(smem_u32(&full_bar[s]), (it / STAGES) & 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + ts * kPairN;
                    const uint64_t da = sdesc_kmajor_sw128(a_base + s * S::A_BYTES);
                    const uint64_t db = sdesc_kmajor_sw128(b_base + s * S::B_BYTES);
                    if (elect_one_sync()) {
                        #pragma unroll
                        for (int k = 0; k < 4; ++k)   // 32-byte steps inside the 128-byte rows
                            mma_f8_pair(d, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                        mma_commit_pair(smem_u32(&empty_bar[s]), 0x3);
                        mma_commit_pair(smem_u32(&tfull_bar[ts]), 0x3);
                    }
                    __syncwarp();
                }
            }
            // every MMA of the pair completes before either CTA frees its TMEM
            if (elect_one_sync()) mma_commit_pair(smem_u32(drain_bar), 0x1);
            __syncwarp();
            volatile int no_abort = 0;
            mbar_wait(smem_u32(drain_bar), 0, p.timeout_ns, &no_abort);
        }
    } else {
        warpgroup_reg_alloc<pair_reg_hi(EPI)>();
        // ------------------------------------------------------------ epilogue warps
        const int ew = warp - 4;                 // 0 .. EPI-1
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int col_base = (ew >> 2) * COLS;   // first column of this thread
        const int row_local = quad * 32 + lane;
        const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
        const uint32_t tempty0 = mapa_shared(smem_u32(tempty_bar), 0);   // the leader's
        constexpr int NBX = pair_boxes(EPI);
        uint32_t acc_it = 0, g_done = 0, box_it = 0;
        bool ok = true;
        for (int item = cid; ok && item < num_items; item += ncl) {
            const PairTile t = pair_tile(p, m_pairs, item);
            float2 acc[COLS / 2];
            #pragma unroll
            for (int c = 0; c < COLS / 2; ++c) acc[c] = make_float2(0.0f, 0.0f);

            for (int kb = 0; kb < p.nkb; ++kb, ++acc_it) {
                const uint32_t gi = S::SG == 1 ? acc_it : g_done;
                const uint32_t ss = gi % NS;
                const uint32_t ts = acc_it % kPairBufs;
                const int q = kb % S::SG;
                const bool g_first = q == 0;
                const bool g_last = kb + 1 == p.nkb || q == S::SG - 1;
                bool got = true;
                if (g_first) got = mbar_wait(smem_u32(&sfull_bar[ss]), (gi / NS) & 1, p.timeout_ns, abort_flag);
                got = got && mbar_wait(smem_u32(&tfull_bar[ts]), (acc_it / kPairBufs) & 1, p.timeout_ns, abort_flag);
                ok = __all_sync(0xffffffffu, got);
                if (!ok) break;
                tc_fence_after();
                const float* slot = ring + ss * S::SLOT;
                const uint32_t tb = tmem_base + t_lane + ts * kPairN + col_base;
                const float fa = slot[q * 128 + row_local];
                float2 f2 = make_float2(fa, fa);
                if constexpr (B_MODE != SCALE_ROW) {
                    // the block scale of B for this thread's 128-column block
                    const int cb = (t.nt * kPairN + col_base) >> 7;
                    const float fb = (p.sb_kb == 1) ? slot[S::SLOT_A + (cb - ((t.nt * kPairN) >> 7)) * 4 + (kb & 3)]
                                                    : slot[S::SLOT_A + q * 4 + (cb & 3)];
                    f2 = make_float2(fa * fb, fa * fb);
                }
                if constexpr (B_MODE == SCALE_ROW) {
                    // 16x256b fragments: rows g8 + 8h (h = 0..3) of the warp's 32 and columns
                    // 8j + 2tq + {0,1}; parts of 16 rows x 32 columns, the next part's TMEM
                    // load in flight while this one is promoted
                    const int g8 = lane >> 2, tq = lane & 3;
                    float fr[4];
                    const uint32_t fra = smem_u32(slot) + 4u * (uint32_t)(q * 128 + quad * 32 + g8);
                    #pragma unroll
                    for (int h = 0; h < 4; ++h)
                        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(fr[h]) : "r"(fra + 32u * h));
                    const uint32_t sba = smem_u32(slot) + 4u * (uint32_t)(S::SLOT_A + q * kPairN + col_base + 2 * tq);
                    const uint32_t tb0 = tmem_base + ((uint32_t)(quad * 32) << 16) + ts * kPairN + col_base;
                    const uint32_t tb1 = tb0 + (16u << 16);
                    constexpr int NP = 2 * (COLS / 32);
                    uint32_t ra[16], rb[16];
                    float2 sc[4];
                    tmem_ld_16x256b_x4(tb0, ra);
                    tmem_ld_wait(ra);
                    #pragma unroll
                    for (int pp = 0; pp < NP; ++pp) {
                        const int jq = pp >> 1, hh = pp & 1;
                        uint32_t (&cur)[16] = (pp & 1) ? rb : ra;
                        uint32_t (&nxt)[16] = (pp & 1) ? ra : rb;
                        if (pp + 1 < NP) {
                            tmem_ld_16x256b_x4((((pp + 1) & 1) ? tb1 : tb0) + ((pp + 1) >> 1) * 32, nxt);
                        } else {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive_cluster(tempty0 + 8 * ts);
                        }
                        if (hh == 0) {
                            #pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(sc[jj].x), "=f"(sc[jj].y) : "r"(sba + 32u * (jq * 4 + jj)));
                        }
                        #pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            #pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const int h = 2 * hh + h2;
                                const int o = 4 * jj + 2 * h2;
                                const float2 s2 = __fmul2_rn(make_float2(fr[h], fr[h]), sc[jj]);
                                acc[h * (COLS / 8) + jq * 4 + jj] = __ffma2_rn(make_float2(__uint_as_float(cur[o]), __uint_as_float(cur[o + 1])),
                                                                               s2, acc[h * (COLS / 8) + jq * 4 + jj]);
                            }
                        }
                        if (pp + 1 < NP) tmem_ld_wait(nxt);
                    }
                } else {
                    // 32x32b loads: one row and COLS columns per thread, LPW loads per wait
                    #pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        uint32_t r[LPW][32];
                        #pragma unroll
                        for (int h = 0; h < LPW; ++h) tmem_ld_32x32b_x32(tb + (g * LPW + h) * 32, r[h]);
                        #pragma unroll
                        for (int h = 0; h < LPW; ++h) tmem_ld_wait(r[h]);
                        if (g == NG - 1) {
                            // the whole partial is in registers: hand the buffer back to the leader
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive_cluster(tempty0 + 8 * ts);
                        }
                        #pragma unroll
                        for (int h = 0; h < LPW; ++h) {
                            const int c0 = (g * LPW + h) * 32;   // first of these 32 columns
                            #pragma unroll
                            for (int j = 0; j < 32; j += 2)
                                acc[(c0 + j) / 2] = __ffma2_rn(make_float2(__uint_as_float(r[h][j]), __uint_as_float(r[h][j + 1])),
                                                               f2, acc[(c0 + j) / 2]);
                        }
                    }
                }
                if (g_last) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sempty_bar[ss]));
                    if (S::SG > 1) ++g_done;
                }
            }
            if (!ok) break;

            // ---- the warp's 32 rows x COLS columns go out as 32 x 32 BF16 boxes, staged in
            // the warp's own 2 KB buffers in turn (64-byte swizzle: the 16-byte chunk c of row
            // r sits at chunk c ^ ((r >> 1) & 3)) and written by TMA, which clips rows and
            // columns outside C.  One bulk group per box: before a buffer is refilled, the
            // store that last read it has finished reading.
            const int y0 = t.mp * 256 + (int)rank * 128 + quad * 32;
            #pragma unroll
            for (int b = 0; b < COLS / 32; ++b, ++box_it) {
                const uint32_t buf = smem_u32(stage_c + (ew * NBX + (int)(box_it % NBX)) * 2048);
                if (lane == 0) bulk_wait_read<NBX - 1>();
                __syncwarp();
                if constexpr (B_MODE == SCALE_ROW) {
                    // rows g + 8h, columns 8j + 2tq + {0,1}: one BF16 pair per (row, chunk)
                    const int g8 = lane >> 2, tq = lane & 3;
                    #pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int rl = g8 + 8 * h;
                        #pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float2 v = acc[h * (COLS / 8) + b * 4 + c];
                            st_shared_b32(buf + rl * 64 + ((c ^ ((rl >> 1) & 3)) << 4) + 4 * tq, pack_bf16x2(v.x, v.y));
                        }
                    }
                } else {
                    #pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int cc = b * 32 + c * 8;    // first of these 8 columns
                        uint4 v;
                        v.x = pack_bf16x2(acc[cc / 2 + 0].x, acc[cc / 2 + 0].y);
                        v.y = pack_bf16x2(acc[cc / 2 + 1].x, acc[cc / 2 + 1].y);
                        v.z = pack_bf16x2(acc[cc / 2 + 2].x, acc[cc / 2 + 2].y);
                        v.w = pack_bf16x2(acc[cc / 2 + 3].x, acc[cc / 2 + 3].y);
                        st_shared_v4(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4), v);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int x = t.nt * kPairN + col_base + b * 32;
                    if (y0 < p.R1 && x < p.R2) tma_store_2d(&tmC, buf, x, y0);
                    bulk_commit();
                }
            }
        }
        if (lane == 0) bulk_wait_all();   // tile stores complete before exit
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();   // the pair's MMAs and remote arrivals are done in both CTAs
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int B_MODE, int EPI, int STAGES, int PN>
cudaError_t launch_pair_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                          const CUtensorMap& tsb, const CUtensorMap& tc, const GemmParams& p, int clusters,
                          cudaStream_t st) {
    auto kern = k_gemm_pair<B_MODE, EPI, STAGES, PN>;
    constexpr size_t smem = PairSmem<B_MODE, EPI, STAGES, PN>::BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<2 * clusters, pair_threads(EPI), smem, st>>>(ta, tb, tsa, tsb, tc, p);
    return cudaGetLastError();
}

}  // namespace

// Launch contract (checked by the caller): A's tensor map has 128 x 128-byte boxes, B's
// pn/2 x 128-byte boxes; tsa is A's row-scale map with boxes of 128 x min(4 or 1,
// K-blocks); tsb B's scale map as for the one-SM kernel with a tile width of pn; tc the
// BF16 output map (32 x 32 boxes).  p.m_tiles counts 128-row tiles, p.n_tiles pn-column
// tiles.  pn is 128 or 256.
cudaError_t launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                             const CUtensorMap& tsb, const CUtensorMap& tc, const GemmParams& p, int b_mode,
                             int epi_warps, int pn, int clusters, cudaStream_t st) {
    if (pn == 256) {
        if (b_mode == SCALE_ROW) {
            if (epi_warps == 8) return launch_pair_t<SCALE_ROW, 8, 5, 256>(ta, tb, tsa, tsb, tc, p, clusters, st);
            return launch_pair_t<SCALE_ROW, 16, 5, 256>(ta, tb, tsa, tsb, tc, p, clusters, st);
        }
        if (epi_warps == 16) return launch_pair_t<SCALE_BLOCK, 16, 5, 256>(ta, tb, tsa, tsb, tc, p, clusters, st);
        return launch_pair_t<SCALE_BLOCK, 8, 5, 256>(ta, tb, tsa, tsb, tc, p, clusters, st);
    }
    if (b_mode == SCALE_ROW) {
        if (epi_warps == 8) return launch_pair_t<SCALE_ROW, 8, 7, 128>(ta, tb, tsa, tsb, tc, p, clusters, st);
        return launch_pair_t<SCALE_ROW, 16, 7, 128>(ta, tb, tsa, tsb, tc, p, clusters, st);
    }
    if (epi_warps == 16) return launch_pair_t<SCALE_BLOCK, 16, 7, 128>(ta, tb, tsa, tsb, tc, p, clusters, st);
    return launch_pair_t<SCALE_BLOCK, 8, 7, 128>(ta, tb, tsa, tsb, tc, p, clusters, st);
}

// Reads and clears this translation unit's device status word (the pair kernel's bounded
// waits record their timeouts in it).  The caller has synchronized the stream.
fp8rl_status read_and_clear_pair_status() {
    unsigned int v = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return FP8RL_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) return FP8RL_ERR_CUDA;
    return static_cast<fp8rl_status>(v);
}

}  // namespace fp8rl
