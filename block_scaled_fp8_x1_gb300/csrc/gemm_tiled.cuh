// gemm_tiled.cuh -- the one-SM block-scaled FP8 GEMM kernel (tcgen05 + TMEM + TMA), shared
// by the plain form (gemm.cu) and the form whose CTA pairs share B tiles (gemm_mc.cu).
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
// Structure (one CTA of 384 threads per SM, persistent over work items):
//   warp 0      copies (lane 0): TMA loads of the 128x128 A tile and the BNx128 B tile of
//               each K-block into a STAGES-deep shared-memory ring (128-byte swizzle); when
//               B has one scale per row (WGrad), also that K-block's BN scales of B into an
//               8-slot scale ring that the epilogue releases.
//   warp 1      allocates all 512 TMEM columns and issues, per K-block, four tcgen05.mma
//               (K = 32 each) into one of 512/BN partial-sum buffers (fresh accumulate per
//               block), so the tensor pipe runs up to 512/BN - 1 blocks ahead of the
//               epilogue.
//   warps 2-3   idle (they complete warpgroup 0, whose registers go to the epilogue).
//   warps 4-11  epilogue, two warps per TMEM lane quadrant, each owning 32 rows x BN/2
//               columns: per K-block, load the FP32 partial from TMEM, release the buffer,
//               and promote it into FP32 registers with the block's scales ("per-block
//               scale promotion"); the scales arrive in the scale ring (or, when they
//               cannot travel by TMA, each thread copies its own a few K-blocks ahead).
//               Finally round to BF16 and store,
//               or, in the split-K form, store FP32 partials and let the last CTA of a tile
//               sum them in split order (deterministic, no spin-wait).
// Every mbarrier wait is bounded; on timeout the CTA records FP8RL_ERR_DEVICE_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and returns.
#pragma once

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

// Items are (output tile, reduction slice) pairs; slices of one tile are adjacent items.
// Tiles follow the grouped order of raster_tile (p.group, p.raster_n), so the CTAs running
// at the same time reuse the same A rows and B columns through L2.
// With clusters of CM CTAs along M (CM = 2: the multicast form), an item is a group of CM
// vertically adjacent tiles, and CTA `rank` of the cluster takes m-tile CM * group + rank
// (past the last m-tile its rows are TMA zero fill and its stores are clipped).
template <int CM>
__device__ __forceinline__ int cta_rank() { return CM > 1 ? (int)cluster_ctarank() : 0; }

template <int CM = 1>
__device__ __forceinline__ WorkItem work_item(const GemmParams& p, int item, int rank = 0) {
    WorkItem w;
    const int splits = p.splits > 1 ? p.splits : 1;
    w.tile = item / splits;
    w.split = item - w.tile * splits;
    int mu, nt;
    raster_tile(w.tile, (p.m_tiles + CM - 1) / CM, p.n_tiles, p.group, p.raster_n, &mu, &nt);
    w.mt = mu * CM + rank;
    w.nt = nt;
    w.kb_begin = (int)(((int64_t)w.split * p.nkb) / splits);
    w.kb_end = (int)(((int64_t)(w.split + 1) * p.nkb) / splits);
    return w;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 4 warps (copies, MMA, two idle) + epi_warps() epilogue warps, a quarter of them per SM
// sub-partition.  With 8 the epilogue threads get 224 registers: room for a 128-column
// accumulator and a partial in flight.  (16 warps of 112 registers measured no faster for
// the row-scaled form and 25% more instructions.)  Register split: warpgroup 0 drops to
// reg_lo(), the epilogue rises to reg_hi(), within the launch_regs() per thread the CTA is
// launched with.
__host__ __device__ constexpr int epi_warps(int) { return 8; }
__host__ __device__ constexpr int gemm_threads(int b_mode) { return 128 + 32 * epi_warps(b_mode); }
__host__ __device__ constexpr int launch_regs(int) { return 168; }
__host__ __device__ constexpr uint32_t reg_lo(int) { return 56; }
__host__ __device__ constexpr uint32_t reg_hi(int) { return 224; }
static_assert(128 * reg_lo(0) + 32 * epi_warps(0) * reg_hi(0) <= gemm_threads(0) * launch_regs(0), "register split");
constexpr int kScalePD = 4;   // K-blocks of scale prefetch per epilogue thread

// How the epilogue gets the per-K-block scales of A's rows and of B's column blocks.
enum ScaleDelivery {
    SD_TMA = 0,     // the copy warp's TMA puts each K-block's scales in the scale ring
    SD_THREAD = 1   // each epilogue thread copies its own (any M; B rows still by TMA)
};

// Shared-memory plan of one CTA.  Scale-ring slot (SD_TMA), one per group of SG K-blocks:
// A's row scales [K-block of the group][128], then B's scales: [K-block][BN] row scales
// for SCALE_ROW, or a box of at most 16 block scales for SCALE_BLOCK.
template <int BN, int STAGES, int B_MODE, int SD, bool SPLITK>
struct GemmSmem {
    static constexpr int A_BYTES = 128 * 128;                 // one 128x128 E4M3 tile of A
    static constexpr int B_BYTES = BN * 128;                  // one BNx128 E4M3 tile of B
    static constexpr int SG = scale_group(B_MODE, SPLITK);    // K-blocks per scale group
    static constexpr int NS = (B_MODE == SCALE_ROW) ? 8 : 4;   // scale-ring slots (groups)
    static constexpr int SLOT_A = (SD == SD_TMA) ? 128 * SG : 0;   // floats
    // (a box of block scales takes at most 16 floats; padded so that every TMA destination
    // in the ring starts on a 128-byte boundary, as tensor copies require)
    static constexpr int SLOT_B = (B_MODE == SCALE_ROW) ? BN * SG : ((SD == SD_TMA) ? 32 : 0);
    static constexpr int SLOT = SLOT_A + SLOT_B;
    static_assert((SLOT_A * 4) % 128 == 0 && (SLOT * 4) % 128 == 0, "TMA destinations 128-byte aligned");
    static constexpr bool RING = SLOT > 0;
    static constexpr int RING_BYTES = NS * SLOT * 4;
    static constexpr int NTB = 512 / BN;                      // TMEM partial-sum buffers
    // SD_THREAD: per epilogue thread, kScalePD slots of its scale words: A row (+ B block)
    static constexpr int SC_WORDS = (B_MODE == SCALE_BLOCK) ? 2 : 1;
    static constexpr int SC_BYTES = (SD == SD_THREAD) ? kScalePD * SC_WORDS * 32 * epi_warps(B_MODE) * 4 : 0;
    static constexpr int NBARS = 2 * STAGES + 2 * NTB + 2 * NS + 1;
    // BF16 output staging for the TMA store: one 32 x 32 box per epilogue warp (the split-K
    // form writes FP32 partials straight to global memory instead)
    static constexpr int STAGE_C_BYTES = SPLITK ? 0 : epi_warps(B_MODE) * 2048;
    static constexpr size_t BYTES = 1024 /* alignment slack */ + (size_t)STAGES * (A_BYTES + B_BYTES) +
                                    STAGE_C_BYTES + RING_BYTES + SC_BYTES + NBARS * 8 + 16;
};

// The scales one epilogue thread applies per K-block: the scale of its row of A and, when
// B has one scale per 128-row block, the scale of the block its columns fall in.  The
// cursor walks the (work item, K-block) sequence of the CTA in processing order; each
// thread copies its own scale words (cp.async, one commit group per K-block) kScalePD
// K-blocks ahead into private shared-memory slots, so no register ever waits on a load.
template <int BN, int B_MODE>
struct ScaleCursor {
    int item, kb, kb_end;
    int r1;      // row of A this thread scales
    int col;     // first column of C this thread owns

    __device__ __forceinline__ void enter(const GemmParams& p, int row_local, int col_base) {
        if (item < p.num_items) {
            const WorkItem w = work_item(p, item);
            kb = w.kb_begin;
            kb_end = w.kb_end;
            r1 = w.mt * 128 + row_local;
            col = w.nt * BN + col_base;
        }
    }
    // Copy the scales of the current position into slot words `dst_a` (and `dst_b`); zero
    // past the end of the sequence or outside A/C.  Then advance and close the group.
    __device__ __forceinline__ void issue(const GemmParams& p, uint32_t dst_a, uint32_t dst_b,
                                          int row_local, int col_base) {
        const bool live = item < p.num_items;
        const bool va = live && r1 < p.R1;
        cp_async_4(dst_a, p.sa + (va ? (int64_t)kb * p.sa_kb + r1 : 0), va ? 4u : 0u);
        if (B_MODE == SCALE_BLOCK) {
            const bool vb = live && col < p.R2;
            cp_async_4(dst_b, p.sb + (vb ? (int64_t)(col >> 7) * p.sb_r + (int64_t)kb * p.sb_kb : 0),
                       vb ? 4u : 0u);
        }
        cp_async_commit();
        if (live && ++kb >= kb_end) {
            item += gridDim.x;
            enter(p, row_local, col_base);
        }
    }
};

// CM: CTAs per cluster along M (1, or 2 for the multicast form, whose two CTAs share
// every B tile).  Ops supplies the B-tile copy and the commit that frees a stage:
//   Ops::load_b<BN>(dst, map, bar, x, y, policy, rank)  -- B rows [y, y + BN) into dst
//   Ops::commit_stage(bar)                               -- arrives when the MMAs complete
template <int BN, int SD, int B_MODE, int STAGES, bool SPLITK, int CM, class Ops>
__global__ void __launch_bounds__(gemm_threads(B_MODE), 1)
    k_gemm_bs(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
              const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    using S = GemmSmem<BN, STAGES, B_MODE, SD, SPLITK>;
    constexpr int kEpiWarps = epi_warps(B_MODE);
    constexpr int COLS = BN / (kEpiWarps / 4);   // columns per epilogue thread
    constexpr int LW = kEpiWarps == 16 ? 16 : 32; // columns per TMEM load
    constexpr int LPW = 1;                        // loads per wait
    constexpr int NG = COLS / (LW * LPW);         // waits per K-block
    constexpr int NS = S::NS;
    constexpr int NTB = S::NTB;
    constexpr int PD = kScalePD;
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t IDESC = idesc_e4m3_f32(128, BN);
    static_assert(COLS % (LW * LPW) == 0, "BN must be 128 or 256");
    static_assert(B_MODE == SCALE_ROW || BN >= 128, "block scales of B need whole 128-column blocks");
    static_assert(CM == 1 || (SD == SD_TMA && !SPLITK), "the multicast form copies its scales by TMA, unsplit");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * S::A_BYTES;
    uint8_t* stage_c = sB + STAGES * S::B_BYTES;                     // [epilogue warp][2048]
    float* ring = reinterpret_cast<float*>(stage_c + S::STAGE_C_BYTES);   // [NS][SLOT]
    float* sc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ring) + S::RING_BYTES);  // [PD][W][thr]
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sc) + S::SC_BYTES);
    uint64_t* full_bar = bars;                 // [STAGES] TMA -> MMA
    uint64_t* empty_bar = bars + STAGES;       // [STAGES] MMA -> TMA
    uint64_t* tfull_bar = bars + 2 * STAGES;   // [NTB] MMA -> epilogue
    uint64_t* tempty_bar = tfull_bar + NTB;    // [NTB] epilogue -> MMA
    uint64_t* sfull_bar = tempty_bar + NTB;    // [NS] scale copies -> epilogue
    uint64_t* sempty_bar = sfull_bar + NS;     // [NS] epilogue -> scale copies
    uint64_t* drain_bar = sempty_bar + NS;     // [1] MMA completion at exit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // this cluster's items: blockIdx.x / CM, stepping by gridDim.x / CM (read where used)

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), CM);   // every CTA whose copies fill the stage
        }
        for (int t = 0; t < NTB; ++t) {
            mbar_init(smem_u32(&tfull_bar[t]), 1);
            mbar_init(smem_u32(&tempty_bar[t]), kEpiWarps);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&sfull_bar[s]), 1);
            mbar_init(smem_u32(&sempty_bar[s]), kEpiWarps);
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (SD == SD_TMA) tma_prefetch_desc(&tmSA);
        if (S::SLOT_B > 0) tma_prefetch_desc(&tmSB);
        if (!SPLITK) tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    if (CM > 1)
        cluster_sync_all();   // the peer's barriers are initialised before any copy reaches them
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    constexpr uint32_t REG_LO = reg_lo(B_MODE), REG_HI = reg_hi(B_MODE);
    if (warp < 4) {
      warpgroup_reg_dealloc<REG_LO>();
      if (warp == 0) {
        // ------------------------------------------------------------ copies (lane 0)
        // TMA tiles of A and B per K-block, and that K-block's scales into the scale ring:
        // the 128 row scales of A (SD_TMA) and B's scales (its BN row scales, or a box of
        // block scales that holds the tile's column blocks).
        if (lane == 0) {
            // split-K (decode) streams the weights (B) once: let them leave L2 first
            const uint64_t pol_a = l2_policy_evict_last();
            const uint64_t pol_b = SPLITK ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_s = pol_a;   // scales
            // K-blocks per scale box: the group size, or all of them when K is shorter
            const int sgrp = p.nkb < S::SG ? p.nkb : S::SG;
            uint32_t it = 0, s_issued = 0;
            bool ok = true;
            for (int item = (int)blockIdx.x / CM; ok && item < p.num_items; item += (int)gridDim.x / CM) {
                const WorkItem w = work_item<CM>(p, item, cta_rank<CM>());
                const int m0 = w.mt * 128;
                const int n0 = w.nt * BN;
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    if (!mbar_wait(smem_u32(&empty_bar[s]), ((it / STAGES) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[s]);
                    mbar_arrive_expect_tx(fb, S::A_BYTES + S::B_BYTES);
                    tma_load_2d(smem_u32(sA + s * S::A_BYTES), &tmA, fb, kb * 128, m0, pol_a);
                    Ops::template load_b<BN>(smem_u32(sB + s * S::B_BYTES), &tmB, fb, kb * 128, n0, pol_b, cta_rank<CM>());
                    if (S::RING && (kb == w.kb_begin || kb % S::SG == 0)) {
                        // first K-block of a scale group: the scales of the whole group
                        const uint32_t ss = s_issued % NS;
                        if (!mbar_wait(smem_u32(&sempty_bar[ss]), ((s_issued / NS) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                            ok = false;
                            ++it;   // this K-block's tiles are in flight: drain them below
                            break;
                        }
                        const uint32_t sb = smem_u32(&sfull_bar[ss]);
                        float* slot = ring + ss * S::SLOT;
                        const int kb0 = kb - kb % S::SG;
                        const uint32_t a_bytes = (SD == SD_TMA) ? 128u * 4u * (uint32_t)sgrp : 0u;
                        if (B_MODE == SCALE_ROW) {
                            mbar_arrive_expect_tx(sb, a_bytes + (uint32_t)BN * 4u * (uint32_t)sgrp);
                            tma_load_2d(smem_u32(slot + S::SLOT_A), &tmSB, sb, n0, kb0, pol_s);
                        } else if (p.sb_kb == 1) {
                            // block scales stored [column block][K-block]: 4 K-blocks from a
                            // 4-aligned one (the box's x is a K-block index: x * 4 bytes must
                            // be a multiple of 16 whatever the group size) x the tile's
                            // BN/128 column blocks
                            mbar_arrive_expect_tx(sb, a_bytes + 16u * (BN / 128));
                            tma_load_2d(smem_u32(slot + S::SLOT_A), &tmSB, sb, kb & ~3, n0 >> 7, pol_s);
                        } else {
                            // block scales stored [K-block][column block]: 4 column blocks
                            // from a 4-aligned one, for each K-block of the group
                            mbar_arrive_expect_tx(sb, a_bytes + 16u * (uint32_t)sgrp);
                            tma_load_2d(smem_u32(slot + S::SLOT_A), &tmSB, sb, (n0 >> 7) & ~3, kb0, pol_s);
                        }
                        if (SD == SD_TMA) tma_load_2d(smem_u32(slot), &tmSA, sb, m0, kb0, pol_s);
                        ++s_issued;
                    }
                }
            }
            // Drain: every issued copy lands before the CTA can exit.
            volatile int no_abort = 0;
            const uint32_t n_out = it < STAGES ? it : STAGES;
            for (uint32_t j = it - n_out; j < it; ++j)
                mbar_wait(smem_u32(&full_bar[j % STAGES]), (j / STAGES) & 1, p.timeout_ns, &no_abort);
            if (S::RING) {
                const uint32_t s_out = s_issued < NS ? s_issued : NS;
                for (uint32_t j = s_issued - s_out; j < s_issued; ++j)
                    mbar_wait(smem_u32(&sfull_bar[j % NS]), (j / NS) & 1, p.timeout_ns, &no_abort);
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
            for (int item = (int)blockIdx.x / CM; ok && item < p.num_items; item += (int)gridDim.x / CM) {
                const WorkItem w = work_item<CM>(p, item, cta_rank<CM>());
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++it) {
                    const uint32_t ts = it % NTB;
                    if (!mbar_wait(smem_u32(&tempty_bar[ts]), ((it / NTB) & 1) ^ 1, p.timeout_ns, abort_flag)) {
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
                    const uint64_t da = sdesc_kmajor_sw128(a_base + s * S::A_BYTES);
                    const uint64_t db = sdesc_kmajor_sw128(b_base + s * S::B_BYTES);
                    #pragma unroll
                    for (int k = 0; k < 4; ++k)  // 32-byte steps inside the 128-byte row
                        mma_f8(d, da + 2 * k, db + 2 * k, IDESC, k > 0 ? 1u : 0u);
                    Ops::commit_stage(smem_u32(&empty_bar[s]));
                    mma_commit(smem_u32(&tfull_bar[ts]));
                }
            }
            // All MMAs issued by this thread complete before TMEM is freed.
            mma_commit(smem_u32(drain_bar));
            volatile int no_abort = 0;
            mbar_wait(smem_u32(drain_bar), 0, p.timeout_ns, &no_abort);
        }
      }
    } else {
        warpgroup_reg_alloc<REG_HI>();
        // ------------------------------------------------------------ epilogue warps
        // After an abort every warp keeps walking the same items and blocks (no waits, no
        // TMEM loads) so that all of them reach the same named barriers.
        const int ew = warp - 4;            // 0 .. kEpiWarps-1
        const int quad = warp & 3;          // TMEM lane quadrant this warp may access
        const int col_base = (ew >> 2) * COLS;
        const int row_local = quad * 32 + lane;
        const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
        // SD_THREAD: scale slots of this thread, word (slot, w) at sc[(slot * SC_WORDS + w) * ET + et]
        const int et = threadIdx.x - 128;
        constexpr int ET = 32 * kEpiWarps;
        const uint32_t sc_base = smem_u32(sc) + 4u * (uint32_t)et;
        ScaleCursor<BN, B_MODE> cur;
        if (SD == SD_THREAD) {
            cur.item = blockIdx.x;
            cur.enter(p, row_local, col_base);
            #pragma unroll
            for (int i = 0; i < PD; ++i)
                cur.issue(p, sc_base + 4u * ET * (i * S::SC_WORDS), sc_base + 4u * ET * (i * S::SC_WORDS + 1),
                          row_local, col_base);
        }
        uint32_t acc_it = 0;
        uint32_t g_done = 0;   // scale groups consumed
        bool ok = true;
        for (int item = (int)blockIdx.x / CM; item < p.num_items; item += (int)gridDim.x / CM) {
            const WorkItem w = work_item<CM>(p, item, cta_rank<CM>());
            const int64_t r1 = (int64_t)w.mt * 128 + row_local;
            const int64_t n0 = (int64_t)w.nt * BN + col_base;  // first column of this thread
            float2 acc[COLS / 2];
            #pragma unroll
            for (int c = 0; c < COLS / 2; ++c) acc[c] = make_float2(0.0f, 0.0f);

            for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++acc_it) {
                float f = 0.0f;
                if (SD == SD_THREAD) {
                    // this K-block's scales: its copy group is the oldest of the PD in flight
                    const uint32_t slot = acc_it % PD;
                    cp_async_wait_group<PD - 1>();
                    const float* scw = sc + slot * S::SC_WORDS * ET + et;
                    f = (B_MODE == SCALE_BLOCK) ? scw[0] * scw[ET] : scw[0];
                    cur.issue(p, sc_base + 4u * ET * (slot * S::SC_WORDS), sc_base + 4u * ET * (slot * S::SC_WORDS + 1),
                              row_local, col_base);
                }
                if (!ok) continue;
                const uint32_t gi = S::SG == 1 ? acc_it : g_done;   // scale group index
                const uint32_t ss = gi % NS;
                const uint32_t ts = acc_it % NTB;
                const int q = kb % S::SG;   // this K-block's place in its scale group
                const bool g_first = kb == w.kb_begin || q == 0;
                const bool g_last = kb + 1 == w.kb_end || q == S::SG - 1;
                bool got = true;
                if (S::RING && g_first)
                    got = mbar_wait(smem_u32(&sfull_bar[ss]), (gi / NS) & 1, p.timeout_ns, abort_flag);
                got = got && mbar_wait(smem_u32(&tfull_bar[ts]), (acc_it / NTB) & 1, p.timeout_ns, abort_flag);
                ok = __all_sync(0xffffffffu, got);
                if (!ok) continue;
                tc_fence_after();
                const float* slot = ring + ss * S::SLOT;
                if constexpr (B_MODE == SCALE_ROW) {
                    // 16x256b fragments: this thread holds rows g + 8h (h = 0..3) of the warp's
                    // 32 and columns 8j + 2tq + {0,1}, so it needs 4 row and 32 column scales
                    // per K-block instead of 1 and 128 (read with shared-space loads).
                    const int g = lane >> 2, tq = lane & 3;
                    float fr[4];
                    const uint32_t fra = smem_u32(slot) + 4u * (uint32_t)(q * 128 + quad * 32 + g);
                    #pragma unroll
                    for (int h = 0; h < 4; ++h)
                        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(fr[h]) : "r"(fra + 32u * h));
                    const uint32_t sba = smem_u32(slot) + 4u * (uint32_t)(S::SLOT_A + q * BN + col_base + 2 * tq);
                    const uint32_t tb0 = tmem_base + ((uint32_t)(quad * 32) << 16) + ts * BN + col_base;
                    const uint32_t tb1 = tb0 + (16u << 16);
                    // parts of 16 rows x 32 columns, the next part's TMEM load in flight
                    // while this one is promoted
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
                            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[ts]));
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
                    if (SD == SD_TMA) {
                        f = slot[q * 128 + row_local];
                        if (B_MODE == SCALE_BLOCK) {
                            const int cb = (int)(n0 >> 7);   // column block of this thread
                            f *= slot[S::SLOT_A + (p.sb_kb == 1 ? ((cb - ((w.nt * BN) >> 7)) * 4 + (kb & 3)) : (q * 4 + (cb & 3)))];
                        }
                    }
                    const float2 f2 = make_float2(f, f);
                    const uint32_t tbase = tmem_base + t_lane + ts * BN + col_base;
                    // LPW loads of LW columns per wait
                    #pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        uint32_t r[LPW][LW];
                        #pragma unroll
                        for (int h = 0; h < LPW; ++h) tmem_ld_cols(tbase + (g * LPW + h) * LW, r[h]);
                        #pragma unroll
                        for (int h = 0; h < LPW; ++h) tmem_ld_wait(r[h]);
                        if (g == NG - 1) {
                            // the whole partial is in registers: hand the TMEM buffer back
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[ts]));
                        }
                        #pragma unroll
                        for (int h = 0; h < LPW; ++h) {
                            const int c0 = (g * LPW + h) * LW;   // first column of these LW
                            #pragma unroll
                            for (int j = 0; j < LW; j += 2)
                                acc[(c0 + j) / 2] = __ffma2_rn(make_float2(__uint_as_float(r[h][j]), __uint_as_float(r[h][j + 1])),
                                                               f2, acc[(c0 + j) / 2]);
                        }
                    }
                }
                if (S::RING && g_last) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sempty_bar[ss]));
                    if (S::SG > 1) ++g_done;
                }
            }

            if (!SPLITK) {
                // ---- whole reduction in this CTA: the warp's 32 rows x COLS columns go out
                // as 32 x 32 BF16 boxes staged in its own 2 KB buffer (64-byte swizzle: the
                // 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3)) and written by
                // TMA, which clips rows and columns outside C.
                const uint32_t buf = smem_u32(stage_c + ew * 2048);
                const int y0 = w.mt * 128 + quad * 32;
                #pragma unroll
                for (int q = 0; q < COLS / 32; ++q) {
                    if (lane == 0) bulk_wait_read<0>();   // the previous box has left the buffer
                    __syncwarp();
                    if constexpr (B_MODE == SCALE_ROW) {
                        // rows g + 8h, columns 8j + 2tq + {0,1}: one BF16 pair per (row, chunk)
                        const int g = lane >> 2, tq = lane & 3;
                        #pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const int rl = g + 8 * h;
                            #pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const float2 v = acc[h * (COLS / 8) + q * 4 + c];
                                st_shared_b32(buf + rl * 64 + ((c ^ ((rl >> 1) & 3)) << 4) + 4 * tq,
                                              pack_bf16x2(v.x, v.y));
                            }
                        }
                    } else {
                        #pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int cc = q * 32 + c * 8;    // first of these 8 columns
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
                    const int x = w.nt * BN + col_base + q * 32;
                    if (ok && lane == 0 && x < p.R2 && y0 < p.R1) {
                        tma_store_2d(&tmC, buf, x, y0);
                        bulk_commit();
                    }
                }
            } else if (p.splits <= 1) {
                // ---- split-K form run unsplit: BF16 row segment of this thread
                if (ok && r1 < p.R1 && n0 < p.R2) {
                    uint16_t* dst = p.c + r1 * p.ldc + n0;
                    #pragma unroll
                    for (int c = 0; c < COLS; c += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(acc[c / 2 + 0].x, acc[c / 2 + 0].y);
                        v.y = pack_bf16x2(acc[c / 2 + 1].x, acc[c / 2 + 1].y);
                        v.z = pack_bf16x2(acc[c / 2 + 2].x, acc[c / 2 + 2].y);
                        v.w = pack_bf16x2(acc[c / 2 + 3].x, acc[c / 2 + 3].y);
                        *reinterpret_cast<uint4*>(dst + c) = v;
                    }
                }
            } else {
                // ---- split-K: this slice's FP32 partial sums; k_splitk_reduce adds the slices
                // in slice order.  Partials are laid out [tile][slice][BN/4][128 rows][4] so
                // that a warp's float4 accesses cover 32 consecutive rows: fully coalesced
                // 512-byte transactions.  Rows past R1 are not needed.
                if (ok && r1 < p.R1) {
                    float4* part = reinterpret_cast<float4*>(p.ws) +
                                   ((int64_t)w.tile * p.splits + w.split) * (int64_t)(BN * 32) +
                                   (int64_t)(col_base / 4) * 128 + row_local;
                    #pragma unroll
                    for (int c = 0; c < COLS; c += 4)
                        __stcg(part + (c / 4) * 128, make_float4(acc[c / 2].x, acc[c / 2].y, acc[c / 2 + 1].x, acc[c / 2 + 1].y));
                }
            }
        }
        if (SD == SD_THREAD) cp_async_wait_all();   // own scale copies land before exit
        if (!SPLITK && lane == 0) bulk_wait_all();   // tile stores complete before exit
    }

    tc_fence_before();
    if (CM > 1)
        cluster_sync_all();   // no copy or commit of the peer is still headed for this CTA
    else
        __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// The one-SM form's copy and commit: the whole B tile into this CTA's stage.
struct PlainOps {
    template <int BN>
    static __device__ __forceinline__ void load_b(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y,
                                                  uint64_t pol, int) {
        tma_load_2d(dst, m, bar, x, y, pol);
    }
    static __device__ __forceinline__ void commit_stage(uint32_t bar) { mma_commit(bar); }
};

}  // namespace fp8rl
