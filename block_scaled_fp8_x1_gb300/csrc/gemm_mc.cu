// gemm_mc.cu -- the one-SM block-scaled FP8 GEMM on clusters of two CTAs that share every
// B tile through TMA multicast.  Single-GPU code: every tensor map here covers this GPU's
// own memory, and the multicast copies go only to the two CTAs of a cluster on this GPU.
//
// "Technical summary: Jet-RL", section "Quantization Scheme": the same forward, DGrad and
// WGrad GEMMs as gemm.cu (1x128 / 128x128 / 128x1 operand quantization, FP32 promotion per
// 128-long reduction block, BF16 out); only the copies of B change.
//
// Two CTAs on vertically adjacent output tiles (m-tiles 2g and 2g + 1, the same n-tile)
// need the same BN x 128 B tile per K-block.  CTA r copies B rows [r*BN/2, (r+1)*BN/2) of
// it with a multicast TMA into the same stage of both CTAs, so each CTA reads half of B
// from L2 and both stages fill completely (each CTA's stage barrier counts the whole
// tile: its own half and the peer's).  A CTA may overwrite a stage only when both CTAs'
// MMAs have finished reading it, so each MMA commit that frees a stage arrives on the
// stage barrier of both CTAs (count 2).  A cluster barrier after the barriers are
// initialised and another before exit keep every copy and commit inside live CTAs.
#include "gemm_tiled.cuh"

namespace fp8rl {

namespace {

struct McOps {
    // This CTA's half of the B tile, multicast to both CTAs of the cluster (mask 0b11):
    // the data and the byte count land at the same shared-memory offsets in each.
    template <int BN>
    static __device__ __forceinline__ void load_b(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y,
                                                  uint64_t pol, int rank) {
        const uint32_t d = dst + (uint32_t)(rank * (BN / 2) * 128);
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
            ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5, %6;" ::"r"(d),
            "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y + rank * (BN / 2)), "h"((uint16_t)0x3),
            "l"(pol)
            : "memory");
    }
    // The stage is free once this CTA's MMAs complete: tell both CTAs' stage barriers.
    static __device__ __forceinline__ void commit_stage(uint32_t bar) {
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                bar),
            "h"((uint16_t)0x3)
            : "memory");
    }
};

template <int BN, int B_MODE, int STAGES>
cudaError_t launch_mc_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa, const CUtensorMap& tsb,
                        const CUtensorMap& tc, const GemmParams& p, int clusters, cudaStream_t st) {
    auto kern = k_gemm_bs<BN, SD_TMA, B_MODE, STAGES, false, 2, McOps>;
    constexpr size_t smem = GemmSmem<BN, STAGES, B_MODE, SD_TMA, false>::BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2u * (unsigned)clusters, 1, 1);
    cfg.blockDim = dim3(gemm_threads(B_MODE), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, tc, p);
}

}  // namespace

// Launch contract (checked by the caller): as launch_gemm_tiled with BN = 256 and both
// scale maps, except that B's tensor map has boxes of 128 rows (half a tile), p.m_tiles
// counts 128-row tiles and p.num_items counts pairs of m-tiles x n-tiles; `clusters`
// persistent pairs of CTAs.
cudaError_t launch_gemm_mc(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                           const CUtensorMap& tsb, const CUtensorMap& tc, const GemmParams& p, int b_mode,
                           int clusters, cudaStream_t st) {
    if (b_mode == SCALE_ROW) return launch_mc_t<256, SCALE_ROW, 3>(ta, tb, tsa, tsb, tc, p, clusters, st);
    return launch_mc_t<256, SCALE_BLOCK, 4>(ta, tb, tsa, tsb, tc, p, clusters, st);
}

// Reads and clears this translation unit's device status word (the bounded waits of the
// multicast form record their timeouts in it).  The caller has synchronized the stream.
fp8rl_status read_and_clear_mc_status() {
    unsigned int v = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return FP8RL_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) return FP8RL_ERR_CUDA;
    return static_cast<fp8rl_status>(v);
}

}  // namespace fp8rl
