// gemm.h -- parameters and launchers of the block-scaled GEMM kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8rl.h"

namespace fp8rl {

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry point.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// How an operand's per-K-block scale is indexed.
enum ScaleMode : int {
    SCALE_ROW = 0,    // one scale per row of the operand: s[kb*s_kb + row]
    SCALE_BLOCK = 1   // one scale per 128-row block:      s[(row/128)*s_r + kb*s_kb]
};

// K-blocks whose scales the GEMM's copy warp fetches with one TMA copy per operand (one
// scale-ring slot and one barrier round trip per group): 4 for the tiled block-scaled
// form; 1 for row-scaled B (WGrad, whose per-K-block slots measured faster) and for the
// split-K form (short K slices).  Groups start at K-block multiples of the group size, so
// a box of block scales stored [column block][K-block] lines up with them; a work item's
// first and last groups may be partial.  Scale tensor maps use boxes of
// min(group, K-blocks) K-blocks.
__host__ __device__ constexpr int scale_group(int b_mode, bool splitk) {
    return (b_mode == SCALE_ROW || splitk) ? 1 : 4;
}

struct GemmParams {
    int64_t R1, R2, Kr;      // C is R1 x R2; reduction length Kr (multiple of 128)
    const float* sa;         // scales of A, one per row: sa[kb*sa_kb + r1]
    int64_t sa_kb;
    const float* sb;         // scales of B (rows r2)
    int64_t sb_kb, sb_r;
    uint16_t* c;             // c[r1*ldc + r2]
    int64_t ldc;
    float* ws;               // split-K partials [tiles][splits][BN/4][128 rows][4]
    int splits;              // reduction slices per output tile (<= 1: none)
    int m_tiles, n_tiles, nkb;
    int num_items;
    int group;               // tile order (see raster_tile): units per group
    int raster_n;            // 0: groups of row units sweep the column tiles; 1: the converse
    uint64_t timeout_ns;
};

// Tile order of the persistent GEMMs.  Output tiles are numbered in groups: with
// raster_n == 0 a group is `group` consecutive row units (128-row tiles, or pairs of them)
// and its tiles are numbered row unit first, then column tile, so the CTAs running at the
// same time share the group's rows of A from L2 while the column tiles of B stream past;
// raster_n == 1 is the same with the roles of rows and columns exchanged.  The host picks
// the orientation and size that read the operands from HBM the fewest times.
__host__ __device__ inline void raster_tile(int tile, int m_units, int n_units, int group, int raster_n, int* m,
                                            int* n) {
    const int g_units = raster_n ? n_units : m_units;   // the grouped dimension
    const int s_units = raster_n ? m_units : n_units;   // the swept one
    const int per_group = group * s_units;
    const int g = tile / per_group;
    const int first = g * group;
    const int gs = (group < g_units - first) ? group : g_units - first;
    const int r = tile - g * per_group;
    const int a = first + r % gs, b = r / gs;
    *m = raster_n ? b : a;
    *n = raster_n ? a : b;
}

// The tile order of raster_tile for an m_units x n_units grid of tiles whose row unit holds
// a_unit_bytes of A and column tile b_unit_bytes of B (each across the whole reduction),
// with `wave` tiles running at once.
void choose_raster(int64_t m_units, int64_t n_units, int64_t a_unit_bytes, int64_t b_unit_bytes, int wave,
                   int* group, int* raster_n);

// Scale tensor maps (FP32; g = min(scale_group(), K-blocks) K-blocks per box): tsa over A's
// row scales [K-block][R1], box 128 x g; tsb over B's scales, box BN x g for row scales
// [K-block][R2], 4 x BN/128 for block scales stored [column block][K-block] (sb_kb == 1),
// 4 x g for block scales stored [K-block][column block].  With both maps the scales travel by TMA; when
// either is null (strides that are not multiples of 16 bytes) each epilogue thread copies
// its own.  B row scales (WGrad) always need both maps.
// tc: tensor map of C (BF16 [R1][ldc], box 32 x 32, 64-byte swizzle) for the tile stores.
cudaError_t launch_gemm_tiled(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap* tsa,
                              const CUtensorMap* tsb, const CUtensorMap& tc, const GemmParams& p, int b_mode,
                              int bn, int grid, cudaStream_t st);
cudaError_t launch_gemm_splitk(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap* tsa,
                               const CUtensorMap* tsb, const GemmParams& p, int grid, cudaStream_t st);
cudaError_t launch_debug_wait_timeout(uint64_t timeout_ns, cudaStream_t st);

// gemm_pair.cu: the same GEMM on clusters of two CTAs (256 x pn tiles, M = 256 MMAs,
// pn = 128 or 256).  ta: A map with 128 x 128-byte boxes; tb: B map with pn/2 x 128-byte
// boxes; tsa, tsb: the scale maps of scale_maps() for a tile width of pn; tc: the BF16
// output map.  p.m_tiles / p.n_tiles count 128-row / pn-column tiles; `clusters`
// persistent pairs.
cudaError_t launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                             const CUtensorMap& tsb, const CUtensorMap& tc, const GemmParams& p, int b_mode,
                             int epi_warps, int pn, int clusters, cudaStream_t st);
fp8rl_status read_and_clear_pair_status();

// gemm_mc.cu: the one-SM kernel on clusters of two CTAs along M that share each B tile by
// TMA multicast (this GPU's memory only).  As launch_gemm_tiled with BN = 256 and both scale
// maps, except: tb has 128-row boxes (half a tile), p.num_items counts pairs of m-tiles x
// n-tiles, `clusters` persistent pairs.
cudaError_t launch_gemm_mc(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                           const CUtensorMap& tsb, const CUtensorMap& tc, const GemmParams& p, int b_mode,
                           int clusters, cudaStream_t st);
fp8rl_status read_and_clear_mc_status();

// decode.cu: decode-shaped forward GEMM (M <= 256 tokens), weights on the MMA's M side,
// split-K reduced inside a cluster of `splits` CTAs (1..8) through distributed shared
// memory.  tw: weight codes [N][K] with 128 x 128-byte boxes; tx: activation codes [M][K]
// with boxes of decode_mp(M) rows x 128 bytes.  grid_clusters: p.tiles when splits > 1
// (one tile per cluster), any count up to p.tiles when splits == 1 (persistent CTAs).
struct DecodeParams {
    int M;                   // tokens, 1..256
    int nkb;                 // K / 128
    int tiles;               // N / 128
    const float* sx;         // activation scales sx[kb * sx_kb + m]
    int64_t sx_kb;
    const float* sw;         // weight block scales sw[(n / 128) * sw_r + kb]
    int64_t sw_r;
    uint16_t* y;             // y[m * ldy + n]
    int64_t ldy;
    uint64_t timeout_ns;
};
int decode_mp(int M);
int decode_max_clusters(int M, int splits);
// pdl: launch as a programmatic dependent of the stream's previous kernel (the kernel
// requests its first weight tiles, then waits for that kernel before reading the activation).
cudaError_t launch_decode(const CUtensorMap& tw, const CUtensorMap& tx, const DecodeParams& p, int grid_clusters,
                          int splits, bool pdl, cudaStream_t st);
fp8rl_status read_and_clear_decode_status();

// quantize.cu
cudaError_t launch_quant_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                               float* s, int num_sms, cudaStream_t st);
cudaError_t launch_quant_dual(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                              float* s, uint8_t* qT, float* sT, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_silu_mul_quant(const uint16_t* gu, int64_t M, int64_t I, uint8_t* q, float* s,
                                  uint8_t* qT, float* sT, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M,
                                 int64_t K, uint8_t* q, float* s, uint8_t* qT, float* sT,
                                 float* rstd, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_silu_mul_bwd_quant(const uint16_t* gu, const uint16_t* dh, int64_t M, int64_t I, uint8_t* q,
                                      float* s, uint8_t* qT, float* sT, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_rmsnorm_bwd(const uint16_t* x, const uint16_t* gamma, const float* rstd, const uint16_t* dy,
                               int64_t M, int64_t K, uint16_t* dx, float* dgamma, float* ws, int nblocks,
                               cudaStream_t st);
int rmsnorm_bwd_blocks(int64_t M, int num_sms);
cudaError_t launch_requant_128x1(const uint8_t* q, const float* s, int64_t M, int64_t K, uint8_t* qT, float* sT,
                                 uint64_t timeout_ns, cudaStream_t st);
fp8rl_status read_and_clear_quant_status();
cudaError_t launch_quant_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                 float* s, uint8_t* qT, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_debug_e4m3(const float* in, uint8_t* out, int64_t n, cudaStream_t st);
cudaError_t launch_debug_encode_check(uint32_t amax_lo, uint32_t amax_hi,
                                      unsigned long long* mismatches, uint32_t* first_bad,
                                      cudaStream_t st);

}  // namespace fp8rl
