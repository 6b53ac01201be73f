// rollout.h -- launchers of the NVFP4 rollout path (internal): the NVFP4 quantizer and the
// FP4 decode GEMM.
#pragma once

#include "gemm.h"

namespace fp8rl {

// nvfp4.cu: NVFP4 row quantizer and the decode-shaped FP4 GEMM (weights on the MMA's M
// side, split-K inside a cluster of `splits` CTAs as for launch_decode).  tw: weight codes
// [N][K/2] bytes with 128 x 128-byte boxes; tx: activation codes [M][K/2] with boxes of
// nvf4_token_tile(M) rows x 128 bytes.  Scale factors in the tensor core's atom layout.
struct Nvf4Params {
    int M;                   // tokens, 1..256
    int nkb;                 // K / 256
    int tiles;               // N / 128
    const uint8_t* sfw;      // weight block scales, 2 KB per (tile, K-block)
    const uint8_t* sfx;      // activation block scales, 2 KB per (128-token group, K-block)
    const float* gw;         // per-row scales of W [N] and X [M]
    const float* gx;
    uint16_t* y;             // y[m * ldy + n]
    int64_t ldy;
    uint64_t timeout_ns;
};
int nvf4_token_tile(int M);
int nvf4_max_clusters(int M, int splits);
cudaError_t launch_gemm_nvf4(const CUtensorMap& tw, const CUtensorMap& tx, const Nvf4Params& p, int grid_clusters,
                             int splits, bool pdl, cudaStream_t st);
cudaError_t launch_quant_nvfp4(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q, uint8_t* sf,
                               float* g, cudaStream_t st);
cudaError_t launch_debug_e2m1(const float* in, uint8_t* out, int64_t n, cudaStream_t st);
fp8rl_status read_and_clear_nvf4_status();

}  // namespace fp8rl
