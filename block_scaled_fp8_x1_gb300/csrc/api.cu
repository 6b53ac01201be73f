// api.cu -- the extern "C" boundary of libfp8rl (declared in include/fp8rl.h).
//
// Validates arguments on the host (nothing is launched on an error), checks that the
// current device is compute capability 10.3, builds the TMA descriptors of the GEMM
// operands and picks the kernel form.  All compute happens in the CUDA kernels of
// quantize.cu and gemm.cu.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/fp8rl.h"
#include "gemm.h"
#include "rollout.h"

namespace fp8rl {
fp8rl_status read_and_clear_device_status(cudaStream_t st);  // gemm.cu
size_t noalloc_scratch_bytes();                              // gemm_noalloc.cu
cudaError_t noalloc_scratch(void** out);                     // gemm_noalloc.cu
}

using namespace fp8rl;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int state = 0;  // 0 unknown, 1 supported, -1 unsupported
    int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

fp8rl_status current_device(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8RL_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FP8RL_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.state == 0) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8RL_ERR_CUDA;
        d.state = (major == 10 && minor == 3) ? 1 : -1;
        d.num_sms = n;
    }
    if (d.state < 0) return FP8RL_ERR_UNSUPPORTED_DEVICE;
    if (sms) *sms = d.num_sms;
    return FP8RL_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline fp8rl_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA; }

// ---------------------------------------------------------------- TMA descriptors

}  // namespace

EncodeTiledFn fp8rl::encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

namespace {

// Row-major byte matrix [rows][cols] (row stride ld bytes), box of box_rows x 128 bytes,
// 128-byte swizzle (the K-major layout the tcgen05 descriptors expect).
fp8rl_status make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld,
                       int box_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return FP8RL_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8RL_OK : FP8RL_ERR_CUDA;
}

// 2-D tensor map of an FP32 scale array [outer][inner] (inner a multiple of 4, so that the
// row stride is a multiple of 16 bytes), boxes of box_outer x box_inner scales.
fp8rl_status make_tmap_scales(CUtensorMap* m, const float* base, int64_t outer, int64_t inner,
                              int box_inner, int box_outer) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return FP8RL_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 4};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8RL_OK : FP8RL_ERR_CUDA;
}

// ---------------------------------------------------------------- GEMM planning

// The decode form is the tiled kernel (tokens as rows, weights as 256-wide columns) with
// the reduction split into slices so that a handful of output tiles still occupy every SM.
constexpr int kDecodeBN = 256;

int64_t decode_tiles(int64_t M, int64_t N) { return ((M + 127) / 128) * ((N + kDecodeBN - 1) / kDecodeBN); }

// Slices per tile: as many as keep all (tile, slice) items within one wave of CTAs, at
// most 16, and at least two K-blocks per slice.  Problems with a wave of tiles or more are
// not split: writing and re-reading the FP32 partial sums and the last CTA's serial
// reduction cost more than the unbalanced last wave (256 x 28672 x 4096: 62 us with two
// slices, 44 us with one).
int choose_splits(int64_t tiles, int64_t nkb, int num_sms) {
    if (tiles >= num_sms) return 1;
    int64_t s = num_sms / tiles;
    s = std::min<int64_t>(s, 16);
    s = std::min<int64_t>(s, std::max<int64_t>(nkb / 2, 1));
    return (int)std::max<int64_t>(s, 1);
}

// Workspace of the decode form: the FP32 partial sums of every (tile, slice) when the
// reduction is split, nothing otherwise.
size_t decode_ws_bytes(int64_t M, int64_t N, int64_t K, int splits) {
    (void)K;
    if (splits <= 1) return 0;
    return (size_t)decode_tiles(M, N) * splits * kDecodeBN * 128 * sizeof(float);
}

// 2-D tensor map of the BF16 output C [rows][ld] (ld a multiple of 8) for the GEMM's tile
// stores: 32 x 32 boxes, 64-byte swizzle.
fp8rl_status make_tmap_out(CUtensorMap* m, uint16_t* base, int64_t rows, int64_t cols, int64_t ld) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return FP8RL_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8RL_OK : FP8RL_ERR_CUDA;
}

// Tensor maps that let the GEMM's copy warp move the scales by TMA (see launch_gemm_tiled):
// A's row scales [K-block][R1] need R1 % 4 == 0; B's block scales need 4 | K-blocks
// ([column block][K-block] storage) or 4 | column blocks ([K-block][column block]); B's
// row scales [K-block][R2] always qualify (R2 % 128 == 0).  Returns false when they do not
// all qualify, in which case the kernel takes the per-thread scale path.
bool scale_maps(const GemmParams& p, int b_mode, int bn, bool splitk, CUtensorMap* tsa, CUtensorMap* tsb,
                fp8rl_status* err) {
    *err = FP8RL_OK;
    const int64_t nkb = p.Kr / 128;
    if (p.R1 % 4 != 0 || p.sa_kb != p.R1) return false;
    if (b_mode == SCALE_ROW) {
        if (p.sb_kb != p.R2 || p.R2 % 4 != 0) return false;
    } else if (p.sb_kb == 1) {
        if (nkb % 4 != 0 || p.sb_r != nkb) return false;
    } else {
        if (p.sb_r != 1 || p.sb_kb % 4 != 0) return false;
    }
    // boxes of one scale group of K-blocks (all of them when K is shorter): the kernel
    // fetches a group's scales with one copy per operand
    const int grp = (int)std::min<int64_t>(nkb, scale_group(b_mode, splitk));
    *err = make_tmap_scales(tsa, p.sa, nkb, p.R1, 128, grp);
    if (*err != FP8RL_OK) return false;
    if (b_mode == SCALE_ROW)
        *err = make_tmap_scales(tsb, p.sb, nkb, p.R2, bn, grp);
    else if (p.sb_kb == 1)
        *err = make_tmap_scales(tsb, p.sb, (p.R2 + 127) / 128, nkb, 4, bn / 128);
    else
        *err = make_tmap_scales(tsb, p.sb, nkb, p.sb_kb, 4, grp);
    return *err == FP8RL_OK;
}

struct TiledArgs {
    const uint8_t* A; const float* sa; int64_t sa_kb;
    const uint8_t* B; const float* sb; int64_t sb_kb, sb_r; int b_mode;
    uint16_t* c; int64_t ldc;
    int64_t R1, R2, Kr;
};

// Column-tile width of the tiled form: 256 halves the re-reads of A, 128 gives the tensor
// pipe four TMEM buffers of lead over the promotion epilogue.
int tiled_bn(int req) { return req == 128 ? 128 : 256; }

fp8rl_status run_tiled(const TiledArgs& t, int grid_req, int bn_req, int num_sms, cudaStream_t st);

// Paired-SM form (gemm_pair.cu): 256 x pn tiles (pn = 128 or 256) on clusters of two
// CTAs.  Returns FP8RL_ERR_SHAPE, launching nothing, when a scale array cannot be moved by
// TMA.
fp8rl_status run_pair(const TiledArgs& t, int clusters_req, int epi_req, int pn_req, int num_sms, cudaStream_t st) {
    const int pn = pn_req == 128 ? 128 : 256;
    GemmParams p = {};
    p.R1 = t.R1; p.R2 = t.R2; p.Kr = t.Kr;
    p.sa = t.sa; p.sa_kb = t.sa_kb;
    p.sb = t.sb; p.sb_kb = t.sb_kb; p.sb_r = t.sb_r;
    p.c = t.c; p.ldc = t.ldc;
    p.splits = 0;
    CUtensorMap tsa, tsb;
    fp8rl_status e = FP8RL_OK;
    if (!scale_maps(p, t.b_mode, pn, false, &tsa, &tsb, &e)) return e != FP8RL_OK ? e : FP8RL_ERR_SHAPE;
    if (t.ldc % 8 != 0) return FP8RL_ERR_ALIGN;
    CUtensorMap ta, tb, tc;
    if ((e = make_tmap(&ta, t.A, t.R1, t.Kr, t.Kr, 128)) != FP8RL_OK) return e;
    if ((e = make_tmap(&tb, t.B, t.R2, t.Kr, t.Kr, pn / 2)) != FP8RL_OK) return e;
    if ((e = make_tmap_out(&tc, t.c, t.R1, t.R2, t.ldc)) != FP8RL_OK) return e;
    p.m_tiles = (int)((t.R1 + 127) / 128);
    p.n_tiles = (int)((t.R2 + pn - 1) / pn);
    p.nkb = (int)(t.Kr / 128);
    const int items = ((p.m_tiles + 1) / 2) * p.n_tiles;
    p.num_items = items;
    int clusters = clusters_req > 0 ? clusters_req : num_sms / 2;
    clusters = std::max(1, std::min(clusters, items));
    choose_raster((p.m_tiles + 1) / 2, p.n_tiles, 256 * t.Kr, (int64_t)pn * t.Kr, clusters, &p.group, &p.raster_n);
    p.timeout_ns = g_timeout_ns.load();
    const int epi = epi_req == 8 || epi_req == 16 ? epi_req : 8;
    return cuda_status(launch_gemm_pair(ta, tb, tsa, tsb, tc, p, t.b_mode, epi, pn, clusters, st));
}

// Multicast form (gemm_mc.cu): 128 x 256 one-SM tiles, two CTAs of a cluster on vertically
// adjacent tiles sharing each B tile.  Needs TMA-able scales (FP8RL_ERR_SHAPE otherwise).
fp8rl_status run_mc(const TiledArgs& t, int clusters_req, int num_sms, cudaStream_t st) {
    constexpr int bn = 256;
    GemmParams p = {};
    p.R1 = t.R1; p.R2 = t.R2; p.Kr = t.Kr;
    p.sa = t.sa; p.sa_kb = t.sa_kb;
    p.sb = t.sb; p.sb_kb = t.sb_kb; p.sb_r = t.sb_r;
    p.c = t.c; p.ldc = t.ldc;
    p.splits = 0;
    CUtensorMap tsa, tsb;
    fp8rl_status e = FP8RL_OK;
    if (!scale_maps(p, t.b_mode, bn, false, &tsa, &tsb, &e)) return e != FP8RL_OK ? e : FP8RL_ERR_SHAPE;
    if (t.ldc % 8 != 0) return FP8RL_ERR_ALIGN;
    CUtensorMap ta, tb, tc;
    if ((e = make_tmap(&ta, t.A, t.R1, t.Kr, t.Kr, 128)) != FP8RL_OK) return e;
    if ((e = make_tmap(&tb, t.B, t.R2, t.Kr, t.Kr, bn / 2)) != FP8RL_OK) return e;
    if ((e = make_tmap_out(&tc, t.c, t.R1, t.R2, t.ldc)) != FP8RL_OK) return e;
    p.m_tiles = (int)((t.R1 + 127) / 128);
    p.n_tiles = (int)((t.R2 + bn - 1) / bn);
    p.nkb = (int)(t.Kr / 128);
    p.num_items = ((p.m_tiles + 1) / 2) * p.n_tiles;
    int clusters = clusters_req > 0 ? clusters_req : num_sms / 2;
    clusters = std::max(1, std::min(clusters, p.num_items));
    choose_raster((p.m_tiles + 1) / 2, p.n_tiles, 256 * t.Kr, (int64_t)bn * t.Kr, clusters, &p.group, &p.raster_n);
    p.timeout_ns = g_timeout_ns.load();
    return cuda_status(launch_gemm_mc(ta, tb, tsa, tsb, tc, p, t.b_mode, clusters, st));
}

// Whether every scale array of the problem can be moved by TMA (the paired form's need).
bool pair_eligible(const TiledArgs& t) {
    const int64_t nkb = t.Kr / 128;
    if (t.R1 % 4 != 0 || t.sa_kb != t.R1) return false;
    if (t.b_mode == SCALE_ROW) return t.sb_kb == t.R2 && t.R2 % 4 == 0;
    if (t.sb_kb == 1) return nkb % 4 == 0 && t.sb_r == nkb;
    return t.sb_r == 1 && t.sb_kb % 4 == 0;
}

// The tiled forms: PAIR, MULTICAST or TILED on request.  AUTO takes 256 x 256 pair tiles
// when every scale array can travel by TMA and the tiles fill every pair of SMs at least
// once: per SM the tensor pipe then reads 32 KB of operands per K-block instead of 48 KB.
// On the 32B layer's shapes that measured 3-10% faster than the one-SM form for forward
// and DGrad (8 epilogue warps: one FMA per element) and 13% faster for WGrad (16 epilogue
// warps: a multiply and an FMA per element, in 16-row x 32-column parts).
fp8rl_status run_gemm(const TiledArgs& t, const fp8rl_gemm_opts* opts, int num_sms, cudaStream_t st) {
    const int variant = opts ? opts->variant : FP8RL_VARIANT_AUTO;
    if (variant == FP8RL_VARIANT_PAIR)
        return pair_eligible(t) ? run_pair(t, opts->grid, opts->epi_warps, opts->tile_n, num_sms, st) : FP8RL_ERR_SHAPE;
    if (variant == FP8RL_VARIANT_MULTICAST)
        return pair_eligible(t) ? run_mc(t, opts->grid, num_sms, st) : FP8RL_ERR_SHAPE;
    if (variant == FP8RL_VARIANT_AUTO && pair_eligible(t)) {
        const int64_t pair_tiles = ((t.R1 + 255) / 256) * ((t.R2 + 255) / 256);
        if (pair_tiles >= num_sms / 2)
            return run_pair(t, opts ? opts->grid : 0, t.b_mode == SCALE_ROW ? 16 : 8, 256, num_sms, st);
    }
    return run_tiled(t, opts ? opts->grid : 0, opts ? opts->tile_n : 0, num_sms, st);
}

fp8rl_status run_tiled(const TiledArgs& t, int grid_req, int bn_req, int num_sms, cudaStream_t st) {
    int bn = tiled_bn(bn_req);
    GemmParams p = {};
    p.R1 = t.R1; p.R2 = t.R2; p.Kr = t.Kr;
    p.sa = t.sa; p.sa_kb = t.sa_kb;
    p.sb = t.sb; p.sb_kb = t.sb_kb; p.sb_r = t.sb_r;
    p.c = t.c; p.ldc = t.ldc;
    p.splits = 0;
    CUtensorMap tsa, tsb;
    fp8rl_status e = FP8RL_OK;
    bool tma_scales = scale_maps(p, t.b_mode, bn, false, &tsa, &tsb, &e);
    if (e != FP8RL_OK) return e;
    if (t.b_mode == SCALE_ROW && !tma_scales) return FP8RL_ERR_INVALID_ARG;
    if (!tma_scales) bn = 256;   // the per-thread scale path is built for 256-wide tiles only
    CUtensorMap ta, tb;
    e = make_tmap(&ta, t.A, t.R1, t.Kr, t.Kr, 128);
    if (e != FP8RL_OK) return e;
    e = make_tmap(&tb, t.B, t.R2, t.Kr, t.Kr, bn);
    if (e != FP8RL_OK) return e;
    p.m_tiles = (int)((t.R1 + 127) / 128);
    p.n_tiles = (int)((t.R2 + bn - 1) / bn);
    p.nkb = (int)(t.Kr / 128);
    p.num_items = p.m_tiles * p.n_tiles;
    int grid = grid_req > 0 ? grid_req : num_sms;
    grid = std::max(1, std::min(grid, p.num_items));
    choose_raster(p.m_tiles, p.n_tiles, 128 * t.Kr, (int64_t)bn * t.Kr, grid, &p.group, &p.raster_n);
    p.timeout_ns = g_timeout_ns.load();
    if (t.ldc % 8 != 0) return FP8RL_ERR_ALIGN;
    CUtensorMap tc;
    e = make_tmap_out(&tc, t.c, t.R1, t.R2, t.ldc);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_gemm_tiled(ta, tb, tma_scales ? &tsa : nullptr, tma_scales ? &tsb : nullptr, tc,
                                         p, t.b_mode, bn, grid, st));
}

fp8rl_status run_decode(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw,
                        uint16_t* y, int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes,
                        int splits_req, int num_sms, cudaStream_t st) {
    const int64_t tiles = decode_tiles(M, N);
    const int64_t nkb = K / 128;
    const int splits = splits_req > 0 ? (int)std::min<int64_t>(splits_req, nkb)
                                      : choose_splits(tiles, nkb, num_sms);
    const size_t need = decode_ws_bytes(M, N, K, splits);
    if (need > 0) {
        if (ws == nullptr || ws_bytes < need) return FP8RL_ERR_WORKSPACE;
        if (!aligned16(ws)) return FP8RL_ERR_ALIGN;
    }
    CUtensorMap ta, tb;
    fp8rl_status e = make_tmap(&ta, qx, M, K, K, 128);
    if (e != FP8RL_OK) return e;
    e = make_tmap(&tb, qw, N, K, K, kDecodeBN);
    if (e != FP8RL_OK) return e;
    GemmParams p = {};
    p.R1 = M; p.R2 = N; p.Kr = K;
    p.sa = sx; p.sa_kb = M;
    p.sb = sw; p.sb_kb = 1; p.sb_r = K / 128;
    p.c = y; p.ldc = N;
    p.ws = reinterpret_cast<float*>(ws);
    p.splits = splits;
    p.m_tiles = (int)((M + 127) / 128);
    p.n_tiles = (int)((N + kDecodeBN - 1) / kDecodeBN);
    p.nkb = (int)nkb;
    p.num_items = (int)(tiles * splits);
    p.group = p.m_tiles;   // at most two row tiles: every weight tile streams once
    p.raster_n = 0;
    p.timeout_ns = g_timeout_ns.load();
    const int grid = std::max(1, std::min(num_sms, p.num_items));
    CUtensorMap tsa, tsb;
    const bool tma_scales = scale_maps(p, SCALE_BLOCK, kDecodeBN, true, &tsa, &tsb, &e);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_gemm_splitk(ta, tb, tma_scales ? &tsa : nullptr, tma_scales ? &tsb : nullptr, p,
                                          grid, st));
}

// Whether the automatic choice takes the decode form with the weights on the MMA's M side
// (else the split-K form with the tokens there).  Measured on the 7B decode shapes:
// up to 64 tokens it is the faster form; at 128 tokens it is for the narrow layers (qkv,
// o: 12.8 against 16.6 us) but not for gate_up (38 against 30 us), whose 296 weight tiles
// each re-read a 128-token activation tile as large as themselves; at 256 tokens the
// split-K form wins on every layer.
bool decode_swapped_auto(int64_t M, int64_t N) { return M <= 64 || (M <= 128 && N <= 8192); }

// 129-256 tokens against a wide weight: one 256-row pair tile per column tile already
// fills every pair of SMs, reads each weight tile once and needs no reduction of slices,
// so the paired training form beats the split-K form (Qwen2.5-7B gate_up 37888x3584 at
// 256 tokens: 35.1 against 40.4 us per GEMM on GB300).
bool decode_pair_auto(const TiledArgs& t, int num_sms) {
    if (t.R1 <= 128 || !pair_eligible(t)) return false;
    const int64_t pair_tiles = ((t.R1 + 255) / 256) * ((t.R2 + 255) / 256);
    return pair_tiles >= num_sms / 2;
}

// Decode form with the weights on the MMA's M side (decode.cu).  Cluster size (split of
// the reduction): the one that minimises waves x K-blocks per CTA, with one K-block of cost
// for the cluster reduction, among the sizes whose clusters fit on the GPU at once.
struct DecodeChoice {
    int cached = 0;
    int max_clusters[9] = {};
};
DecodeChoice g_dec_choice[kMaxDevices][4];
std::mutex g_dec_mu;

int decode_splits(int64_t M, int64_t tiles, int64_t nkb) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int mp = decode_mp((int)M);
    const int cls = mp == 32 ? 0 : (mp == 64 ? 1 : (mp == 128 ? 2 : 3));
    int maxc[9];
    {
        std::lock_guard<std::mutex> lk(g_dec_mu);
        DecodeChoice& c = g_dec_choice[dev < kMaxDevices ? dev : 0][cls];
        if (!c.cached) {
            for (int sz = 1; sz <= 8; ++sz) c.max_clusters[sz] = decode_max_clusters((int)M, sz);
            c.cached = 1;
        }
        for (int sz = 1; sz <= 8; ++sz) maxc[sz] = c.max_clusters[sz];
    }
    int best = 1;
    double best_cost = 1e30;
    for (int sz = 1; sz <= 8 && sz <= nkb; ++sz) {
        if (maxc[sz] <= 0) continue;
        // the busiest CTA's K-blocks: S = 1 runs persistent CTAs (one pipeline across their
        // tiles, one fill); S > 1 one wave per maxc[sz] clusters, each wave paying a pipeline
        // fill and the cluster reduction
        const int64_t waves = (tiles + maxc[sz] - 1) / maxc[sz];
        const double cost = sz == 1 ? (double)(waves * nkb) + 2.0
                                    : (double)waves * ((double)((nkb + sz - 1) / sz) + 3.0);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = sz;
        }
    }
    return best;
}

// pdl: the kernel is launched as a programmatic dependent of the previous kernel on the
// stream (the fused linear's quantizer); it then streams its first weight tiles while that
// kernel finishes.  Used without a cluster split only: the split form's clusters, launched
// early, take the SMs the quantizer still needs (measured 25-55% slower).
fp8rl_status run_decode_swap(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw,
                             uint16_t* y, int64_t M, int64_t N, int64_t K, int splits_req, cudaStream_t st,
                             bool pdl = false) {
    const int64_t nkb = K / 128;
    const int64_t tiles = N / 128;
    const int splits = splits_req > 0 ? (int)std::min<int64_t>(std::min(splits_req, 8), nkb)
                                      : decode_splits(M, tiles, nkb);
    CUtensorMap tw, tx;
    fp8rl_status e = make_tmap(&tw, qw, N, K, K, 128);
    if (e != FP8RL_OK) return e;
    e = make_tmap(&tx, qx, M, K, K, decode_mp((int)M));
    if (e != FP8RL_OK) return e;
    DecodeParams p = {};
    p.M = (int)M;
    p.nkb = (int)nkb;
    p.tiles = (int)tiles;
    p.sx = sx; p.sx_kb = M;
    p.sw = sw; p.sw_r = nkb;
    p.y = y; p.ldy = N;
    p.timeout_ns = g_timeout_ns.load();
    // one cluster per tile when the reduction is split; else persistent CTAs, one per SM
    int sms = 0;
    current_device(&sms);
    const int grid = splits > 1 ? (int)tiles : (int)std::min<int64_t>(tiles, std::max(sms, 1));
    return cuda_status(launch_decode(tw, tx, p, grid, splits, pdl && splits == 1, st));
}

// NVFP4 decode GEMM (nvfp4.cu): the same split rule as the FP8 decode form, over K-blocks
// of 256 elements and the clusters of the FP4 kernel that fit.
DecodeChoice g_nvf4_choice[kMaxDevices][4];

int nvf4_splits(int64_t M, int64_t tiles, int64_t nkb) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int mp = nvf4_token_tile((int)M);
    const int cls = mp == 32 ? 0 : (mp == 64 ? 1 : (mp == 128 ? 2 : 3));
    int maxc[9];
    {
        std::lock_guard<std::mutex> lk(g_dec_mu);
        DecodeChoice& c = g_nvf4_choice[dev < kMaxDevices ? dev : 0][cls];
        if (!c.cached) {
            for (int sz = 1; sz <= 8; ++sz) c.max_clusters[sz] = nvf4_max_clusters((int)M, sz);
            c.cached = 1;
        }
        for (int sz = 1; sz <= 8; ++sz) maxc[sz] = c.max_clusters[sz];
    }
    int best = 1;
    double best_cost = 1e30;
    for (int sz = 1; sz <= 8 && sz <= nkb; ++sz) {
        if (maxc[sz] <= 0) continue;
        const int64_t waves = (tiles + maxc[sz] - 1) / maxc[sz];
        const double cost = sz == 1 ? (double)(waves * nkb) + 2.0
                                    : (double)waves * ((double)((nkb + sz - 1) / sz) + 3.0);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = sz;
        }
    }
    return best;
}

fp8rl_status run_gemm_nvf4(const uint8_t* qx, const uint8_t* sfx, const float* gx, const uint8_t* qw,
                           const uint8_t* sfw, const float* gw, uint16_t* y, int64_t M, int64_t N, int64_t K,
                           int64_t ldy, int splits_req, bool pdl, cudaStream_t st) {
    const int64_t nkb = K / 256;
    const int64_t tiles = N / 128;
    const int splits = splits_req > 0 ? (int)std::min<int64_t>(std::min(splits_req, 8), nkb)
                                      : nvf4_splits(M, tiles, nkb);
    CUtensorMap tw, tx;
    fp8rl_status e = make_tmap(&tw, qw, N, K / 2, K / 2, 128);
    if (e != FP8RL_OK) return e;
    e = make_tmap(&tx, qx, M, K / 2, K / 2, nvf4_token_tile((int)M));
    if (e != FP8RL_OK) return e;
    Nvf4Params p = {};
    p.M = (int)M;
    p.nkb = (int)nkb;
    p.tiles = (int)tiles;
    p.sfw = sfw;
    p.sfx = sfx;
    p.gw = gw;
    p.gx = gx;
    p.y = y;
    p.ldy = ldy;
    p.timeout_ns = g_timeout_ns.load();
    int sms = 0;
    current_device(&sms);
    const int grid = splits > 1 ? (int)tiles : (int)std::min<int64_t>(tiles, std::max(sms, 1));
    return cuda_status(launch_gemm_nvf4(tw, tx, p, grid, splits, pdl && splits == 1, st));
}

}  // namespace

// ====================================================================================
extern "C" {

int fp8rl_version(void) { return (0 << 16) | 1; }

const char* fp8rl_status_string(fp8rl_status st) {
    switch (st) {
        case FP8RL_OK: return "FP8RL_OK";
        case FP8RL_ERR_INVALID_ARG: return "FP8RL_ERR_INVALID_ARG";
        case FP8RL_ERR_SHAPE: return "FP8RL_ERR_SHAPE";
        case FP8RL_ERR_ALIGN: return "FP8RL_ERR_ALIGN";
        case FP8RL_ERR_UNSUPPORTED_DEVICE: return "FP8RL_ERR_UNSUPPORTED_DEVICE";
        case FP8RL_ERR_WORKSPACE: return "FP8RL_ERR_WORKSPACE";
        case FP8RL_ERR_CUDA: return "FP8RL_ERR_CUDA";
        case FP8RL_ERR_DEVICE_TIMEOUT: return "FP8RL_ERR_DEVICE_TIMEOUT";
        case FP8RL_ERR_DEVICE_BOUNDS: return "FP8RL_ERR_DEVICE_BOUNDS";
    }
    return "FP8RL_ERR_UNKNOWN";
}

fp8rl_status fp8rl_init(int device) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess) return FP8RL_ERR_CUDA;
    if (device < 0 || device >= n) return FP8RL_ERR_INVALID_ARG;
    if (cudaSetDevice(device) != cudaSuccess) return FP8RL_ERR_CUDA;
    return current_device(nullptr);
}

void fp8rl_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns > 0 ? ns : 1); }

fp8rl_status fp8rl_check_status(fp8rl_stream_t stream) {
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    const fp8rl_status g = read_and_clear_device_status(stream);  // synchronizes the stream
    const fp8rl_status q = read_and_clear_quant_status();
    const fp8rl_status pr = read_and_clear_pair_status();
    const fp8rl_status dc = read_and_clear_decode_status();
    const fp8rl_status mc = read_and_clear_mc_status();
    const fp8rl_status nv = read_and_clear_nvf4_status();
    if (g != FP8RL_OK) return g;
    if (pr != FP8RL_OK) return pr;
    if (mc != FP8RL_OK) return mc;
    if (nv != FP8RL_OK) return nv;
    return dc != FP8RL_OK ? dc : q;
}

// ---------------------------------------------------------------- quantizers

fp8rl_status fp8rl_quantize_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                                  float* s, uint8_t* qT, float* sT, fp8rl_stream_t stream) {
    if (M < 0 || K <= 0 || ldx < K) return FP8RL_ERR_INVALID_ARG;
    if ((qT == nullptr) != (sT == nullptr)) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0) return FP8RL_ERR_SHAPE;
    if (qT && M % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0) return FP8RL_OK;
    if (!x || !q || !s) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s) || (ldx * 2) % 16 != 0) return FP8RL_ERR_ALIGN;
    if (qT && (!aligned16(qT) || !aligned16(sT))) return FP8RL_ERR_ALIGN;
    int sms = 0;
    fp8rl_status e = current_device(&sms);
    if (e != FP8RL_OK) return e;
    if (qT) return cuda_status(launch_quant_dual(x, M, K, ldx, q, s, qT, sT, g_timeout_ns.load(), stream));
    return cuda_status(launch_quant_1x128(x, M, K, ldx, q, s, sms, stream));
}

fp8rl_status fp8rl_quantize_128x1(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* qT, float* sT, fp8rl_stream_t stream) {
    if (M < 0 || K <= 0 || ldx < K) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || M % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0) return FP8RL_OK;
    if (!x || !qT || !sT) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(qT) || !aligned16(sT) || (ldx * 2) % 16 != 0) return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_quant_dual(x, M, K, ldx, nullptr, nullptr, qT, sT, g_timeout_ns.load(), stream));
}

fp8rl_status fp8rl_requantize_128x1(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                    uint8_t* qT, float* sT, fp8rl_stream_t stream) {
    if (M < 0 || K <= 0) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || M % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0) return FP8RL_OK;
    if (!q || !s || !qT || !sT) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(s) || !aligned16(qT) || !aligned16(sT)) return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_requant_128x1(q, s, M, K, qT, sT, g_timeout_ns.load(), stream));
}

fp8rl_status fp8rl_quantize_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw,
                                    uint8_t* q, float* s, uint8_t* qT, fp8rl_stream_t stream) {
    if (N < 0 || K <= 0 || ldw < K) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0) return FP8RL_ERR_SHAPE;
    if (N == 0) return FP8RL_OK;
    if (!w || !q || !s) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || !aligned16(s) || (ldw * 2) % 16 != 0) return FP8RL_ERR_ALIGN;
    if (qT && !aligned16(qT)) return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_quant_128x128(w, N, K, ldw, q, s, qT, g_timeout_ns.load(), stream));
}

fp8rl_status fp8rl_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M,
                                 int64_t K, uint8_t* q, float* s, uint8_t* qT, float* sT,
                                 float* rstd, fp8rl_stream_t stream) {
    if (M < 0 || K <= 0 || !(eps >= 0.0f) || eps > 3.0e38f) return FP8RL_ERR_INVALID_ARG;
    if ((qT == nullptr) != (sT == nullptr)) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0) return FP8RL_ERR_SHAPE;
    if (qT && M % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0) return FP8RL_OK;
    if (!x || !gamma || !q || !s) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(q) || !aligned16(s)) return FP8RL_ERR_ALIGN;
    if (qT && (!aligned16(qT) || !aligned16(sT))) return FP8RL_ERR_ALIGN;
    if (rstd && !aligned16(rstd)) return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_rmsnorm_quant(x, gamma, eps, M, K, q, s, qT, sT, rstd, g_timeout_ns.load(), stream));
}

fp8rl_status fp8rl_silu_mul_quant(const uint16_t* gu, int64_t M, int64_t I, uint8_t* q, float* s,
                                  uint8_t* qT, float* sT, fp8rl_stream_t stream) {
    if (M < 0 || I <= 0) return FP8RL_ERR_INVALID_ARG;
    if ((qT == nullptr) != (sT == nullptr)) return FP8RL_ERR_INVALID_ARG;
    if (I % 128 != 0) return FP8RL_ERR_SHAPE;
    if (qT && M % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0) return FP8RL_OK;
    if (!gu || !q || !s) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(gu) || !aligned16(q) || !aligned16(s)) return FP8RL_ERR_ALIGN;
    if (qT && (!aligned16(qT) || !aligned16(sT))) return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_silu_mul_quant(gu, M, I, q, s, qT, sT, g_timeout_ns.load(), stream));
}

// ---------------------------------------------------------------- backward steps

fp8rl_status fp8rl_silu_mul_bwd_quant(const uint16_t* gu, const uint16_t* dh, int64_t M, int64_t I,
                                      uint8_t* q, float* s, uint8_t* qT, float* sT,
                                      fp8rl_stream_t stream) {
    if (M < 0 || I <= 0) return FP8RL_ERR_INVALID_ARG;
    if ((qT == nullptr) != (sT == nullptr)) return FP8RL_ERR_INVALID_ARG;
    if (I % 128 != 0) return FP8RL_ERR_SHAPE;
    if (qT && M % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0) return FP8RL_OK;
    if (!gu || !dh || !q || !s) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(gu) || !aligned16(dh) || !aligned16(q) || !aligned16(s)) return FP8RL_ERR_ALIGN;
    if (qT && (!aligned16(qT) || !aligned16(sT))) return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_silu_mul_bwd_quant(gu, dh, M, I, q, s, qT, sT, g_timeout_ns.load(), stream));
}

size_t fp8rl_rmsnorm_bwd_workspace_bytes(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0) return 0;
    int sms = 0;
    if (current_device(&sms) != FP8RL_OK) sms = 148;
    return (size_t)rmsnorm_bwd_blocks(M, sms) * (size_t)K * sizeof(float);
}

fp8rl_status fp8rl_rmsnorm_bwd(const uint16_t* x, const uint16_t* gamma, const float* rstd,
                               const uint16_t* dy, int64_t M, int64_t K, uint16_t* dx,
                               float* dgamma, void* ws, size_t ws_bytes, fp8rl_stream_t stream) {
    if (M < 0 || K <= 0) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > 8192) return FP8RL_ERR_SHAPE;
    if (M == 0) {
        if (dgamma) return cuda_status(cudaMemsetAsync(dgamma, 0, (size_t)K * sizeof(float), stream));
        return FP8RL_OK;
    }
    if (!x || !gamma || !rstd || !dy || !dx) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(rstd) || !aligned16(dy) || !aligned16(dx))
        return FP8RL_ERR_ALIGN;
    int sms = 0;
    fp8rl_status e = current_device(&sms);
    if (e != FP8RL_OK) return e;
    const int nblocks = rmsnorm_bwd_blocks(M, sms);
    if (dgamma) {
        if (!aligned16(dgamma)) return FP8RL_ERR_ALIGN;
        if (!ws || ws_bytes < (size_t)nblocks * (size_t)K * sizeof(float)) return FP8RL_ERR_WORKSPACE;
        if (!aligned16(ws)) return FP8RL_ERR_ALIGN;
    }
    return cuda_status(launch_rmsnorm_bwd(x, gamma, rstd, dy, M, K, dx, dgamma, reinterpret_cast<float*>(ws),
                                          nblocks, stream));
}

// ---------------------------------------------------------------- GEMMs

size_t fp8rl_gemm_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
    return fp8rl_gemm_workspace_bytes_ex(op, M, N, K, nullptr);
}

size_t fp8rl_gemm_workspace_bytes_ex(int op, int64_t M, int64_t N, int64_t K,
                                     const fp8rl_gemm_opts* opts) {
    if (op != FP8RL_OP_FWD || M <= 0 || N <= 0 || K <= 0 || K % 128 != 0) return 0;
    const int variant = opts ? opts->variant : FP8RL_VARIANT_AUTO;
    // only the split-K form uses one
    if (M > 256 || !(variant == FP8RL_VARIANT_SPLITK || (variant == FP8RL_VARIANT_AUTO && !decode_swapped_auto(M, N))))
        return 0;
    int sms = 0;
    if (current_device(&sms) != FP8RL_OK) sms = 148;
    if (variant == FP8RL_VARIANT_AUTO && N % 128 == 0) {
        TiledArgs t = {};   // the shape alone decides the route
        t.sa_kb = M; t.sb_kb = 1; t.sb_r = K / 128; t.b_mode = SCALE_BLOCK;
        t.R1 = M; t.R2 = N; t.Kr = K;
        if (decode_pair_auto(t, sms)) return 0;
    }
    const int64_t tiles = decode_tiles(M, N), nkb = K / 128;
    const int splits = (opts && opts->splits > 0) ? (int)std::min<int64_t>(opts->splits, nkb)
                                                  : choose_splits(tiles, nkb, sms);
    return decode_ws_bytes(M, N, K, splits);
}

fp8rl_status fp8rl_gemm_fwd_ex(const uint8_t* qx, const float* sx, const uint8_t* qw,
                               const float* sw, uint16_t* y, int64_t M, int64_t N, int64_t K,
                               void* ws, size_t ws_bytes, const fp8rl_gemm_opts* opts,
                               fp8rl_stream_t stream) {
    if (M < 0 || N < 0 || K <= 0) return FP8RL_ERR_INVALID_ARG;
    const int variant = opts ? opts->variant : FP8RL_VARIANT_AUTO;
    if (variant < FP8RL_VARIANT_AUTO || variant > FP8RL_VARIANT_MULTICAST) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8RL_OK;
    if (!qx || !sx || !qw || !sw || !y) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(qx) || !aligned16(sx) || !aligned16(qw) || !aligned16(sw) || !aligned16(y))
        return FP8RL_ERR_ALIGN;
    int sms = 0;
    fp8rl_status e = current_device(&sms);
    if (e != FP8RL_OK) return e;
    TiledArgs t;
    t.A = qx; t.sa = sx; t.sa_kb = M;
    t.B = qw; t.sb = sw; t.sb_kb = 1; t.sb_r = K / 128; t.b_mode = SCALE_BLOCK;
    t.c = y; t.ldc = N;
    t.R1 = M; t.R2 = N; t.Kr = K;
    const bool swapped = variant == FP8RL_VARIANT_DECODE || (variant == FP8RL_VARIANT_AUTO && decode_swapped_auto(M, N));
    const bool splitk = variant == FP8RL_VARIANT_SPLITK ||
                        (variant == FP8RL_VARIANT_AUTO && !swapped && M <= 256 && !decode_pair_auto(t, sms));
    if ((swapped || splitk) && M > 256) return FP8RL_ERR_SHAPE;
    if (swapped)
        return run_decode_swap(qx, sx, qw, sw, y, M, N, K, opts ? opts->splits : 0, stream);
    if (splitk)
        return run_decode(qx, sx, qw, sw, y, M, N, K, ws, ws_bytes, opts ? opts->splits : 0, sms, stream);
    return run_gemm(t, opts, sms, stream);
}

fp8rl_status fp8rl_gemm_fwd(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw,
                            uint16_t* y, int64_t M, int64_t N, int64_t K, void* ws,
                            size_t ws_bytes, fp8rl_stream_t stream) {
    return fp8rl_gemm_fwd_ex(qx, sx, qw, sw, y, M, N, K, ws, ws_bytes, nullptr, stream);
}

fp8rl_status fp8rl_gemm_dgrad(const uint8_t* qdy, const float* sdy, const uint8_t* qwT,
                              const float* sw, uint16_t* dx, int64_t M, int64_t N, int64_t K,
                              void* ws, size_t ws_bytes, fp8rl_stream_t stream) {
    return fp8rl_gemm_dgrad_ex(qdy, sdy, qwT, sw, dx, M, N, K, ws, ws_bytes, nullptr, stream);
}

// The forms DGrad and WGrad take: AUTO, TILED, PAIR, MULTICAST (not the decode-shaped ones).
static bool training_variant(int v) {
    return v == FP8RL_VARIANT_AUTO || v == FP8RL_VARIANT_TILED || v == FP8RL_VARIANT_PAIR ||
           v == FP8RL_VARIANT_MULTICAST;
}

fp8rl_status fp8rl_gemm_dgrad_ex(const uint8_t* qdy, const float* sdy, const uint8_t* qwT,
                                 const float* sw, uint16_t* dx, int64_t M, int64_t N, int64_t K,
                                 void* ws, size_t ws_bytes, const fp8rl_gemm_opts* opts,
                                 fp8rl_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (M < 0 || N < 0 || K <= 0) return FP8RL_ERR_INVALID_ARG;
    if (opts && !training_variant(opts->variant)) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0) return FP8RL_OK;
    if (N == 0) return FP8RL_ERR_SHAPE;
    if (!qdy || !sdy || !qwT || !sw || !dx) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(qdy) || !aligned16(sdy) || !aligned16(qwT) || !aligned16(sw) || !aligned16(dx))
        return FP8RL_ERR_ALIGN;
    int sms = 0;
    fp8rl_status e = current_device(&sms);
    if (e != FP8RL_OK) return e;
    TiledArgs t;
    t.A = qdy; t.sa = sdy; t.sa_kb = M;
    t.B = qwT; t.sb = sw; t.sb_kb = K / 128; t.sb_r = 1; t.b_mode = SCALE_BLOCK;
    t.c = dx; t.ldc = K;
    t.R1 = M; t.R2 = K; t.Kr = N;
    return run_gemm(t, opts, sms, stream);
}

fp8rl_status fp8rl_gemm_wgrad(const uint8_t* qdyT, const float* sdyT, const uint8_t* qxT,
                              const float* sxT, uint16_t* dw, int64_t M, int64_t N, int64_t K,
                              void* ws, size_t ws_bytes, fp8rl_stream_t stream) {
    return fp8rl_gemm_wgrad_ex(qdyT, sdyT, qxT, sxT, dw, M, N, K, ws, ws_bytes, nullptr, stream);
}

fp8rl_status fp8rl_gemm_wgrad_ex(const uint8_t* qdyT, const float* sdyT, const uint8_t* qxT,
                                 const float* sxT, uint16_t* dw, int64_t M, int64_t N, int64_t K,
                                 void* ws, size_t ws_bytes, const fp8rl_gemm_opts* opts,
                                 fp8rl_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (M < 0 || N < 0 || K <= 0) return FP8RL_ERR_INVALID_ARG;
    if (opts && !training_variant(opts->variant)) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0 || M % 128 != 0) return FP8RL_ERR_SHAPE;
    if (N == 0) return FP8RL_OK;
    if (!qdyT || !sdyT || !qxT || !sxT || !dw) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(qdyT) || !aligned16(sdyT) || !aligned16(qxT) || !aligned16(sxT) || !aligned16(dw))
        return FP8RL_ERR_ALIGN;
    int sms = 0;
    fp8rl_status e = current_device(&sms);
    if (e != FP8RL_OK) return e;
    if (M == 0) return cuda_status(cudaMemsetAsync(dw, 0, (size_t)N * K * 2, stream));
    TiledArgs t;
    t.A = qdyT; t.sa = sdyT; t.sa_kb = N;
    t.B = qxT; t.sb = sxT; t.sb_kb = K; t.sb_r = 0; t.b_mode = SCALE_ROW;
    t.c = dw; t.ldc = K;
    t.R1 = N; t.R2 = K; t.Kr = M;
    return run_gemm(t, opts, sms, stream);
}

// ---------------------------------------------------------------- fused linear

fp8rl_status fp8rl_linear_fwd(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* qw,
                              const float* sw, int64_t N, uint8_t* qx, float* sx, uint16_t* y,
                              void* ws, size_t ws_bytes, fp8rl_stream_t stream) {
    if (M < 0 || N < 0 || K <= 0 || ldx < K) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0) return FP8RL_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8RL_OK;
    if (!x || !qw || !sw || !qx || !sx || !y) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(qw) || !aligned16(sw) || !aligned16(qx) || !aligned16(sx) ||
        !aligned16(y) || (ldx * 2) % 16 != 0)
        return FP8RL_ERR_ALIGN;
    int sms = 0;
    fp8rl_status e = current_device(&sms);
    if (e != FP8RL_OK) return e;
    e = cuda_status(launch_quant_1x128(x, M, K, ldx, qx, sx, sms, stream));
    if (e != FP8RL_OK) return e;
    TiledArgs t;
    t.A = qx; t.sa = sx; t.sa_kb = M;
    t.B = qw; t.sb = sw; t.sb_kb = 1; t.sb_r = K / 128; t.b_mode = SCALE_BLOCK;
    t.c = y; t.ldc = N;
    t.R1 = M; t.R2 = N; t.Kr = K;
    if (decode_swapped_auto(M, N))
        return run_decode_swap(qx, sx, qw, sw, y, M, N, K, 0, stream, true);
    if (M <= 256 && !decode_pair_auto(t, sms))
        return run_decode(qx, sx, qw, sw, y, M, N, K, ws, ws_bytes, 0, sms, stream);
    return run_gemm(t, nullptr, sms, stream);
}

// ---------------------------------------------------------------- NVFP4 rollout path

size_t fp8rl_nvfp4_scale_bytes(int64_t R, int64_t K) {
    if (R <= 0 || K <= 0 || K % 256 != 0) return 0;
    return (size_t)((R + 127) / 128) * (size_t)(K / 256) * 2048u;
}

fp8rl_status fp8rl_quantize_nvfp4(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q, uint8_t* sf,
                                  float* g, fp8rl_stream_t stream) {
    if (R < 0 || K <= 0 || ldx < K) return FP8RL_ERR_INVALID_ARG;
    if (K % 256 != 0) return FP8RL_ERR_SHAPE;
    if (R == 0) return FP8RL_OK;
    if (!x || !q || !sf || !g) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf) || (ldx * 2) % 16 != 0) return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_quant_nvfp4(x, R, K, ldx, q, sf, g, stream));
}

fp8rl_status fp8rl_gemm_nvfp4(const uint8_t* qx, const uint8_t* sfx, const float* gx, const uint8_t* qw,
                              const uint8_t* sfw, const float* gw, uint16_t* y, int64_t M, int64_t N, int64_t K,
                              int64_t ldy, int splits, fp8rl_stream_t stream) {
    if (M < 0 || N < 0 || K <= 0 || ldy < N || splits < 0) return FP8RL_ERR_INVALID_ARG;
    if (K % 256 != 0 || N % 128 != 0 || M > 256) return FP8RL_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8RL_OK;
    if (!qx || !sfx || !gx || !qw || !sfw || !gw || !y) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(qx) || !aligned16(sfx) || !aligned16(qw) || !aligned16(sfw) || !aligned16(gw) ||
        !aligned16(y) || ldy % 8 != 0)
        return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return run_gemm_nvf4(qx, sfx, gx, qw, sfw, gw, y, M, N, K, ldy, splits, false, stream);
}

fp8rl_status fp8rl_linear_nvfp4(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* qw,
                                const uint8_t* sfw, const float* gw, int64_t N, uint8_t* qx, uint8_t* sfx, float* gx,
                                uint16_t* y, fp8rl_stream_t stream) {
    if (M < 0 || N < 0 || K <= 0 || ldx < K) return FP8RL_ERR_INVALID_ARG;
    if (K % 256 != 0 || N % 128 != 0 || M > 256) return FP8RL_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8RL_OK;
    if (!x || !qw || !sfw || !gw || !qx || !sfx || !gx || !y) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(qw) || !aligned16(sfw) || !aligned16(gw) || !aligned16(qx) ||
        !aligned16(sfx) || !aligned16(y) || (ldx * 2) % 16 != 0)
        return FP8RL_ERR_ALIGN;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    e = cuda_status(launch_quant_nvfp4(x, M, K, ldx, qx, sfx, gx, stream));
    if (e != FP8RL_OK) return e;
    return run_gemm_nvf4(qx, sfx, gx, qw, sfw, gw, y, M, N, K, N, 0, true, stream);
}

// ---------------------------------------------------------------- no-allocation decode

// Decode-shaped forward GEMM on the library's own fixed scratch array (see
// gemm_noalloc.cu): the same kernel, split and reduction order as fp8rl_gemm_fwd_ex with
// FP8RL_VARIANT_SPLITK and automatic splits, but no workspace argument and no allocation.
fp8rl_status fp8rl_gemm_fwd_decode_noalloc(const uint8_t* qx, const float* sx, const uint8_t* qw,
                                           const float* sw, uint16_t* y, int64_t M, int64_t N,
                                           int64_t K, fp8rl_stream_t stream) {
    if (M < 0 || N < 0 || K <= 0) return FP8RL_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0 || M > 256) return FP8RL_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8RL_OK;
    if (!qx || !sx || !qw || !sw || !y) return FP8RL_ERR_INVALID_ARG;
    if (!aligned16(qx) || !aligned16(sx) || !aligned16(qw) || !aligned16(sw) || !aligned16(y))
        return FP8RL_ERR_ALIGN;
    int sms = 0;
    fp8rl_status e = current_device(&sms);
    if (e != FP8RL_OK) return e;
    const int64_t tiles = decode_tiles(M, N);
    const size_t have = noalloc_scratch_bytes();
    // The automatic split keeps tiles x slices <= SMs, so the partial sums never exceed
    // SMs x 128 KiB (19 MiB at 152 SMs): they fit the 32 MiB array on any GPU with up to
    // 256 SMs.  A larger GPU would be refused here rather than overrun the array.
    const int splits = choose_splits(tiles, K / 128, sms);
    if (decode_ws_bytes(M, N, K, splits) > have) return FP8RL_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return FP8RL_ERR_CUDA;
    // the array keeps the previous call's partial sums; every slice rewrites its own before
    // the reduction reads it, so nothing needs clearing
    return run_decode(qx, sx, qw, sw, y, M, N, K, scratch, have, splits, sms, stream);
}

size_t fp8rl_gemm_noalloc_scratch_bytes(void) { return noalloc_scratch_bytes(); }

// ---------------------------------------------------------------- diagnostics

fp8rl_status fp8rl_debug_e4m3_encode(const float* in, uint8_t* out, int64_t n,
                                     fp8rl_stream_t stream) {
    if (n < 0) return FP8RL_ERR_INVALID_ARG;
    if (n == 0) return FP8RL_OK;
    if (!in || !out) return FP8RL_ERR_INVALID_ARG;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_debug_e4m3(in, out, n, stream));
}

fp8rl_status fp8rl_debug_e2m1_encode(const float* in, uint8_t* out, int64_t n, fp8rl_stream_t stream) {
    if (n < 0) return FP8RL_ERR_INVALID_ARG;
    if (n == 0) return FP8RL_OK;
    if (!in || !out) return FP8RL_ERR_INVALID_ARG;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_debug_e2m1(in, out, n, stream));
}

fp8rl_status fp8rl_debug_encode_check(uint32_t amax_lo, uint32_t amax_hi,
                                      unsigned long long* mismatches, uint32_t* first_bad,
                                      fp8rl_stream_t stream) {
    if (!mismatches || !first_bad || amax_hi > 0x7F80u || amax_lo > amax_hi) return FP8RL_ERR_INVALID_ARG;
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_debug_encode_check(amax_lo, amax_hi, mismatches, first_bad, stream));
}

fp8rl_status fp8rl_debug_wait_timeout(uint64_t timeout_ns, fp8rl_stream_t stream) {
    fp8rl_status e = current_device(nullptr);
    if (e != FP8RL_OK) return e;
    return cuda_status(launch_debug_wait_timeout(timeout_ns, stream));
}

}  // extern "C"
