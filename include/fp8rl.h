/*
 * fp8rl.h -- C ABI of libfp8rl, the GB300 (sm_103a) unified-precision FP8 linear layer.
 *
 * The scheme is the one stated in "Technical summary: Jet-RL" (gist.science, paper
 * 2601.14243), section "Quantization Scheme":
 *   - activations are quantized per 1x128 group,
 *   - weights are quantized per 128x128 block,
 *   - activations saved for the backward pass are stored in FP8 by the preceding (fused)
 *     operator, gradients passed between operators stay BF16,
 *   - DGrad and WGrad run in FP8, WGrad with 1x128 and 128x1 operand quantization.
 * Section "Core architecture" requires the inference (rollout) graph to be a sub-graph of
 * the training forward graph with the same quantization granularity and precision: the
 * same quantizers and GEMM numerics below serve both, including the small-M decode path.
 * Section "Implementation" names fused activation (SiLU-mul) and RMSNorm operators that
 * feed the quantizer; fp8rl_rmsnorm_quant and fp8rl_silu_mul_quant are those operators.
 *
 * Number formats and readings the pages leave open:
 *   - FP8 is OCP E4M3 ("FN": bias 7, max 448, no infinities).
 *   - A group's scale is s = fl32(amax / 448) in IEEE single precision; a group whose amax
 *     is 0 has s = 0 and all codes 0x00.
 *   - code = E4M3 round-to-nearest-even of fl32(x / s) (IEEE single division), saturated
 *     to +-448.  Dequantized value = decode(code) * s.
 *   - GEMMs multiply E4M3 codes exactly, accumulate each 128-long reduction block in FP32
 *     on the tensor cores, promote it into an FP32 accumulator with the product of the two
 *     operands' scales for that block, and round the result to BF16 (nearest even).
 *
 * Layouts (all row-major, element = one byte for codes, 4 bytes for scales, 2 bytes for
 * BF16 which travels as uint16_t bit patterns):
 *   1x128 codes of A[R,C]   : q[R][C]                 scales s[C/128][R]
 *   128x1 codes of X[M,K]   : emitted TRANSPOSED, qT[K][M]   scales sT[M/128][K]
 *                             (this is the 1x128 quantization of X^T along M)
 *   128x128 codes of W[N,K] : q[N][K]                 scales s[N/128][K/128]
 *                             optional transposed copy qT[K][N] uses the same scales.
 *
 * Shape rules: K % 128 == 0 always; N % 128 == 0 for weights and GEMM outputs; M % 128 == 0
 * wherever M is grouped 128x1 (the transposed outputs and WGrad).  M may be any value >= 0
 * elsewhere; M == 0 is a no-op that returns FP8RL_OK.  Other shapes return FP8RL_ERR_SHAPE.
 *
 * Memory and execution: the caller owns every buffer (device memory unless stated).  All
 * device pointers must be 16-byte aligned and every leading dimension a multiple of 16
 * bytes, else FP8RL_ERR_ALIGN.  Every call is asynchronous on the given stream; argument
 * errors are returned synchronously and launch nothing.  Device-side errors (a bounded
 * wait that ran out) are recorded in a per-device status word and returned by
 * fp8rl_check_status.  Inputs must be finite; NaN or Inf inputs give unspecified codes.
 * The library allocates no device memory of its own: split-K partial sums live in the
 * caller's workspace (fp8rl_gemm_workspace_bytes).
 *
 * Threading: the entry points are stateless apart from the status word and a per-device
 * cache of kernel attributes; they may be called from several host threads.  Each call
 * runs on the CUDA device that is current in the calling thread.
 */
#ifndef FP8RL_H
#define FP8RL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported from libfp8rl.so (the library is built with hidden visibility otherwise). */
#if defined(__GNUC__)
#define FP8RL_API __attribute__((visibility("default")))
#else
#define FP8RL_API
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* fp8rl_stream_t;

typedef enum {
    FP8RL_OK = 0,
    FP8RL_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum */
    FP8RL_ERR_SHAPE = 2,              /* a shape rule above is broken */
    FP8RL_ERR_ALIGN = 3,              /* pointer or leading dimension not 16-byte aligned */
    FP8RL_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
    FP8RL_ERR_WORKSPACE = 5,          /* workspace null or smaller than required */
    FP8RL_ERR_CUDA = 6,               /* a CUDA runtime/driver call failed */
    FP8RL_ERR_DEVICE_TIMEOUT = 7,     /* a kernel's bounded wait ran out (device status) */
    FP8RL_ERR_DEVICE_BOUNDS = 8       /* a kernel's own bounds check fired (device status) */
} fp8rl_status;

/* Library version, (major << 16) | minor. */
FP8RL_API int fp8rl_version(void);

/* Human-readable name of a status code (static string, never NULL). */
FP8RL_API const char* fp8rl_status_string(fp8rl_status st);

/* Checks that `device` is a compute-capability 10.3 GPU, makes it current in the calling
 * thread and prepares the kernels for it (function attributes).  Optional: every entry
 * point performs the same check for the current device on first use.  Returns
 * FP8RL_ERR_UNSUPPORTED_DEVICE on any other device, FP8RL_ERR_CUDA if CUDA fails. */
FP8RL_API fp8rl_status fp8rl_init(int device);

/* Upper bound, in nanoseconds, of every spin-wait inside the GEMM kernels (mbarrier waits
 * between the copy, tensor-core and epilogue warps).  When a wait runs out the kernel
 * records FP8RL_ERR_DEVICE_TIMEOUT, drains its own copies and returns.  Default 2e9 ns.
 * Applies to launches made after the call, on every device. */
FP8RL_API void fp8rl_set_wait_timeout_ns(uint64_t ns);

/* Waits for `stream`, then reads and clears the current device's status word.
 * Returns FP8RL_OK or the first device-side error recorded since the last check.
 * FP8RL_ERR_DEVICE_TIMEOUT means that the outputs of the GEMM calls made since the
 * previous check are not valid: a CTA whose wait ran out skips its stores (the split-K
 * reduction writes NaN instead once a timeout is on record). */
FP8RL_API fp8rl_status fp8rl_check_status(fp8rl_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Quantizers ("Quantization Scheme": activations 1x128, weights 128x128, WGrad operands
 * 128x1; the transposed 128x1 output is the layout WGrad consumes).
 * -------------------------------------------------------------------------------------- */

/* Activation quantization, 1x128 groups along K.
 *   x  : BF16 [M][ldx] (first K columns used), ldx >= K
 *   q  : E4M3 [M][K];  s : float [K/128][M]
 *   qT, sT (both NULL or both set; then M % 128 == 0): the 128x1 quantization of the same
 *        x, transposed: qT [K][M], sT [M/128][K].  One read of x feeds both outputs. */
FP8RL_API fp8rl_status fp8rl_quantize_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* q, float* s, uint8_t* qT, float* sT,
                                  fp8rl_stream_t stream);

/* 128x1 quantization along M (WGrad operand), transposed output.
 *   x : BF16 [M][ldx], M % 128 == 0;  qT : E4M3 [K][M];  sT : float [M/128][K] */
FP8RL_API fp8rl_status fp8rl_quantize_128x1(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* qT, float* sT, fp8rl_stream_t stream);

/* 128x1 WGrad operand rebuilt from a saved 1x128 quantization (the memory-saving variant of
 * "Quantization Scheme": the activation saved for the backward pass is its FP8 form).
 *   q : E4M3 [M][K], s : float [K/128][M]  (an fp8rl_quantize_1x128 output)
 *   x^ = bf16_rne( fl32(decode(q) * s) ) is quantized 128x1 along M, transposed:
 *   qT : E4M3 [K][M], sT : float [M/128][K].  M % 128 == 0, K % 128 == 0.
 * The result differs from fp8rl_quantize_128x1 of the original BF16 X by the 1x128
 * rounding error it starts from. */
FP8RL_API fp8rl_status fp8rl_requantize_128x1(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                              uint8_t* qT, float* sT, fp8rl_stream_t stream);

/* Weight quantization, 128x128 blocks (re-run from the BF16 master weights after each
 * optimizer step: "Core architecture", master weights stay BF16).
 *   w : BF16 [N][ldw];  q : E4M3 [N][K];  s : float [N/128][K/128]
 *   qT (nullable): E4M3 [K][N], the transposed copy DGrad reads; same scales. */
FP8RL_API fp8rl_status fp8rl_quantize_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw,
                                    uint8_t* q, float* s, uint8_t* qT,
                                    fp8rl_stream_t stream);

/* Fused RMSNorm -> quantize ("Implementation": fused RMSNorm kernel; "Quantization
 * Scheme": the saved activation is FP8, produced by the preceding operator).
 *   y[m,k] = bf16_rne( (x[m,k] * rstd[m]) * gamma[k] ),
 *   rstd[m] = 1 / sqrt( fl32(sum_k x[m,k]^2 / K) + eps )   (IEEE single sqrt and divide)
 * then y is quantized 1x128 (q [M][K], s [K/128][M]) and, if qT/sT are set, 128x1
 * transposed (qT [K][M], sT [M/128][K]; needs M % 128 == 0).  y itself is not stored.
 *   x : BF16 [M][K] (contiguous);  gamma : BF16 [K];  rstd (nullable): float [M] */
FP8RL_API fp8rl_status fp8rl_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, float eps,
                                 int64_t M, int64_t K, uint8_t* q, float* s, uint8_t* qT,
                                 float* sT, float* rstd, fp8rl_stream_t stream);

/* Fused SiLU-mul -> quantize ("Implementation": fused activation kernel).
 *   gu : BF16 [M][2*I], gate = columns [0, I), up = columns [I, 2I)
 *   h[m,i] = bf16_rne( silu(g) * u ), silu(g) = g / (1 + exp(-g)) evaluated in FP32
 * then h is quantized 1x128 (q [M][I], s [I/128][M]) and, if qT/sT are set, 128x1
 * transposed (qT [I][M], sT [M/128][I]).  I % 128 == 0. */
FP8RL_API fp8rl_status fp8rl_silu_mul_quant(const uint16_t* gu, int64_t M, int64_t I, uint8_t* q,
                                  float* s, uint8_t* qT, float* sT, fp8rl_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Backward operators either side of the gradient quantizer ("Quantization Scheme":
 * gradients between operators stay BF16; DGrad and WGrad consume quantized gradients).
 * -------------------------------------------------------------------------------------- */

/* Fused SiLU-mul backward -> quantize: the gradient of the gate_up output from the forward's
 * gate_up output and the gradient of h (the down projection's DGrad output):
 *   gu : BF16 [M][2*I] (gate = columns [0, I), up = [I, 2I));  dh : BF16 [M][I]
 *   with s = sigmoid(g):  dg = bf16(dh*u*s*(1 + g*(1 - s))),  du = bf16(dh*g*s)
 *   evaluated in FP32; dgu = [dg | du] ([M][2I]) is quantized 1x128 along its 2I columns
 *   (q [M][2I], s [2I/128][M], the DGrad operand) and, if qT/sT are set (M % 128 == 0),
 *   128x1 transposed (qT [2I][M], sT [M/128][2I], the WGrad operand).  dgu itself is not
 *   stored.  I % 128 == 0. */
FP8RL_API fp8rl_status fp8rl_silu_mul_bwd_quant(const uint16_t* gu, const uint16_t* dh, int64_t M,
                                                int64_t I, uint8_t* q, float* s, uint8_t* qT,
                                                float* sT, fp8rl_stream_t stream);

/* RMSNorm backward from the forward's saved rstd (fp8rl_rmsnorm_quant's rstd output):
 *   x : BF16 [M][K];  gamma : BF16 [K];  rstd : float [M];  dy : BF16 [M][K] (the gradient
 *   of the normalised output)
 *   dx[m,j]   = bf16( r*gamma_j*dy_j - r^3*x_j*S/K ),  S = sum_k dy_k*gamma_k*x_k   (FP32)
 *   dgamma[k] = sum_m dy[m,k]*x[m,k]*r_m   (FP32; nullable: then ws is unused)
 * K % 128 == 0 and K <= 8192, else FP8RL_ERR_SHAPE.  dgamma needs
 * fp8rl_rmsnorm_bwd_workspace_bytes(M, K) bytes of workspace (no initial contents); the
 * sums run in a fixed order, so repeated calls give the same bits. */
FP8RL_API fp8rl_status fp8rl_rmsnorm_bwd(const uint16_t* x, const uint16_t* gamma, const float* rstd,
                                         const uint16_t* dy, int64_t M, int64_t K, uint16_t* dx,
                                         float* dgamma, void* ws, size_t ws_bytes,
                                         fp8rl_stream_t stream);
FP8RL_API size_t fp8rl_rmsnorm_bwd_workspace_bytes(int64_t M, int64_t K);

/* ----------------------------------------------------------------------------------------
 * Block-scaled FP8 GEMMs ("Quantization Scheme": forward, DGrad and WGrad in FP8).
 * Output element = bf16_rne( sum_kb sA(kb,row) * sB(kb,col) * sum_{k in kb} a*b ), with
 * the inner block sum in FP32 on the tensor cores and the outer sum in FP32 registers.
 * -------------------------------------------------------------------------------------- */

/* Operation selector for fp8rl_gemm_workspace_bytes and fp8rl_gemm_opts. */
typedef enum { FP8RL_OP_FWD = 0, FP8RL_OP_DGRAD = 1, FP8RL_OP_WGRAD = 2 } fp8rl_gemm_op;

/* Forward Y = X W^T.
 *   qx : E4M3 [M][K] (1x128), sx : float [K/128][M]
 *   qw : E4M3 [N][K] (128x128), sw : float [N/128][K/128]
 *   y  : BF16 [M][N]
 * Small M takes a decode-shaped form.  Up to 64 tokens (and up to 128 when N <= 8192),
 * FP8RL_VARIANT_DECODE: each CTA streams 128 weight rows of one reduction slice, and the
 * slices of a tile are added in rank order inside a cluster (the result does not depend
 * on timing); no workspace.  From 129 to 256 tokens against a weight wide enough that
 * the paired-SM form's 256-row tiles alone cover every pair of SMs, that form (below).
 * Otherwise up to 256 tokens, FP8RL_VARIANT_SPLITK: tokens on the tensor core's M side,
 * the reduction split over CTAs whose FP32 partial sums a second kernel adds in slice
 * order; it needs fp8rl_gemm_workspace_bytes(FP8RL_OP_FWD, M, N, K) bytes of workspace (no
 * initial contents required; calls that overlap in time need separate workspaces).  A
 * size of 0 means ws may be NULL.
 * Larger M takes the paired-SM form (FP8RL_VARIANT_PAIR, 256 x 256 tiles) when every
 * scale array can be moved by TMA -- M % 4 == 0 and (K/128) % 4 == 0 for the forward GEMM,
 * M % 4 == 0 and (K/128) % 4 == 0 on the weight's block-scale rows for DGrad -- and its
 * tiles cover every pair of SMs at least once; otherwise the one-SM tiled form
 * (FP8RL_VARIANT_TILED).  WGrad chooses the same way (its scale arrays always qualify). */
FP8RL_API fp8rl_status fp8rl_gemm_fwd(const uint8_t* qx, const float* sx, const uint8_t* qw,
                            const float* sw, uint16_t* y, int64_t M, int64_t N, int64_t K,
                            void* ws, size_t ws_bytes, fp8rl_stream_t stream);

/* DGrad dX = dY W.
 *   qdy : E4M3 [M][N] (1x128 along N), sdy : float [N/128][M]
 *   qwT : E4M3 [K][N], the transposed weight copy from fp8rl_quantize_128x128
 *   sw  : float [N/128][K/128] (the weight's block scales)
 *   dx  : BF16 [M][K]
 * ws may be NULL (no workspace is used at present). */
FP8RL_API fp8rl_status fp8rl_gemm_dgrad(const uint8_t* qdy, const float* sdy, const uint8_t* qwT,
                              const float* sw, uint16_t* dx, int64_t M, int64_t N,
                              int64_t K, void* ws, size_t ws_bytes, fp8rl_stream_t stream);

/* WGrad dW = dY^T X, both operands quantized 128x1 along the token dimension M.
 *   qdyT : E4M3 [N][M], sdyT : float [M/128][N]   (fp8rl_quantize_128x1 of dY)
 *   qxT  : E4M3 [K][M], sxT  : float [M/128][K]   (128x1 of the saved activation)
 *   dw   : BF16 [N][K];  M % 128 == 0. */
FP8RL_API fp8rl_status fp8rl_gemm_wgrad(const uint8_t* qdyT, const float* sdyT, const uint8_t* qxT,
                              const float* sxT, uint16_t* dw, int64_t M, int64_t N,
                              int64_t K, void* ws, size_t ws_bytes, fp8rl_stream_t stream);

/* Workspace bytes the given GEMM needs with the automatic kernel choice (0 if none). */
FP8RL_API size_t fp8rl_gemm_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);

/* Explicit kernel choice, for tests and benchmarks. */
typedef enum {
    FP8RL_VARIANT_AUTO = 0,   /* what fp8rl_gemm_fwd / _dgrad / _wgrad pick */
    FP8RL_VARIANT_TILED = 1,  /* one SM per output tile: persistent 128 x BN tiles */
    FP8RL_VARIANT_SPLITK = 2, /* decode-shaped: the reduction of each 128x256 output tile
                                 is split over `splits` CTAs (forward only, M <= 256) */
    FP8RL_VARIANT_PAIR = 3,   /* two SMs per output tile: persistent 256 x 256 (or, with
                                 tile_n = 128, 256 x 128) tiles on clusters of two CTAs
                                 (M = 256 tensor-core MMAs); needs
                                 scale arrays whose rows are multiples of 16 bytes (the
                                 rule under fp8rl_gemm_fwd), else FP8RL_ERR_SHAPE */
    FP8RL_VARIANT_DECODE = 4, /* forward only, M <= 256: weights on the MMA's M side (one
                                 CTA per 128 weight rows and reduction slice), the
                                 reduction split over a cluster of `splits` CTAs (1..8, 0 =
                                 choose) and summed in the cluster's shared memory in rank
                                 order; no workspace */
    FP8RL_VARIANT_MULTICAST = 5 /* the TILED form's 128 x 256 tiles on clusters of two CTAs
                                 (vertically adjacent tiles) that share each B tile: every
                                 CTA copies half of it with a TMA multicast into both CTAs;
                                 the same scale-array rule as PAIR (FP8RL_ERR_SHAPE
                                 otherwise); this GPU's memory only */
} fp8rl_variant;

typedef struct {
    int variant;    /* fp8rl_variant */
    int splits;     /* SPLITK: number of reduction slices (0 = choose); ignored otherwise */
    int grid;       /* TILED: persistent CTAs (0 = one per SM); PAIR, MULTICAST: persistent
                       clusters of two (0 = one per two SMs); ignored otherwise */
    int tile_n;     /* TILED: output tile width, 128 or 256 (0 = choose); PAIR: the pair
                       tile's width, 128 or 256 (0 = 256); ignored otherwise */
    int epi_warps;  /* PAIR: epilogue warps per CTA, 8 or 16 (0 = 8); ignored otherwise */
} fp8rl_gemm_opts;

/* Workspace bytes fp8rl_gemm_fwd_ex needs with these options (opts may be NULL = AUTO). */
FP8RL_API size_t fp8rl_gemm_workspace_bytes_ex(int op, int64_t M, int64_t N, int64_t K,
                                     const fp8rl_gemm_opts* opts);

/* fp8rl_gemm_fwd with an explicit variant; opts may be NULL (= AUTO). */
FP8RL_API fp8rl_status fp8rl_gemm_fwd_ex(const uint8_t* qx, const float* sx, const uint8_t* qw,
                               const float* sw, uint16_t* y, int64_t M, int64_t N,
                               int64_t K, void* ws, size_t ws_bytes,
                               const fp8rl_gemm_opts* opts, fp8rl_stream_t stream);

/* fp8rl_gemm_dgrad / fp8rl_gemm_wgrad with an explicit variant (AUTO, TILED, PAIR or
 * MULTICAST);
 * opts may be NULL (= AUTO). */
FP8RL_API fp8rl_status fp8rl_gemm_dgrad_ex(const uint8_t* qdy, const float* sdy, const uint8_t* qwT,
                                 const float* sw, uint16_t* dx, int64_t M, int64_t N,
                                 int64_t K, void* ws, size_t ws_bytes,
                                 const fp8rl_gemm_opts* opts, fp8rl_stream_t stream);
FP8RL_API fp8rl_status fp8rl_gemm_wgrad_ex(const uint8_t* qdyT, const float* sdyT, const uint8_t* qxT,
                                 const float* sxT, uint16_t* dw, int64_t M, int64_t N,
                                 int64_t K, void* ws, size_t ws_bytes,
                                 const fp8rl_gemm_opts* opts, fp8rl_stream_t stream);

/* One linear layer from the BF16 activation ("Core architecture": rollout and the
 * training forward pass run the same FP8 linear): x is quantized 1x128 into qx / sx
 * (exactly fp8rl_quantize_1x128), then Y = X W^T with the form fp8rl_gemm_fwd picks.  In
 * the decode form without a cluster split, the GEMM kernel starts streaming its weights
 * while the quantizer finishes (programmatic dependent launch on the same stream).
 *   x : BF16 [M][ldx];  qw, sw, y, ws as for fp8rl_gemm_fwd;  qx : E4M3 [M][K] and
 *   sx : float [K/128][M] receive the quantized activation (caller-owned). */
FP8RL_API fp8rl_status fp8rl_linear_fwd(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                        const uint8_t* qw, const float* sw, int64_t N,
                                        uint8_t* qx, float* sx, uint16_t* y, void* ws,
                                        size_t ws_bytes, fp8rl_stream_t stream);

/* Decode-shaped forward GEMM that allocates nothing and takes no workspace.  It has no
 * counterpart in the scheme's pages; it exists for callers that cannot provide device
 * memory: a C/C++ decode loop that links only this library and owns no allocator, or a
 * serving loop that must not allocate between decode steps (allocating and freeing
 * device memory can synchronize the device and stall the loop).
 * Same operands, layouts and numerics as fp8rl_gemm_fwd_ex with FP8RL_VARIANT_SPLITK
 * and automatic splits (M <= 256); the result equals it within the GEMM tolerance (the
 * split, and with it the summation order, may differ).  Its split-K partial sums live in
 * a fixed scratch array inside the library,
 * fp8rl_gemm_noalloc_scratch_bytes() bytes (32 MiB) per device, reserved on every GPU
 * that loads the library and held until the process exits.
 *   - The automatic split keeps at most one (tile, slice) pair per SM, so the partial
 *     sums take at most SMs x 128 KiB (19 MiB on a 152-SM GB300); a GPU where they would
 *     not fit gets FP8RL_ERR_WORKSPACE.  M > 256 returns FP8RL_ERR_SHAPE.  Neither
 *     launches anything.
 *   - The first call in each CUDA context of a device looks up the array's device
 *     address (with that device current) and caches it; make that first call before any
 *     stream capture.
 *   - Every call on a device shares the array, which keeps the last call's partial sums
 *     (each call writes its own before reading them, so nothing needs clearing); calls
 *     whose kernels overlap on the GPU race on the array and give wrong results, so order
 *     them on one stream. */
FP8RL_API fp8rl_status fp8rl_gemm_fwd_decode_noalloc(const uint8_t* qx, const float* sx,
                                                     const uint8_t* qw, const float* sw,
                                                     uint16_t* y, int64_t M, int64_t N,
                                                     int64_t K, fp8rl_stream_t stream);

/* Size in bytes of the scratch array fp8rl_gemm_fwd_decode_noalloc uses on each device. */
FP8RL_API size_t fp8rl_gemm_noalloc_scratch_bytes(void);

/* ----------------------------------------------------------------------------------------
 * NVFP4 rollout path.  "QeRL" (chatpaper.ai), abstract: rollout runs with NVFP4-quantized
 * weights.  The page names the format only; the format is FP4 E2M1 elements (0, 0.5, 1,
 * 1.5, 2, 3, 4, 6 and negatives), one E4M3 scale per 16 consecutive elements along K, and
 * an FP32 scale on top, here one per row.  The tensor core's FP4 path multiplies FP4 by
 * FP4, so the activation is quantized to NVFP4 as well, per call.
 *
 * Quantization of a row with maximum |x| = a (IEEE single precision, no FMA):
 *   g = a / 2688;  block of 16 with maximum b: sb = E4M3_rne_satfinite(b / (6 g)) (0 when
 *   g = 0), d = decode(sb) * g;  code = E2M1_rne_satfinite(x / d), 0 when d = 0.
 * Layouts:
 *   q  : [R][K/2] bytes; element k of a row in bits 4(k%2) .. 4(k%2)+3 of byte k/2.
 *   sf : the tensor core's scale-factor layout, fp8rl_nvfp4_scale_bytes(R, K) bytes:
 *        512-byte atoms of 128 rows x 4 scales (64 elements of K); atom (row group rg =
 *        r/128, K-atom ka = k/64) at byte 512 (rg K/64 + ka); inside it the scale of row
 *        r, K-elements 16j .. 16j+15 of the atom, at byte 16 (r%32) + 4 ((r%128)/32) + j.
 *        Rows from R up to the next multiple of 128 hold zeros.
 *   g  : float [R].
 * -------------------------------------------------------------------------------------- */

/* Bytes of the sf buffer of an R x K NVFP4 operand: ceil(R/128) * K/256 * 2048 (0 for
 * R <= 0 or K not a positive multiple of 256). */
FP8RL_API size_t fp8rl_nvfp4_scale_bytes(int64_t R, int64_t K);

/* NVFP4 quantization of the rows of x (BF16 [R][ldx], ldx >= K, ldx % 8 == 0; K % 256 == 0)
 * into q, sf, g (layouts above; caller-owned device memory, 16-byte aligned).  Used for
 * weights (R = N output channels, once per weight update) and activations (R = M tokens,
 * per call).  Errors: FP8RL_ERR_SHAPE (K % 256), FP8RL_ERR_ALIGN, FP8RL_ERR_INVALID_ARG. */
FP8RL_API fp8rl_status fp8rl_quantize_nvfp4(const uint16_t* x, int64_t R, int64_t K, int64_t ldx,
                                            uint8_t* q, uint8_t* sf, float* g, fp8rl_stream_t stream);

/* Decode-shaped NVFP4 GEMM: y[m][n] = bf16_rne(gx[m] gw[n] sum_k x^(m,k) w^(n,k)), x^ and
 * w^ the codes times their block scales, accumulated in FP32 by the tensor core (within
 * the GEMM tolerance of the exact sum).  Operands from fp8rl_quantize_nvfp4: qx / sfx / gx
 * of X [M][K], qw / sfw / gw of W [N][K].  y: BF16 [M][ldy], ldy >= N, ldy % 8 == 0.
 * 1 <= M <= 256, N % 128 == 0, K % 256 == 0.  splits: slices of the reduction, one cluster
 * of CTAs per 128-row weight tile (1..8; 0 = automatic).  No workspace. */
FP8RL_API fp8rl_status fp8rl_gemm_nvfp4(const uint8_t* qx, const uint8_t* sfx, const float* gx,
                                        const uint8_t* qw, const uint8_t* sfw, const float* gw,
                                        uint16_t* y, int64_t M, int64_t N, int64_t K, int64_t ldy,
                                        int splits, fp8rl_stream_t stream);

/* One NVFP4 linear layer from the BF16 activation: x is quantized into qx / sfx / gx
 * (exactly fp8rl_quantize_nvfp4; caller-owned), then y = fp8rl_gemm_nvfp4 with automatic
 * splits.  The GEMM kernel starts streaming its weights while the quantizer finishes
 * (programmatic dependent launch on the same stream) when the reduction is not split. */
FP8RL_API fp8rl_status fp8rl_linear_nvfp4(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                          const uint8_t* qw, const uint8_t* sfw, const float* gw,
                                          int64_t N, uint8_t* qx, uint8_t* sfx, float* gx,
                                          uint16_t* y, fp8rl_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Diagnostics (used by the tests).
 * -------------------------------------------------------------------------------------- */

/* The device's E4M3 encoder (the exact routine the quantizers use) applied to n binary32
 * values: out[i] = E4M3_rne_satfinite(in[i]).  Device pointers. */
FP8RL_API fp8rl_status fp8rl_debug_e4m3_encode(const float* in, uint8_t* out, int64_t n,
                                     fp8rl_stream_t stream);

/* The device's E2M1 encoder (the routine fp8rl_quantize_nvfp4 uses) applied to n binary32
 * values: out[i] = E2M1_rne_satfinite(in[i]) in bits 0-3.  Device pointers. */
FP8RL_API fp8rl_status fp8rl_debug_e2m1_encode(const float* in, uint8_t* out, int64_t n,
                                               fp8rl_stream_t stream);

/* Checks the quantizers' division-free encode against IEEE division on the device: for
 * every BF16 group maximum with bits in [amax_lo, amax_hi) (positive finite: below 0x7F80)
 * and every BF16 x with |x| <= amax, both signs, the code of E4M3(fl32(x / s)) with
 * s = fl32(amax / 448) must equal the production encode.  Adds the number of mismatching
 * pairs to *mismatches and stores the first one as (amax_bits << 16) | |x|_bits into
 * *first_bad if that still holds 0xFFFFFFFF.  Device pointers. */
FP8RL_API fp8rl_status fp8rl_debug_encode_check(uint32_t amax_lo, uint32_t amax_hi,
                                                unsigned long long* mismatches,
                                                uint32_t* first_bad, fp8rl_stream_t stream);

/* Launches one CTA that waits, with the GEMM kernels' bounded wait, on an mbarrier that
 * nothing completes; after `timeout_ns` it records FP8RL_ERR_DEVICE_TIMEOUT and returns.
 * Exercises the failure path without faulting or hanging the GPU. */
FP8RL_API fp8rl_status fp8rl_debug_wait_timeout(uint64_t timeout_ns, fp8rl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8RL_H */
