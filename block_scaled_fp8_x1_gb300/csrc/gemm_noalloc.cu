// gemm_noalloc.cu -- scratch memory for fp8rl_gemm_fwd_decode_noalloc.
//
// Some callers cannot hand the library a workspace: a C or C++ decode loop that links
// only this library and owns no device allocator, or a serving loop that must not
// allocate between decode steps (allocating and freeing device memory can synchronize
// the device and stall the loop).  For them the
// decode-shaped forward GEMM can run on a fixed scratch area that lives in the library
// itself: a file-scope device array, reserved on every GPU that loads the library and
// held until the process exits.
//
// The array keeps whatever the last call left in it, and every call on a device uses the
// same array.  Nothing in it needs clearing (each call's slices write their partial sums
// before its reduction reads them), but calls whose kernels overlap on the GPU (different
// streams, no ordering) race on the array and give wrong results.
#include <mutex>

#include "common.cuh"
#include "gemm.h"

namespace fp8rl {

// FP32 split-K partial tiles: 32 MiB holds 256 partial 128x256 tiles.  The automatic split
// keeps (tiles x slices) within one wave of CTAs, at most one per SM, so the partial sums
// of any decode problem take at most SMs x 128 KiB: 19 MiB on a 152-SM GB300.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_mu;
// Per device: the context the address was looked up in, and the address.  A device reset
// (cudaDeviceReset) makes a new primary context with the module loaded afresh, so the
// address is looked up again whenever the current context's id changes.
unsigned long long g_scratch_ctx[kMaxDev] = {};
void* g_scratch_ptr[kMaxDev] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (CUDA 12+), 0 when it cannot be read.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}
}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device.  Looked up with that device
// current on the first call in each context (the host-side name of the array is only a
// stand-in and must never be passed to a kernel), then served from the cache.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace fp8rl
