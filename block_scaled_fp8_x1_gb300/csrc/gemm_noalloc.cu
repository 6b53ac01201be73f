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

// FP32 split-K partial tiles: 32 MiB holds 256 partial 128x256 tiles, which covers the
// automatic split of the 7B and 32B decode shapes up to 256 tokens; a problem that would
// need more runs with a smaller split.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDev] = {};
}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device.  Looked up once per device
// (the first call), with that device current; the host-side name of the array is only a
// stand-in and must never be passed to a kernel.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace fp8rl
