// noalloc.cu -- a backward entry point that needs no caller-provided scratch.
//
// adaln_bwd needs a device workspace for its per-chunk column partials and its
// status word.  Some callers cannot allocate one: a plugin running inside a
// host framework that owns every byte of device memory and offers no
// allocation hook, or a latency-critical path that must not call cudaMalloc
// (it can synchronise the device and stall other streams).  For them this file
// keeps one fixed scratch buffer in the library's own device memory and runs
// the regular backward on it.
//
// The buffer is a file-scope __device__ array, so every GPU that loads this
// library holds it until the process exits.  Host code cannot use the array's
// name as a device address; the address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.
#include "adaln.h"

#include <mutex>

namespace {

// Largest workspace the built-in scratch can stand in for (16 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_ptr[kMaxDevices];

// Device address of the scratch array on the current device (set up on first use).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_ptr[dev] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_ptr[dev] = p;
    }
    *out = g_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" size_t adaln_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" adaln_status adaln_bwd_noalloc(const void *x, const float *mean, const float *rstd,
                                          const void *scale, const void *dy, void *dx,
                                          float *d_scale, float *d_shift, int64_t B, int64_t N,
                                          int64_t D, adaln_dtype dtype, cudaStream_t stream) {
    // the size query validates B, N, D and dtype (0 means invalid) and needs no allocation
    const size_t need = adaln_bwd_workspace_size(B, N, D, dtype);
    if (need == 0) return ADALN_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes) return ADALN_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return ADALN_ERR_CUDA;
    // the regular backward clears the status word and overwrites every partial it reads
    return adaln_bwd(x, mean, rstd, scale, dy, dx, d_scale, d_shift, scratch,
                     kNoAllocScratchBytes, B, N, D, dtype, stream);
}
