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
// name as a device address: the address is looked up with cudaGetSymbolAddress
// (with the device current) and remembered per device together with the
// identity of the context it was looked up in.  A call made in another context
// of that device (after cudaDeviceReset, say, which destroys the context the
// array lived in) looks the address up again instead of using a stale one.
#include "adaln.h"
#include "launch.h"

#include <cuda.h>  // CUcontext / CUresult types only: the driver is reached through the runtime

#include <mutex>

namespace {

// Largest workspace the built-in scratch can stand in for (16 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct Slot {
    void *ptr = nullptr;
    unsigned long long ctx = 0;  // unique id of the context ptr belongs to
};

std::mutex g_mu;
Slot g_slot[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_get_current = nullptr;
CtxGetIdFn g_get_id = nullptr;

// Unique id of the calling thread's current context (0: none is current yet).
// The two driver calls are taken from the runtime's entry-point table, so the
// library needs no link against the driver library.  Called with g_mu held.
cudaError_t current_context_id(unsigned long long *id) {
    if (g_get_current == nullptr || g_get_id == nullptr) {
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        cudaError_t err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000,
                                                           cudaEnableDefault, &q1);
        if (err != cudaSuccess || q1 != cudaDriverEntryPointSuccess || f1 == nullptr)
            return err != cudaSuccess ? err : cudaErrorNotSupported;
        err = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
        if (err != cudaSuccess || q2 != cudaDriverEntryPointSuccess || f2 == nullptr)
            return err != cudaSuccess ? err : cudaErrorNotSupported;
        g_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
        g_get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    CUcontext ctx = nullptr;
    if (g_get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
    *id = 0;
    if (ctx != nullptr && g_get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorUnknown;
    return cudaSuccess;
}

// Device address of the scratch array in the current device's current context:
// the remembered one if it was looked up in this same context, else looked up now.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long ctx = 0;
    err = current_context_id(&ctx);
    if (err != cudaSuccess) return err;
    Slot &s = g_slot[dev];
    if (s.ptr == nullptr || ctx == 0 || s.ctx != ctx) {
        // set-up: also makes the device's context current if it was not yet
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        err = current_context_id(&ctx);
        if (err != cudaSuccess) return err;
        s.ptr = p;
        s.ctx = ctx;
    }
    *out = s.ptr;
    return cudaSuccess;
}

}  // namespace

namespace adaln {

// First word of the scratch: the status the last adaln_bwd_noalloc call on this
// device wrote (its workspace header).  Synchronous; -1 if the read fails.
int noalloc_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_noalloc_scratch, sizeof(int)) != cudaSuccess) return -1;
    return v;
}

}  // namespace adaln

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
