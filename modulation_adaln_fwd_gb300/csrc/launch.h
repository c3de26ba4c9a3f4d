// launch.h -- internal interface between the C ABI (api.cpp) and the kernels.
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

namespace adaln {

enum class DType { F32 = 0, BF16 = 1 };

// How rows are grouped into segments: either `nseg` uniform segments of
// `seg_rows` rows (dense [B, N, D]) or explicit packed offsets on the device.
struct Segments {
    int64_t rows = 0;          // total rows
    int64_t nseg = 0;          // number of segments
    int64_t seg_rows = 0;      // dense: rows per segment; ragged: unused
    const int64_t *offsets = nullptr;  // ragged: device offsets [nseg + 1]; dense: nullptr
    // modulation rows: segment k uses row mod_index[k] of [nmod, D] tables (device
    // int32 [nseg]), or row k when mod_index is nullptr (then nmod == nseg)
    const int32_t *mod_index = nullptr;
    int64_t nmod = 0;
};

// Chunking of the rows for the column (parameter-gradient) reductions: the rows
// are cut into chunks of `L` consecutive rows (the last one shorter), whatever
// the segment boundaries; the piece of chunk c that lies in segment k produces
// partial row c + k (one per reduced quantity).
struct Chunking {
    int64_t L = 1;             // rows per chunk
    int64_t nchunks = 0;       // ceil(rows / L)
    int64_t npart = 0;         // partial rows: nchunks + nseg - 1 (0 without rows)
    int ctas = 0;              // CTAs of the pipelined kernel: min(SMs, nchunks)
};

// Device facts the launchers size grids with (queried once per device).
struct DeviceInfo {
    int sms = 0;
    int max_smem_optin = 0;   // shared memory one CTA may opt in to
    int smem_per_sm = 0;      // shared memory of one SM (all its CTAs)
};
cudaError_t device_info(DeviceInfo &out);

// Largest D the kernels support for a dtype.
int64_t max_dim(DType dt);

// Chunk length for `rows` rows (host-side, deterministic for a given SM count).
int64_t choose_chunk_rows(int64_t rows, int sms);

// Gated-residual epilogue fused into the forward: out = r + gate[k] * y, with y
// in fp32 (not rounded to the I/O type first).  out == nullptr: no epilogue.
// With an epilogue the forward's y may be nullptr (then it is not written).
struct GateEpilogue {
    const void *gate = nullptr;
    const void *r = nullptr;
    void *out = nullptr;
};

// Kernel launchers: enqueue on `stream`, return the launch status.  `rms`: the
// RMSNorm statistics (rstd = 1/sqrt(mean_d x^2 + eps), no mean; mean may be
// nullptr); not combined with a gate epilogue.
cudaError_t launch_fwd(DType dt, const void *x, const void *shift, const void *scale, void *y,
                       float *mean, float *rstd, const Segments &seg, int64_t D, float eps,
                       cudaStream_t stream, const GateEpilogue &ge = GateEpilogue(),
                       bool rms = false);
cudaError_t launch_gate(DType dt, const void *r, const void *z, const void *gate, void *out,
                        const Segments &seg, int64_t D, cudaStream_t stream);
// Backward launchers.  Device scratch: `partial` (npart * nq * D floats),
// `cta_status` (ch.ctas ints, one per CTA of the pipelined kernel, cleared by
// that CTA) and `header` (one int, written by the column sums: the OR of the
// status words, non-zero if a bounded wait inside the pipelined kernel gave up;
// the parameter gradients are then NaN).  Nothing is launched when nseg == 0.
// The fused gated chain's backward (dy is then the gradient of out = r + gate * y):
// with `gate` set, d_scale and d_shift are those of y with dy := gate * dout and
// d_gate = sum_n dout * y, which needs `shift` too.
struct BwdGate {
    const void *shift = nullptr;
    const void *gate = nullptr;
    float *d_gate = nullptr;
};
// `rowcoef`: 4 floats per row of scratch, needed (not nullptr) only where
// bwd_ring_fits is false.
cudaError_t launch_bwd(DType dt, const void *x, const float *mean, const float *rstd,
                       const void *scale, const void *dy, void *dx, float *d_scale,
                       float *d_shift, float *partial, int *header, int *cta_status,
                       float *rowcoef, const Segments &seg, const Chunking &ch, int64_t D,
                       cudaStream_t stream, const BwdGate &bg = BwdGate());
cudaError_t launch_gate_bwd(DType dt, const void *dout, const void *z, const void *gate, void *dz,
                            float *d_gate, float *partial, int *header, int *cta_status,
                            const Segments &seg, const Chunking &ch, int64_t D,
                            cudaStream_t stream);

// Pipelined LayerNorm (or RMSNorm, mean == nullptr) backward and gated-residual
// backward for one dtype: launch the ring kernel that writes dx (dz) and the
// chunk partials; the column sums are launched by the caller.
cudaError_t bwd_ring_bf16(const void *x, const float *mean, const float *rstd, const void *scale,
                          const void *dy, void *dx, float *partial, int *status,
                          const Segments &sg, const Chunking &ch, int D, const void *gate,
                          cudaStream_t s);
cudaError_t bwd_ring_f32(const void *x, const float *mean, const float *rstd, const void *scale,
                         const void *dy, void *dx, float *partial, int *status,
                         const Segments &sg, const Chunking &ch, int D, const void *gate,
                         cudaStream_t s);
cudaError_t gate_bwd_ring_bf16(const void *dout, const void *z, const void *gate, void *dz,
                               float *partial, int *status, const Segments &sg,
                               const Chunking &ch, int D, cudaStream_t s);
cudaError_t gate_bwd_ring_f32(const void *dout, const void *z, const void *gate, void *dz,
                              float *partial, int *status, const Segments &sg,
                              const Chunking &ch, int D, cudaStream_t s);

// CTAs of the pipelined backward per SM for rows of D elements (1, or 2-3 for
// narrow rows whose few consumer warps leave a single CTA latency-bound).  The
// chunking of the column reductions is cut for SMs x this many CTAs.  `gate`:
// the gated-residual backward, otherwise the LayerNorm backward.
int bwd_ring_ctas_per_sm(DType dt, int64_t D, bool gate);

// Whether the pipelined backward kernels hold rows of D elements of this dtype
// (two ring slots of a row of x and dy; at most four vectors per consumer thread
// with the column partials in registers, six with the LayerNorm backward's
// partials in tensor memory).  `gate`: the gated-residual backward, which keeps
// four at most.  Wider rows take the wide backward below.
bool bwd_ring_fits(DType dt, int64_t D, bool gate = false);

// Wide rows (wide.cu).  The forward for rows of more than 768 vectors (a CTA
// per row); the backward in two launches (per-row coefficients into `coef`,
// 4 floats per row, then column slabs that write dx and the chunk partials)
// and the gated-residual backward in one (column slabs); the column sums are
// launched by the caller, as for the pipelined kernels.
cudaError_t launch_fwd_wide(DType dt, const void *x, const void *shift, const void *scale,
                            void *y, float *mean, float *rstd, const Segments &sg, int D,
                            float eps, const GateEpilogue &ge, bool rms, cudaStream_t stream);
cudaError_t bwd_wide(DType dt, const void *x, const float *mean, const float *rstd,
                     const void *scale, const void *dy, void *dx, float *partial, int *cta_status,
                     float *coef, const Segments &sg, const Chunking &ch, int D, const void *gate,
                     cudaStream_t s);
cudaError_t gate_bwd_wide(DType dt, const void *dout, const void *z, const void *gate, void *dz,
                          float *partial, int *cta_status, const Segments &sg, const Chunking &ch,
                          int D, cudaStream_t s);
int64_t wide_max_dim();

// The pipelined forward (bf16 whole-vector shapes that fit its ring); sets
// `launched` to false, queueing nothing, for shapes it does not take.
cudaError_t launch_fwd_ring(const void *x, const void *shift, const void *scale, void *y,
                            float *mean, float *rstd, const Segments &sg, int D, float eps,
                            const GateEpilogue &ge, bool rms, const DeviceInfo &di,
                            cudaStream_t stream, bool &launched);

// Non-zero once a bounded wait inside the pipelined forward gave up (reads a
// device word: synchronous).
int pipeline_status();
// The header word of the no-allocation backward's built-in scratch on the
// current device: the status its last launching call wrote (synchronous).
int noalloc_status();

// Process-wide count of kernel launches issued by the library.
void count_launch(uint64_t n = 1);
uint64_t launch_count();

}  // namespace adaln
