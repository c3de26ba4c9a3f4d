// bwd.cu -- AdaLN backward and gated-residual backward (sm_103a).
//
// Both follow the "(d_tile, n_tile)" layout of the "AdaptiveLoad" summary,
// section 2.B, "Paso Atras": a CTA owns a chunk of consecutive rows of one
// segment; each thread is pinned to the same feature columns for every row of
// the chunk and accumulates the parameter-gradient partials "vertically" in
// registers, so each warp load is 512 contiguous bytes of one row.  A chunk
// writes one fp32 partial row per reduced quantity; a second kernel sums the
// partials of each segment in a fixed order (no floating-point atomics), so
// the results are bitwise reproducible.
//
// adaln_bwd additionally needs two row reductions for dx,
//     dx = rstd * (g - mean_d(g) - xhat * mean_d(g * xhat)),  g = dy * (1 + scale),
// done per tile of R rows: warp shuffles, then one barrier and a fixed-order
// sum over the warps.  x and dy are read from HBM once; dx is written once.
//
// This file holds the host side, the column sums and the launchers; the
// pipelined kernels live in bwd_ring.cuh, instantiated per dtype in
// bwd_bf16.cu and bwd_f32.cu; rows too wide for their ring go to the
// column-slab kernels of wide.cu, which fill the same partials.
#include "common.cuh"
#include "launch.h"

#include <atomic>
#include <mutex>

namespace adaln {

// ------------------------------------------------------------------ host helpers

namespace {
std::atomic<uint64_t> g_launches{0};
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_info_ok[kMaxDevices];
std::mutex g_info_mu;
}  // namespace

void count_launch(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

cudaError_t device_info(DeviceInfo &out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_info_mu);
    if (!g_info_ok[dev]) {
        DeviceInfo di;
        err = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                     dev);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&di.smem_per_sm,
                                     cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (err != cudaSuccess) return err;
        g_info[dev] = di;
        g_info_ok[dev] = true;
    }
    out = g_info[dev];
    return cudaSuccess;
}

namespace {
constexpr int64_t kMaxChunkRows = 4096;
}  // namespace

// Rows are cut into chunks of L consecutive rows regardless of segment
// boundaries, about one chunk per CTA of the pipelined kernel (a whole number
// of chunks per CTA when rows exceed ctas * kMaxChunkRows), so a static
// round-robin over the persistent CTAs is balanced whatever the segment lengths.
int64_t choose_chunk_rows(int64_t rows, int ctas) {
    const int64_t n = ctas > 0 ? ctas : 1;
    if (rows <= 0) return 1;
    const int64_t waves = (rows + n * kMaxChunkRows - 1) / (n * kMaxChunkRows);
    return (rows + n * waves - 1) / (n * waves);
}

namespace {

// ------------------------------------------------------------------ column sums
// out_q[m][d] = sum, over the segments k whose modulation row is m (k = m
// without an index; in ascending k with one) and over the chunks c that hold
// rows of segment k (in chunk order), of partial[c + k][q][d].  Lane = column
// (32 columns per CTA).  Two mappings, chosen per call, each a fixed order, so
// results are reproducible:
//   per-row (rows spanning many chunks): CTA = (modulation row, column block);
//     warp w sums chunks w, w+8, ... of each segment (eight loads in flight),
//     then the eight warp sums are added in warp order;
//   per-warp (many rows of a few chunks each, e.g. the buckets of short
//     sequences): CTA = (eight modulation rows, column block); warp w takes row
//     8 b + w alone and sums its chunks in order, eight loads in flight.
// The CTAs also fold the status words of the pipelined kernel: any non-zero
// word turns the outputs into NaN, and CTA 0 writes their OR to the workspace
// header.  Gated chain (out2 != nullptr, NQ = 2): the sums are A = sum dout *
// xhat and B = sum dout, and the outputs are d_scale = gate * A, d_shift =
// gate * B and d_gate = (1 + scale) * A + shift * B (d_gate = sum dout * y
// with y = xhat * (1 + scale) + shift).
template <int NQ, typename T>
__global__ void __launch_bounds__(256)
    colsum_kernel(const float *__restrict__ partial, float *__restrict__ out0,
                  float *__restrict__ out1, int D, int64_t nseg, int64_t nmod, int64_t ncb,
                  int64_t L, int64_t nchunks, int64_t seg_rows,
                  const int64_t *__restrict__ offsets, const int32_t *__restrict__ mod_index,
                  const int *__restrict__ cta_status, int nctas, int *__restrict__ header,
                  float *__restrict__ out2, const T *__restrict__ shift,
                  const T *__restrict__ scale, const T *__restrict__ gate, bool per_warp) {
    __shared__ float sm[8][NQ][32];
    __shared__ int s_code;
    if (threadIdx.x == 0) s_code = 0;
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t blk = div_nonneg(blockIdx.x, ncb);
    const int64_t cb = blockIdx.x - blk * ncb;
    const int col = (int)(cb * 32) + lane;
    // this warp's modulation row and its share of each segment's chunks
    const int64_t mrow = per_warp ? blk * 8 + warp : blk;
    const int64_t first = per_warp ? 0 : warp;    // first chunk offset
    const int64_t stride = per_warp ? 1 : 8;      // between a warp's chunks
    int code = 0;
    for (int i = threadIdx.x; i < nctas; i += blockDim.x) code |= cta_status[i];
    float acc[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) acc[q] = 0.f;
    // the segments of this modulation row: k = mrow alone, or every k with
    // mod_index[k] == mrow (the same test across the warp: no divergence)
    const bool live = mrow < nmod;
    const int64_t k_begin = mod_index ? 0 : mrow;
    const int64_t k_end = !live ? k_begin : mod_index ? nseg : (mrow < nseg ? mrow + 1 : mrow);
    for (int64_t seg = k_begin; seg < k_end; ++seg) {
        if (mod_index && __ldg(mod_index + seg) != mrow) continue;
        int64_t s0, s1;
        if (offsets == nullptr) {
            s0 = seg * seg_rows;
            s1 = s0 + seg_rows;
        } else {
            s0 = __ldg(offsets + seg);
            s1 = __ldg(offsets + seg + 1);
        }
        int64_t c0 = 0, c1 = 0;
        if (s1 > s0 && s0 >= 0) {
            c0 = div_nonneg(s0, L);
            c1 = div_nonneg(s1 - 1, L) + 1;
        }
        c1 = min(c1, nchunks);  // never read past the partials, even if offsets were inconsistent
        if (col < D) {
            const float *base = partial + seg * NQ * (int64_t)D + col;  // row c + seg
            // eight chunks of this warp in flight per iteration (chunks past the end
            // read as 0, which leaves the ascending-order sum unchanged)
            for (int64_t cc = c0 + first; cc < c1; cc += 8 * stride) {
                float p[8][NQ];
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int q = 0; q < NQ; ++q)
                        p[u][q] = cc + stride * u < c1
                                      ? __ldg(base + ((cc + stride * u) * NQ + q) * D)
                                      : 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int q = 0; q < NQ; ++q) acc[q] += p[u][q];
            }
        }
    }
    if (!per_warp) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) sm[warp][q][lane] = acc[q];
    }
    __syncthreads();  // s_code is initialised
    if (code) atomicOr(&s_code, code);
    __syncthreads();
    const int bad = s_code;
    if (blockIdx.x == 0 && threadIdx.x == 0) *header = bad;
    if ((per_warp || warp == 0) && live && col < D) {
        float t[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            t[q] = acc[q];
            if (!per_warp) {
                t[q] = sm[0][q][lane];
                for (int w = 1; w < 8; ++w) t[q] += sm[w][q][lane];
            }
            if (bad) t[q] = __int_as_float(0x7fffffff);
        }
        if (NQ == 2 && out2 != nullptr) {
            const int64_t m = mrow * D + col;
            const float g = to_f32(gate[m]), s1 = 1.0f + to_f32(scale[m]), b = to_f32(shift[m]);
            out0[m] = g * t[0];
            out1[m] = g * t[NQ - 1];
            out2[m] = fmaf(s1, t[0], b * t[NQ - 1]);
        } else {
#pragma unroll
            for (int q = 0; q < NQ; ++q) (q == 0 ? out0 : out1)[mrow * D + col] = t[q];
        }
    }
}

template <int NQ, typename T>
cudaError_t colsum(const float *partial, float *o0, float *o1, const Segments &sg,
                   const Chunking &ch, int D, const int *cta_status, int *header,
                   const void *scale, const BwdGate &bg, cudaStream_t s) {
    const int64_t ncb = (D + 31) / 32;
    // a warp per modulation row where rows average at most eight chunk pieces (one
    // round of loads per warp; the segments hold chunks + segments - 1 pieces in
    // all), else a CTA per row
    const bool per_warp = sg.nmod >= 8 && ch.nchunks + sg.nseg <= 8 * sg.nmod;
    const int64_t blocks = per_warp ? (sg.nmod + 7) / 8 : sg.nmod;
    const cudaError_t err = launch_pdl(
        colsum_kernel<NQ, T>, dim3((unsigned)(blocks * ncb)), dim3(256), 0, s, partial, o0, o1, D,
        sg.nseg, sg.nmod, ncb, ch.L, ch.nchunks, sg.seg_rows, sg.offsets, sg.mod_index,
        (const int *)cta_status, ch.nchunks > 0 ? ch.ctas : 0, header, bg.d_gate,
        (const T *)bg.shift, (const T *)scale, (const T *)bg.gate, per_warp);
    count_launch();
    return err;
}

}  // namespace

// Two launches: the pipelined kernel (each CTA clears its own status word), then
// the column sums, which also write the workspace header word.
cudaError_t launch_bwd(DType dt, const void *x, const float *mean, const float *rstd,
                       const void *scale, const void *dy, void *dx, float *d_scale,
                       float *d_shift, float *partial, int *header, int *cta_status,
                       float *rowcoef, const Segments &sg, const Chunking &ch, int64_t D64,
                       cudaStream_t stream, const BwdGate &bg) {
    const int D = (int)D64;
    if (sg.nmod == 0) return cudaSuccess;  // no parameter gradients to write
    const bool bf = dt == DType::BF16;
    if (ch.nchunks > 0 && !bwd_ring_fits(dt, D)) {
        const cudaError_t err = bwd_wide(dt, x, mean, rstd, scale, dy, dx, partial, cta_status,
                                         rowcoef, sg, ch, D, bg.gate, stream);
        if (err != cudaSuccess) return err;
    } else if (ch.nchunks > 0) {
        const cudaError_t err =
            bf ? bwd_ring_bf16(x, mean, rstd, scale, dy, dx, partial, cta_status, sg, ch, D,
                               bg.gate, stream)
               : bwd_ring_f32(x, mean, rstd, scale, dy, dx, partial, cta_status, sg, ch, D,
                              bg.gate, stream);
        if (err != cudaSuccess) return err;
    }
    return bf ? colsum<2, __nv_bfloat16>(partial, d_scale, d_shift, sg, ch, D, cta_status, header,
                                         scale, bg, stream)
              : colsum<2, float>(partial, d_scale, d_shift, sg, ch, D, cta_status, header, scale,
                                 bg, stream);
}

cudaError_t launch_gate_bwd(DType dt, const void *dout, const void *z, const void *gate, void *dz,
                            float *d_gate, float *partial, int *header, int *cta_status,
                            const Segments &sg, const Chunking &ch, int64_t D64,
                            cudaStream_t stream) {
    const int D = (int)D64;
    if (sg.nmod == 0) return cudaSuccess;  // no parameter gradients to write
    if (ch.nchunks > 0 && !bwd_ring_fits(dt, D, true)) {
        const cudaError_t err = gate_bwd_wide(dt, dout, z, gate, dz, partial, cta_status, sg, ch,
                                              D, stream);
        if (err != cudaSuccess) return err;
    } else if (ch.nchunks > 0) {
        const cudaError_t err =
            dt == DType::BF16 ? gate_bwd_ring_bf16(dout, z, gate, dz, partial, cta_status, sg, ch,
                                                   D, stream)
                              : gate_bwd_ring_f32(dout, z, gate, dz, partial, cta_status, sg, ch,
                                                  D, stream);
        if (err != cudaSuccess) return err;
    }
    return colsum<1, float>(partial, d_gate, nullptr, sg, ch, D, cta_status, header, nullptr,
                            BwdGate(), stream);
}

}  // namespace adaln
