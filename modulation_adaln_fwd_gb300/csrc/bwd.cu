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
        g_info[dev] = di;
        g_info_ok[dev] = true;
    }
    out = g_info[dev];
    return cudaSuccess;
}

namespace {
constexpr int kTile = 4;           // chunk lengths are multiples of this (and of every row tile)
constexpr int kMaxThreads = 640;   // CTA size cap of the backward kernels (<= 102 registers)
constexpr int kChunkWaves = 4;     // target chunks ~ kChunkWaves CTAs per SM
constexpr int64_t kMaxChunkRows = 1024;
}  // namespace

int64_t choose_chunk_rows(int64_t rows, int64_t nseg, int sms) {
    (void)nseg;
    const int64_t target = (int64_t)(sms > 0 ? sms : 1) * kChunkWaves;
    int64_t L = (rows + target - 1) / target;
    L = (L + kTile - 1) / kTile * kTile;
    if (L < kTile) L = kTile;
    if (L > kMaxChunkRows) L = kMaxChunkRows;
    return L;
}

int64_t count_chunks(const int64_t *offsets_host, int64_t nseg, int64_t seg_rows, int64_t L) {
    if (!offsets_host) return nseg * ((seg_rows + L - 1) / L);
    int64_t n = 0;
    for (int64_t k = 0; k < nseg; ++k) n += (offsets_host[k + 1] - offsets_host[k] + L - 1) / L;
    return n;
}

namespace {

// ------------------------------------------------------------------ chunk map

struct ChunkRange {
    int64_t seg, row0, row1;
};

__device__ __forceinline__ ChunkRange chunk_range(int64_t c, int64_t rows, int64_t seg_rows,
                                                  const int64_t *__restrict__ offsets,
                                                  int64_t nseg, int64_t L, int64_t cps,
                                                  const int64_t *__restrict__ prefix) {
    ChunkRange cr;
    if (offsets == nullptr) {
        cr.seg = c / cps;
        const int64_t j = c - cr.seg * cps;
        const int64_t s0 = cr.seg * seg_rows;
        cr.row0 = s0 + j * L;
        cr.row1 = min(cr.row0 + L, s0 + seg_rows);
    } else {
        cr.seg = find_segment(prefix, nseg, c);
        const int64_t j = c - __ldg(prefix + cr.seg);
        const int64_t s1 = min(__ldg(offsets + cr.seg + 1), rows);
        cr.row0 = __ldg(offsets + cr.seg) + j * L;
        cr.row1 = min(cr.row0 + L, s1);
    }
    if (cr.row0 < 0) cr.row0 = 0;
    if (cr.row1 > rows) cr.row1 = rows;
    return cr;
}

// prefix[k] = number of chunks of segments 0..k-1 (one CTA, block-wide scan)
__global__ void __launch_bounds__(1024)
    chunk_prefix_kernel(const int64_t *__restrict__ offsets, int64_t nseg, int64_t L,
                        int64_t *__restrict__ prefix) {
    __shared__ int64_t part[1024];
    const int t = threadIdx.x;
    const int64_t per = (nseg + blockDim.x - 1) / blockDim.x;
    const int64_t k0 = min((int64_t)t * per, nseg), k1 = min(k0 + per, nseg);
    int64_t s = 0;
    for (int64_t k = k0; k < k1; ++k) {
        const int64_t len = offsets[k + 1] - offsets[k];
        s += len > 0 ? (len + L - 1) / L : 0;
    }
    part[t] = s;
    __syncthreads();
    if (t == 0) {  // serial scan over the per-thread totals (nthreads values)
        int64_t run = 0;
        for (int i = 0; i < (int)blockDim.x; ++i) {
            const int64_t v = part[i];
            part[i] = run;
            run += v;
        }
    }
    __syncthreads();
    int64_t run = part[t];
    for (int64_t k = k0; k < k1; ++k) {
        prefix[k] = run;
        const int64_t len = offsets[k + 1] - offsets[k];
        run += len > 0 ? (len + L - 1) / L : 0;
    }
    if (k1 == nseg && k0 < k1) prefix[nseg] = run;
    if (nseg == 0 && t == 0) prefix[0] = 0;
}

// ------------------------------------------------------------------ bwd main

template <int NV>
__device__ __forceinline__ void warp_allreduce(float (&v)[NV]) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], off);
}

template <typename T, int K, int R>
__global__ void __launch_bounds__(kMaxThreads)
    adaln_bwd_kernel(const T *__restrict__ x, const float *__restrict__ mean,
                     const float *__restrict__ rstd, const T *__restrict__ scale,
                     const T *__restrict__ dy, T *__restrict__ dx, float *__restrict__ partial,
                     int64_t rows, int D, int64_t seg_rows, const int64_t *__restrict__ offsets,
                     int64_t nseg, int64_t L, int64_t cps, const int64_t *__restrict__ prefix) {
    constexpr int VEC = IO<T>::VEC;
    __shared__ float red[2][kMaxThreads / 32][2 * R];
    const int V = D / VEC;
    const int nthr = blockDim.x;
    const int nwarps = nthr >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = blockIdx.x;
    const ChunkRange cr = chunk_range(c, rows, seg_rows, offsets, nseg, L, cps, prefix);
    const float invD = 1.0f / (float)D;

    float s1[K][VEC], acc_s[K][VEC], acc_b[K][VEC];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int v = threadIdx.x + k * nthr;
        if (v < V) {
            IO<T>::unpack(ld_cached(scale + cr.seg * D + (int64_t)v * VEC), s1[k]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) s1[k][e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            s1[k][e] = 1.0f + s1[k][e];
            acc_s[k][e] = 0.f;
            acc_b[k][e] = 0.f;
        }
    }

    int buf = 0;
    for (int64_t r0 = cr.row0; r0 < cr.row1; r0 += R) {
        const int nr = (int)min((int64_t)R, cr.row1 - r0);
        V16 xv[R][K], gv[R][K];
        float mu[R], rs[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            mu[r] = 0.f;
            rs[r] = 0.f;
            if (r < nr) {
                mu[r] = __ldg(mean + r0 + r);
                rs[r] = __ldg(rstd + r0 + r);
            }
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int v = threadIdx.x + k * nthr;
                if (r < nr && v < V) {
                    const int64_t o = (r0 + r) * (int64_t)D + (int64_t)v * VEC;
                    xv[r][k] = ld_stream(x + o);
                    gv[r][k] = ld_stream(dy + o);
                } else {
                    xv[r][k] = V16{{0u, 0u, 0u, 0u}};
                    gv[r][k] = V16{{0u, 0u, 0u, 0u}};
                }
            }
        }
        // pass 1: row partial sums and column accumulation (zero rows add nothing)
        float red_v[2 * R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float pg = 0.f, pgx = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                float xf[VEC], gf[VEC];
                IO<T>::unpack(xv[r][k], xf);
                IO<T>::unpack(gv[r][k], gf);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float xh = (xf[e] - mu[r]) * rs[r];
                    const float g = gf[e] * s1[k][e];
                    pg += g;
                    pgx = fmaf(g, xh, pgx);
                    acc_s[k][e] = fmaf(gf[e], xh, acc_s[k][e]);
                    acc_b[k][e] += gf[e];
                }
            }
            red_v[2 * r] = pg;
            red_v[2 * r + 1] = pgx;
        }
        warp_allreduce<2 * R>(red_v);
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < 2 * R; ++i) red[buf][warp][i] = red_v[i];
        }
        __syncthreads();
        float tot[2 * R];
#pragma unroll
        for (int i = 0; i < 2 * R; ++i) tot[i] = 0.f;
        for (int w = 0; w < nwarps; ++w) {
#pragma unroll
            for (int i = 0; i < 2 * R; ++i) tot[i] += red[buf][w][i];
        }
        buf ^= 1;
        // pass 2: dx
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < nr) {
                const float mg = tot[2 * r] * invD;
                const float mgx = tot[2 * r + 1] * invD;
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int v = threadIdx.x + k * nthr;
                    if (v < V) {
                        float xf[VEC], gf[VEC], o[VEC];
                        IO<T>::unpack(xv[r][k], xf);
                        IO<T>::unpack(gv[r][k], gf);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const float xh = (xf[e] - mu[r]) * rs[r];
                            const float g = gf[e] * s1[k][e];
                            o[e] = rs[r] * (g - mg - xh * mgx);
                        }
                        st_vec(dx + (r0 + r) * (int64_t)D + (int64_t)v * VEC, IO<T>::pack(o));
                    }
                }
            }
        }
    }
    // chunk partials: [c][0][:] = sum dy*xhat, [c][1][:] = sum dy
    float *p0 = partial + (c * 2 + 0) * (int64_t)D;
    float *p1 = partial + (c * 2 + 1) * (int64_t)D;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int v = threadIdx.x + k * nthr;
        if (v < V) {
#pragma unroll
            for (int e = 0; e < VEC; e += 4) {
                *reinterpret_cast<float4 *>(p0 + v * VEC + e) =
                    make_float4(acc_s[k][e], acc_s[k][e + 1], acc_s[k][e + 2], acc_s[k][e + 3]);
                *reinterpret_cast<float4 *>(p1 + v * VEC + e) =
                    make_float4(acc_b[k][e], acc_b[k][e + 1], acc_b[k][e + 2], acc_b[k][e + 3]);
            }
        }
    }
}

// ------------------------------------------------------------------ gate bwd main
// dz = gate * dout; partial d_gate = sum over the chunk of dout * z.
template <typename T, int K, int U>
__global__ void __launch_bounds__(kMaxThreads)
    gate_bwd_kernel(const T *__restrict__ dout, const T *__restrict__ z,
                    const T *__restrict__ gate, T *__restrict__ dz, float *__restrict__ partial,
                    int64_t rows, int D, int64_t seg_rows, const int64_t *__restrict__ offsets,
                    int64_t nseg, int64_t L, int64_t cps, const int64_t *__restrict__ prefix) {
    constexpr int VEC = IO<T>::VEC;
    const int V = D / VEC;
    const int nthr = blockDim.x;
    const int64_t c = blockIdx.x;
    const ChunkRange cr = chunk_range(c, rows, seg_rows, offsets, nseg, L, cps, prefix);

    float gk[K][VEC], acc[K][VEC];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int v = threadIdx.x + k * nthr;
        if (v < V) {
            IO<T>::unpack(ld_cached(gate + cr.seg * D + (int64_t)v * VEC), gk[k]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) gk[k][e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[k][e] = 0.f;
    }
    for (int64_t r0 = cr.row0; r0 < cr.row1; r0 += U) {
        const int nr = (int)min((int64_t)U, cr.row1 - r0);
        V16 dv[U][K], zv[U][K];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int v = threadIdx.x + k * nthr;
                if (u < nr && v < V) {
                    const int64_t o = (r0 + u) * (int64_t)D + (int64_t)v * VEC;
                    dv[u][k] = ld_stream(dout + o);
                    zv[u][k] = ld_stream(z + o);
                } else {
                    dv[u][k] = V16{{0u, 0u, 0u, 0u}};
                    zv[u][k] = V16{{0u, 0u, 0u, 0u}};
                }
            }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int v = threadIdx.x + k * nthr;
                float df[VEC], zf[VEC], o[VEC];
                IO<T>::unpack(dv[u][k], df);
                IO<T>::unpack(zv[u][k], zf);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    o[e] = gk[k][e] * df[e];
                    acc[k][e] = fmaf(df[e], zf[e], acc[k][e]);
                }
                if (u < nr && v < V)
                    st_vec(dz + (r0 + u) * (int64_t)D + (int64_t)v * VEC, IO<T>::pack(o));
            }
    }
    float *p0 = partial + c * (int64_t)D;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int v = threadIdx.x + k * nthr;
        if (v < V) {
#pragma unroll
            for (int e = 0; e < VEC; e += 4)
                *reinterpret_cast<float4 *>(p0 + v * VEC + e) =
                    make_float4(acc[k][e], acc[k][e + 1], acc[k][e + 2], acc[k][e + 3]);
        }
    }
}

// ------------------------------------------------------------------ column sums
// out_q[seg][d] = sum over the chunks of seg, in chunk order, of partial[c][q][d].
// CTA = (segment, 128-column block); warp w sums chunks w, w+8, ...; the eight
// warp sums are then added in warp order.
template <int NQ>
__global__ void __launch_bounds__(256)
    colsum_kernel(const float *__restrict__ partial, float *__restrict__ out0,
                  float *__restrict__ out1, int D, int64_t nseg, int64_t ncb, int64_t nchunks,
                  int64_t cps, const int64_t *__restrict__ offsets,
                  const int64_t *__restrict__ prefix) {
    __shared__ float4 sm[8][NQ][32];
    const int64_t seg = blockIdx.x / ncb;
    const int64_t cb = blockIdx.x - seg * ncb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = (int)(cb * 128) + lane * 4;
    int64_t c0, c1;
    if (offsets == nullptr) {
        c0 = seg * cps;
        c1 = c0 + cps;
    } else {
        c0 = __ldg(prefix + seg);
        c1 = __ldg(prefix + seg + 1);
    }
    c1 = min(c1, nchunks);  // never read past the partials, even if offsets were inconsistent
    c0 = max(c0, (int64_t)0);
    float4 acc[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < D) {
        for (int64_t cc = c0 + warp; cc < c1; cc += 8) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4 p =
                    __ldg(reinterpret_cast<const float4 *>(partial + (cc * NQ + q) * D + col));
                acc[q].x += p.x;
                acc[q].y += p.y;
                acc[q].z += p.z;
                acc[q].w += p.w;
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) sm[warp][q][lane] = acc[q];
    __syncthreads();
    if (warp == 0 && col < D) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            float4 s = sm[0][q][lane];
            for (int w = 1; w < 8; ++w) {
                const float4 p = sm[w][q][lane];
                s.x += p.x;
                s.y += p.y;
                s.z += p.z;
                s.w += p.w;
            }
            float *o = (q == 0 ? out0 : out1) + seg * D + col;
            *reinterpret_cast<float4 *>(o) = s;
        }
    }
}

// ------------------------------------------------------------------ dispatch

// Threads per CTA and vectors per thread for V 16-byte vectors per row: the
// fewest vectors per thread (K <= 4) with at most 1024 threads, threads a
// multiple of 32 and as few idle slots as possible.
void pick_threads(int V, int &threads, int &K) {
    int best_t = 0, best_k = 0, best_waste = 1 << 30;
    for (int k = 1; k <= 4; ++k) {
        int t = (V + k - 1) / k;
        t = (t + 31) / 32 * 32;
        if (t > kMaxThreads) continue;
        if (t < 64) t = 64;
        const int waste = t * k - V;
        // prefer fewer idle slots; among equal, prefer more threads (more loads in flight)
        if (waste < best_waste) {
            best_waste = waste;
            best_t = t;
            best_k = k;
        }
    }
    threads = best_t;
    K = best_k;
}

template <typename T>
cudaError_t bwd_dispatch(const void *x, const float *mean, const float *rstd, const void *scale,
                         const void *dy, void *dx, float *partial, const Segments &sg,
                         const Chunking &ch, int D, cudaStream_t s) {
    constexpr int VEC = IO<T>::VEC;
    int threads, K;
    pick_threads(D / VEC, threads, K);
    if (threads == 0) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)ch.nchunks;
#define ADALN_BWD_CASE(KK)                                                                      \
    case KK:                                                                                    \
        adaln_bwd_kernel<T, KK, (KK == 1 ? 4 : KK == 2 ? 2 : 1)><<<blocks, threads, 0, s>>>(                                     \
            (const T *)x, mean, rstd, (const T *)scale, (const T *)dy, (T *)dx, partial, sg.rows, \
            D, sg.seg_rows, sg.offsets, sg.nseg, ch.L, ch.cps, ch.prefix);                       \
        break;
    switch (K) {
        ADALN_BWD_CASE(1)
        ADALN_BWD_CASE(2)
        ADALN_BWD_CASE(3)
        ADALN_BWD_CASE(4)
        default:
            return cudaErrorInvalidValue;
    }
#undef ADALN_BWD_CASE
    count_launch();
    return cudaGetLastError();
}

template <typename T>
cudaError_t gate_bwd_dispatch(const void *dout, const void *z, const void *gate, void *dz,
                              float *partial, const Segments &sg, const Chunking &ch, int D,
                              cudaStream_t s) {
    constexpr int VEC = IO<T>::VEC;
    int threads, K;
    pick_threads(D / VEC, threads, K);
    if (threads == 0) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)ch.nchunks;
#define ADALN_GBWD_CASE(KK)                                                                    \
    case KK:                                                                                   \
        gate_bwd_kernel<T, KK, (KK == 1 ? 4 : KK == 2 ? 2 : 1)><<<blocks, threads, 0, s>>>(                                     \
            (const T *)dout, (const T *)z, (const T *)gate, (T *)dz, partial, sg.rows, D,       \
            sg.seg_rows, sg.offsets, sg.nseg, ch.L, ch.cps, ch.prefix);                         \
        break;
    switch (K) {
        ADALN_GBWD_CASE(1)
        ADALN_GBWD_CASE(2)
        ADALN_GBWD_CASE(3)
        ADALN_GBWD_CASE(4)
        default:
            return cudaErrorInvalidValue;
    }
#undef ADALN_GBWD_CASE
    count_launch();
    return cudaGetLastError();
}

template <int NQ>
cudaError_t colsum(const float *partial, float *o0, float *o1, const Segments &sg,
                   const Chunking &ch, int D, cudaStream_t s) {
    if (sg.nseg == 0) return cudaSuccess;
    const int64_t ncb = (D + 127) / 128;
    colsum_kernel<NQ><<<(unsigned)(sg.nseg * ncb), 256, 0, s>>>(
        partial, o0, o1, D, sg.nseg, ncb, ch.nchunks, ch.cps, sg.offsets, ch.prefix);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_prefix(const Segments &sg, const Chunking &ch, cudaStream_t stream) {
    chunk_prefix_kernel<<<1, 1024, 0, stream>>>(sg.offsets, sg.nseg, ch.L, ch.prefix);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_bwd(DType dt, const void *x, const float *mean, const float *rstd,
                       const void *scale, const void *dy, void *dx, float *d_scale,
                       float *d_shift, float *partial, const Segments &sg, const Chunking &ch,
                       int64_t D64, cudaStream_t stream) {
    const int D = (int)D64;
    cudaError_t err = cudaSuccess;
    if (ch.nchunks > 0) {
        err = dt == DType::BF16
                  ? bwd_dispatch<__nv_bfloat16>(x, mean, rstd, scale, dy, dx, partial, sg, ch, D,
                                                stream)
                  : bwd_dispatch<float>(x, mean, rstd, scale, dy, dx, partial, sg, ch, D, stream);
        if (err != cudaSuccess) return err;
    }
    return colsum<2>(partial, d_scale, d_shift, sg, ch, D, stream);
}

cudaError_t launch_gate_bwd(DType dt, const void *dout, const void *z, const void *gate, void *dz,
                            float *d_gate, float *partial, const Segments &sg,
                            const Chunking &ch, int64_t D64, cudaStream_t stream) {
    const int D = (int)D64;
    cudaError_t err = cudaSuccess;
    if (ch.nchunks > 0) {
        err = dt == DType::BF16
                  ? gate_bwd_dispatch<__nv_bfloat16>(dout, z, gate, dz, partial, sg, ch, D, stream)
                  : gate_bwd_dispatch<float>(dout, z, gate, dz, partial, sg, ch, D, stream);
        if (err != cudaSuccess) return err;
    }
    return colsum<1>(partial, d_gate, nullptr, sg, ch, D, stream);
}

}  // namespace adaln
