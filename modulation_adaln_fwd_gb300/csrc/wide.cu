// wide.cu -- AdaLN for rows too wide for the single-warp and pipelined kernels
// (up to 16,384 elements): the forward of fp32 rows above 3,072 elements and of
// the bf16 rows above 6,144 that the warp-group forward of fwd_ring.cu does not
// take; the LayerNorm backward of fp32 rows above 8,448 elements (below that the
// pipelined kernels hold the row, with their partials in tensor memory when
// registers do not); the gated-residual backward of bf16 rows above 11,264 and
// fp32 rows above 5,632.
//
// Forward: a CTA of four warps (eight for fp32 rows of more than 8,192
// elements) owns a row and holds it in registers (8 or 16 vectors of 16 bytes
// per thread).  The exact row statistics of fwd_stats.cuh run with the
// CTA-wide merge; the modulation (and the fused gated residual) is then
// applied from the registers.  x is read from HBM once and y written once, as
// in the narrow kernels.
//
// Backward (LayerNorm or RMSNorm, plain or fused gated): the column partials of
// a whole row no longer fit one SM's registers next to the row, so the work is
// cut by columns as well.  A first kernel (a warp per row) reduces each row to
// the three sums the dx formula needs and stores three per-row coefficients.
// A second kernel gives each CTA one chunk of rows and a slab of 256 column
// vectors: it writes dx for those columns and the chunk's column partials, in
// the workspace layout of the pipelined kernels, so that the same column sums
// finish d_scale and d_shift (and d_gate).  x and dy are read twice: 5 D E
// bytes per row instead of 3.
//
// Gated-residual backward: the slab kernel alone (it needs no row reduction),
// with one read of dout and z and one write of dz.
#include "fwd_stats.cuh"

namespace adaln {
namespace {

constexpr int64_t kWideMaxGrid = int64_t(1) << 20;  // forward CTAs; more rows loop
constexpr int kSlabThreads = 256;                   // column vectors per slab

// ------------------------------------------------------------------ forward

// A row per CTA of W warps: thread t holds vectors t, t + 32 W, ... of the row
// (nv of them, at most NVMAX).  GATED / RMS as in the register kernel of
// fwd.cu.  bf16 rows take the packed-pair statistics; the modulation runs on
// packed pairs,
//     y = (x rstd + n) (1 + scale) + shift,  n = -mean rstd,
// except for fp32 rows and rows with |n| > 4 (|mean| >> std), which centre
// first: y = (x - mean) rstd (1 + scale) + shift.  Each row costs the CTA a
// fixed number of merges and barriers, so a thread holds as many vectors as its
// registers allow (fewer warps per row, more rows in flight per SM).
template <typename T, int W, int NVMAX, bool GATED, bool RMS>
__global__ void __launch_bounds__(32 * W, W == 4 ? 4 : 2)
    adaln_fwd_wide_kernel(const T *__restrict__ x, const T *__restrict__ shift,
                          const T *__restrict__ scale, T *__restrict__ y,
                          float *__restrict__ mean, float *__restrict__ rstd, int64_t rows, int D,
                          int nv, float eps, int64_t seg_rows, const int64_t *__restrict__ offsets,
                          int64_t nseg, const int32_t *__restrict__ mod_index,
                          const T *__restrict__ gate, const T *__restrict__ r,
                          T *__restrict__ out) {
    constexpr int VEC = IO<T>::VEC;
    constexpr int NP = Pairs<T>::NP;
    constexpr int NT = 32 * W;
    constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
    __shared__ CtaGroupSmem<W> gsm;
    pdl_wait();
    pdl_trigger();
    const int li = threadIdx.x;
    const int V = D / VEC;
    auto has = [&](int k) { return k < nv && li + k * NT < V; };
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const T *xr = x + row * (int64_t)D;
        V16 xv[NVMAX];
#pragma unroll
        for (int k = 0; k < NVMAX; ++k) {
            if (has(k))
                xv[k] = ld_stream(xr + (int64_t)(li + k * NT) * VEC);
            else
                xv[k] = V16{{0u, 0u, 0u, 0u}};
        }
        float mh, ml, rs;
        auto xreg = [&](int k) -> const V16 & { return xv[k]; };
        // bf16: packed sums (vectors the thread does not own are zero and add nothing)
        row_stats<T, NT, NVMAX, BF, false, !BF, NVMAX, decltype(xreg), BF, RMS, CtaGroup<W>>(
            xreg, li, nv, V, D, eps, mh, ml, rs, CtaGroup<W>(&gsm));
        if (li == 0) {
            if (!RMS) mean[row] = mh;
            rstd[row] = rs;
        }
        const int64_t k_seg =
            mod_row(mod_index, offsets ? find_segment(offsets, nseg, row) : div_nonneg(row, seg_rows));
        const T *shr = shift + k_seg * D;
        const T *scr = scale + k_seg * D;
        const float nh = __fmul_rn(-mh, rs);
        const bool centred = !BF || !(fabsf(nh) <= 4.0f);  // the same in every thread
        const f2 RS = f2_make(rs, rs), NH = f2_make(nh, nh);
        const f2 MH = f2_make(mh, mh), ML = f2_make(ml, ml), ONE = f2_make(1.0f, 1.0f);
        T *yr = y != nullptr ? y + row * (int64_t)D : nullptr;
#pragma unroll
        for (int k = 0; k < NVMAX; ++k) {
            const int v = li + k * NT;
            if (has(k)) {
                f2 xp[NP], sp[NP], bp[NP], o[NP];
                Pairs<T>::unpack(xv[k], xp);
                Pairs<T>::unpack(ld_cached(scr + (int64_t)v * VEC), sp);
                Pairs<T>::unpack(ld_cached(shr + (int64_t)v * VEC), bp);
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    const f2 U = centred ? f2_mul(f2_sub(f2_sub(xp[i], MH), ML), RS)
                                         : f2_fma(xp[i], RS, NH);
                    o[i] = f2_fma(U, f2_add(ONE, sp[i]), bp[i]);
                }
                if (yr != nullptr) st_vec(yr + (int64_t)v * VEC, Pairs<T>::pack(o));
                if constexpr (GATED) {
                    f2 gp[NP], rp[NP];
                    Pairs<T>::unpack(ld_cached(gate + k_seg * D + (int64_t)v * VEC), gp);
                    Pairs<T>::unpack(ld_stream(r + row * (int64_t)D + (int64_t)v * VEC), rp);
#pragma unroll
                    for (int i = 0; i < NP; ++i) o[i] = f2_fma(gp[i], o[i], rp[i]);
                    st_vec(out + row * (int64_t)D + (int64_t)v * VEC, Pairs<T>::pack(o));
                }
            }
        }
        __syncthreads();  // the next row's merges reuse the shared buffers
    }
}

// ------------------------------------------------------------------ backward

// Per-row coefficients.  With xh = x rstd - mean rstd and g = dy (1 + scale)
// (times gate in the fused chain), the row sums sx = sum xh, sg = sum g and
// sgx = sum g xh give delta = sx / D (the mean of xh: zero up to the rounding
// of the stored mean), c1 = rstd (sgx - delta sg) / D and c0 = c1 delta -
// rstd sg / D, so that dx = g rstd - c1 xh + c0
//                          = rstd (g - mean_d g - (xh - delta) mean_d(g (xh - delta))).
// RMS: no mean, so delta = 0 and there is no mean_d g term.  A warp per row;
// each lane sums its columns in order, then the lanes in a fixed butterfly.
template <typename T, bool GATED, bool RMS>
__global__ void __launch_bounds__(256)
    bwd_rowcoef_kernel(const T *__restrict__ x, const float *__restrict__ mean,
                       const float *__restrict__ rstd, const T *__restrict__ scale,
                       const T *__restrict__ dy, const T *__restrict__ gate,
                       float4 *__restrict__ coef, int64_t rows, int D, int64_t seg_rows,
                       const int64_t *__restrict__ offsets, int64_t nseg,
                       const int32_t *__restrict__ mod_index) {
    constexpr int VEC = IO<T>::VEC;
    constexpr int U = 4;  // vectors of each tensor in flight per lane
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int V = D / VEC;
    const float invD = 1.0f / (float)D;
    const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += wstride) {
        const int64_t k =
            mod_row(mod_index, offsets ? find_segment(offsets, nseg, row) : div_nonneg(row, seg_rows));
        const float rs = __ldg(rstd + row);
        const float nmr = RMS ? 0.f : -__ldg(mean + row) * rs;
        const T *xr = x + row * (int64_t)D;
        const T *gr = dy + row * (int64_t)D;
        const T *sr = scale + k * D;
        float sx = 0.f, sg = 0.f, sgx = 0.f;
        for (int v0 = lane; v0 < V; v0 += 32 * U) {
            V16 xv[U], dv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + 32 * u;
                if (v < V) {
                    xv[u] = ld_stream(xr + (int64_t)v * VEC);
                    dv[u] = ld_stream(gr + (int64_t)v * VEC);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + 32 * u;
                if (v < V) {
                    float xf[VEC], df[VEC], s1[VEC];
                    IO<T>::unpack(xv[u], xf);
                    IO<T>::unpack(dv[u], df);
                    IO<T>::unpack(ld_cached(sr + (int64_t)v * VEC), s1);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) s1[e] = 1.0f + s1[e];
                    if constexpr (GATED) {
                        float gf[VEC];
                        IO<T>::unpack(ld_cached(gate + k * D + (int64_t)v * VEC), gf);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) s1[e] = s1[e] * gf[e];
                    }
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float xh = fmaf(xf[e], rs, nmr);
                        const float g = df[e] * s1[e];
                        sx += xh;
                        sg += g;
                        sgx = fmaf(g, xh, sgx);
                    }
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            sx += __shfl_xor_sync(kFull, sx, off);
            sg += __shfl_xor_sync(kFull, sg, off);
            sgx += __shfl_xor_sync(kFull, sgx, off);
        }
        if (lane == 0) {
            const float delta = RMS ? 0.f : sx * invD;
            const float mg = RMS ? 0.f : sg * invD;
            const float mgx = fmaf(-delta, sg, sgx) * invD;
            const float c1 = rs * mgx;
            const float c0 = fmaf(c1, delta, -rs * mg);
            coef[row] = make_float4(c1, c0, delta, 0.f);
        }
    }
}

// Slab kernel.  CTA (c, j) takes chunk c of the rows (L consecutive rows, cut at
// segment boundaries into pieces, as for the pipelined kernels) and slab j of
// 256 column vectors; each thread owns one column vector and walks the rows of
// every piece four at a time, with all their loads in flight.
//   LN:   a = x, b = dy, mod = scale: dx from the per-row coefficients; the
//         piece of segment k writes partial rows (c + k, 0) = sum dy (xh - delta)
//         and (c + k, 1) = sum dy.  GATED (fused chain): the modulation column is
//         (1 + scale) gate, and the column sums turn the two sums into d_scale,
//         d_shift and d_gate.
//   !LN:  a = dout, b = z, mod = gate: dz = gate dout and partial row c + k holds
//         sum dout z.
// Nothing here waits, so the status words the column sums fold are cleared.
template <typename T, bool LN, bool GATED, bool RMS>
__global__ void __launch_bounds__(kSlabThreads)
    bwd_slab_kernel(const T *__restrict__ a, const T *__restrict__ b, const T *__restrict__ mod,
                    const T *__restrict__ gate, const float *__restrict__ mean,
                    const float *__restrict__ rstd, const float4 *__restrict__ coef,
                    T *__restrict__ out, float *__restrict__ partial, int *__restrict__ cta_status,
                    int nctas, int64_t rows, int D, int64_t seg_rows,
                    const int64_t *__restrict__ offsets, int64_t nseg,
                    const int32_t *__restrict__ mod_index, int64_t L, int nslabs) {
    constexpr int VEC = IO<T>::VEC;
    constexpr int NQ = LN ? 2 : 1;
    constexpr int U = 4;  // rows in flight
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0 && blockIdx.x < (unsigned)nctas) cta_status[blockIdx.x] = 0;
    const int64_t c = blockIdx.x / nslabs;
    const int j = (int)(blockIdx.x - c * nslabs);
    const int V = D / VEC;
    const int v = j * kSlabThreads + threadIdx.x;
    if (v >= V) return;  // no barriers below
    const int64_t col = (int64_t)v * VEC;
    int64_t r = c * L;
    const int64_t cend = min(r + L, rows);
    int64_t k = offsets ? find_segment(offsets, nseg, r) : div_nonneg(r, seg_rows);
    while (r < cend) {
        // piece [r, e) of segment k
        int64_t e;
        if (offsets) {
            while (k + 1 < nseg && __ldg(offsets + k + 1) <= r) ++k;
            e = k + 1 < nseg ? min(cend, __ldg(offsets + k + 1)) : cend;
        } else {
            e = min(cend, (k + 1) * seg_rows);
        }
        if (e <= r) e = cend;
        float m[VEC], acc0[VEC], acc1[VEC];
        const int64_t mr = mod_row(mod_index, k);
        IO<T>::unpack(ld_cached(mod + mr * D + col), m);
        if constexpr (LN) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) m[i] = 1.0f + m[i];
            if constexpr (GATED) {
                float gf[VEC];
                IO<T>::unpack(ld_cached(gate + mr * D + col), gf);
#pragma unroll
                for (int i = 0; i < VEC; ++i) m[i] = m[i] * gf[i];
            }
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            acc0[i] = 0.f;
            acc1[i] = 0.f;
        }
        for (int64_t r0 = r; r0 < e; r0 += U) {
            V16 av[U], bv[U];
            float rs[U], nmr[U];
            float4 cf[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (r0 + u < e) {
                    const int64_t row = r0 + u;
                    if constexpr (LN) {
                        rs[u] = __ldg(rstd + row);
                        nmr[u] = RMS ? 0.f : -__ldg(mean + row);
                        cf[u] = __ldg(coef + row);
                    }
                    av[u] = ld_stream(a + row * (int64_t)D + col);
                    bv[u] = ld_stream(b + row * (int64_t)D + col);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (r0 + u < e) {
                    const int64_t row = r0 + u;
                    float af[VEC], bf[VEC], o[VEC];
                    IO<T>::unpack(av[u], af);
                    IO<T>::unpack(bv[u], bf);
                    if constexpr (LN) {
                        const float R = rs[u], NMR = nmr[u] * rs[u];
#pragma unroll
                        for (int i = 0; i < VEC; ++i) {
                            const float xh = fmaf(af[i], R, NMR);
                            const float g = bf[i] * m[i];
                            o[i] = fmaf(g, R, fmaf(xh, -cf[u].x, cf[u].y));
                            acc0[i] = fmaf(bf[i], xh - cf[u].z, acc0[i]);
                            acc1[i] += bf[i];
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < VEC; ++i) {
                            o[i] = m[i] * af[i];
                            acc0[i] = fmaf(af[i], bf[i], acc0[i]);
                        }
                    }
                    st_vec(out + row * (int64_t)D + col, IO<T>::pack(o));
                }
            }
        }
        float *p = partial + (c + k) * NQ * (int64_t)D + col;
#pragma unroll
        for (int i = 0; i < VEC; i += 4) {
            *reinterpret_cast<float4 *>(p + i) =
                make_float4(acc0[i], acc0[i + 1], acc0[i + 2], acc0[i + 3]);
            if constexpr (LN)
                *reinterpret_cast<float4 *>(p + D + i) =
                    make_float4(acc1[i], acc1[i + 1], acc1[i + 2], acc1[i + 3]);
        }
        r = e;
        if (!offsets) ++k;
    }
}

// ------------------------------------------------------------------ launchers

template <typename T, int W, int NVMAX>
cudaError_t fwd_wide_one(const void *x, const void *shift, const void *scale, void *y,
                         float *mean, float *rstd, const Segments &sg, int D, float eps,
                         const GateEpilogue &ge, bool rms, cudaStream_t stream) {
    const int V = D / IO<T>::VEC;
    const int nv = (V + 32 * W - 1) / (32 * W);
    if (nv > NVMAX) return cudaErrorInvalidValue;
    auto kern = ge.out != nullptr ? adaln_fwd_wide_kernel<T, W, NVMAX, true, false>
                : rms        ? adaln_fwd_wide_kernel<T, W, NVMAX, false, true>
                             : adaln_fwd_wide_kernel<T, W, NVMAX, false, false>;
    const int64_t grid = sg.rows < kWideMaxGrid ? sg.rows : kWideMaxGrid;
    const cudaError_t err = launch_pdl(
        kern, dim3((unsigned)grid), dim3(32 * W), 0, stream, (const T *)x, (const T *)shift,
        (const T *)scale, (T *)y, mean, rstd, sg.rows, D, nv, eps, sg.seg_rows, sg.offsets,
        sg.nseg, sg.mod_index, (const T *)ge.gate, (const T *)ge.r, (T *)ge.out);
    count_launch();
    return err;
}

template <typename T, bool LN, bool GATED, bool RMS>
cudaError_t slab_launch(const void *a, const void *b, const void *mod, const void *gate,
                        const float *mean, const float *rstd, const float *coef, void *out,
                        float *partial, int *cta_status, const Segments &sg, const Chunking &ch,
                        int D, cudaStream_t s) {
    const int V = D / IO<T>::VEC;
    const int nslabs = (V + kSlabThreads - 1) / kSlabThreads;
    const cudaError_t err = launch_pdl(
        bwd_slab_kernel<T, LN, GATED, RMS>, dim3((unsigned)(ch.nchunks * nslabs)),
        dim3(kSlabThreads), 0, s, (const T *)a, (const T *)b, (const T *)mod, (const T *)gate,
        mean, rstd, reinterpret_cast<const float4 *>(coef), (T *)out, partial, cta_status,
        ch.ctas, sg.rows, D, sg.seg_rows, sg.offsets, sg.nseg, sg.mod_index, ch.L, nslabs);
    count_launch();
    return err;
}

template <typename T, bool GATED, bool RMS>
cudaError_t bwd_wide_t(const void *x, const float *mean, const float *rstd, const void *scale,
                       const void *dy, void *dx, float *partial, int *cta_status, float *coef,
                       const Segments &sg, const Chunking &ch, int D, const void *gate,
                       cudaStream_t s) {
    DeviceInfo di;
    cudaError_t err = device_info(di);
    if (err != cudaSuccess) return err;
    // a warp per row, enough CTAs to fill every SM several times over
    const int64_t blocks_needed = (sg.rows + 7) / 8;
    const int64_t cap = (int64_t)di.sms * 16;
    const int64_t blocks = blocks_needed < cap ? blocks_needed : cap;
    err = launch_pdl(bwd_rowcoef_kernel<T, GATED, RMS>, dim3((unsigned)blocks), dim3(256), 0, s,
                     (const T *)x, mean, rstd, (const T *)scale, (const T *)dy, (const T *)gate,
                     reinterpret_cast<float4 *>(coef), sg.rows, D, sg.seg_rows, sg.offsets,
                     sg.nseg, sg.mod_index);
    count_launch();
    if (err != cudaSuccess) return err;
    return slab_launch<T, true, GATED, RMS>(x, dy, scale, gate, mean, rstd, coef, dx, partial,
                                            cta_status, sg, ch, D, s);
}

// Four warps per row up to 2048 vectors (8 or 16 vectors per thread), eight
// warps above that (fp32 rows of more than 8192 elements).  Measured against
// eight warps at every width: four are 10-30% faster wherever they fit, since
// the merges and barriers of a row are paid once per 64-128 elements of a
// thread instead of once per 32-64.
template <typename T>
cudaError_t fwd_wide_t(const void *x, const void *shift, const void *scale, void *y, float *mean,
                       float *rstd, const Segments &sg, int D, float eps, const GateEpilogue &ge,
                       bool rms, cudaStream_t stream) {
    const int V = D / IO<T>::VEC;
#define ADALN_WIDE_FWD(WW, NVM)                                                              \
    if (V <= 32 * (WW) * (NVM))                                                             \
        return fwd_wide_one<T, WW, NVM>(x, shift, scale, y, mean, rstd, sg, D, eps, ge, rms, \
                                        stream);
    ADALN_WIDE_FWD(4, 8)
    ADALN_WIDE_FWD(4, 16)
    if constexpr (IO<T>::VEC == 4) {  // bf16 rows stop at 2048 vectors
        ADALN_WIDE_FWD(8, 16)
    }
#undef ADALN_WIDE_FWD
    return cudaErrorInvalidValue;
}

}  // namespace

int64_t wide_max_dim() { return 16384; }

cudaError_t launch_fwd_wide(DType dt, const void *x, const void *shift, const void *scale,
                            void *y, float *mean, float *rstd, const Segments &sg, int D,
                            float eps, const GateEpilogue &ge, bool rms, cudaStream_t stream) {
    if (sg.rows == 0) return cudaSuccess;
    return dt == DType::BF16
               ? fwd_wide_t<__nv_bfloat16>(x, shift, scale, y, mean, rstd, sg, D, eps, ge, rms, stream)
               : fwd_wide_t<float>(x, shift, scale, y, mean, rstd, sg, D, eps, ge, rms, stream);
}

cudaError_t bwd_wide(DType dt, const void *x, const float *mean, const float *rstd,
                     const void *scale, const void *dy, void *dx, float *partial, int *cta_status,
                     float *coef, const Segments &sg, const Chunking &ch, int D, const void *gate,
                     cudaStream_t s) {
    if (ch.nchunks == 0) return cudaSuccess;
    if (coef == nullptr) return cudaErrorInvalidValue;
    const bool rms = mean == nullptr;
#define ADALN_WIDE_BWD(TT)                                                                     \
    return gate != nullptr ? bwd_wide_t<TT, true, false>(x, mean, rstd, scale, dy, dx, partial, \
                                                          cta_status, coef, sg, ch, D, gate, s) \
           : rms ? bwd_wide_t<TT, false, true>(x, mean, rstd, scale, dy, dx, partial,          \
                                               cta_status, coef, sg, ch, D, gate, s)           \
                 : bwd_wide_t<TT, false, false>(x, mean, rstd, scale, dy, dx, partial,         \
                                                cta_status, coef, sg, ch, D, gate, s);
    if (dt == DType::BF16) {
        ADALN_WIDE_BWD(__nv_bfloat16)
    }
    ADALN_WIDE_BWD(float)
#undef ADALN_WIDE_BWD
}

cudaError_t gate_bwd_wide(DType dt, const void *dout, const void *z, const void *gate, void *dz,
                          float *partial, int *cta_status, const Segments &sg, const Chunking &ch,
                          int D, cudaStream_t s) {
    if (ch.nchunks == 0) return cudaSuccess;
    if (dt == DType::BF16)
        return slab_launch<__nv_bfloat16, false, false, false>(dout, z, gate, nullptr, nullptr,
                                                               nullptr, nullptr, dz, partial,
                                                               cta_status, sg, ch, D, s);
    return slab_launch<float, false, false, false>(dout, z, gate, nullptr, nullptr, nullptr,
                                                   nullptr, dz, partial, cta_status, sg, ch, D, s);
}

}  // namespace adaln
