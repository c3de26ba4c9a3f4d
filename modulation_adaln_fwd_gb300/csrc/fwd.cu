// fwd.cu -- AdaLN forward (register kernels, dispatch) and the gated residual.
//
// The row statistics and modulation are in fwd_stats.cuh; the pipelined
// forward, which takes every bf16 shape it has an instance for (a warp per row,
// or a group of four warps per row for rows of 8,192 to 16,384 elements), is in
// fwd_ring.cu; the other rows of more than 768 vectors go to the CTA-per-row
// kernel of wide.cu.  This file holds the register kernel
// (a warp per row, the row in registers) for the other shapes and fp32, the
// gated-residual stream and the launchers.
#include "fwd_stats.cuh"

namespace adaln {
namespace {

// y = LN(x) * (1 + scale) + shift for rows of D elements; a row is owned by LPR
// lanes (32 / LPR rows per warp), each holding up to NVMAX 16-byte vectors.
// EXACT: D == LPR * NVMAX * VEC, so no lane needs a bounds predicate.
// GATED: also out = r + gate[k] * y from the fp32 y (the gated residual applied
// to the modulated output itself); y is then written only if it is not null.
// RMS: the RMSNorm statistics (no mean; mean is not written).
template <typename T, int LPR, int NVMAX, bool FAST, bool EXACT, bool GATED, bool RMS>
__global__ void __launch_bounds__(kFwdThreads, 2)
    adaln_fwd_kernel(const T *__restrict__ x, const T *__restrict__ shift,
                     const T *__restrict__ scale, T *__restrict__ y, float *__restrict__ mean,
                     float *__restrict__ rstd, int64_t rows, int D, int nv, float eps,
                     int64_t seg_rows, const int64_t *__restrict__ offsets, int64_t nseg,
                     const int32_t *__restrict__ mod_index, const T *__restrict__ gate,
                     const T *__restrict__ r, T *__restrict__ out) {
    constexpr int VEC = IO<T>::VEC;
    constexpr int RPW = 32 / LPR;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int li = lane % LPR;
    const int V = EXACT ? LPR * NVMAX : D / VEC;
    const int64_t row =
        ((int64_t)blockIdx.x * (kFwdThreads / 32) + (threadIdx.x >> 5)) * RPW + lane / LPR;
    const bool active = row < rows;
    const T *xr = x + (active ? row : 0) * (int64_t)D;
    // (the runtime count nv also splits the unrolled loops into per-vector blocks,
    // which keeps the scheduler from hoisting every unpack and blowing registers)
    auto has = [&](int k) { return k < nv && (EXACT || li + k * LPR < V); };

    // ---- one HBM read of the row: NVMAX 16-byte vectors per lane
    V16 xv[NVMAX];
#pragma unroll
    for (int k = 0; k < NVMAX; ++k) {
        if (active && has(k))
            xv[k] = ld_stream(xr + (int64_t)(li + k * LPR) * VEC);
        else
            xv[k] = V16{{0u, 0u, 0u, 0u}};
    }
    float mh, ml, rs;
    auto xreg = [&](int k) -> const V16 & { return xv[k]; };
    row_stats<T, LPR, NVMAX, FAST, EXACT, true, NVMAX, decltype(xreg), false, RMS>(
        xreg, li, nv, V, D, eps, mh, ml, rs);

    if (!active) return;
    if (li == 0) {
        if (!RMS) mean[row] = mh;
        rstd[row] = rs;
    }
    // ---- modulation: one more traversal of the registers, one HBM write
    const int64_t k_seg =
        mod_row(mod_index, offsets ? find_segment(offsets, nseg, row) : div_nonneg(row, seg_rows));
    const T *shr = shift + k_seg * D;
    const T *scr = scale + k_seg * D;
    const bool wide = !(fabsf(mh * rs) <= 4.0f);
    T *yr = y != nullptr ? y + row * (int64_t)D : nullptr;
#pragma unroll
    for (int k = 0; k < NVMAX; ++k) {
        const int v = li + k * LPR;
        if (has(k)) {
            float s[VEC], b[VEC], yv[VEC];
            IO<T>::unpack(ld_cached(scr + (int64_t)v * VEC), s);
            IO<T>::unpack(ld_cached(shr + (int64_t)v * VEC), b);
            modulate_vals<T, FAST>(xv[k], s, b, mh, ml, rs, wide, yv);
            if (yr != nullptr) st_vec(yr + (int64_t)v * VEC, IO<T>::pack(yv));
            if constexpr (GATED) {
                float g[VEC], rv[VEC];
                IO<T>::unpack(ld_cached(gate + k_seg * D + (int64_t)v * VEC), g);
                IO<T>::unpack(ld_stream(r + row * (int64_t)D + (int64_t)v * VEC), rv);
#pragma unroll
                for (int e = 0; e < VEC; ++e) yv[e] = fmaf(g[e], yv[e], rv[e]);
                st_vec(out + row * (int64_t)D + (int64_t)v * VEC, IO<T>::pack(yv));
            }
        }
    }
}

// ------------------------------------------------------------------ gate fwd
// out = r + gate[k] * z: pure stream.  A warp walks a contiguous block of
// rows (segment looked up once, then advanced), 4 vectors in flight per lane.
template <typename T>
__global__ void __launch_bounds__(256)
    gate_fwd_kernel(const T *__restrict__ r, const T *__restrict__ z, const T *__restrict__ gate,
                    T *__restrict__ out, int64_t rows, int D, int64_t rows_per_warp,
                    int64_t seg_rows, const int64_t *__restrict__ offsets, int64_t nseg,
                    const int32_t *__restrict__ mod_index) {
    constexpr int VEC = IO<T>::VEC;
    constexpr int U = 4;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int V = D / VEC;
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t r0 = w * rows_per_warp;
    const int64_t r1 = min(rows, r0 + rows_per_warp);
    if (r0 >= r1) return;
    int64_t k_seg = offsets ? find_segment(offsets, nseg, r0) : div_nonneg(r0, seg_rows);
    int64_t seg_end = offsets ? __ldg(offsets + k_seg + 1) : (k_seg + 1) * seg_rows;
    for (int64_t row = r0; row < r1; ++row) {
        while (row >= seg_end && k_seg + 1 < nseg) {  // next non-empty segment
            ++k_seg;
            seg_end = offsets ? __ldg(offsets + k_seg + 1) : (k_seg + 1) * seg_rows;
        }
        const T *gr = gate + mod_row(mod_index, k_seg) * D;
        const int64_t base = row * (int64_t)D;
        for (int v0 = lane; v0 < V; v0 += 32 * U) {
            V16 rv[U], zv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * 32;
                if (v < V) {
                    rv[u] = ld_stream(r + base + (int64_t)v * VEC);
                    zv[u] = ld_stream(z + base + (int64_t)v * VEC);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * 32;
                if (v < V) {
                    float a[VEC], b[VEC], g[VEC], o[VEC];
                    IO<T>::unpack(rv[u], a);
                    IO<T>::unpack(zv[u], b);
                    IO<T>::unpack(ld_cached(gr + (int64_t)v * VEC), g);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = fmaf(g[e], b[e], a[e]);
                    st_vec(out + base + (int64_t)v * VEC, IO<T>::pack(o));
                }
            }
        }
    }
}

// out = r + gate[k] * z for bf16 rows, by column slabs: CTA (c, j) takes row
// chunk c (L rows, cut at segment boundaries) and slab j of 256 column vectors;
// each thread owns one vector, keeps the piece's gate column and walks the rows
// four at a time.  The CTAs of one chunk read the same rows side by side, where
// the row-per-warp stream has every warp in a different row (measured on GB300
// against it, fraction of the copy bandwidth: D = 16,384 0.83 -> 0.95, 12,288
// 0.87 -> 0.93, 8,192 0.89 -> 0.93, 3072 0.964 -> 0.978, MMDiT 0.84 -> 0.87,
// DiT 0.47 -> 0.51, the ragged buckets 0.969 -> 0.978; Wan even).  MINB: CTAs
// per SM the registers are sized for (1: as the compiler likes, 78 registers,
// three CTAs an SM, which the widest rows prefer; 4: 64 registers, four CTAs).
template <typename T, int MINB>
__global__ void __launch_bounds__(256, MINB)
    gate_fwd_slab_kernel(const T *__restrict__ r, const T *__restrict__ z,
                         const T *__restrict__ gate, T *__restrict__ out, int64_t rows, int D,
                         int64_t seg_rows, const int64_t *__restrict__ offsets, int64_t nseg,
                         const int32_t *__restrict__ mod_index, int64_t L, int nslabs) {
    constexpr int VEC = IO<T>::VEC;
    constexpr int U = 4;
    pdl_wait();
    pdl_trigger();
    const int64_t c = blockIdx.x / nslabs;
    const int j = (int)(blockIdx.x - c * nslabs);
    const int V = D / VEC;
    const int v = j * 256 + threadIdx.x;
    if (v >= V) return;
    const int64_t col = (int64_t)v * VEC;
    int64_t row0 = c * L;
    const int64_t cend = min(row0 + L, rows);
    int64_t k = offsets ? find_segment(offsets, nseg, row0) : div_nonneg(row0, seg_rows);
    while (row0 < cend) {
        int64_t e;
        if (offsets) {
            while (k + 1 < nseg && __ldg(offsets + k + 1) <= row0) ++k;
            e = k + 1 < nseg ? min(cend, __ldg(offsets + k + 1)) : cend;
        } else {
            e = min(cend, (k + 1) * seg_rows);
        }
        if (e <= row0) e = cend;
        float m[VEC];
        IO<T>::unpack(ld_cached(gate + mod_row(mod_index, k) * D + col), m);
        for (int64_t q = row0; q < e; q += U) {
            V16 av[U], bv[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (q + u < e) {
                    av[u] = ld_stream(r + (q + u) * (int64_t)D + col);
                    bv[u] = ld_stream(z + (q + u) * (int64_t)D + col);
                }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (q + u < e) {
                    float a[VEC], b[VEC], o[VEC];
                    IO<T>::unpack(av[u], a);
                    IO<T>::unpack(bv[u], b);
#pragma unroll
                    for (int i = 0; i < VEC; ++i) o[i] = fmaf(m[i], b[i], a[i]);
                    st_vec(out + (q + u) * (int64_t)D + col, IO<T>::pack(o));
                }
        }
        row0 = e;
        if (!offsets) ++k;
    }
}

// ------------------------------------------------------------------ dispatch

template <typename T, int LPR, int NVMAX, bool FAST, bool EXACT>
cudaError_t fwd_launch_one(const void *x, const void *shift, const void *scale, void *y,
                           float *mean, float *rstd, const Segments &sg, int D, int nv,
                           float eps, const GateEpilogue &ge, bool rms, cudaStream_t stream) {
    constexpr int rows_per_block = (kFwdThreads / 32) * (32 / LPR);
    const int64_t blocks = (sg.rows + rows_per_block - 1) / rows_per_block;
    auto kern = ge.out != nullptr ? adaln_fwd_kernel<T, LPR, NVMAX, FAST, EXACT, true, false>
                : rms        ? adaln_fwd_kernel<T, LPR, NVMAX, FAST, EXACT, false, true>
                             : adaln_fwd_kernel<T, LPR, NVMAX, FAST, EXACT, false, false>;
    const cudaError_t err = launch_pdl(
        kern, dim3((unsigned)blocks), dim3(kFwdThreads), 0, stream, (const T *)x,
        (const T *)shift, (const T *)scale, (T *)y, mean, rstd, sg.rows, D, nv, eps, sg.seg_rows,
        sg.offsets, sg.nseg, sg.mod_index, (const T *)ge.gate, (const T *)ge.r, (T *)ge.out);
    count_launch();
    return err;
}

// rows whose vector count is not an exact multiple: NVMAX classes with a runtime count
template <typename T, int LPR, bool FAST>
cudaError_t fwd_by_nv(const void *x, const void *shift, const void *scale, void *y, float *mean,
                      float *rstd, const Segments &sg, int D, int nv, float eps,
                      const GateEpilogue &ge, bool rms, cudaStream_t s) {
#define ADALN_NV_CASE(NVM)                                                                  \
    if (nv <= NVM)                                                                          \
        return fwd_launch_one<T, LPR, NVM, FAST, false>(x, shift, scale, y, mean, rstd, sg, D, \
                                                        nv, eps, ge, rms, s);
    // 8 lanes per row only for rows of at most 64 vectors (nv <= 8); a full warp
    // per row only above that (nv >= 3)
    if constexpr (LPR == 8) {
        ADALN_NV_CASE(2)
        ADALN_NV_CASE(4)
        ADALN_NV_CASE(6)
        ADALN_NV_CASE(8)
    } else {
        ADALN_NV_CASE(4)
        ADALN_NV_CASE(6)
        ADALN_NV_CASE(8)
        ADALN_NV_CASE(12)
        ADALN_NV_CASE(16)
        ADALN_NV_CASE(20)
        ADALN_NV_CASE(24)
    }
#undef ADALN_NV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

int64_t max_dim(DType) {
    // the wide kernels (a CTA per row in the forward, column slabs in the backward)
    return wide_max_dim();
}

cudaError_t launch_fwd(DType dt, const void *x, const void *shift, const void *scale, void *y,
                       float *mean, float *rstd, const Segments &sg, int64_t D64, float eps,
                       cudaStream_t stream, const GateEpilogue &ge, bool rms) {
    if (sg.rows == 0) return cudaSuccess;
    const int D = (int)D64;
    // bf16 rows the pipelined forward takes (a warp, or a group of four warps, per row)
    if (dt == DType::BF16) {
        DeviceInfo di;
        cudaError_t err = device_info(di);
        if (err != cudaSuccess) return err;
        bool launched = false;
        err = launch_fwd_ring(x, shift, scale, y, mean, rstd, sg, D, eps, ge, rms, di, stream,
                              launched);
        if (err != cudaSuccess || launched) return err;
    }
    // other rows of more than 24 vectors per lane of a warp: a CTA per row
    if (D / (dt == DType::BF16 ? 8 : 4) > 24 * 32)
        return launch_fwd_wide(dt, x, shift, scale, y, mean, rstd, sg, D, eps, ge, rms, stream);
    if (dt == DType::BF16) {
        using B16 = __nv_bfloat16;
        const int V = D / 8;
        DeviceInfo di;
        cudaError_t err = device_info(di);
        if (err != cudaSuccess) return err;
        // exact shapes: a warp per row with a whole number of vectors per lane
#define ADALN_EXACT(LPR, NV)                                                                  \
    if (V == (LPR) * (NV))                                                                    \
        return fwd_launch_one<B16, LPR, NV, true, true>(x, shift, scale, y, mean, rstd, sg, D, \
                                                        NV, eps, ge, rms, stream);
        ADALN_EXACT(32, 24)
#undef ADALN_EXACT
        // small rows: 8 lanes per row (4 rows per warp); otherwise a full warp per row
        if (V <= 8 * 8) {
            const int nv = (V + 7) / 8;
            return fwd_by_nv<B16, 8, true>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, ge,
                                           rms, stream);
        }
        const int nv = (V + 31) / 32;
        return fwd_by_nv<B16, 32, true>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, ge, rms,
                                        stream);
    }
    const int V = D / 4;
    if (V <= 8 * 8) {
        const int nv = (V + 7) / 8;
        return fwd_by_nv<float, 8, false>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, ge,
                                          rms, stream);
    }
    const int nv = (V + 31) / 32;
    return fwd_by_nv<float, 32, false>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, ge, rms,
                                       stream);
}

cudaError_t launch_gate(DType dt, const void *r, const void *z, const void *gate, void *out,
                        const Segments &sg, int64_t D64, cudaStream_t stream) {
    if (sg.rows == 0) return cudaSuccess;
    DeviceInfo di;
    cudaError_t err = device_info(di);
    if (err != cudaSuccess) return err;
    const int D = (int)D64;
    if (dt == DType::BF16) {
        // column slabs; chunks of rows for about 64 CTAs per SM (16 for rows of
        // four slabs and more, whose chunks already take that many CTAs each),
        // at least one chunk per SM and four rows per chunk.  Measured on GB300
        // against eight CTAs per SM: Wan 0.954 -> 1.017 of the copy bandwidth,
        // D = 3072 0.986 -> 1.008, MMDiT 0.871 -> 0.888, ragged 0.987 -> 1.008;
        // 64 at D = 16,384 was 0.909 (16: 0.948) and 64 on DiT's 1,152-wide
        // rows, a row per chunk, 0.339 (four rows: 0.508).
        const int V = D / 8, nslabs = (V + 255) / 256;
        int64_t target = (int64_t)di.sms * (nslabs >= 4 ? 16 : 64) / nslabs;
        if (target < di.sms) target = di.sms;
        int64_t L = (sg.rows + target - 1) / target;
        if (L < 4) L = 4;
        const int64_t nch = (sg.rows + L - 1) / L;
        using B16 = __nv_bfloat16;
        auto kern = V >= 1536 ? gate_fwd_slab_kernel<B16, 1> : gate_fwd_slab_kernel<B16, 4>;
        err = launch_pdl(kern, dim3((unsigned)(nch * nslabs)), dim3(256), 0, stream,
                         (const B16 *)r, (const B16 *)z, (const B16 *)gate, (B16 *)out, sg.rows, D,
                         sg.seg_rows, sg.offsets, sg.nseg, sg.mod_index, L, nslabs);
        count_launch();
        return err;
    }
    // enough warps to fill every SM several times over; each warp a contiguous block of rows
    const int64_t target_warps = (int64_t)di.sms * 64;
    int64_t rpw = (sg.rows + target_warps - 1) / target_warps;
    if (rpw < 1) rpw = 1;
    const int64_t warps = (sg.rows + rpw - 1) / rpw;
    const int64_t blocks = (warps + 7) / 8;
    if (dt == DType::BF16)
        err = launch_pdl(gate_fwd_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0,
                         stream, (const __nv_bfloat16 *)r, (const __nv_bfloat16 *)z,
                         (const __nv_bfloat16 *)gate, (__nv_bfloat16 *)out, sg.rows, D, rpw,
                         sg.seg_rows, sg.offsets, sg.nseg, sg.mod_index);
    else
        err = launch_pdl(gate_fwd_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, stream,
                         (const float *)r, (const float *)z, (const float *)gate, (float *)out,
                         sg.rows, D, rpw, sg.seg_rows, sg.offsets, sg.nseg, sg.mod_index);
    count_launch();
    return err;
}

}  // namespace adaln
