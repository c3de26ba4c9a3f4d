// fwd.cu -- AdaLN forward and the gated-residual epilogue (sm_103a).
//
// Forward ("AdaptiveLoad" summary, section 2.B, "Paso Adelante"): one launch
// reads every row of x from HBM exactly once, keeps it in registers, reduces
// the row statistics with warp shuffles, and applies the modulation in a
// further traversal of the registers:
//     y = (x - mean) * rstd * (1 + scale[k]) + shift[k].
// A row is owned by LPR lanes of one warp (LPR = 32 for D >= 1024 bf16), so no
// block-level barrier sits on the critical path; each lane holds up to NVMAX
// 16-byte vectors of its row.
//
// Row statistics are exact to the float rounding: each lane accumulates
// sum(x) and sum(x^2) as double-float pairs with TwoSum (for bf16 inputs x^2
// is exact in fp32), lanes merge with an accurate double-float addition, and
// mean/var/rstd are finished in double-float with a Newton step on rsqrt.
// When var is small against mean^2 (cancellation in E[x^2] - mean^2) the row
// falls back to a compensated two-pass sum of (x - mean)^2 from registers;
// fp32 inputs always use the two-pass form.
#include "common.cuh"
#include "launch.h"

#include <math.h>

namespace adaln {
namespace {

constexpr int kFwdThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

// Merge a double-float pair across the LPR lanes that own a row (xor butterfly;
// df_add is commutative bit-for-bit, so every lane ends with the same pair).
template <int LPR>
__device__ __forceinline__ void lane_merge(float &h, float &l) {
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
        const float oh = __shfl_xor_sync(kFull, h, off);
        const float ol = __shfl_xor_sync(kFull, l, off);
        df_add(h, l, oh, ol, h, l);
    }
}

// 1 / sqrt(v) for v = vh + vl > 0: hardware estimate, one fp32 Newton step,
// then one Newton step with the residual 1 - v*r^2 evaluated in double-float,
// rounded once to float (relative error of the unrounded value ~2^-45).
__device__ __forceinline__ float rsqrt_df(float vh, float vl) {
    if (!(vh > 0.0f)) return vh == 0.0f ? __int_as_float(0x7f800000) : __int_as_float(0x7fffffff);
    const float r0 = rsqrtf(vh);
    if (!(vh >= 0x1p-100f && vh <= 0x1p100f)) return r0;  // keep r^2 and v*r^2 normal
    const float t = __fmul_rn(vh, r0);
    const float r1 = __fmaf_rn(__fmul_rn(0.5f, r0), __fmaf_rn(-t, r0, 1.0f), r0);
    float a, b, c, ce;
    two_prod(r1, r1, a, b);  // r1^2 = a + b
    two_prod(vh, a, c, ce);  // vh * a = c + ce
    const float cl = __fmaf_rn(vh, b, __fmaf_rn(vl, a, ce));
    const float res = __fsub_rn(__fsub_rn(1.0f, c), cl);  // 1 - c is exact (c ~ 1)
    return __fadd_rn(r1, __fmul_rn(__fmul_rn(0.5f, r1), res));
}

template <typename T, int LPR, int NVMAX, bool FAST>
__global__ void __launch_bounds__(kFwdThreads)
    adaln_fwd_kernel(const T *__restrict__ x, const T *__restrict__ shift,
                     const T *__restrict__ scale, T *__restrict__ y, float *__restrict__ mean,
                     float *__restrict__ rstd, int64_t rows, int D, int nv, float eps,
                     int64_t seg_rows, const int64_t *__restrict__ offsets, int64_t nseg) {
    constexpr int VEC = IO<T>::VEC;
    constexpr int RPW = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int li = lane % LPR;
    const int V = D / VEC;
    const int64_t row =
        ((int64_t)blockIdx.x * (kFwdThreads / 32) + (threadIdx.x >> 5)) * RPW + lane / LPR;
    const bool active = row < rows;
    const T *xr = x + (active ? row : 0) * (int64_t)D;

    // ---- one HBM read of the row: NVMAX 16-byte vectors per lane
    V16 xv[NVMAX];
#pragma unroll
    for (int k = 0; k < NVMAX; ++k) {
        const int v = li + k * LPR;
        if (k < nv && active && v < V)
            xv[k] = ld_stream(xr + (int64_t)v * VEC);
        else
            xv[k] = V16{{0u, 0u, 0u, 0u}};
    }

    const float Df = (float)D;
    float sh = 0.f, sl = 0.f;  // sum(x) as a double-float
    float qh = 0.f, ql = 0.f;  // sum(x^2) (FAST only)
#pragma unroll
    for (int k = 0; k < NVMAX; ++k) {
        if (k < nv) {
            float f[VEC];
            IO<T>::unpack(xv[k], f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float t;
                two_sum(sh, f[e], sh, t);
                sl = __fadd_rn(sl, t);
                if (FAST) {
                    two_sum(qh, __fmul_rn(f[e], f[e]), qh, t);
                    ql = __fadd_rn(ql, t);
                }
            }
            two_sum(sh, sl, sh, sl);
            if (FAST) fast_two_sum(qh, ql, qh, ql);
        }
    }
    lane_merge<LPR>(sh, sl);
    float mh, ml;
    df_div_f(sh, sl, Df, mh, ml);

    float vh = 0.f, vl = 0.f;
    bool two_pass = !FAST;
    if (FAST) {
        lane_merge<LPR>(qh, ql);
        float q2h, q2l, ph, pl;
        df_div_f(qh, ql, Df, q2h, q2l);
        two_prod(mh, mh, ph, pl);
        pl = __fmaf_rn(__fmul_rn(2.0f, mh), ml, pl);
        fast_two_sum(ph, pl, ph, pl);
        df_add(q2h, q2l, -ph, -pl, vh, vl);
        // E[x^2] - mean^2 loses log2(mean^2/var) bits: keep it only when that is small.
        two_pass = !(ph <= 4.0f * vh);
    }
    // Warp-uniform branch: every lane takes part in the shuffles; rows that did
    // not ask for the two-pass result keep their one-pass value.
    if (__any_sync(kFull, two_pass)) {
        float s2h = 0.f, s2l = 0.f;
#pragma unroll
        for (int k = 0; k < NVMAX; ++k) {
            const int v = li + k * LPR;
            if (k < nv && v < V) {
                float f[VEC];
                IO<T>::unpack(xv[k], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    float dh, de, p, pe, t;
                    two_sum(f[e], -mh, dh, de);  // x - mh exactly
                    de = __fsub_rn(de, ml);      // d = dh + de ~ x - mean
                    two_prod(dh, dh, p, pe);
                    // d^2 = dh^2 + de (2 dh + de): de^2 matters when |mean| >> std
                    pe = __fmaf_rn(de, __fmaf_rn(2.0f, dh, de), pe);
                    two_sum(s2h, p, s2h, t);
                    s2l = __fadd_rn(s2l, __fadd_rn(t, pe));
                }
                fast_two_sum(s2h, s2l, s2h, s2l);
            }
        }
        lane_merge<LPR>(s2h, s2l);
        if (two_pass) df_div_f(s2h, s2l, Df, vh, vl);
    }

    // rstd = 1 / sqrt(var + eps), var + eps as a double-float
    float eh, el;
    two_sum(vh, eps, eh, el);
    el = __fadd_rn(el, vl);
    fast_two_sum(eh, el, eh, el);
    const float rs = rsqrt_df(eh, el);

    if (!active) return;
    if (li == 0) {
        mean[row] = mh;
        rstd[row] = rs;
    }

    // ---- modulation: one more traversal of the registers, one HBM write
    const int64_t k_seg = offsets ? find_segment(offsets, nseg, row) : row / seg_rows;
    const T *shr = shift + k_seg * D;
    const T *scr = scale + k_seg * D;
    T *yr = y + row * (int64_t)D;
#pragma unroll
    for (int k = 0; k < NVMAX; ++k) {
        const int v = li + k * LPR;
        if (k < nv && v < V) {
            float f[VEC], s[VEC], b[VEC], o[VEC];
            IO<T>::unpack(xv[k], f);
            IO<T>::unpack(ld_cached(scr + (int64_t)v * VEC), s);
            IO<T>::unpack(ld_cached(shr + (int64_t)v * VEC), b);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                // x - mean with the mean's low word: x - mh is exact near the mean
                // (Sterbenz), so rows whose |mean| >> std keep full fp32 accuracy.
                // bf16 outputs cannot see the low word; skip it there.
                const float d = FAST ? __fsub_rn(f[e], mh) : __fsub_rn(__fsub_rn(f[e], mh), ml);
                o[e] = fmaf(d * rs, 1.0f + s[e], b[e]);
            }
            st_vec(yr + (int64_t)v * VEC, IO<T>::pack(o));
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
                    int64_t seg_rows, const int64_t *__restrict__ offsets, int64_t nseg) {
    constexpr int VEC = IO<T>::VEC;
    constexpr int U = 4;
    const int lane = threadIdx.x & 31;
    const int V = D / VEC;
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t r0 = w * rows_per_warp;
    const int64_t r1 = min(rows, r0 + rows_per_warp);
    if (r0 >= r1) return;
    int64_t k_seg = offsets ? find_segment(offsets, nseg, r0) : r0 / seg_rows;
    int64_t seg_end = offsets ? __ldg(offsets + k_seg + 1) : (k_seg + 1) * seg_rows;
    for (int64_t row = r0; row < r1; ++row) {
        while (row >= seg_end && k_seg + 1 < nseg) {  // next non-empty segment
            ++k_seg;
            seg_end = offsets ? __ldg(offsets + k_seg + 1) : (k_seg + 1) * seg_rows;
        }
        const T *gr = gate + k_seg * D;
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

// ------------------------------------------------------------------ dispatch

constexpr int kNvClasses[] = {2, 4, 6, 8, 12, 16, 20, 24};

template <typename T, int LPR, int NVMAX, bool FAST>
cudaError_t fwd_launch_one(const void *x, const void *shift, const void *scale, void *y,
                           float *mean, float *rstd, const Segments &sg, int D, int nv,
                           float eps, cudaStream_t stream) {
    constexpr int rows_per_block = (kFwdThreads / 32) * (32 / LPR);
    const int64_t blocks = (sg.rows + rows_per_block - 1) / rows_per_block;
    adaln_fwd_kernel<T, LPR, NVMAX, FAST><<<(unsigned)blocks, kFwdThreads, 0, stream>>>(
        (const T *)x, (const T *)shift, (const T *)scale, (T *)y, mean, rstd, sg.rows, D, nv,
        eps, sg.seg_rows, sg.offsets, sg.nseg);
    count_launch();
    return cudaGetLastError();
}

template <typename T, int LPR, bool FAST>
cudaError_t fwd_by_nv(const void *x, const void *shift, const void *scale, void *y, float *mean,
                      float *rstd, const Segments &sg, int D, int nv, float eps,
                      cudaStream_t s) {
#define ADALN_NV_CASE(NVM)                                                                     \
    if (nv <= NVM)                                                                             \
        return fwd_launch_one<T, LPR, NVM, FAST>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, \
                                                 s);
    ADALN_NV_CASE(2)
    ADALN_NV_CASE(4)
    ADALN_NV_CASE(6)
    ADALN_NV_CASE(8)
    ADALN_NV_CASE(12)
    ADALN_NV_CASE(16)
    ADALN_NV_CASE(20)
    ADALN_NV_CASE(24)
#undef ADALN_NV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

int64_t max_dim(DType dt) {
    // 24 vectors of 16 bytes per lane, 32 lanes per row
    return dt == DType::BF16 ? 24 * 32 * 8 : 24 * 32 * 4;
}

cudaError_t launch_fwd(DType dt, const void *x, const void *shift, const void *scale, void *y,
                       float *mean, float *rstd, const Segments &sg, int64_t D64, float eps,
                       cudaStream_t stream) {
    if (sg.rows == 0) return cudaSuccess;
    const int D = (int)D64;
    if (dt == DType::BF16) {
        const int V = D / 8;
        // small rows: 8 lanes per row (4 rows per warp); otherwise a full warp per row
        if (V <= 8 * 8) {
            const int nv = (V + 7) / 8;
            return fwd_by_nv<__nv_bfloat16, 8, true>(x, shift, scale, y, mean, rstd, sg, D, nv, eps,
                                                     stream);
        }
        const int nv = (V + 31) / 32;
        return fwd_by_nv<__nv_bfloat16, 32, true>(x, shift, scale, y, mean, rstd, sg, D, nv, eps,
                                                  stream);
    }
    const int V = D / 4;
    if (V <= 8 * 8) {
        const int nv = (V + 7) / 8;
        return fwd_by_nv<float, 8, false>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, stream);
    }
    const int nv = (V + 31) / 32;
    return fwd_by_nv<float, 32, false>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, stream);
}

cudaError_t launch_gate(DType dt, const void *r, const void *z, const void *gate, void *out,
                        const Segments &sg, int64_t D64, cudaStream_t stream) {
    if (sg.rows == 0) return cudaSuccess;
    DeviceInfo di;
    cudaError_t err = device_info(di);
    if (err != cudaSuccess) return err;
    const int D = (int)D64;
    // enough warps to fill every SM several times over; each warp a contiguous block of rows
    const int64_t target_warps = (int64_t)di.sms * 64;
    int64_t rpw = (sg.rows + target_warps - 1) / target_warps;
    if (rpw < 1) rpw = 1;
    const int64_t warps = (sg.rows + rpw - 1) / rpw;
    const int64_t blocks = (warps + 7) / 8;
    if (dt == DType::BF16)
        gate_fwd_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(
            (const __nv_bfloat16 *)r, (const __nv_bfloat16 *)z, (const __nv_bfloat16 *)gate,
            (__nv_bfloat16 *)out, sg.rows, D, rpw, sg.seg_rows, sg.offsets, sg.nseg);
    else
        gate_fwd_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(
            (const float *)r, (const float *)z, (const float *)gate, (float *)out, sg.rows, D, rpw,
            sg.seg_rows, sg.offsets, sg.nseg);
    count_launch();
    return cudaGetLastError();
}

}  // namespace adaln
