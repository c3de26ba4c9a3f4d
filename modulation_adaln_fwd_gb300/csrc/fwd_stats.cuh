// fwd_stats.cuh -- row statistics and modulation shared by the forward kernels
// (fwd.cu: register kernels and dispatch; fwd_ring.cu: the pipelined kernel).
//
// Forward ("AdaptiveLoad" summary, section 2.B, "Paso Adelante"): one launch
// reads every row of x from HBM exactly once, keeps it in registers, reduces
// the row statistics with warp shuffles, and applies the modulation in a
// further traversal of the registers:
//     y = (x - mean) * rstd * (1 + scale[k]) + shift[k].
// A row is owned by LPR lanes of one warp (LPR = 32 for D >= 1024 bf16), so no
// block-level barrier sits on the critical path; each lane holds up to NVMAX
// 16-byte vectors of its row.  Rows too wide for one warp (wide.cu) are owned
// by a whole CTA, whose lanes merge through shared memory (CtaGroup below).
//
// Row statistics are exact to the float rounding: each lane accumulates
// sum(x) and sum(x^2) as double-float pairs with TwoSum (for bf16 inputs x^2
// is exact in fp32), lanes merge with an accurate double-float addition, and
// mean/var/rstd are finished in double-float with a Newton step on rsqrt.
// When var is small against mean^2 (cancellation in E[x^2] - mean^2) the row
// falls back to a compensated two-pass sum of (x - mean)^2 from registers;
// fp32 inputs always use the two-pass form.
#pragma once

#include "common.cuh"
#include "launch.h"

#include <math.h>

#include <type_traits>

namespace adaln {
namespace {

constexpr int kFwdThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

// Merge a double-float pair across the LPR lanes that own a row (xor butterfly).
// The addition is TwoSum on the high words plus the low words, renormalised;
// it is commutative bit-for-bit, so every lane ends with the same pair.
template <int LPR>
__device__ __forceinline__ void lane_merge(float &h, float &l) {
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
        const float oh = __shfl_xor_sync(kFull, h, off);
        const float ol = __shfl_xor_sync(kFull, l, off);
        float s, e;
        two_sum(h, oh, s, e);
        e = __fadd_rn(e, __fadd_rn(l, ol));
        fast_two_sum(s, e, h, l);
    }
}

// Two such merges at once on packed pairs: (ah, al) and (bh, bl) ride in the
// two halves, so each butterfly level is one packed TwoSum.
template <int LPR>
__device__ __forceinline__ void lane_merge2(float &ah, float &al, float &bh, float &bl) {
    f2 H = f2_make(ah, bh), L = f2_make(al, bl);
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
        float h0, h1, l0, l1;
        f2_split(H, h0, h1);
        f2_split(L, l0, l1);
        const f2 OH = f2_make(__shfl_xor_sync(kFull, h0, off), __shfl_xor_sync(kFull, h1, off));
        const f2 OL = f2_make(__shfl_xor_sync(kFull, l0, off), __shfl_xor_sync(kFull, l1, off));
        f2 sum, err;
        f2_two_sum(H, OH, sum, err);
        err = f2_add(err, f2_add(L, OL));
        H = f2_add(sum, err);  // Fast2Sum: |sum| >= |err|
        L = f2_sub(err, f2_sub(H, sum));
    }
    f2_split(H, ah, bh);
    f2_split(L, al, bl);
}

// How the lanes that own a row combine their per-lane results.  LaneGroup: LPR
// lanes of one warp (shuffles only).  CtaGroup: every thread of a CTA of W warps
// (shuffles within each warp, then a fixed-order fold of the W warp results
// through shared memory, so every thread ends with the same bits).  Both merge
// double-float pairs with the same TwoSum + Fast2Sum addition.
template <int LPR>
struct LaneGroup {
    __device__ __forceinline__ void merge(float &h, float &l) { lane_merge<LPR>(h, l); }
    __device__ __forceinline__ void merge2(float &ah, float &al, float &bh, float &bl) {
        lane_merge2<LPR>(ah, al, bh, bl);
    }
    __device__ __forceinline__ bool any(bool p) { return __any_sync(kFull, p); }
    __device__ __forceinline__ int max(int v) {
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) v = ::max(v, __shfl_xor_sync(kFull, v, off));
        return v;
    }
};

// (h, l) += (oh, ol) for double-float pairs: the addition lane_merge uses
__device__ __forceinline__ void df_merge(float &h, float &l, float oh, float ol) {
    float s, e;
    two_sum(h, oh, s, e);
    e = __fadd_rn(e, __fadd_rn(l, ol));
    fast_two_sum(s, e, h, l);
}

template <int W>
struct CtaGroupSmem {
    float2 p[2][W][2];  // [buffer][warp][value]: per-warp double-float pairs
    int m[2][W];
};

// Every call is a CTA-wide barrier, so all threads of the CTA make the same
// calls.  The two buffers alternate: a thread writes buffer b only after the
// barrier of the call before, which every thread reaches only once it has read
// what the call before that left in b.
template <int W>
struct CtaGroup {
    CtaGroupSmem<W> *s;
    int t;
    __device__ explicit CtaGroup(CtaGroupSmem<W> *sm) : s(sm), t(0) {}
    __device__ __forceinline__ void merge(float &h, float &l) {
        lane_merge<32>(h, l);
        if ((threadIdx.x & 31) == 0) s->p[t][threadIdx.x >> 5][0] = make_float2(h, l);
        __syncthreads();
        float2 v = s->p[t][0][0];
        h = v.x;
        l = v.y;
#pragma unroll
        for (int w = 1; w < W; ++w) {
            v = s->p[t][w][0];
            df_merge(h, l, v.x, v.y);
        }
        t ^= 1;
    }
    __device__ __forceinline__ void merge2(float &ah, float &al, float &bh, float &bl) {
        lane_merge2<32>(ah, al, bh, bl);
        if ((threadIdx.x & 31) == 0) {
            s->p[t][threadIdx.x >> 5][0] = make_float2(ah, al);
            s->p[t][threadIdx.x >> 5][1] = make_float2(bh, bl);
        }
        __syncthreads();
        float2 a = s->p[t][0][0], b = s->p[t][0][1];
        ah = a.x;
        al = a.y;
        bh = b.x;
        bl = b.y;
#pragma unroll
        for (int w = 1; w < W; ++w) {
            a = s->p[t][w][0];
            b = s->p[t][w][1];
            df_merge(ah, al, a.x, a.y);
            df_merge(bh, bl, b.x, b.y);
        }
        t ^= 1;
    }
    __device__ __forceinline__ bool any(bool p) { return __syncthreads_or(p ? 1 : 0) != 0; }
    __device__ __forceinline__ int max(int v) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = ::max(v, __shfl_xor_sync(kFull, v, off));
        if ((threadIdx.x & 31) == 0) s->m[t][threadIdx.x >> 5] = v;
        __syncthreads();
        v = s->m[t][0];
#pragma unroll
        for (int w = 1; w < W; ++w) v = ::max(v, s->m[t][w]);
        t ^= 1;
        return v;
    }
};

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

// Row statistics of a row held in registers by LPR lanes (NVMAX 16-byte vectors
// per lane; vectors a lane does not own are zero).  Returns the float mean mh,
// the double-float low word ml and the float rstd, identical in all LPR lanes.
// FAST (bf16 only): one-pass compensated sums of x and x^2 (x^2 is exact in
// fp32 for bf16 x), with the two-pass fallback for ill-conditioned rows.
// `xv(k)` returns vector k of this lane (zero where the lane owns none).  OFFSET
// picks the x^2 accumulation: Fast2Sum against a power-of-two offset >= every
// x^2 (one extra pass over the vectors to find it), or Fast2Sum of the pair
// ordered by size (no extra pass, two more operations per element).
// UNR: how far the loops over the lane's vectors are unrolled (fully when xv(k)
// indexes a register array; partially when it reads shared memory, to keep the
// code small enough for the instruction cache).
// X2 (bf16, FAST, not OFFSET): both sums in packed f32x2 arithmetic; the even
// and odd elements of a word accumulate in the two halves of a register pair,
// which are merged with an accurate double-float addition at the end.  sum(x)
// uses TwoSum; sum(x^2) uses Fast2Sum against a power-of-two offset, found by
// an integer pass over the words (as for OFFSET).
// RMS: root-mean-square statistics (no mean): mh = ml = 0 and var = mean_d x^2.
// GRP: how the row's lanes merge (LaneGroup<LPR> by default; CtaGroup for a row
// spread over a whole CTA, LPR then being the CTA's thread count).
template <typename T, int LPR, int NVMAX, bool FAST, bool EXACT, bool OFFSET, int UNR,
          typename XV, bool X2 = false, bool RMS = false, typename GRP = LaneGroup<LPR>>
__device__ __forceinline__ void row_stats(XV xv, int li, int nv, int V, int D, float eps,
                                          float &mh, float &ml, float &rs, GRP grp = GRP()) {
    constexpr int VEC = IO<T>::VEC;
    static_assert(!X2 || (FAST && !OFFSET && VEC == 8), "packed sums: bf16 one-pass only");
    auto has = [&](int k) { return k < nv && (EXACT || li + k * LPR < V); };
    const float Df = (float)D;
    float sh = 0.f, sl = 0.f;  // sum(x) as a double-float
    float qh = 0.f, ql = 0.f;  // sum(x^2) as a double-float, offset by qsub
    float qc = 0.f;            // the offset (OFFSET, X2): a power of two >= every x^2
    float qsub = 0.f;          // what is still to be removed from qh
    int emax = -127;           // exponent of this lane's largest |x| (big-row check)
    float xmax = 0.f;          // fp32 inputs: this lane's largest |x|
    if constexpr (X2) {
        // the largest |x| in each half: max of absolute values (the sign bits of the
        // running value are meaningless and masked off at the end)
        uint32_t m = 0;
#pragma unroll(UNR)
        for (int k = 0; k < NVMAX; ++k)
            if (k < nv) {
                const V16 v = xv(k);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.w[i]));
            }
        // for non-negative bf16 the bit patterns order like the values
        const uint32_t m2 = max(m & 0x7fffu, (m >> 16) & 0x7fffu);
        const int ex = (int)((m2 >> 7) & 0xffu) - 127;  // exponent of max |x|
        emax = ex;
        qc = __int_as_float((min(max(2 * (ex + 1), -120), 120) + 127) << 23);
        const f2 QC = f2_make(qc, qc);
        f2 S = 0ull, E = 0ull, Q = QC, QE = 0ull;  // all-zero bits: (0.f, 0.f)
#pragma unroll(UNR)
        for (int k = 0; k < NVMAX; ++k) {
            if (k < nv) {
                const V16 v = xv(k);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const f2 X = f2_from_bf16x2(v.w[i]);
                    f2 t, e;
                    f2_two_sum(S, X, t, e);
                    S = t;
                    E = f2_add(E, e);
                    // Fast2Sum is exact: Q >= qc >= x^2 (x^2 is exact in fp32 for bf16 x)
                    const f2 X2v = f2_mul(X, X);
                    t = f2_add(Q, X2v);
                    QE = f2_add(QE, f2_sub(X2v, f2_sub(t, Q)));
                    Q = t;
                }
                if (k & 1) {  // renormalise every two vectors
                    f2_two_sum(S, E, S, E);
                    const f2 t = f2_add(Q, QE);
                    QE = f2_sub(QE, f2_sub(t, Q));
                    Q = t;
                }
            }
        }
        // Q - qc is exact in each half: Q >= qc, qc a power of two, Q < 2^24 qc
        Q = f2_sub(Q, QC);
        float a, b, c, d;
        f2_split(S, a, b);
        f2_split(E, c, d);
        two_sum(a, c, a, c);
        two_sum(b, d, b, d);
        df_add(a, c, b, d, sh, sl);
        f2_split(Q, a, b);
        f2_split(QE, c, d);
        two_sum(a, c, a, c);
        two_sum(b, d, b, d);
        df_add(a, c, b, d, qh, ql);
    }
    if (FAST && OFFSET) {
        // qc: a power of two >= every x^2 of this lane, so that Fast2Sum(qh, x^2)
        // is exact at every step (|qh| >= qc >= x^2); removed exactly at the end
        __nv_bfloat162 mm = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll(UNR)
        for (int k = 0; k < NVMAX; ++k)
            if (k < nv)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t a = xv(k).w[i] & 0x7fff7fffu;  // |x| of both halves
                    mm = __hmax2(mm, *reinterpret_cast<const __nv_bfloat162 *>(&a));
                }
        const uint32_t mw = *reinterpret_cast<const uint32_t *>(&mm);
        // for non-negative bf16 the bit patterns order like the values
        const uint32_t m2 = max(mw & 0xffffu, mw >> 16);
        const int e = (int)((m2 >> 7) & 0xffu) - 127;  // exponent of max |x|
        emax = e;
        const int ce = min(max(2 * (e + 1), -120), 120);
        qc = __int_as_float((ce + 127) << 23);
        qh = qc;
        qsub = qc;
    }
#pragma unroll(UNR)
    for (int k = 0; k < NVMAX; ++k) {
        if (!X2 && k < nv) {
            float f[VEC];
            IO<T>::unpack(xv(k), f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float t;
                two_sum(sh, f[e], sh, t);
                sl = __fadd_rn(sl, t);
                if (!FAST) xmax = fmaxf(xmax, fabsf(f[e]));
                if (FAST) {
                    const float q = __fmul_rn(f[e], f[e]);
                    if (OFFSET)
                        fast_two_sum(qh, q, qh, t);
                    else  // x^2 >= 0: order the pair by size and Fast2Sum is exact
                        fast_two_sum(fmaxf(qh, q), fminf(qh, q), qh, t);
                    ql = __fadd_rn(ql, t);
                }
            }
            if (k & 1) {  // renormalise every two vectors
                two_sum(sh, sl, sh, sl);
                if (FAST) fast_two_sum(qh, ql, qh, ql);
            }
        }
    }
    two_sum(sh, sl, sh, sl);
    if constexpr (X2) {
        grp.merge2(sh, sl, qh, ql);  // (qh, ql): already normalised, offset removed
    } else {
        grp.merge(sh, sl);
    }
    if constexpr (RMS) {
        mh = 0.f;
        ml = 0.f;
    } else {
        df_div_f(sh, sl, Df, mh, ml);
    }

    float vh = 0.f, vl = 0.f;
    bool two_pass = !FAST;
    if (FAST) {
        if constexpr (!X2) {
            // remove the offset: qh - qc is exact (qh >= qc, qc a power of two)
            two_sum(__fsub_rn(qh, qsub), ql, qh, ql);
            grp.merge(qh, ql);
        }
        float q2h, q2l, ph, pl;
        df_div_f(qh, ql, Df, q2h, q2l);
        if constexpr (RMS) {
            vh = q2h;  // mean_d x^2 itself: no cancellation
            vl = q2l;
            two_pass = (OFFSET || X2) && qc >= 0x1p120f;
        } else {
            two_prod(mh, mh, ph, pl);
            pl = __fmaf_rn(__fmul_rn(2.0f, mh), ml, pl);
            fast_two_sum(ph, pl, ph, pl);
            df_add(q2h, q2l, -ph, -pl, vh, vl);
            // E[x^2] - mean^2 loses log2(mean^2/var) bits: keep it only when that is small
            // (this also sends rows with |x| beyond 2^60 to the two-pass form)
            two_pass = !(ph <= 4.0f * vh) || ((OFFSET || X2) && qc >= 0x1p120f);
        }
    }
    // Warp-uniform branch: every lane takes part in the shuffles; rows that did
    // not ask for the two-pass result keep their one-pass value.
    if (grp.any(two_pass)) {
        float s2h = 0.f, s2l = 0.f;
#pragma unroll(UNR)
        for (int k = 0; k < NVMAX; ++k) {
            if (has(k)) {
                float f[VEC];
                IO<T>::unpack(xv(k), f);
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
        grp.merge(s2h, s2l);
        if (two_pass) df_div_f(s2h, s2l, Df, vh, vl);
    }

    // rstd = 1 / sqrt(var + eps), var + eps as a double-float
    float eh, el;
    two_sum(vh, eps, eh, el);
    el = __fadd_rn(el, vl);
    fast_two_sum(eh, el, eh, el);
    rs = rsqrt_df(eh, el);

    // Rows whose largest |x| reaches 2^59: x^2, the sums or the variance can leave
    // the float range.  Redo the statistics two-pass on x * 2^-k, a power of two
    // (exact) with k from the row's largest exponent, and scale the results back.
    // eps * 2^-2k is below 2^-70 of any non-zero scaled variance (bf16 or fp32
    // spacing at the row's largest value), so it only matters for a constant row.
    if constexpr (!FAST) emax = xmax > 0.f ? (int)((__float_as_uint(xmax) >> 23) & 0xffu) - 127 : -127;
    const bool big = emax >= 59;
    if (grp.any(big)) {
        emax = grp.max(emax);
        const int ks = min(max(emax - 2, 0), 126);
        const float down = __int_as_float((127 - ks) << 23), up = __int_as_float((127 + ks) << 23);
        float s1h = 0.f, s1l = 0.f;
#pragma unroll(UNR)
        for (int k = 0; k < NVMAX; ++k) {
            if (has(k)) {
                float f[VEC];
                IO<T>::unpack(xv(k), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    float t;
                    two_sum(s1h, __fmul_rn(f[e], down), s1h, t);
                    s1l = __fadd_rn(s1l, t);
                }
                two_sum(s1h, s1l, s1h, s1l);
            }
        }
        grp.merge(s1h, s1l);
        float msh = 0.f, msl = 0.f;
        if (!RMS) df_div_f(s1h, s1l, Df, msh, msl);
        float s2h = 0.f, s2l = 0.f;
#pragma unroll(UNR)
        for (int k = 0; k < NVMAX; ++k) {
            if (has(k)) {
                float f[VEC];
                IO<T>::unpack(xv(k), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    float dh, de, p, pe, t;
                    two_sum(__fmul_rn(f[e], down), -msh, dh, de);
                    de = __fsub_rn(de, msl);
                    two_prod(dh, dh, p, pe);
                    pe = __fmaf_rn(de, __fmaf_rn(2.0f, dh, de), pe);
                    two_sum(s2h, p, s2h, t);
                    s2l = __fadd_rn(s2l, __fadd_rn(t, pe));
                }
                fast_two_sum(s2h, s2l, s2h, s2l);
            }
        }
        grp.merge(s2h, s2l);
        float vsh, vsl;
        df_div_f(s2h, s2l, Df, vsh, vsl);
        if (big) {
            mh = __fmul_rn(msh, up);
            ml = __fmul_rn(msl, up);
            rs = (vsh == 0.0f) ? rsqrt_df(eps, 0.0f) : __fmul_rn(rsqrt_df(vsh, vsl), down);
        }
    }
}

// y for one 16-byte vector given the row statistics, as fp32 values; s, b are
// (scale, shift).  `wide` rows (|mean| * rstd > 4: the mean is far from the
// values' spread, or so large that x * rstd would overflow) always take the
// centred form (x - mean) * rstd.
template <typename T, bool FAST>
__device__ __forceinline__ void modulate_vals(const V16 &xvk, const float *s, const float *b,
                                              float mh, float ml, float rs, bool wide,
                                              float (&o)[IO<T>::VEC]) {
    constexpr int VEC = IO<T>::VEC;
    float f[VEC];
    IO<T>::unpack(xvk, f);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const float s1 = 1.0f + s[e];
        if (FAST && !wide) {
            // y = A x + B with A = rstd (1 + scale), B = shift - mean A: |mean| rstd <= 4,
            // so B's rounding stays far below bf16's
            const float A = __fmul_rn(rs, s1);
            o[e] = __fmaf_rn(f[e], A, __fmaf_rn(-mh, A, b[e]));
        } else {
            // x - mean with the mean's low word: x - mh is exact near the mean
            // (Sterbenz), so rows whose |mean| >> std keep full fp32 accuracy
            const float d = __fsub_rn(__fsub_rn(f[e], mh), ml);
            o[e] = fmaf(d * rs, s1, b[e]);
        }
    }
}

}  // namespace
}  // namespace adaln
