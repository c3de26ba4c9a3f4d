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
template <typename T, int LPR, int NVMAX, bool FAST, bool EXACT, bool OFFSET, int UNR,
          typename XV, bool X2 = false>
__device__ __forceinline__ void row_stats(XV xv, int li, int nv, int V, int D, float eps,
                                          float &mh, float &ml, float &rs) {
    constexpr int VEC = IO<T>::VEC;
    static_assert(!X2 || (FAST && !OFFSET && VEC == 8), "packed sums: bf16 one-pass only");
    auto has = [&](int k) { return k < nv && (EXACT || li + k * LPR < V); };
    const float Df = (float)D;
    float sh = 0.f, sl = 0.f;  // sum(x) as a double-float
    float qh = 0.f, ql = 0.f;  // sum(x^2) as a double-float, offset by qsub
    float qc = 0.f;            // the offset (OFFSET, X2): a power of two >= every x^2
    float qsub = 0.f;          // what is still to be removed from qh
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
        lane_merge2<LPR>(sh, sl, qh, ql);  // (qh, ql): already normalised, offset removed
    } else {
        lane_merge<LPR>(sh, sl);
    }
    df_div_f(sh, sl, Df, mh, ml);

    float vh = 0.f, vl = 0.f;
    bool two_pass = !FAST;
    if (FAST) {
        if constexpr (!X2) {
            // remove the offset: qh - qc is exact (qh >= qc, qc a power of two)
            two_sum(__fsub_rn(qh, qsub), ql, qh, ql);
            lane_merge<LPR>(qh, ql);
        }
        float q2h, q2l, ph, pl;
        df_div_f(qh, ql, Df, q2h, q2l);
        two_prod(mh, mh, ph, pl);
        pl = __fmaf_rn(__fmul_rn(2.0f, mh), ml, pl);
        fast_two_sum(ph, pl, ph, pl);
        df_add(q2h, q2l, -ph, -pl, vh, vl);
        // E[x^2] - mean^2 loses log2(mean^2/var) bits: keep it only when that is small
        // (this also sends rows with |x| beyond 2^60 to the two-pass form)
        two_pass = !(ph <= 4.0f * vh) || ((OFFSET || X2) && qc >= 0x1p120f);
    }
    // Warp-uniform branch: every lane takes part in the shuffles; rows that did
    // not ask for the two-pass result keep their one-pass value.
    if (__any_sync(kFull, two_pass)) {
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
        lane_merge<LPR>(s2h, s2l);
        if (two_pass) df_div_f(s2h, s2l, Df, vh, vl);
    }

    // rstd = 1 / sqrt(var + eps), var + eps as a double-float
    float eh, el;
    two_sum(vh, eps, eh, el);
    el = __fadd_rn(el, vl);
    fast_two_sum(eh, el, eh, el);
    rs = rsqrt_df(eh, el);
}

// y for one 16-byte vector given the row statistics, as fp32 values; s, b are
// (scale, shift).
template <typename T, bool FAST>
__device__ __forceinline__ void modulate_vals(const V16 &xvk, const float *s, const float *b,
                                              float mh, float ml, float rs,
                                              float (&o)[IO<T>::VEC]) {
    constexpr int VEC = IO<T>::VEC;
    float f[VEC];
    IO<T>::unpack(xvk, f);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const float s1 = 1.0f + s[e];
        if (FAST) {
            // y = A x + B with A = rstd (1 + scale), B = shift - mean A; the fast path
            // has |mean| rstd <= 2, so B's rounding stays far below bf16's
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

// y = LN(x) * (1 + scale) + shift for rows of D elements; a row is owned by LPR
// lanes (32 / LPR rows per warp), each holding up to NVMAX 16-byte vectors.
// EXACT: D == LPR * NVMAX * VEC, so no lane needs a bounds predicate.
// GATED: also out = r + gate[k] * y from the fp32 y (the gated residual applied
// to the modulated output itself); y is then written only if it is not null.
template <typename T, int LPR, int NVMAX, bool FAST, bool EXACT, bool GATED>
__global__ void __launch_bounds__(kFwdThreads, 2)
    adaln_fwd_kernel(const T *__restrict__ x, const T *__restrict__ shift,
                     const T *__restrict__ scale, T *__restrict__ y, float *__restrict__ mean,
                     float *__restrict__ rstd, int64_t rows, int D, int nv, float eps,
                     int64_t seg_rows, const int64_t *__restrict__ offsets, int64_t nseg,
                     const T *__restrict__ gate, const T *__restrict__ r, T *__restrict__ out) {
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
    row_stats<T, LPR, NVMAX, FAST, EXACT, true, NVMAX>(
        [&](int k) -> const V16 & { return xv[k]; }, li, nv, V, D, eps, mh, ml, rs);

    if (!active) return;
    if (li == 0) {
        mean[row] = mh;
        rstd[row] = rs;
    }
    // ---- modulation: one more traversal of the registers, one HBM write
    const int64_t k_seg = offsets ? find_segment(offsets, nseg, row) : row / seg_rows;
    const T *shr = shift + k_seg * D;
    const T *scr = scale + k_seg * D;
    T *yr = y != nullptr ? y + row * (int64_t)D : nullptr;
#pragma unroll
    for (int k = 0; k < NVMAX; ++k) {
        const int v = li + k * LPR;
        if (has(k)) {
            float s[VEC], b[VEC], yv[VEC];
            IO<T>::unpack(ld_cached(scr + (int64_t)v * VEC), s);
            IO<T>::unpack(ld_cached(shr + (int64_t)v * VEC), b);
            modulate_vals<T, FAST>(xv[k], s, b, mh, ml, rs, yv);
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

// ------------------------------------------------------------------ fwd ring
//
// Persistent forward for bf16 rows with a whole number of vectors per lane.
// Each CTA owns a contiguous range of rows, cut at segment boundaries into
// pieces.  For every piece the consumers stage the segment's modulation row in
// shared memory as fp32 (1 + scale, shift), then process the piece's "units"
// (32/LPR consecutive rows, one per warp row-group): the CTA's units are
// numbered across pieces and unit g goes to consumer warp g % C (computed, not
// counted per warp, so the producer keeps no per-warp state in local memory).  One producer lane streams the units with
// cp.async.bulk into per-warp rings of one or two shared-memory slots; a warp
// reads its unit from shared memory in each pass (statistics, then modulation)
// and then frees the slot.  Every mbarrier wait is bounded.
constexpr int kFwdRingWarps = 16;
constexpr int kFwdMaxSlots = 2;

// non-zero once a bounded wait in the pipelined forward gave up (never expected)
__device__ int g_fwd_status;

// slots, the (1+scale, shift) table, the barriers and (gated) the raw gate row
__host__ __device__ inline uint32_t fwd_ring_smem(int D, int RPW, int slots, bool gated) {
    const uint32_t unit = (uint32_t)RPW * D * 2u;
    return (uint32_t)kFwdRingWarps * slots * unit + 2u * D * 4u +
           2u * kFwdRingWarps * kFwdMaxSlots * 8u + (gated ? (uint32_t)D * 2u : 0u);
}

// L2 prefetch of `bytes` (a multiple of 16) at a 16-byte aligned global address
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// [start, end) of the segment holding `row` (32-bit: the ring runs below 2^31 rows)
__device__ __forceinline__ void segment_of(int row, int seg_rows, const int64_t *offsets,
                                           int nseg, int &seg, int &end) {
    if (offsets) {
        seg = (int)find_segment(offsets, nseg, row);
        end = (int)__ldg(offsets + seg + 1);
    } else {
        seg = row / seg_rows;
        end = (seg + 1) * seg_rows;
    }
}

// GATED: out = r + gate[k] * y from the fp32 y; the producer prefetches each
// unit's rows of r into L2 when it issues the unit, the consumers read them
// with streaming loads and take the gate row from shared memory; y is written
// only if it is not null.
template <int LPR, int NV, bool GATED>
__global__ void __launch_bounds__(32 * (kFwdRingWarps + 1), 1)
    adaln_fwd_ring_kernel(const __nv_bfloat16 *__restrict__ x,
                          const __nv_bfloat16 *__restrict__ shift,
                          const __nv_bfloat16 *__restrict__ scale, __nv_bfloat16 *__restrict__ y,
                          float *__restrict__ mean, float *__restrict__ rstd, int rows,
                          int D, float eps, int seg_rows, const int64_t *__restrict__ offsets,
                          int nseg, int rows_per_cta, int slots,
                          const __nv_bfloat16 *__restrict__ gate,
                          const __nv_bfloat16 *__restrict__ r, __nv_bfloat16 *__restrict__ out) {
    using T = __nv_bfloat16;
    constexpr int VEC = 8;
    constexpr int RPW = 32 / LPR;
    constexpr int C = kFwdRingWarps;
    int *status = &g_fwd_status;
    extern __shared__ __align__(128) unsigned char smem[];
    const int V = D / VEC;
    const uint32_t unit_bytes = (uint32_t)RPW * D * 2u;
    // modulation table, interleaved so that consecutive lanes read consecutive
    // 16-byte words: (1+scale) columns 8v..8v+3 at [v], 8v+4..8v+7 at [V+v];
    // shift likewise at [2V+v] and [3V+v]
    float4 *tab = reinterpret_cast<float4 *>(smem + (size_t)C * slots * unit_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(tab + 4 * V);
    uint64_t *empty = full + C * kFwdMaxSlots;
    V16 *gtab = reinterpret_cast<V16 *>(empty + C * kFwdMaxSlots);  // gated: raw gate row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 32-bit row arithmetic (the launcher uses this kernel only below 2^30 rows)
    const int r_begin = blockIdx.x * rows_per_cta;
    const int r_end = min(rows, r_begin + rows_per_cta);
    if (r_begin >= r_end) return;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C * kFwdMaxSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    if (warp == C) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        int g = 0;  // units handed out so far (unit g goes to warp g % C)
        for (int p0 = r_begin; p0 < r_end;) {
            int seg, p1;
            segment_of(p0, seg_rows, offsets, nseg, seg, p1);
            p1 = min(p1, r_end);
            const int nu = (p1 - p0 + RPW - 1) / RPW;
            for (int u = 0; u < nu; ++u, ++g) {
                const int w = g % C;
                const int j = g / C;
                const int s = j % slots;
                uint64_t *f = &full[w * kFwdMaxSlots + s];
                if (j >= slots &&
                    !mbar_wait(&empty[w * kFwdMaxSlots + s], (uint32_t)((j / slots) - 1) & 1u)) {
                    atomicExch(status, 3);
                    return;
                }
                const int row0 = p0 + u * RPW;
                const uint32_t bytes = (uint32_t)min(RPW, p1 - row0) * (uint32_t)D * 2u;
                mbar_arrive_expect_tx(f, bytes);
                bulk_g2s(smem + (size_t)(w * slots + s) * unit_bytes, x + (int64_t)row0 * D,
                         bytes, f);
                if (GATED) prefetch_l2(r + (int64_t)row0 * D, bytes);
            }
            p0 = p1;
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int li = lane % LPR;
    const int sub = lane / LPR;
    const int ncons = C * 32;
    int g0 = 0;  // global index of the piece's first unit
    for (int p0 = r_begin; p0 < r_end;) {
        int seg, p1;
        segment_of(p0, seg_rows, offsets, nseg, seg, p1);
        p1 = min(p1, r_end);
        // stage this piece's modulation row (after every warp is done with the last one)
        named_barrier(1, ncons);
        for (int v = threadIdx.x; v < V; v += ncons) {
            float sc[VEC], sh[VEC];
            IO<T>::unpack(ld_cached(scale + (int64_t)seg * D + v * VEC), sc);
            IO<T>::unpack(ld_cached(shift + (int64_t)seg * D + v * VEC), sh);
            tab[v] = make_float4(1.0f + sc[0], 1.0f + sc[1], 1.0f + sc[2], 1.0f + sc[3]);
            tab[V + v] = make_float4(1.0f + sc[4], 1.0f + sc[5], 1.0f + sc[6], 1.0f + sc[7]);
            tab[2 * V + v] = make_float4(sh[0], sh[1], sh[2], sh[3]);
            tab[3 * V + v] = make_float4(sh[4], sh[5], sh[6], sh[7]);
            if (GATED) gtab[v] = ld_cached(gate + (int64_t)seg * D + v * VEC);
        }
        named_barrier(1, ncons);

        const int nu = (p1 - p0 + RPW - 1) / RPW;
        for (int u = ((warp - g0) % C + C) % C; u < nu; u += C) {
            const int j = (g0 + u) / C;
            const int s = j % slots;
            if (!mbar_wait(&full[warp * kFwdMaxSlots + s], (uint32_t)(j / slots) & 1u)) {
                atomicExch(status, 4);
                return;
            }
            const int row = p0 + u * RPW + sub;
            const bool active = row < p1;
            const unsigned char *src =
                smem + (size_t)(warp * slots + s) * unit_bytes + (size_t)sub * D * 2u;
            // the row stays in shared memory and is read once per pass
            auto xv = [&](int k) -> V16 {
                return active ? lds128(src + (size_t)(li + k * LPR) * 16) : V16{{0u, 0u, 0u, 0u}};
            };
            float mh, ml, rs;
            row_stats<T, LPR, NV, true, true, false, 2, decltype(xv), true>(xv, li, NV, LPR * NV,
                                                                           D, eps, mh, ml, rs);
            // y = (x rstd + n) (1 + scale) + shift with n = -mean rstd as a double-float
            // (nh + nl), in packed pairs: x rstd + nh is one rounding of a value of the
            // order of the normalised x.  nl matters only where |n| is large (|mean| >>
            // std); elsewhere it is below the half-ulp of y and the add is skipped.
            const float nh = __fmul_rn(-mh, rs);
            const float nl = __fmaf_rn(-ml, rs, __fmaf_rn(-mh, rs, -nh));
            const bool wide = __any_sync(kFull, active && !(fabsf(nh) <= 4.0f));
            const f2 RS = f2_make(rs, rs), NH = f2_make(nh, nh), NL = f2_make(nl, nl);
            T *yr = y != nullptr ? y + (int64_t)row * D : nullptr;
            auto modulate = [&](auto wide_c) {
                constexpr bool W = decltype(wide_c)::value;
#pragma unroll 2
                for (int k = 0; k < NV; ++k) {
                    const int v = li + k * LPR;
                    // (volatile shared loads keep the table reads next to their use)
                    const V16 t0 = lds128(tab + v), t1 = lds128(tab + V + v);
                    const V16 t2 = lds128(tab + 2 * V + v), t3 = lds128(tab + 3 * V + v);
                    const V16 xk = xv(k);
                    V16 o, og;
                    V16 rk, gk;
                    if constexpr (GATED) {
                        rk = ld_stream(r + (int64_t)row * D + v * VEC);
                        gk = lds128(gtab + v);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const V16 &ts = i < 2 ? t0 : t1;
                        const V16 &tb = i < 2 ? t2 : t3;
                        const int j = 2 * (i & 1);
                        f2 U = f2_fma(f2_from_bf16x2(xk.w[i]), RS, NH);
                        if (W) U = f2_add(U, NL);
                        const f2 Y = f2_fma(U, f2_from_words(ts.w[j], ts.w[j + 1]),
                                            f2_from_words(tb.w[j], tb.w[j + 1]));
                        o.w[i] = f2_to_bf16x2(Y);
                        if constexpr (GATED)
                            og.w[i] = f2_to_bf16x2(f2_fma(f2_from_bf16x2(gk.w[i]), Y,
                                                          f2_from_bf16x2(rk.w[i])));
                    }
                    if (yr != nullptr) st_vec(yr + v * VEC, o);
                    if constexpr (GATED) st_vec(out + (int64_t)row * D + v * VEC, og);
                }
            };
            if (active) {
                if (li == 0) {
                    mean[row] = mh;
                    rstd[row] = rs;
                }
                if (wide)
                    modulate(std::true_type{});
                else
                    modulate(std::false_type{});
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[warp * kFwdMaxSlots + s]);  // done with the slot
        }
        g0 += nu;
        p0 = p1;
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
    pdl_wait();
    pdl_trigger();
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

template <typename T, int LPR, int NVMAX, bool FAST, bool EXACT>
cudaError_t fwd_launch_one(const void *x, const void *shift, const void *scale, void *y,
                           float *mean, float *rstd, const Segments &sg, int D, int nv,
                           float eps, const GateEpilogue &ge, cudaStream_t stream) {
    constexpr int rows_per_block = (kFwdThreads / 32) * (32 / LPR);
    const int64_t blocks = (sg.rows + rows_per_block - 1) / rows_per_block;
    auto kern = ge.out != nullptr ? adaln_fwd_kernel<T, LPR, NVMAX, FAST, EXACT, true>
                                  : adaln_fwd_kernel<T, LPR, NVMAX, FAST, EXACT, false>;
    const cudaError_t err = launch_pdl(
        kern, dim3((unsigned)blocks), dim3(kFwdThreads), 0, stream, (const T *)x,
        (const T *)shift, (const T *)scale, (T *)y, mean, rstd, sg.rows, D, nv, eps, sg.seg_rows,
        sg.offsets, sg.nseg, (const T *)ge.gate, (const T *)ge.r, (T *)ge.out);
    count_launch();
    return err;
}

// rows whose vector count is not an exact multiple: NVMAX classes with a runtime count
template <typename T, int LPR, bool FAST>
cudaError_t fwd_by_nv(const void *x, const void *shift, const void *scale, void *y, float *mean,
                      float *rstd, const Segments &sg, int D, int nv, float eps,
                      const GateEpilogue &ge, cudaStream_t s) {
#define ADALN_NV_CASE(NVM)                                                                  \
    if (nv <= NVM)                                                                          \
        return fwd_launch_one<T, LPR, NVM, FAST, false>(x, shift, scale, y, mean, rstd, sg, D, \
                                                        nv, eps, ge, s);
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

// shared-memory slots per consumer warp that fit (0: the ring does not fit)
inline int fwd_ring_slots(int D, int RPW, bool gated, int smem_optin) {
    for (int sl = kFwdMaxSlots; sl >= 1; --sl)
        if (fwd_ring_smem(D, RPW, sl, gated) + 1024 <= (uint32_t)smem_optin) return sl;
    return 0;
}

template <int LPR, int NV>
cudaError_t fwd_ring_launch(const void *x, const void *shift, const void *scale, void *y,
                            float *mean, float *rstd, const Segments &sg, int D, float eps,
                            const GateEpilogue &ge, const DeviceInfo &di, cudaStream_t stream) {
    constexpr int RPW = 32 / LPR;
    constexpr int C = kFwdRingWarps;
    const bool gated = ge.out != nullptr;
    const int slots = fwd_ring_slots(D, RPW, gated, di.max_smem_optin);
    const uint32_t smem = fwd_ring_smem(D, RPW, slots, gated);
    auto kern = gated ? adaln_fwd_ring_kernel<LPR, NV, true> : adaln_fwd_ring_kernel<LPR, NV, false>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int64_t units = (sg.rows + RPW - 1) / RPW;
    int64_t grid = (units + C - 1) / C;
    if (grid > di.sms) grid = di.sms;
    int64_t rpc = (sg.rows + grid - 1) / grid;
    rpc = (rpc + RPW - 1) / RPW * RPW;
    grid = (sg.rows + rpc - 1) / rpc;
    using B16 = __nv_bfloat16;
    err = launch_pdl(kern, dim3((unsigned)grid), dim3(32 * (C + 1)), smem, stream, (const B16 *)x,
                     (const B16 *)shift, (const B16 *)scale, (B16 *)y, mean, rstd, (int)sg.rows, D,
                     eps, (int)sg.seg_rows, sg.offsets, (int)sg.nseg, (int)rpc, slots,
                     (const B16 *)ge.gate, (const B16 *)ge.r, (B16 *)ge.out);
    count_launch();
    return err;
}

}  // namespace

int64_t max_dim(DType dt) {
    // 24 vectors of 16 bytes per lane, 32 lanes per row
    return dt == DType::BF16 ? 24 * 32 * 8 : 24 * 32 * 4;
}

int pipeline_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fwd_status, sizeof(int)) != cudaSuccess) return -1;
    return v;
}

cudaError_t launch_fwd(DType dt, const void *x, const void *shift, const void *scale, void *y,
                       float *mean, float *rstd, const Segments &sg, int64_t D64, float eps,
                       cudaStream_t stream, const GateEpilogue &ge) {
    if (sg.rows == 0) return cudaSuccess;
    const int D = (int)D64;
    const bool gated = ge.out != nullptr;
    if (dt == DType::BF16) {
        using B16 = __nv_bfloat16;
        const int V = D / 8;
        DeviceInfo di;
        cudaError_t err = device_info(di);
        if (err != cudaSuccess) return err;
        // pipelined forward for whole-vector shapes that fit the shared-memory ring
        const bool ring_ok = sg.rows < (int64_t)1 << 30 && sg.nseg < (int64_t)1 << 30 &&
                             sg.seg_rows < (int64_t)1 << 30;
#define ADALN_RING(LPR, NV)                                                                \
    if (ring_ok && V == (LPR) * (NV) &&                                                    \
        fwd_ring_slots(D, 32 / (LPR), gated, di.max_smem_optin) > 0)                       \
        return fwd_ring_launch<LPR, NV>(x, shift, scale, y, mean, rstd, sg, D, eps, ge, di, \
                                        stream);
        ADALN_RING(16, 24)  // D = 3072: two rows per unit halve the per-row work per element
        ADALN_RING(32, 4)
        ADALN_RING(32, 8)
        ADALN_RING(32, 12)
        ADALN_RING(32, 16)
        ADALN_RING(32, 20)
        ADALN_RING(32, 24)
        ADALN_RING(16, 9)
#undef ADALN_RING
        // exact shapes: a warp per row with a whole number of vectors per lane
#define ADALN_EXACT(LPR, NV)                                                                  \
    if (V == (LPR) * (NV))                                                                    \
        return fwd_launch_one<B16, LPR, NV, true, true>(x, shift, scale, y, mean, rstd, sg, D, \
                                                        NV, eps, ge, stream);
        ADALN_EXACT(32, 24)
#undef ADALN_EXACT
        // small rows: 8 lanes per row (4 rows per warp); otherwise a full warp per row
        if (V <= 8 * 8) {
            const int nv = (V + 7) / 8;
            return fwd_by_nv<B16, 8, true>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, ge,
                                           stream);
        }
        const int nv = (V + 31) / 32;
        return fwd_by_nv<B16, 32, true>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, ge, stream);
    }
    const int V = D / 4;
    if (V <= 8 * 8) {
        const int nv = (V + 7) / 8;
        return fwd_by_nv<float, 8, false>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, ge,
                                          stream);
    }
    const int nv = (V + 31) / 32;
    return fwd_by_nv<float, 32, false>(x, shift, scale, y, mean, rstd, sg, D, nv, eps, ge, stream);
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
        err = launch_pdl(gate_fwd_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0,
                         stream, (const __nv_bfloat16 *)r, (const __nv_bfloat16 *)z,
                         (const __nv_bfloat16 *)gate, (__nv_bfloat16 *)out, sg.rows, D, rpw,
                         sg.seg_rows, sg.offsets, sg.nseg);
    else
        err = launch_pdl(gate_fwd_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, stream,
                         (const float *)r, (const float *)z, (const float *)gate, (float *)out,
                         sg.rows, D, rpw, sg.seg_rows, sg.offsets, sg.nseg);
    count_launch();
    return err;
}

}  // namespace adaln
