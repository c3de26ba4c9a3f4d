// common.cuh -- device helpers shared by the AdaLN kernels (sm_103a).
//
// * 16-byte vector I/O: every activation access is one 128-bit load or store
//   per thread, so a warp touches 512 contiguous bytes per instruction.
// * bf16 <-> fp32 conversion (bf16 is the top half of an fp32 word, so widening
//   is a shift or a mask; narrowing rounds to nearest-even once).
// * Error-free transformations for the compensated row statistics: Knuth's
//   TwoSum, Dekker's Fast2Sum and the FMA-based TwoProd, and a double-float
//   (pair of floats) addition built from them.  Written with explicit
//   round-to-nearest intrinsics so the compiler cannot contract or reorder them.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace adaln {

struct alignas(16) V16 {
    uint32_t w[4];
};

// Streaming load (read once): no L1 allocation, read-only path.
__device__ __forceinline__ V16 ld_stream(const void *p) {
    V16 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
        : "l"(p));
    return v;
}

// Cached read-only load (modulation rows, reused by every row of a segment).
// volatile: kept in program order, so the compiler does not hoist a whole row
// of these loads ahead of their use (which costs registers, not latency: they
// hit in L1).
__device__ __forceinline__ V16 ld_cached(const void *p) {
    V16 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_vec(void *p, const V16 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]),
                 "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
}

// ----------------------------------------------------------------- element I/O

// Element-type traits: VEC elements per 16-byte vector; unpack to / pack from fp32.
template <typename T>
struct IO;

template <>
struct IO<float> {
    static constexpr int VEC = 4;
    __device__ __forceinline__ static void unpack(const V16 &v, float (&f)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(v.w[i]);
    }
    __device__ __forceinline__ static V16 pack(const float (&f)[4]) {
        V16 v;
#pragma unroll
        for (int i = 0; i < 4; ++i) v.w[i] = __float_as_uint(f[i]);
        return v;
    }
};

template <>
struct IO<__nv_bfloat16> {
    static constexpr int VEC = 8;
    // element 2i is the low half of word i, element 2i+1 the high half
    __device__ __forceinline__ static void unpack(const V16 &v, float (&f)[8]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(v.w[i] << 16);
            f[2 * i + 1] = __uint_as_float(v.w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static V16 pack(const float (&f)[8]) {
        V16 v;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            v.w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return v;
    }
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// ----------------------------------------------------------------- error-free transforms

// Knuth TwoSum: s + e == a + b exactly, s = fl(a + b).  No ordering precondition.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float ea = __fsub_rn(a, __fsub_rn(s, bb));
    const float eb = __fsub_rn(b, bb);
    e = __fadd_rn(ea, eb);
}

// Dekker Fast2Sum: exact when |a| >= |b| (or a == 0).
__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

// TwoProd with FMA: p + e == a * b exactly (barring under/overflow).
__device__ __forceinline__ void two_prod(float a, float b, float &p, float &e) {
    p = __fmul_rn(a, b);
    e = __fmaf_rn(a, b, -p);
}

// Accurate double-float addition (Shewchuk/Dekker style, both pairs normalised).
__device__ __forceinline__ void df_add(float ah, float al, float bh, float bl, float &rh,
                                       float &rl) {
    float s, e, t, f;
    two_sum(ah, bh, s, e);
    two_sum(al, bl, t, f);
    e = __fadd_rn(e, t);
    fast_two_sum(s, e, s, e);
    e = __fadd_rn(e, f);
    fast_two_sum(s, e, rh, rl);
}

// Double-float divided by a float d (exactly representable, > 0).
__device__ __forceinline__ void df_div_f(float ah, float al, float d, float &qh, float &ql) {
    qh = __fdiv_rn(ah, d);
    // remainder of a correctly rounded quotient is exact and the FMA returns it exactly
    const float rem = __fmaf_rn(-qh, d, ah);
    ql = __fdiv_rn(__fadd_rn(rem, al), d);
    fast_two_sum(qh, ql, qh, ql);
}

// ----------------------------------------------------------------- packed pairs
//
// Two fp32 lanes in one 64-bit register (sm_100+ f32x2 arithmetic): one
// instruction does the same correctly rounded operation on both halves, which
// halves the issue slots of the compensated sums and of the modulation.  The
// operations are written with .rn so nothing contracts or reorders them.
typedef unsigned long long f2;

__device__ __forceinline__ f2 f2_make(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f2 a, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f2 f2_from_words(uint32_t lo, uint32_t hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
// the two bf16 of a 32-bit word (element 2i low, 2i+1 high) widened to fp32
__device__ __forceinline__ f2 f2_from_bf16x2(uint32_t w) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(w << 16), "r"(w & 0xffff0000u));
    return r;
}
// both halves rounded to bf16 (nearest-even) into one word, low half first
__device__ __forceinline__ uint32_t f2_to_bf16x2(f2 a) {
    float lo, hi;
    f2_split(a, lo, hi);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// A 16-byte vector as packed element pairs (element 2i low, 2i+1 high): four
// pairs of bf16, two pairs of fp32.
template <typename T>
struct Pairs;

template <>
struct Pairs<__nv_bfloat16> {
    static constexpr int NP = 4;
    __device__ __forceinline__ static void unpack(const V16 &v, f2 (&p)[4]);
    __device__ __forceinline__ static V16 pack(const f2 (&p)[4]);
};

template <>
struct Pairs<float> {
    static constexpr int NP = 2;
    __device__ __forceinline__ static void unpack(const V16 &v, f2 (&p)[2]);
    __device__ __forceinline__ static V16 pack(const f2 (&p)[2]);
};

// TwoSum on both halves: s + e == a + b exactly, s = fl(a + b)
__device__ __forceinline__ void f2_two_sum(f2 a, f2 b, f2 &s, f2 &e) {
    s = f2_add(a, b);
    const f2 bb = f2_sub(s, a);
    e = f2_add(f2_sub(a, f2_sub(s, bb)), f2_sub(b, bb));
}

__device__ __forceinline__ void Pairs<__nv_bfloat16>::unpack(const V16 &v, f2 (&p)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = f2_from_bf16x2(v.w[i]);
}
__device__ __forceinline__ V16 Pairs<__nv_bfloat16>::pack(const f2 (&p)[4]) {
    V16 v;
#pragma unroll
    for (int i = 0; i < 4; ++i) v.w[i] = f2_to_bf16x2(p[i]);
    return v;
}
__device__ __forceinline__ void Pairs<float>::unpack(const V16 &v, f2 (&p)[2]) {
#pragma unroll
    for (int i = 0; i < 2; ++i) p[i] = f2_from_words(v.w[2 * i], v.w[2 * i + 1]);
}
__device__ __forceinline__ V16 Pairs<float>::pack(const f2 (&p)[2]) {
    V16 v;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float lo, hi;
        f2_split(p[i], lo, hi);
        v.w[2 * i] = __float_as_uint(lo);
        v.w[2 * i + 1] = __float_as_uint(hi);
    }
    return v;
}

// ----------------------------------------------------------------- segments

// Segment of `row` among packed segments: the largest k with offsets[k] <= row
// (empty segments are skipped because their start equals the next one's).
__device__ __forceinline__ int64_t find_segment(const int64_t *__restrict__ offsets,
                                                int64_t nseg, int64_t row) {
    int64_t lo = 0, hi = nseg;  // invariant: offsets[lo] <= row < offsets[hi]
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if (__ldg(offsets + mid) <= row)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// a / b for a >= 0 and b > 0, by 32-bit division when both fit in 32 bits: the
// 64-bit integer division is a far longer instruction sequence, and in the
// short kernels (column sums, the gated residual on small rows) it was most of
// a warp's instructions
__device__ __forceinline__ int64_t div_nonneg(int64_t a, int64_t b) {
    if ((((uint64_t)a | (uint64_t)b) >> 32) == 0)
        return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

// Modulation row of segment k: mod_index[k], or k itself when there is no index.
__device__ __forceinline__ int64_t mod_row(const int32_t *__restrict__ mod_index, int64_t k) {
    return mod_index != nullptr ? (int64_t)__ldg(mod_index + k) : k;
}

// The same search done by a whole warp (every lane calls it with the same
// arguments and gets the same result): each round probes 32 evenly spaced
// offsets at once and keeps the sub-range after the last probe <= row, so 1024
// segments take two rounds of loads instead of ten dependent ones.  Whatever
// the offsets hold, the result stays in [0, nseg).
__device__ __forceinline__ int64_t find_segment_warp(const int64_t *__restrict__ offsets,
                                                     int64_t nseg, int64_t row, int lane) {
    int64_t lo = 0, hi = nseg;
    while (hi - lo > 1) {
        const int64_t step = (hi - lo + 31) / 32;
        const int64_t p = lo + (int64_t)lane * step;
        const bool le = p < hi && __ldg(offsets + p) <= row;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        const int j = m ? 31 - __clz((int)m) : 0;
        lo += (int64_t)j * step;
        hi = min(hi, lo + step);
    }
    return lo;
}

}  // namespace adaln

// ----------------------------------------------------------------- launches

namespace adaln {

// Launch `kern` on `stream` with programmatic stream serialisation allowed
// (see pdl_wait).  Returns the launch status.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace adaln

// ----------------------------------------------------------------- async copies (sm_90+)
//
// Bulk copies global -> shared complete on an mbarrier (transaction bytes);
// every wait on an mbarrier is bounded: after kWaitLimit polls the caller gets
// `false` and must record an error and stop instead of spinning forever.
namespace adaln {

// Polls before a wait gives up.  ADALN_TEST_WAIT_LIMIT shortens it in the test
// build whose producers drop their last copy (ADALN_TEST_DROP_LAST_COPY), so that
// a test can watch a wait run out and the kernel return with an error status.
#ifdef ADALN_TEST_WAIT_LIMIT
constexpr uint32_t kWaitLimit = ADALN_TEST_WAIT_LIMIT;
#else
constexpr uint32_t kWaitLimit = 1u << 24;
#endif
#ifdef ADALN_TEST_DROP_LAST_COPY
constexpr bool kTestDropLastCopy = true;
#else
constexpr bool kTestDropLastCopy = false;
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// L2 prefetch of `bytes` (a multiple of 16) at a 16-byte aligned global address
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// make barrier initialisation visible to the async (bulk-copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          uint32_t limit = kWaitLimit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// the shorter limit of a wait that only drains a copy already issued, once a
// wait of the same thread has given up (a copy in flight lands in microseconds)
constexpr uint32_t kDrainLimit = 1u << 12;

// 1-D bulk copy global -> shared; src, dst 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 4-byte asynchronous copy global -> shared (no register round trip)
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}

// one arrival on `bar` once all of this thread's earlier cp.async copies have landed
// (.noinc: the arrival is part of the barrier's initial count)
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 16-byte shared load at a 32-bit shared-window address
__device__ __forceinline__ V16 lds128_at(uint32_t a) {
    V16 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "r"(a));
    return v;
}

__device__ __forceinline__ V16 lds128(const void *p) {
    V16 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "r"(smem_u32(p)));
    return v;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation, so it may start while the kernel before it
// on the stream drains.  pdl_wait() blocks until that kernel has completed and
// its memory is visible; each kernel calls it before its first global access
// (only CTA-local setup runs earlier).  pdl_trigger() lets the next kernel on
// the stream be scheduled; a kernel that never calls it triggers on exit.
// The persistent kernels that take most of an SM's shared memory (the bulk-copy
// rings) never trigger early: the next kernel's CTAs would become resident
// beside them and run under their shared-memory/L1 split, with a small L1.  The
// gated-residual stream, whose loads go through L1, lost about 15% of its
// bandwidth that way on the Wan and ragged chains.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// barrier among `nthreads` threads (a multiple of 32) on hardware barrier `id` (1..15)
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// the same barrier, which also returns whether any of the `nthreads` threads
// passed a non-zero `flag` (a reduction done by the barrier itself)
__device__ __forceinline__ bool named_barrier_any(int id, int nthreads, int flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(flag), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

}  // namespace adaln
