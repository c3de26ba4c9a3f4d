// fwd_ring.cu -- the pipelined (bulk-copy ring) AdaLN forward, bf16 rows.
#include "fwd_stats.cuh"
#include "tmem.cuh"

namespace adaln {
namespace {

// ------------------------------------------------------------------ fwd ring
//
// Persistent forward for bf16 rows with a whole number of vectors per lane.
// Each CTA owns a contiguous range of rows, cut at segment boundaries into
// pieces.  For every piece the consumers stage the segment's modulation row as
// fp32 (1 + scale, shift), then process the piece's "units" (32/LPR
// consecutive rows, one per warp row-group): the CTA's units are numbered
// across pieces and unit g goes to consumer warp g % C (computed, not counted
// per warp, so the producer keeps no per-warp state in local memory).
// One producer lane streams the units with cp.async.bulk into a pool of as many
// shared-memory slots as fit (at least one per consumer warp, or per group of GW
// warps when a row is spread over GW warps): unit g lands in slot g % slots.  A
// warp reads its unit from shared memory in each pass
// (statistics, then modulation) and then frees the slot, and the producer
// refills it at once with the unit `slots` places further on.  With more slots
// than warps, the spare slots are copies in flight while every warp computes.
// Every mbarrier wait is bounded.
//
// The modulation table sits in shared memory (TT = false) or in tensor memory
// (TT = true).  In tensor memory it leaves the whole of shared memory to the
// slots (D = 3072: 18 slots instead of 16; D = 5120: 22 instead of 18) and its
// reads leave the shared-memory pipe, which the slots' three passes keep busy;
// it costs an allocation and a heavier staging per piece, which the short
// launches of narrow rows do not recover.
constexpr int kFwdRingWarps = 16;  // consumer warps, unless an instance takes more
constexpr int kFwdMaxPool = 64;

// non-zero once a bounded wait in the pipelined forward gave up (never expected)
__device__ int g_fwd_status;

// ------------------------------------------------------------------ tensor memory
// (tmem.cuh) Thread l of warp w owns TMEM lane 32 (w % 4) + l; its columns
// 16k .. 16k+15 hold (1 + scale, shift) of its k-th vector.  The four warps of a
// quarter read the same values (same lane, same columns), so one copy serves
// them all.

// Rows split over a group of GW warps (GW > 1): the warps' partial statistics
// meet in shared memory behind a named barrier of the group's 32 GW threads.
// Two buffers alternate, as in CtaGroup: a warp writes buffer b only after the
// barrier of the call before, which every warp of the group reaches only once
// it has read what the call before that left in b.  Every warp combines the
// partials in warp order, so all end with the same bits.
template <int GW>
struct GroupXch {
    float2 p[2][GW][2];  // [buffer][warp][value]
    int m[2][GW];        // [buffer][warp]
};
template <int GW>
struct WarpGroup {
    GroupXch<GW> *x;
    int h, bar, t;
    __device__ WarpGroup(GroupXch<GW> *xx, int pos, int id) : x(xx), h(pos), bar(id), t(0) {}
    __device__ __forceinline__ void merge(float &hh, float &ll) {
        lane_merge<32>(hh, ll);
        if ((threadIdx.x & 31) == 0) x->p[t][h][0] = make_float2(hh, ll);
        named_barrier(bar, 32 * GW);
        float2 a = x->p[t][0][0];
        hh = a.x;
        ll = a.y;
#pragma unroll
        for (int w = 1; w < GW; ++w) {
            a = x->p[t][w][0];
            df_merge(hh, ll, a.x, a.y);
        }
        t ^= 1;
    }
    __device__ __forceinline__ void merge2(float &ah, float &al, float &bh, float &bl) {
        lane_merge2<32>(ah, al, bh, bl);
        if ((threadIdx.x & 31) == 0) {
            x->p[t][h][0] = make_float2(ah, al);
            x->p[t][h][1] = make_float2(bh, bl);
        }
        named_barrier(bar, 32 * GW);
        float2 a = x->p[t][0][0], b = x->p[t][0][1];
        ah = a.x;
        al = a.y;
        bh = b.x;
        bl = b.y;
#pragma unroll
        for (int w = 1; w < GW; ++w) {
            a = x->p[t][w][0];
            b = x->p[t][w][1];
            df_merge(ah, al, a.x, a.y);
            df_merge(bh, bl, b.x, b.y);
        }
        t ^= 1;
    }
    __device__ __forceinline__ bool any(bool p) {
        const int v = __any_sync(kFull, p);
        if ((threadIdx.x & 31) == 0) x->m[t][h] = v;
        named_barrier(bar, 32 * GW);
        int r = 0;
#pragma unroll
        for (int w = 0; w < GW; ++w) r |= x->m[t][w];
        t ^= 1;
        return r != 0;
    }
    __device__ __forceinline__ int max(int v) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = ::max(v, __shfl_xor_sync(kFull, v, off));
        if ((threadIdx.x & 31) == 0) x->m[t][h] = v;
        named_barrier(bar, 32 * GW);
        v = x->m[t][0];
#pragma unroll
        for (int w = 1; w < GW; ++w) v = ::max(v, x->m[t][w]);
        t ^= 1;
        return v;
    }
};
constexpr uint32_t kGroupXchBytes = 1024;  // >= (16 / GW) GroupXch<GW> for GW in 2, 4

// cached read-only load the compiler may schedule freely (staging loads)
__device__ __forceinline__ V16 ldg_nc(const void *p) {
    const uint4 q = __ldg(reinterpret_cast<const uint4 *>(p));
    return V16{{q.x, q.y, q.z, q.w}};
}

// Shared memory: the slots; the table (TT: the 16-byte TMEM address word instead);
// (gated) the raw gate row; then the barriers.  Every part before the barriers
// is a whole number of 16-byte vectors, so each starts 16-byte aligned (the
// barriers, 3 per slot, need only 8).
__host__ __device__ inline uint32_t fwd_ring_smem(int D, int RPW, int slots, bool gated,
                                                  bool tt) {
    const uint32_t unit = (uint32_t)RPW * D * 2u;
    return (uint32_t)slots * unit + (tt ? 16u : 2u * D * 4u) + (gated ? (uint32_t)D * 2u : 0u) +
           kGroupXchBytes + 3u * (uint32_t)slots * 8u;
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
template <int LPR, int NV, bool GATED, bool RMS, bool TT, int GW, int C>
__global__ void __launch_bounds__(32 * (C + 1), 1)
    adaln_fwd_ring_kernel(const __nv_bfloat16 *__restrict__ x,
                          const __nv_bfloat16 *__restrict__ shift,
                          const __nv_bfloat16 *__restrict__ scale, __nv_bfloat16 *__restrict__ y,
                          float *__restrict__ mean, float *__restrict__ rstd, int rows,
                          int D, float eps, int seg_rows, const int64_t *__restrict__ offsets,
                          int nseg, const int32_t *__restrict__ mod_index, int rows_per_cta,
                          int slots,
                          const __nv_bfloat16 *__restrict__ gate,
                          const __nv_bfloat16 *__restrict__ r, __nv_bfloat16 *__restrict__ out) {
    using T = __nv_bfloat16;
    constexpr int VEC = 8;
    constexpr int RPW = 32 / LPR;
    static_assert(C % 4 == 0 && C % GW == 0, "whole TMEM quarters and whole warp groups");
    int *status = &g_fwd_status;
    extern __shared__ __align__(128) unsigned char smem[];
    const int V = D / VEC;
    const uint32_t unit_bytes = (uint32_t)RPW * D * 2u;
    // shared-memory table (not TT), interleaved so that consecutive lanes read
    // consecutive 16-byte words: (1+scale) columns 8v..8v+3 at [v], 8v+4..8v+7 at
    // [V+v]; shift likewise at [2V+v] and [3V+v].  TT: the TMEM address word.
    float4 *tab = reinterpret_cast<float4 *>(smem + (size_t)slots * unit_bytes);
    uint32_t *tmem_word = reinterpret_cast<uint32_t *>(tab);
    V16 *gtab = reinterpret_cast<V16 *>(TT ? reinterpret_cast<unsigned char *>(tab) + 16
                                           : reinterpret_cast<unsigned char *>(tab + 4 * V));
    // unit g lands in slot g % slots and completes on full[g % (2 slots)]: two
    // units that share a full barrier are 2 slots apart, so a warp waiting for
    // its unit never sees the barrier more than one phase behind (the parity
    // test is exact) even when copies complete out of order
    unsigned char *xch_raw = reinterpret_cast<unsigned char *>(gtab + (GATED ? V : 0));
    uint64_t *full = reinterpret_cast<uint64_t *>(xch_raw + kGroupXchBytes);
    uint64_t *empty = full + 2 * slots;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 32-bit row arithmetic (the launcher uses this kernel only below 2^30 rows)
    const int r_begin = blockIdx.x * rows_per_cta;
    const int r_end = min(rows, r_begin + rows_per_cta);
    if (r_begin >= r_end) return;

    constexpr uint32_t kCols = tmem_cols(16 * NV);
    if (TT && warp == 0) tmem_alloc(tmem_word, kCols);  // consumer warp 0 frees it at the end
    // one barrier per thread: a pool of up to 64 slots has 192 barriers
    if (threadIdx.x < 3 * slots) {
        // full[0 .. 2 slots): the producer's arrival; empty[0 .. slots): one per warp
        // of the unit's group
        mbar_init(&full[threadIdx.x], threadIdx.x < 2 * slots ? 1 : GW);
        fence_barrier_init();
    }
    if (TT) tmem_fence_before();
    __syncthreads();
    if (TT) tmem_fence_after();
    const uint32_t tbase = TT ? *tmem_word : 0u;
    // no early pdl_trigger: see pdl_trigger in common.cuh (dependents launch at exit)
    pdl_wait();

    if (warp == C) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        int g = 0;  // units handed out so far (unit g goes to warp g % C)
        bool failed = false;
        for (int p0 = r_begin; p0 < r_end;) {
            int seg, p1;
            segment_of(p0, seg_rows, offsets, nseg, seg, p1);
            p1 = min(p1, r_end);
            const int nu = (p1 - p0 + RPW - 1) / RPW;
            for (int u = 0; u < nu; ++u, ++g) {
                const int s = g % slots;
                const int j = g / slots;  // earlier uses of slot s
                uint64_t *f = &full[g % (2 * slots)];
                if (j >= 1 && !mbar_wait(&empty[s], (uint32_t)(j - 1) & 1u)) {
                    atomicExch(status, 3);
                    failed = true;
                    p1 = r_end;  // stop issuing
                    break;
                }
                const int row0 = p0 + u * RPW;
                const uint32_t bytes = (uint32_t)min(RPW, p1 - row0) * (uint32_t)D * 2u;
                // (test build only: the CTA's last unit is never sent, so its
                // consumer's bounded wait runs out)
                if (kTestDropLastCopy && p1 == r_end && u == nu - 1) continue;
                mbar_arrive_expect_tx(f, bytes);
                bulk_g2s(smem + (size_t)s * unit_bytes, x + (int64_t)row0 * D, bytes, f);
                if (GATED) prefetch_l2(r + (int64_t)row0 * D, bytes);
            }
            p0 = p1;
        }
        // after a wait gave up, wait (briefly) for the copies of the last `slots`
        // units before leaving: their consumers may have stopped too, and no copy
        // may land in the CTA's shared memory after the CTA has exited.  (On the
        // normal path the consumers wait for every unit; a consumer whose wait
        // gave up drains its later units itself.)
        if (failed)
            for (int u = g > slots ? g - slots : 0; u < g; ++u)
                mbar_wait(&full[u % (2 * slots)], (uint32_t)(u / (2 * slots)) & 1u, kDrainLimit);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int li = lane % LPR;
    const int sub = lane / LPR;
    const int ncons = C * 32;
    // a unit goes to one group of GW warps; warp h of the group owns the row's
    // column vectors vbase + k VS
    constexpr int G = C / GW;
    constexpr int VS = LPR * GW;
    const int gi = warp / GW, h = warp % GW;
    const int vbase = h * LPR + li;
    [[maybe_unused]] WarpGroup<GW> wg(reinterpret_cast<GroupXch<GW> *>(xch_raw) + gi, h, 2 + gi);
    const uint32_t tlane = tmem_lane_addr(tbase, warp, 0);  // TT: this thread's TMEM lane
    int g0 = 0;  // global index of the piece's first unit
    // set once a wait of this warp gave up: the warp then does no more work but
    // stays in the loops, so the other warps still meet it at the named barrier
    // of every piece
    bool dead = false;
    for (int p0 = r_begin; p0 < r_end;) {
        int seg, p1;
        segment_of(p0, seg_rows, offsets, nseg, seg, p1);
        p1 = min(p1, r_end);
        // stage this piece's modulation row (after every warp is done with the last one)
        if (TT) tmem_fence_before();
        named_barrier(1, ncons);
        if (TT) tmem_fence_after();
        const int64_t mrow = mod_row(mod_index, seg);
        if constexpr (TT) {
            // the four warps of a TMEM quarter share its vectors: warp w writes
            // k = w / 4 + 4 i; all loads first, then the conversions and stores
            constexpr int QW = C / 4;  // warps per TMEM quarter
            constexpr int KW = (NV + QW - 1) / QW;
            V16 scv[KW], shv[KW];
#pragma unroll
            for (int i = 0; i < KW; ++i) {
                const int k = (warp >> 2) + QW * i;
                if (k < NV) {
                    const int v = (warp & 3) % GW * LPR + li + k * VS;
                    scv[i] = ldg_nc(scale + mrow * D + v * VEC);
                    shv[i] = ldg_nc(shift + mrow * D + v * VEC);
                }
            }
#pragma unroll
            for (int i = 0; i < KW; ++i) {
                const int k = (warp >> 2) + QW * i;
                if (k < NV) {
                    float sc[VEC], sh[VEC];
                    uint32_t t[16];
                    IO<T>::unpack(scv[i], sc);
                    IO<T>::unpack(shv[i], sh);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        t[e] = __float_as_uint(1.0f + sc[e]);
                        t[VEC + e] = __float_as_uint(sh[e]);
                    }
                    tmem_st16(tlane + 16u * k, t);
                }
            }
            tmem_wait_st();
        } else {
            for (int v = threadIdx.x; v < V; v += ncons) {
                float sc[VEC], sh[VEC];
                IO<T>::unpack(ld_cached(scale + mrow * D + v * VEC), sc);
                IO<T>::unpack(ld_cached(shift + mrow * D + v * VEC), sh);
                tab[v] = make_float4(1.0f + sc[0], 1.0f + sc[1], 1.0f + sc[2], 1.0f + sc[3]);
                tab[V + v] = make_float4(1.0f + sc[4], 1.0f + sc[5], 1.0f + sc[6], 1.0f + sc[7]);
                tab[2 * V + v] = make_float4(sh[0], sh[1], sh[2], sh[3]);
                tab[3 * V + v] = make_float4(sh[4], sh[5], sh[6], sh[7]);
            }
        }
        if (GATED)
            for (int v = threadIdx.x; v < V; v += ncons) gtab[v] = ld_cached(gate + mrow * D + v * VEC);
        if (TT) tmem_fence_before();
        named_barrier(1, ncons);
        if (TT) tmem_fence_after();

        const int nu = (p1 - p0 + RPW - 1) / RPW;
        for (int u = ((gi - g0) % G + G) % G; u < nu; u += G) {
            const int g = g0 + u;
            if (dead) {
                // no more work; only let the unit's copy (if it was issued) land
                mbar_wait(&full[g % (2 * slots)], (uint32_t)(g / (2 * slots)) & 1u, kDrainLimit);
                continue;
            }
            const int s = g % slots;
            // the whole warp (group) takes the same decision (its lanes poll on their own)
            bool ok = __all_sync(kFull, mbar_wait(&full[g % (2 * slots)],
                                                  (uint32_t)(g / (2 * slots)) & 1u));
            if constexpr (GW > 1) ok = !wg.any(!ok);
            if (!ok) {
                if (lane == 0) atomicExch(status, 4);
                dead = true;
                continue;
            }
            const int row = p0 + u * RPW + sub;
            // a unit of one row is always full; in a unit of two the second row may
            // lie past the piece: its lanes then run on the first row's values (the
            // loads need no guard, and the warp-wide table loads stay warp-wide)
            // and store nothing
            const bool active = RPW == 1 || row < p1;
            const int rrow = active ? row : p0 + u * RPW;
            const unsigned char *src =
                smem + (size_t)s * unit_bytes + (size_t)(active ? sub : 0) * D * 2u;
            // the row stays in shared memory and is read once per pass; the passes
            // are unrolled four vectors deep (two deep was 4-5% slower at D = 3072
            // and 5120)
            auto xv = [&](int k) -> V16 { return lds128(src + (size_t)(vbase + k * VS) * 16); };
            float mh, ml, rs;
            if constexpr (GW > 1)
                row_stats<T, LPR, NV, true, true, false, 4, decltype(xv), true, RMS, WarpGroup<GW>>(
                    xv, li, NV, LPR * NV, D, eps, mh, ml, rs, wg);
            else
                row_stats<T, LPR, NV, true, true, false, 4, decltype(xv), true, RMS>(
                    xv, li, NV, LPR * NV, D, eps, mh, ml, rs);
            // y = (x rstd + n) (1 + scale) + shift with n = -mean rstd, in packed pairs:
            // x rstd + n is one rounding of a value of the order of the normalised x.
            // Rows with |n| > 4 (|mean| >> std) take (x - mean) * rstd instead.
            const float nh = __fmul_rn(-mh, rs);
            const bool wide = __any_sync(kFull, active && !(fabsf(nh) <= 4.0f));
            const f2 RS = f2_make(rs, rs), NH = f2_make(nh, nh);
            const f2 MH = f2_make(mh, mh), ML = f2_make(ml, ml);
            T *yr = (y != nullptr && active) ? y + (int64_t)row * D : nullptr;
            auto modulate = [&](auto wide_c) {
                constexpr bool W = decltype(wide_c)::value;
                // vector k with its table words tw: (1 + scale) of its 8 columns, then shift
                auto one = [&](int k, const uint32_t *tw) {
                    const int v = vbase + k * VS;
                    const V16 xk = xv(k);
                    V16 o;
                    [[maybe_unused]] V16 og, rk, gk;  // gated only
                    if constexpr (GATED) {
                        rk = ld_stream(r + (int64_t)rrow * D + v * VEC);
                        gk = lds128(gtab + v);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        // wide rows: centre first, (x - mean) * rstd, which cannot
                        // overflow where x * rstd would (huge, nearly constant rows)
                        const f2 X = f2_from_bf16x2(xk.w[i]);
                        const f2 U = W ? f2_mul(f2_sub(f2_sub(X, MH), ML), RS)
                                       : f2_fma(X, RS, NH);
                        const f2 Y = f2_fma(U, f2_from_words(tw[2 * i], tw[2 * i + 1]),
                                            f2_from_words(tw[8 + 2 * i], tw[9 + 2 * i]));
                        o.w[i] = f2_to_bf16x2(Y);
                        if constexpr (GATED)
                            og.w[i] = f2_to_bf16x2(f2_fma(f2_from_bf16x2(gk.w[i]), Y,
                                                          f2_from_bf16x2(rk.w[i])));
                    }
                    if (yr != nullptr) st_vec(yr + v * VEC, o);
                    if constexpr (GATED)
                        if (active) st_vec(out + (int64_t)row * D + v * VEC, og);
                };
                if constexpr (TT) {
                    // two vectors' tables per tensor-memory load (one wait for both)
#pragma unroll 2
                    for (int k = 0; k + 1 < NV; k += 2) {
                        uint32_t tw[32];
                        tmem_ld32(tlane + 16u * k, tw);
                        one(k, tw);
                        one(k + 1, tw + 16);
                    }
                    if constexpr (NV & 1) {
                        uint32_t tw[16];
                        tmem_ld16(tlane + 16u * (NV - 1), tw);
                        one(NV - 1, tw);
                    }
                } else {
#pragma unroll 4
                    for (int k = 0; k < NV; ++k) {
                        const int v = vbase + k * VS;
                        // (volatile shared loads keep the table reads next to their use)
                        const V16 t0 = lds128(tab + v), t1 = lds128(tab + V + v);
                        const V16 t2 = lds128(tab + 2 * V + v), t3 = lds128(tab + 3 * V + v);
                        const uint32_t tw[16] = {t0.w[0], t0.w[1], t0.w[2], t0.w[3],
                                                 t1.w[0], t1.w[1], t1.w[2], t1.w[3],
                                                 t2.w[0], t2.w[1], t2.w[2], t2.w[3],
                                                 t3.w[0], t3.w[1], t3.w[2], t3.w[3]};
                        one(k, tw);
                    }
                }
            };
            if (active && li == 0 && h == 0) {
                if (!RMS) mean[row] = mh;
                rstd[row] = rs;
            }
            if (wide)
                modulate(std::true_type{});
            else
                modulate(std::false_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // done with the slot
        }
        g0 += nu;
        p0 = p1;
    }
    if constexpr (TT) {
        // every consumer is done with the table: warp 0 frees the tensor memory
        tmem_fence_before();
        named_barrier(1, ncons);
        if (warp == 0) {
            tmem_fence_after();
            tmem_dealloc(tbase, kCols);
        }
    }
}

// shared-memory slots that fit, at least one per unit a CTA computes at once (a
// warp, or a group of gw warps, of c consumer warps; 0: the ring does not fit)
inline int fwd_ring_slots(int D, int RPW, bool gated, bool tt, int smem_optin, int gw = 1,
                          int c = kFwdRingWarps) {
    for (int sl = kFwdMaxPool; sl >= c / gw; --sl)
        if (fwd_ring_smem(D, RPW, sl, gated, tt) + 1024 <= (uint32_t)smem_optin) return sl;
    return 0;
}

template <int LPR, int NV, bool TT, int GW, int C>
cudaError_t fwd_ring_launch(const void *x, const void *shift, const void *scale, void *y,
                            float *mean, float *rstd, const Segments &sg, int D, float eps,
                            const GateEpilogue &ge, bool rms, const DeviceInfo &di,
                            cudaStream_t stream) {
    constexpr int RPW = 32 / LPR;
    const bool gated = ge.out != nullptr;
    const int slots = fwd_ring_slots(D, RPW, gated, TT, di.max_smem_optin, GW, C);
    const uint32_t smem = fwd_ring_smem(D, RPW, slots, gated, TT);
    auto kern = rms ? adaln_fwd_ring_kernel<LPR, NV, false, true, TT, GW, C>
                    : adaln_fwd_ring_kernel<LPR, NV, false, false, TT, GW, C>;
    if constexpr (C == kFwdRingWarps) {  // (the gated epilogue keeps 16 consumer warps)
        if (gated) kern = adaln_fwd_ring_kernel<LPR, NV, true, false, TT, GW, C>;
    }
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int64_t units = (sg.rows + RPW - 1) / RPW;
    int64_t grid = (units + C / GW - 1) / (C / GW);
    if (grid > di.sms) grid = di.sms;
    int64_t rpc = (sg.rows + grid - 1) / grid;
    rpc = (rpc + RPW - 1) / RPW * RPW;
    grid = (sg.rows + rpc - 1) / rpc;
    using B16 = __nv_bfloat16;
    err = launch_pdl(kern, dim3((unsigned)grid), dim3(32 * (C + 1)), smem, stream, (const B16 *)x,
                     (const B16 *)shift, (const B16 *)scale, (B16 *)y, mean, rstd, (int)sg.rows, D,
                     eps, (int)sg.seg_rows, sg.offsets, (int)sg.nseg, sg.mod_index, (int)rpc, slots,
                     (const B16 *)ge.gate, (const B16 *)ge.r, (B16 *)ge.out);
    count_launch();
    return err;
}

}  // namespace

int pipeline_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fwd_status, sizeof(int)) != cudaSuccess) return -1;
    return v;
}

// The pipelined forward for whole-vector bf16 shapes that fit the shared-memory
// ring; `launched` is false (and nothing is queued) for any other shape.
cudaError_t launch_fwd_ring(const void *x, const void *shift, const void *scale, void *y,
                            float *mean, float *rstd, const Segments &sg, int D, float eps,
                            const GateEpilogue &ge, bool rms, const DeviceInfo &di,
                            cudaStream_t stream, bool &launched) {
    launched = true;
    const int V = D / 8;
    const bool gated = ge.out != nullptr;
    const bool ring_ok = sg.rows < (int64_t)1 << 30 && sg.nseg < (int64_t)1 << 30 &&
                         sg.seg_rows < (int64_t)1 << 30;
#define ADALN_RING_GC(LPR, NV, TT, GW, C)                                                    \
    if (ring_ok && V == (LPR) * (NV) * (GW) && ((C) == kFwdRingWarps || !gated) &&           \
        fwd_ring_slots(D, 32 / (LPR), gated, TT, di.max_smem_optin, GW, C) > 0)              \
        return fwd_ring_launch<LPR, NV, TT, GW, C>(x, shift, scale, y, mean, rstd, sg, D, eps, \
                                                   ge, rms, di, stream);
#define ADALN_RING_G(LPR, NV, TT, GW) ADALN_RING_GC(LPR, NV, TT, GW, kFwdRingWarps)
#define ADALN_RING(LPR, NV, TT) ADALN_RING_G(LPR, NV, TT, 1)
    // table in tensor memory where its shared-memory copy would cost slots the
    // pool needs (measured on GB300: D = 3072 0.93 -> 0.98 of the copy bandwidth,
    // D = 5120 0.91 -> 0.92, MMDiT 0.69 -> 0.73); in shared memory elsewhere (at
    // D = 1152 the allocation and staging cost 2 of 18 us, at D = 4096 1%)
    ADALN_RING(16, 24, true)   // D = 3072: two rows per unit halve the per-row work per element
    // D = 5120 (and the wide rows of 8,192 below): 20 consumer warps where the
    // pool still holds a slot per warp, else 16; the gated epilogue keeps 16 (at
    // 80 registers it would spill).  Measured on GB300 against 16: D = 5120
    // 0.919 -> 0.927 of the copy bandwidth, 8,192 0.643 -> 0.665; at 12,288 two
    // runs disagreed (+3.6%, -1.2%), at 16,384 even; at D = 3072 the pool would
    // be too small for 20.
    ADALN_RING_GC(32, 20, true, 1, 20)
    ADALN_RING(32, 20, true)
    ADALN_RING(32, 24, true)   // D = 6144: the shared-memory table would leave too few slots
    ADALN_RING(32, 4, false)
    ADALN_RING(32, 8, false)
    ADALN_RING(32, 12, false)
    ADALN_RING(32, 16, false)
    ADALN_RING(16, 9, false)
    // rows of 8,192 to 16,384 bf16 elements (multiples of 2,048): a row per group of
    // four warps, 6-12 slots of a row each (measured on GB300: D = 16,384 0.55 -> 0.77
    // of the copy bandwidth, D = 12,288 0.55 -> 0.75, D = 8,192 0.60 -> 0.63 against
    // the CTA-per-row kernel of wide.cu, which takes the other wide rows)
    ADALN_RING_GC(32, 8, true, 4, 20)
    ADALN_RING_G(32, 8, true, 4)
    ADALN_RING_G(32, 12, true, 4)
    ADALN_RING_G(32, 16, true, 4)
#undef ADALN_RING
#undef ADALN_RING_G
#undef ADALN_RING_GC
    launched = false;
    return cudaSuccess;
}

}  // namespace adaln
