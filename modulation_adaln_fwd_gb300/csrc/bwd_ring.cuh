// bwd_ring.cuh -- the pipelined backward kernels and their launch dispatch,
// shared by the per-dtype translation units (bwd_bf16.cu, bwd_f32.cu) so that
// the many kernel instantiations compile in parallel.
#pragma once

#include "common.cuh"
#include "launch.h"
#include "tmem.cuh"

#include <mutex>

namespace adaln {

namespace {

// ------------------------------------------------------------------ bwd main

constexpr unsigned kFull = 0xffffffffu;

constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v >> 1); }
constexpr int pow2_at_least(int v) { return v <= 1 ? 1 : 2 * pow2_at_least((v + 1) >> 1); }

// Transposed butterfly: P per-lane values (P a power of two <= 32) are summed
// over the 32 lanes of the warp with P - 1 + log2(32/P) shuffles in total.
// Afterwards lane l holds the warp total of value index l >> (5 - log2 P).
template <int P>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[P], int lane) {
    int n = P;
#pragma unroll
    for (int o = 16; o >= 32 / P; o >>= 1) {
        const int half = n >> 1;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, o);
        }
        n = half;
    }
    float r = v[0];
#pragma unroll
    for (int o = (32 / P) >> 1; o >= 1; o >>= 1) r += __shfl_xor_sync(kFull, r, o);
    return r;
}

// Sum the per-warp totals red[w][j] (w < nwarps, j < P) in a fixed order; every
// lane l ends with the CTA total of index l % P (identical bits in every warp).
template <int P>
__device__ __forceinline__ float cta_totals(const float (*red)[32], int nwarps, int lane) {
    constexpr int G = 32 / P;  // lane groups that split the warps between them
    const int j = lane & (P - 1);
    float t = 0.f;
    for (int w = lane / P; w < nwarps; w += G) t += red[w][j];
#pragma unroll
    for (int o = P; o < 32; o <<= 1) t += __shfl_xor_sync(kFull, t, o);
    return t;
}

// Shared-memory layout of the ring: `stages` slots, each holding R rows of x,
// R rows of dy, a 32-byte tile header and the R means and rstds of those rows;
// then the full/empty mbarriers of every slot; then the double-buffered
// per-warp reduction rows.
struct TileHdr {
    int chunk;   // -1: no more work
    int nr;      // rows in this tile
    int seg;     // segment (modulation row) of the chunk
    int flags;   // 1: first tile of its chunk, 2: last tile of its chunk
    int64_t r0;  // first row of the tile
    int64_t pad;
};
static_assert(sizeof(TileHdr) == 32, "tile header is 32 bytes");
struct RingLayout {
    uint32_t row_bytes, tile_bytes, stage_bytes, bar_off, red_off, total;
};

__host__ __device__ inline RingLayout ring_layout(int D, int esize, int R, int stages, int cwarps) {
    RingLayout l;
    l.row_bytes = (uint32_t)D * esize;
    l.tile_bytes = (uint32_t)R * l.row_bytes;
    const uint32_t stat = ((32u + 2u * R * 4u) + 15u) & ~15u;
    l.stage_bytes = 2u * l.tile_bytes + stat;
    l.bar_off = (uint32_t)stages * l.stage_bytes;
    // ring barriers (full, empty per slot) + two reduction barriers
    l.red_off = l.bar_off + 8u * (2u * (uint32_t)stages + 2u);
    l.total = l.red_off + 4u * (uint32_t)cwarps * 32u * 4u;  // four reduction buffers
    return l;
}

// consumer threads per CTA: one vector per thread allows 384 (128 registers each);
// two or more vectors per thread need the register room of at most 352
constexpr int ring_max_consumers(int K) { return K == 1 ? 384 : 352; }

// Ring producer (warp 0).  Chunk c covers rows [c L, min((c + 1) L, rows)) and
// the CTA takes chunks c = blockIdx.x, + gridDim.x, ...  A chunk is cut at
// segment boundaries into pieces; the piece of segment k accumulates into
// partial row c + k, which is unique because pieces are visited in row order
// and both c and k grow along the rows (at most nchunks + nseg - 1 rows).  The
// whole warp finds the segment of a chunk's first row (a 32-way search over the
// offsets); lane 0 then walks the pieces and, for every R-row tile, waits for a
// free slot, writes the tile header, bulk-copies the tile's rows of `a` and `b`
// and (STATS) cp.asyncs their mean and rstd, all completing on the slot's `full`
// barrier (whose count is 2 with STATS, else 1).  Past the last chunk it
// publishes an end header.  A timed-out wait writes 1 to *status.  Before it
// leaves, lane 0 waits (bounded) for the copies of its last `stages` slots: the
// consumers may have stopped without waiting for them, and no copy may land in
// the CTA's shared memory after the CTA has exited.
template <typename T, int R, bool STATS>
__device__ __forceinline__ void ring_produce(
    const T *__restrict__ a, const T *__restrict__ b, const float *__restrict__ mean,
    const float *__restrict__ rstd, int *__restrict__ status, unsigned char *smem,
    const RingLayout &lay, uint64_t *full, uint64_t *empty, int stages, int64_t rows, int D,
    int64_t seg_rows, const int64_t *__restrict__ offsets, int64_t nseg, int64_t L,
    int64_t nchunks, int lane) {
    uint32_t it = 0;
    // next free slot (lane 0), or nullptr after a timed-out wait
    auto acquire = [&](int &s) -> unsigned char * {
        s = (int)(it % (uint32_t)stages);
        const uint32_t ph = (it / (uint32_t)stages) & 1u;
        if (it >= (uint32_t)stages && !mbar_wait(&empty[s], ph ^ 1u)) {
            atomicExch(status, 1);
            return nullptr;
        }
        ++it;
        return smem + (size_t)s * lay.stage_bytes;
    };
    for (int64_t c = blockIdx.x;; c += gridDim.x) {
        const bool more = c < nchunks;
        int64_t r = more ? c * L : rows;
        const int64_t cend = more ? min(r + L, rows) : rows;
        int64_t k = 0;
        if (more) k = offsets ? find_segment_warp(offsets, nseg, r, lane) : div_nonneg(r, seg_rows);
        bool ok = true;
        if (lane == 0) {
            if (!more) {  // end of work: header only
                int s;
                unsigned char *sb = acquire(s);
                if (sb != nullptr) {
                    reinterpret_cast<TileHdr *>(sb + 2 * lay.tile_bytes)->chunk = -1;
                    mbar_arrive(&full[s]);
                    if (STATS) mbar_arrive(&full[s]);
                }
            }
            while (ok && r < cend) {
                // piece [r, e) of segment k (empty segments are skipped; offsets that
                // contradict the row count still move r forward)
                int64_t e;
                if (offsets) {
                    while (k + 1 < nseg && __ldg(offsets + k + 1) <= r) ++k;
                    e = k + 1 < nseg ? min(cend, __ldg(offsets + k + 1)) : cend;
                } else {
                    e = min(cend, (k + 1) * seg_rows);
                }
                if (e <= r) e = cend;
                for (int64_t r0 = r; r0 < e;) {
                    int s;
                    unsigned char *sb = acquire(s);
                    if (sb == nullptr) {
                        ok = false;
                        break;
                    }
                    const int nr = (int)min((int64_t)R, e - r0);
                    // (test build only: the CTA's last tile is never sent, so the
                    // consumers' bounded wait for it runs out)
                    if (kTestDropLastCopy && c + gridDim.x >= nchunks && r0 + nr >= cend) {
                        r0 += nr;
                        continue;
                    }
                    TileHdr *hdr = reinterpret_cast<TileHdr *>(sb + 2 * lay.tile_bytes);
                    hdr->chunk = (int)(c + k);
                    hdr->nr = nr;
                    hdr->seg = (int)k;
                    hdr->flags = (r0 == r ? 1 : 0) | (r0 + nr >= e ? 2 : 0);
                    hdr->r0 = r0;
                    const uint32_t bytes = (uint32_t)nr * lay.row_bytes;
                    mbar_arrive_expect_tx(&full[s], 2u * bytes);
                    bulk_g2s(sb, a + r0 * (int64_t)D, bytes, &full[s]);
                    bulk_g2s(sb + lay.tile_bytes, b + r0 * (int64_t)D, bytes, &full[s]);
                    if (STATS) {
                        float *st = reinterpret_cast<float *>(hdr + 1);
                        for (int i = 0; i < nr; ++i) {
                            if (mean != nullptr) cp_async4(st + i, mean + r0 + i);
                            cp_async4(st + R + i, rstd + r0 + i);
                        }
                        cp_async_arrive(&full[s]);
                    }
                    r0 += nr;
                }
                r = e;
                if (!offsets) ++k;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
        if (!ok || !more) break;
    }
    if (lane == 0) {
        const uint32_t first = it > (uint32_t)stages ? it - (uint32_t)stages : 0u;
        for (uint32_t j = first; j < it; ++j)
            if (!mbar_wait(&full[j % (uint32_t)stages], (j / (uint32_t)stages) & 1u))
                atomicExch(status, 1);
    }
}

// Persistent backward.  Warp 0 is the producer (see ring_produce): it streams
// R-row tiles of x and dy, with their mean and rstd, into a ring of
// shared-memory slots.  The other warps consume: each thread owns K 16-byte
// column vectors of the row, reads its columns of the tile from shared memory
// in both passes (row sums, then dx and the column partials), and then releases
// the slot.  A piece's partials go to their own workspace row, so the results
// do not depend on which CTA ran it.  Every mbarrier wait is bounded; on a
// timeout the thread writes a non-zero code to this CTA's status word (cleared
// when the CTA starts) and stops.  With `gate` (the fused gated chain, dy being
// the gradient of out = r + gate * y) the modulation row is gate * (1 + scale),
// so g = gate * dout * (1 + scale) and the partials hold sum dout * xhat and
// sum dout, which the column sums turn into d_scale, d_shift and d_gate.
// RMS (launched without a mean): the RMSNorm backward, xhat = x * rstd and
// dx = rstd * (g - xhat * mean_d(g * xhat)).
template <typename T, int K, int R, bool GATED, bool RMS>
__global__ void __launch_bounds__(32 + ring_max_consumers(K), 1)
    adaln_bwd_ring_kernel(const T *__restrict__ x, const float *__restrict__ mean,
                          const float *__restrict__ rstd, const T *__restrict__ scale,
                          const T *__restrict__ dy, T *__restrict__ dx,
                          float *__restrict__ partial, int *__restrict__ cta_status,
                          int64_t rows, int D, int64_t seg_rows,
                          const int64_t *__restrict__ offsets, int64_t nseg,
                          const int32_t *__restrict__ mod_index, int64_t L, int64_t nchunks,
                          int stages, bool split, const T *__restrict__ gate) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int VEC = IO<T>::VEC;
    constexpr int P = pow2_at_least(3 * R);  // three row sums per row, padded
    static_assert(P <= 32, "row tile too large for one warp-level reduction");
    const int V = D / VEC;
    const int ncons = (int)blockDim.x - 32;
    const int ncw = ncons >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const RingLayout lay = ring_layout(D, (int)sizeof(T), R, stages, ncw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bar_off);
    uint64_t *empty = full + stages;
    uint64_t *redbar = empty + stages;  // [2]: tile k's row sums published on redbar[k % 2]
    float(*red)[32] = reinterpret_cast<float(*)[32]>(smem + lay.red_off);  // [4*ncw][32]
    int *status = cta_status + blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 2);      // producer arrive.expect_tx + cp.async arrival
            mbar_init(&empty[s], ncw);   // one arrival per consumer warp
        }
        mbar_init(&redbar[0], ncons);    // every consumer thread arrives
        mbar_init(&redbar[1], ncons);
        fence_barrier_init();
    }
    pdl_wait();  // before the first global access (the status word included)
    // no early pdl_trigger: see pdl_trigger in common.cuh (dependents launch at exit)
    if (threadIdx.x == 0) *status = 0;
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        ring_produce<T, R, true>(x, dy, mean, rstd, status, smem, lay, full, empty, stages, rows,
                                 D, seg_rows, offsets, nseg, L, nchunks, lane);
        return;
    }

    // ---------------------------------------------------------------- consumers
    //
    // Split-phase row reductions: a tile's per-warp row sums are published (write
    // to reduction buffer k % 4, arrive on redbar[k % 2]) and the warp moves on to
    // the next tile's first pass before it waits for the totals.  Within a chunk the
    // reduction of tile k therefore overlaps the first pass of tile k + 1.  Buffer
    // k % 4 is free again because a warp arrives for tile k only after it has read
    // the totals of tile k - 2, and writes tile k + 1 only after tile k - 1 closed.
    const int ct = threadIdx.x - 32;
    const int cw = ct >> 5;
    const float invD = 1.0f / (float)D;
    // the element math runs on packed pairs (f32x2): NP pairs per 16-byte vector
    constexpr int NP = Pairs<T>::NP;
    f2 s1[K][NP], acc_s[K][NP], acc_b[K][NP];

    struct Tile {
        const unsigned char *sb;
        uint32_t sa;  // shared-window address of the slot
        int slot, chunk, nr, flags, seg;
        int64_t r0;
        float rs[R], nmr[R];
    };
    uint32_t it = 0;  // ring slots consumed so far
    // next tile from the ring (false: the producer published the end of work)
    auto fetch = [&](Tile &t) -> bool {
        const int s = (int)(it % (uint32_t)stages);
        const uint32_t ph = (it / (uint32_t)stages) & 1u;
        ++it;
        // warp-uniform outcome: the lanes poll on their own, the code after shuffles
        if (!__all_sync(kFull, mbar_wait(&full[s], ph))) {
            atomicExch(status, 2);
            return false;
        }
        t.sb = smem + (size_t)s * lay.stage_bytes;
        t.sa = smem_u32(t.sb);
        const TileHdr *hdr = reinterpret_cast<const TileHdr *>(t.sb + 2 * lay.tile_bytes);
        t.slot = s;
        t.chunk = hdr->chunk;
        if (t.chunk < 0) return false;
        t.nr = hdr->nr;
        t.flags = hdr->flags;
        t.r0 = hdr->r0;
        const float *st = reinterpret_cast<const float *>(hdr + 1);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            t.rs[r] = 0.f;
            t.nmr[r] = 0.f;
            if (r < t.nr) {
                t.rs[r] = st[R + r];
                t.nmr[r] = RMS ? 0.f : -st[r] * t.rs[r];
            }
        }
        t.seg = hdr->seg;
        return true;
    };
    // first tile of a chunk: the chunk's modulation row, fresh partials (only after
    // the previous chunk's last tile is finished: it still uses both)
    auto begin_chunk = [&](const Tile &t) {
        const int64_t seg = mod_row(mod_index, t.seg);  // the chunk's modulation row
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int v = ct + k * ncons;
            const V16 sv = v < V ? ld_cached(scale + seg * D + (int64_t)v * VEC)
                                 : V16{{0u, 0u, 0u, 0u}};
            Pairs<T>::unpack(sv, s1[k]);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                s1[k][i] = f2_add(f2_make(1.0f, 1.0f), s1[k][i]);
                acc_s[k][i] = 0ull;
                acc_b[k][i] = 0ull;
            }
            if constexpr (GATED) {  // gated chain: the gradient reaching y is gate * dout
                const V16 gv = v < V ? ld_cached(gate + seg * D + (int64_t)v * VEC)
                                     : V16{{0u, 0u, 0u, 0u}};
                f2 gp[NP];
                Pairs<T>::unpack(gv, gp);
#pragma unroll
                for (int i = 0; i < NP; ++i) s1[k][i] = f2_mul(s1[k][i], gp[i]);
            }
        }
    };
    // the tile stays in shared memory: read once per pass (rows past the tile end
    // and columns past D read as zeros; their rstd is 0 for the former and their
    // xh is masked out of sum(xh) for the latter)
    const uint32_t my_off = (uint32_t)ct * 16u;  // this thread's first column vector
    auto load = [&](const Tile &t, int r, int k, V16 &xvv, V16 &gvv) {
        const int v = ct + k * ncons;
        if (r < t.nr && v < V) {
            const uint32_t a = t.sa + (uint32_t)r * lay.row_bytes + my_off + (uint32_t)(k * ncons) * 16u;
            xvv = lds128_at(a);
            gvv = lds128_at(a + lay.tile_bytes);
        } else {
            xvv = V16{{0u, 0u, 0u, 0u}};
            gvv = V16{{0u, 0u, 0u, 0u}};
        }
    };
    // pass 1 of tile number kk: per row sum(xh), sum(g), sum(g * xh), then publish
    // (each as a pair of half sums over the even and odd columns, added at the end)
    auto pass1 = [&](const Tile &t, uint32_t kk) {
        f2 pv2[3 * R];
#pragma unroll
        for (int i = 0; i < 3 * R; ++i) pv2[i] = 0ull;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const f2 RS = f2_make(t.rs[r], t.rs[r]), NMR = f2_make(t.nmr[r], t.nmr[r]);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                V16 xvv, gvv;
                load(t, r, k, xvv, gvv);
                f2 xp[NP], gp[NP];
                Pairs<T>::unpack(xvv, xp);
                Pairs<T>::unpack(gvv, gp);
                // columns past D are zero-filled: their xh would be -mean * rstd
                const float cwf = (ct + k * ncons < V) ? 1.0f : 0.0f;
                const f2 CW = f2_make(cwf, cwf);
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    const f2 xh = f2_fma(xp[i], RS, NMR);
                    const f2 g = f2_mul(gp[i], s1[k][i]);
                    pv2[3 * r] = f2_fma(CW, xh, pv2[3 * r]);
                    pv2[3 * r + 1] = f2_add(pv2[3 * r + 1], g);
                    pv2[3 * r + 2] = f2_fma(g, xh, pv2[3 * r + 2]);
                }
            }
        }
        float pv[P];
#pragma unroll
        for (int i = 0; i < P; ++i) {
            pv[i] = 0.f;
            if (i < 3 * R) {
                float lo, hi;
                f2_split(pv2[i], lo, hi);
                pv[i] = lo + hi;
            }
        }
        const float wt = warp_transpose_reduce<P>(pv, lane);
        if ((lane & (32 / P - 1)) == 0) red[(kk & 3u) * ncw + cw][lane / (32 / P)] = wt;
        if (split) mbar_arrive(&redbar[kk & 1u]);
    };
    // wait for tile kk's totals, then pass 2: dx and the column partials with xhat
    // recentred on its row mean (sum_d xhat = 0 exactly), which removes the shift
    // the float rounding of the stored mean puts on every xhat of the row
    auto finish = [&](const Tile &t, uint32_t kk) -> bool {
        if (split) {
            if (!__all_sync(kFull, mbar_wait(&redbar[kk & 1u], (kk >> 1) & 1u))) {
                atomicExch(status, 5);
                return false;
            }
        } else if (named_barrier_any(1, ncons, 0)) {
            return false;  // lockstep: a hardware barrier among the consumers, at which
                           // a warp whose wait gave up votes for all to stop
        }
        const float tot = cta_totals<P>(red + (kk & 3u) * ncw, ncw, lane);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float sx = __shfl_sync(kFull, tot, 3 * r);
            const float sg = __shfl_sync(kFull, tot, 3 * r + 1);
            const float sgx = __shfl_sync(kFull, tot, 3 * r + 2);
            if (r < t.nr) {
                // RMSNorm: xhat = x * rstd has no mean to recentre on and dx has
                // no mean(g) term
                const float delta = RMS ? 0.f : sx * invD;
                const float mg = RMS ? 0.f : sg * invD;
                const float mgx = fmaf(-delta, sg, sgx) * invD;
                const float c1 = t.rs[r] * mgx;
                const float c0 = fmaf(c1, delta, -t.rs[r] * mg);
                T *dxr = dx + (t.r0 + r) * (int64_t)D;
                const f2 RS = f2_make(t.rs[r], t.rs[r]), NMR = f2_make(t.nmr[r], t.nmr[r]);
                const f2 NC1 = f2_make(-c1, -c1), C0 = f2_make(c0, c0);
                const f2 DL = f2_make(delta, delta);
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int v = ct + k * ncons;
                    V16 xvv, gvv;
                    load(t, r, k, xvv, gvv);
                    f2 xp[NP], gp[NP], o[NP];
                    Pairs<T>::unpack(xvv, xp);
                    Pairs<T>::unpack(gvv, gp);
#pragma unroll
                    for (int i = 0; i < NP; ++i) {
                        const f2 xh = f2_fma(xp[i], RS, NMR);
                        const f2 g = f2_mul(gp[i], s1[k][i]);
                        o[i] = f2_fma(g, RS, f2_fma(xh, NC1, C0));
                        acc_s[k][i] = f2_fma(gp[i], f2_sub(xh, DL), acc_s[k][i]);
                        acc_b[k][i] = f2_add(acc_b[k][i], gp[i]);
                    }
                    if (v < V) st_vec(dxr + (int64_t)v * VEC, Pairs<T>::pack(o));
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[t.slot]);  // this warp is done with the slot
        if (t.flags & 2) {
            // last tile of the chunk: [c][0][:] = sum dy*xhat, [c][1][:] = sum dy
            float *p0 = partial + ((int64_t)t.chunk * 2 + 0) * D;
            float *p1 = partial + ((int64_t)t.chunk * 2 + 1) * D;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int v = ct + k * ncons;
                if (v < V) {
#pragma unroll
                    for (int i = 0; i < NP; i += 2) {
                        float a0, a1, a2, a3;
                        f2_split(acc_s[k][i], a0, a1);
                        f2_split(acc_s[k][i + 1], a2, a3);
                        *reinterpret_cast<float4 *>(p0 + v * VEC + 2 * i) = make_float4(a0, a1, a2, a3);
                        f2_split(acc_b[k][i], a0, a1);
                        f2_split(acc_b[k][i + 1], a2, a3);
                        *reinterpret_cast<float4 *>(p1 + v * VEC + 2 * i) = make_float4(a0, a1, a2, a3);
                    }
                }
            }
        }
        return true;
    };

    Tile cur, nxt;
    uint32_t kk = 0;  // tiles whose row sums this CTA has published
    if (!split) {
        // lockstep (a ring of only two slots): finish every tile before the next.  A
        // warp whose wait gave up (or whose work ended) still meets the others at
        // the tile's barrier and votes there, so that all leave at the same tile: a
        // warp that left alone would leave the others waiting at the barrier.
        for (;; ++kk) {
            if (!fetch(cur)) {
                named_barrier_any(1, ncons, 1);
                return;
            }
            if (cur.flags & 1) begin_chunk(cur);
            pass1(cur, kk);
            if (!finish(cur, kk)) return;
        }
    }
    if (!fetch(cur)) return;
    begin_chunk(cur);  // a CTA's first tile always starts a chunk
    pass1(cur, kk);
    for (;;) {
        const bool more = fetch(nxt);
        if (more && !(nxt.flags & 1)) {
            // same chunk: overlap this tile's reduction with the next tile's first pass
            pass1(nxt, kk + 1);
            if (!finish(cur, kk)) return;
        } else {
            // end of work or a new chunk (which needs its own modulation row and
            // partials): close the current tile first
            if (!finish(cur, kk)) return;
            if (!more) return;
            begin_chunk(nxt);
            pass1(nxt, kk + 1);
        }
        cur = nxt;
        ++kk;
    }
}

// The same backward for rows too wide for the column partials to stay in
// registers (K > 4 vectors per thread: bf16 rows of up to 16,384 elements, fp32
// rows up to the width whose two ring slots still fit).  Each consumer thread
// keeps its partials in tensor memory instead: warp w of the CTA owns TMEM lanes
// 32 (w % 4) .. +31 and the columns [(w / 4) 2 VEC K, (w / 4 + 1) 2 VEC K) of
// them; vector k's sum dy xhat sits at columns 2 VEC k .. +VEC-1 and its sum dy
// at the next VEC.  The second pass of a tile reads a vector's partials, adds
// the tile's rows and writes them back, one vector at a time.  x and dy are
// read from HBM once, as in the register kernel (the two-kernel column-slab
// backward of wide.cu reads them twice).  The consumers finish each one-row
// tile before the next (lockstep): the register kernel's split-phase schedule,
// tried here, measured no faster at D = 16,384 and 4% slower at 12,288, since
// holding two tiles leaves one ring slot of three in flight.
template <typename T, int K, int R, bool GATED, bool RMS>
__global__ void __launch_bounds__(32 + 352, 1)
    adaln_bwd_ring_tp_kernel(const T *__restrict__ x, const float *__restrict__ mean,
                             const float *__restrict__ rstd, const T *__restrict__ scale,
                             const T *__restrict__ dy, T *__restrict__ dx,
                             float *__restrict__ partial, int *__restrict__ cta_status,
                             int64_t rows, int D, int64_t seg_rows,
                             const int64_t *__restrict__ offsets, int64_t nseg,
                             const int32_t *__restrict__ mod_index, int64_t L, int64_t nchunks,
                             int stages, const T *__restrict__ gate) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t tmem_word;
    constexpr int VEC = IO<T>::VEC;
    constexpr int NP = Pairs<T>::NP;
    constexpr int CPV = 2 * VEC;                       // TMEM columns per vector
    constexpr uint32_t kCols = tmem_cols(3 * K * CPV);  // three warps share a TMEM quarter
    constexpr int P = pow2_at_least(3 * R);
    static_assert(P <= 32, "row tile too large for one warp-level reduction");
    static_assert(CPV == 8 || CPV == 16, "8 or 16 TMEM columns per vector");
    const int V = D / VEC;
    const int ncons = (int)blockDim.x - 32;
    const int ncw = ncons >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const RingLayout lay = ring_layout(D, (int)sizeof(T), R, stages, ncw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bar_off);
    uint64_t *empty = full + stages;
    float(*red)[32] = reinterpret_cast<float(*)[32]>(smem + lay.red_off);  // [4*ncw][32]
    int *status = cta_status + blockIdx.x;

    if (warp == 1) tmem_alloc(&tmem_word, kCols);  // consumer warp 1 frees it at the end
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 2);      // producer arrive.expect_tx + cp.async arrival
            mbar_init(&empty[s], ncw);   // one arrival per consumer warp
        }
        fence_barrier_init();
    }
    pdl_wait();  // before the first global access (the status word included)
    if (threadIdx.x == 0) *status = 0;
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = tmem_word;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        ring_produce<T, R, true>(x, dy, mean, rstd, status, smem, lay, full, empty, stages, rows,
                                 D, seg_rows, offsets, nseg, L, nchunks, lane);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int ct = threadIdx.x - 32;
    const int cw = ct >> 5;
    const float invD = 1.0f / (float)D;
    const uint32_t tp = tmem_lane_addr(tbase, warp, (uint32_t)(warp >> 2) * (uint32_t)(K * CPV));
    f2 s1[K][NP];
    const uint32_t my_off = (uint32_t)ct * 16u;
    auto load = [&](uint32_t sa, int nr, int r, int k, V16 &xvv, V16 &gvv) {
        const int v = ct + k * ncons;
        if (r < nr && v < V) {
            const uint32_t a = sa + (uint32_t)r * lay.row_bytes + my_off + (uint32_t)(k * ncons) * 16u;
            xvv = lds128_at(a);
            gvv = lds128_at(a + lay.tile_bytes);
        } else {
            xvv = V16{{0u, 0u, 0u, 0u}};
            gvv = V16{{0u, 0u, 0u, 0u}};
        }
    };
    // The partials of a pair of vectors k, k + 1 (K is even) are 2 CPV consecutive
    // columns: (sum dy xhat, sum dy) of vector k, then of vector k + 1; one load
    // (and one wait) per pair.
    static_assert(K % 2 == 0, "vectors are handled in pairs");
    auto tp_ld2 = [&](int k, uint32_t (&w)[2 * CPV]) {
        if constexpr (CPV == 16)
            tmem_ld32(tp + (uint32_t)(CPV * k), w);
        else
            tmem_ld16(tp + (uint32_t)(CPV * k), w);
    };
    auto tp_st2 = [&](int k, const uint32_t (&w)[2 * CPV]) {
        if constexpr (CPV == 16) {
            uint32_t a[16], b[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                a[i] = w[i];
                b[i] = w[16 + i];
            }
            tmem_st16(tp + (uint32_t)(CPV * k), a);
            tmem_st16(tp + (uint32_t)(CPV * k + 16), b);
        } else {
            tmem_st16(tp + (uint32_t)(CPV * k), w);
        }
    };
    struct Tile {
        uint32_t sa;  // shared-window address of the slot
        int slot, chunk, nr, flags, seg;
        int64_t r0;
        float rs[R], nmr[R];
    };
    uint32_t it = 0;  // ring slots consumed so far
    // next tile from the ring (false: the end of work, or a wait that gave up)
    auto fetch = [&](Tile &t) -> bool {
        const int s = (int)(it % (uint32_t)stages);
        const uint32_t ph = (it / (uint32_t)stages) & 1u;
        ++it;
        // warp-uniform outcome: the lanes poll on their own, the code after shuffles
        if (!__all_sync(kFull, mbar_wait(&full[s], ph))) {
            atomicExch(status, 2);
            return false;
        }
        const unsigned char *sb = smem + (size_t)s * lay.stage_bytes;
        const TileHdr *hdr = reinterpret_cast<const TileHdr *>(sb + 2 * lay.tile_bytes);
        t.sa = smem_u32(sb);
        t.slot = s;
        t.chunk = hdr->chunk;
        if (t.chunk < 0) return false;
        t.nr = hdr->nr;
        t.flags = hdr->flags;
        t.r0 = hdr->r0;
        t.seg = hdr->seg;
        const float *st = reinterpret_cast<const float *>(hdr + 1);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            t.rs[r] = r < t.nr ? st[R + r] : 0.f;
            t.nmr[r] = (r < t.nr && !RMS) ? -st[r] * t.rs[r] : 0.f;
        }
        return true;
    };
    // first tile of a chunk: the chunk's modulation row, fresh partials (only once
    // the previous chunk's last tile is finished: it still uses both)
    auto begin_chunk = [&](const Tile &t) {
        const int64_t seg = mod_row(mod_index, t.seg);
        uint32_t zero[2 * CPV];
#pragma unroll
        for (int i = 0; i < 2 * CPV; ++i) zero[i] = 0u;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int v = ct + k * ncons;
            const V16 sv = v < V ? ld_cached(scale + seg * D + (int64_t)v * VEC)
                                 : V16{{0u, 0u, 0u, 0u}};
            Pairs<T>::unpack(sv, s1[k]);
#pragma unroll
            for (int i = 0; i < NP; ++i) s1[k][i] = f2_add(f2_make(1.0f, 1.0f), s1[k][i]);
            if constexpr (GATED) {
                const V16 gv = v < V ? ld_cached(gate + seg * D + (int64_t)v * VEC)
                                     : V16{{0u, 0u, 0u, 0u}};
                f2 gp[NP];
                Pairs<T>::unpack(gv, gp);
#pragma unroll
                for (int i = 0; i < NP; ++i) s1[k][i] = f2_mul(s1[k][i], gp[i]);
            }
            if (k % 2 == 1) tp_st2(k - 1, zero);
        }
        tmem_wait_st();
    };
    // pass 1 of tile number kk: per row sum(xh), sum(g), sum(g * xh) over this
    // thread's columns, reduced over the warp and written for the CTA totals
    auto pass1 = [&](const Tile &t, uint32_t kk) {
        f2 pv2[3 * R];
#pragma unroll
        for (int i = 0; i < 3 * R; ++i) pv2[i] = 0ull;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const f2 RS = f2_make(t.rs[r], t.rs[r]), NMR = f2_make(t.nmr[r], t.nmr[r]);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                V16 xvv, gvv;
                load(t.sa, t.nr, r, k, xvv, gvv);
                f2 xp[NP], gp[NP];
                Pairs<T>::unpack(xvv, xp);
                Pairs<T>::unpack(gvv, gp);
                const float cwf = (ct + k * ncons < V) ? 1.0f : 0.0f;
                const f2 CW = f2_make(cwf, cwf);
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    const f2 xh = f2_fma(xp[i], RS, NMR);
                    const f2 g = f2_mul(gp[i], s1[k][i]);
                    pv2[3 * r] = f2_fma(CW, xh, pv2[3 * r]);
                    pv2[3 * r + 1] = f2_add(pv2[3 * r + 1], g);
                    pv2[3 * r + 2] = f2_fma(g, xh, pv2[3 * r + 2]);
                }
            }
        }
        float pv[P];
#pragma unroll
        for (int i = 0; i < P; ++i) {
            pv[i] = 0.f;
            if (i < 3 * R) {
                float lo, hi;
                f2_split(pv2[i], lo, hi);
                pv[i] = lo + hi;
            }
        }
        const float wt = warp_transpose_reduce<P>(pv, lane);
        if ((lane & (32 / P - 1)) == 0) red[(kk & 3u) * ncw + cw][lane / (32 / P)] = wt;
    };
    // wait for tile kk's totals, then pass 2, a pair of vectors at a time: dx, and
    // the pair's partials read, added to and written back (xhat recentred on its
    // row mean, as in the register kernel)
    auto finish = [&](const Tile &t, uint32_t kk) -> bool {
        // every warp's row sums are in, or a warp whose wait gave up voted for all
        // to stop
        if (named_barrier_any(1, ncons, 0)) return false;
        const float tot = cta_totals<P>(red + (kk & 3u) * ncw, ncw, lane);
        float c1v[R], c0v[R], dlv[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float sx = __shfl_sync(kFull, tot, 3 * r);
            const float sg = __shfl_sync(kFull, tot, 3 * r + 1);
            const float sgx = __shfl_sync(kFull, tot, 3 * r + 2);
            const float delta = RMS ? 0.f : sx * invD;
            const float mg = RMS ? 0.f : sg * invD;
            const float mgx = fmaf(-delta, sg, sgx) * invD;
            c1v[r] = t.rs[r] * mgx;
            c0v[r] = fmaf(c1v[r], delta, -t.rs[r] * mg);
            dlv[r] = delta;
        }
#pragma unroll
        for (int k0 = 0; k0 < K; k0 += 2) {
            uint32_t w[2 * CPV];
            tp_ld2(k0, w);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k = k0 + h;
                const int v = ct + k * ncons;
                f2 as[NP], ab[NP];
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    as[i] = f2_from_words(w[h * CPV + 2 * i], w[h * CPV + 2 * i + 1]);
                    ab[i] = f2_from_words(w[h * CPV + VEC + 2 * i], w[h * CPV + VEC + 2 * i + 1]);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r < t.nr) {
                        const f2 RS = f2_make(t.rs[r], t.rs[r]), NMR = f2_make(t.nmr[r], t.nmr[r]);
                        const f2 NC1 = f2_make(-c1v[r], -c1v[r]), C0 = f2_make(c0v[r], c0v[r]);
                        const f2 DL = f2_make(dlv[r], dlv[r]);
                        V16 xvv, gvv;
                        load(t.sa, t.nr, r, k, xvv, gvv);
                        f2 xp[NP], gp[NP], o[NP];
                        Pairs<T>::unpack(xvv, xp);
                        Pairs<T>::unpack(gvv, gp);
#pragma unroll
                        for (int i = 0; i < NP; ++i) {
                            const f2 xh = f2_fma(xp[i], RS, NMR);
                            const f2 g = f2_mul(gp[i], s1[k][i]);
                            o[i] = f2_fma(g, RS, f2_fma(xh, NC1, C0));
                            as[i] = f2_fma(gp[i], f2_sub(xh, DL), as[i]);
                            ab[i] = f2_add(ab[i], gp[i]);
                        }
                        if (v < V)
                            st_vec(dx + (t.r0 + r) * (int64_t)D + (int64_t)v * VEC,
                                   Pairs<T>::pack(o));
                    }
                }
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    float lo, hi;
                    f2_split(as[i], lo, hi);
                    w[h * CPV + 2 * i] = __float_as_uint(lo);
                    w[h * CPV + 2 * i + 1] = __float_as_uint(hi);
                    f2_split(ab[i], lo, hi);
                    w[h * CPV + VEC + 2 * i] = __float_as_uint(lo);
                    w[h * CPV + VEC + 2 * i + 1] = __float_as_uint(hi);
                }
            }
            tp_st2(k0, w);
        }
        tmem_wait_st();  // the next tile's loads of these columns see the stores
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[t.slot]);  // this warp is done with the slot
        if (t.flags & 2) {
            // last tile of the chunk: [c][0][:] = sum dy*xhat, [c][1][:] = sum dy
            float *p0 = partial + ((int64_t)t.chunk * 2 + 0) * D;
            float *p1 = partial + ((int64_t)t.chunk * 2 + 1) * D;
#pragma unroll
            for (int k0 = 0; k0 < K; k0 += 2) {
                uint32_t w[2 * CPV];
                tp_ld2(k0, w);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int v = ct + (k0 + h) * ncons;
                    if (v < V) {
#pragma unroll
                        for (int i = 0; i < VEC; i += 4) {
                            const int b = h * CPV;
                            *reinterpret_cast<float4 *>(p0 + v * VEC + i) = make_float4(
                                __uint_as_float(w[b + i]), __uint_as_float(w[b + i + 1]),
                                __uint_as_float(w[b + i + 2]), __uint_as_float(w[b + i + 3]));
                            *reinterpret_cast<float4 *>(p1 + v * VEC + i) = make_float4(
                                __uint_as_float(w[b + VEC + i]),
                                __uint_as_float(w[b + VEC + i + 1]),
                                __uint_as_float(w[b + VEC + i + 2]),
                                __uint_as_float(w[b + VEC + i + 3]));
                        }
                    }
                }
            }
        }
        return true;
    };

    // Every tile is finished before the next; a warp whose wait gave up (or whose
    // work ended) still meets the others at the tile's barrier and votes there,
    // so all leave at the same tile and no warp frees the tensor memory while
    // another still uses it.
    Tile cur;
    for (uint32_t kk = 0;; ++kk) {
        if (!fetch(cur)) {
            named_barrier_any(1, ncons, 1);
            break;
        }
        if (cur.flags & 1) begin_chunk(cur);
        pass1(cur, kk);
        if (!finish(cur, kk)) break;
    }
    // every consumer is done with its partials: warp 1 frees the tensor memory
    tmem_fence_before();
    named_barrier(1, ncons);
    if (warp == 1) {
        tmem_fence_after();
        tmem_dealloc(tbase, kCols);
    }
}

// Persistent gated-residual backward on the same ring: the producer streams
// R-row tiles of dout and z; every consumer thread owns K column vectors, keeps
// the chunk's gate columns and its d_gate partials in registers, and writes
// dz = gate * dout.  No row reductions, so no barriers among the consumers.
template <typename T, int K, int R>
__global__ void __launch_bounds__(32 + ring_max_consumers(K), 1)
    gate_bwd_ring_kernel(const T *__restrict__ dout, const T *__restrict__ z,
                         const T *__restrict__ gate, T *__restrict__ dz,
                         float *__restrict__ partial, int *__restrict__ cta_status, int64_t rows,
                         int D, int64_t seg_rows, const int64_t *__restrict__ offsets,
                         int64_t nseg, const int32_t *__restrict__ mod_index, int64_t L,
                         int64_t nchunks, int stages) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int VEC = IO<T>::VEC;
    const int V = D / VEC;
    const int ncons = (int)blockDim.x - 32;
    const int ncw = ncons >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const RingLayout lay = ring_layout(D, (int)sizeof(T), R, stages, ncw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bar_off);
    uint64_t *empty = full + stages;
    int *status = cta_status + blockIdx.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);     // producer arrive.expect_tx
            mbar_init(&empty[s], ncw);  // one arrival per consumer warp
        }
        fence_barrier_init();
    }
    pdl_wait();  // before the first global access (the status word included)
    // no early pdl_trigger: see pdl_trigger in common.cuh (dependents launch at exit)
    if (threadIdx.x == 0) *status = 0;
    __syncthreads();
    if (warp == 0) {
        ring_produce<T, R, false>(dout, z, nullptr, nullptr, status, smem, lay, full, empty,
                                  stages, rows, D, seg_rows, offsets, nseg, L, nchunks, lane);
        return;
    }
    const int ct = threadIdx.x - 32;
    const uint32_t my_off = (uint32_t)ct * 16u;
    float gk[K][VEC], acc[K][VEC];
    for (uint32_t it = 0;; ++it) {
        const int s = (int)(it % (uint32_t)stages);
        if (!__all_sync(kFull, mbar_wait(&full[s], (it / (uint32_t)stages) & 1u))) {
            atomicExch(status, 2);
            return;
        }
        const unsigned char *sb = smem + (size_t)s * lay.stage_bytes;
        const TileHdr *hdr = reinterpret_cast<const TileHdr *>(sb + 2 * lay.tile_bytes);
        const int c = hdr->chunk;
        if (c < 0) return;
        const int nr = hdr->nr, flags = hdr->flags;
        const int64_t r0 = hdr->r0;
        if (flags & 1) {  // first tile of a chunk: its gate row, fresh partials
            const int64_t seg = mod_row(mod_index, hdr->seg);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int v = ct + k * ncons;
                if (v < V) {
                    IO<T>::unpack(ld_cached(gate + seg * D + (int64_t)v * VEC), gk[k]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) gk[k][e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[k][e] = 0.f;
            }
        }
        const uint32_t sa = smem_u32(sb);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < nr) {
                T *dzr = dz + (r0 + r) * (int64_t)D;
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int v = ct + k * ncons;
                    if (v < V) {
                        const uint32_t ad = sa + (uint32_t)r * lay.row_bytes + my_off +
                                            (uint32_t)(k * ncons) * 16u;
                        float df[VEC], zf[VEC], o[VEC];
                        IO<T>::unpack(lds128_at(ad), df);
                        IO<T>::unpack(lds128_at(ad + lay.tile_bytes), zf);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            o[e] = gk[k][e] * df[e];
                            acc[k][e] = fmaf(df[e], zf[e], acc[k][e]);
                        }
                        st_vec(dzr + (int64_t)v * VEC, IO<T>::pack(o));
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (flags & 2) {  // last tile of the chunk: [c][:] = sum dout * z
            float *p0 = partial + (int64_t)c * D;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int v = ct + k * ncons;
                if (v < V) {
#pragma unroll
                    for (int e = 0; e < VEC; e += 4)
                        *reinterpret_cast<float4 *>(p0 + v * VEC + e) =
                            make_float4(acc[k][e], acc[k][e + 1], acc[k][e + 2], acc[k][e + 3]);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ dispatch

// Ring geometry for a row of D elements: rows per tile R (about 24 KB of each
// tensor per slot), vectors per consumer thread K, consumer threads, slots.
struct RingGeom {
    int R, K, consumers, stages;
    bool split;  // three or more slots: overlap a tile's reduction with the next tile
    bool tp;     // column partials in tensor memory (K > 4: adaln_bwd_ring_tp_kernel)
    RingLayout lay;
};

// rows per tile: the most (up to 4) for which two slots fit beside each other
inline int ring_rows_for(int64_t row_bytes, int smem_budget) {
    for (int R = 4; R > 1; --R)
        if (2 * (2 * R * row_bytes + 64) + 8192 <= smem_budget) return R;
    return 1;
}

// `tall`: the LayerNorm backward, whose per-tile row reductions and barrier
// cost the same for any tile height; with one vector per thread and rows of at
// least 2048 elements it takes 8-row tiles wherever two slots of them fit.
// `cps`: CTAs that share one SM, each with 1/cps of its shared memory.
bool ring_geometry(int D, int esize, int vec, const DeviceInfo &di, RingGeom &g, bool tall,
                   int cps = 1) {
    const int V = D / vec;
    const int smem_optin = cps > 1 && di.smem_per_sm / cps < di.max_smem_optin
                               ? di.smem_per_sm / cps
                               : di.max_smem_optin;
    g.R = ring_rows_for((int64_t)D * esize, smem_optin - 1024);
    g.K = 0;
    g.tp = false;
    for (int k = 1; k <= 4; k <<= 1)
        if ((V + k - 1) / k <= ring_max_consumers(k)) {
            g.K = k;
            break;
        }
    // wider rows (LayerNorm backward only): six vectors per thread, the column
    // partials in tensor memory
    if (g.K == 0 && tall && (V + 5) / 6 <= 352) {
        g.K = 6;
        g.tp = true;
    }
    if (g.K == 0) return false;
    if (g.K >= 4) g.R = 1;  // keep four vectors per thread within the register budget
    // The gated-residual backward streams with no row reductions: for rows of
    // 8 KB and more it takes 3-row tiles in three slots (measured on GB300 at
    // D = 5120: 0.93 -> 0.96 of the copy bandwidth against two slots of 4 rows;
    // 1- and 2-row tiles were no better).  (Single-row tiles in eight slots were 4%
    // faster on one long D = 3072 call but 20% slower on the ragged buckets,
    // whose short chunks fill the ring more slowly.)
    if (!tall && g.K < 4 && (int64_t)D * esize >= 8192 && g.R > 3) g.R = 3;
    if (tall && g.K == 1 && V >= 256 && 2 * (2 * 8 * (D * esize) + 64) + 8192 <= smem_optin - 1024)
        g.R = 8;
    g.consumers = ((V + g.K - 1) / g.K + 31) / 32 * 32;
    const int cw = g.consumers / 32;
    const int budget = smem_optin - 1024;
    g.stages = 8;
    while (g.stages > 2 && ring_layout(D, esize, g.R, g.stages, cw).total > (uint32_t)budget)
        --g.stages;
    g.lay = ring_layout(D, esize, g.R, g.stages, cw);
    // the split phase holds two slots (a tile and the next) and needs a third to
    // prefetch into; with two slots the consumers finish each tile in turn
    g.split = g.stages >= 3 && !g.tp;
    return g.lay.total <= (uint32_t)budget;
}

// CTAs per SM for rows of D elements: the most (up to kMaxRingCtas) for which
// each CTA keeps the same tile shape and vectors per thread with at least three
// ring slots (the split-phase schedule) in its share of the SM's shared memory,
// and the SM holds that many CTAs' threads and registers (an occupancy query on
// the kernel the shape runs).  Narrow rows only: a row of D elements gives a
// CTA about D / 8 consumer threads, too few warps to hide the latency of a tile.
constexpr int kMaxRingCtas = 3;

// (the kernel's dynamic shared-memory limit is raised first, as its launch does:
// without it the query would count no CTA above 48 KB, and the answer, which
// sizes the workspace, would change after the first launch)
template <typename KERN>
int ring_fits_per_sm_k(KERN kern, int threads, int smem) {
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, (size_t)smem) ==
                   cudaSuccess
               ? n
               : 0;
}

template <typename T, int K, int R>
int ring_fits_per_sm(bool gate, int threads, int smem) {
    return gate ? ring_fits_per_sm_k(gate_bwd_ring_kernel<T, K, R>, threads, smem)
                : ring_fits_per_sm_k(adaln_bwd_ring_kernel<T, K, R, false, false>, threads, smem);
}

template <typename T>
int ctas_per_sm_uncached(int D, bool gate, const DeviceInfo &di) {
    constexpr int VEC = IO<T>::VEC;
    RingGeom g1;
    if (!ring_geometry(D, (int)sizeof(T), VEC, di, g1, !gate, 1)) return 1;
    if (g1.K != 1 || g1.consumers > 256) return 1;
    for (int cps = kMaxRingCtas; cps >= 2; --cps) {
        RingGeom g;
        if (!ring_geometry(D, (int)sizeof(T), VEC, di, g, !gate, cps)) continue;
        if (g.R != g1.R || g.K != g1.K || !g.split) continue;
        const int threads = 32 + g.consumers, smem = (int)g.lay.total;
        int fit = 0;
        if (g.R == 4) fit = ring_fits_per_sm<T, 1, 4>(gate, threads, smem);
        else if (g.R == 3) fit = ring_fits_per_sm<T, 1, 3>(gate, threads, smem);
        else if (g.R == 2) fit = ring_fits_per_sm<T, 1, 2>(gate, threads, smem);
        if (fit >= cps) return cps;
    }
    return 1;
}

// The answer for (device, D, gate), remembered: the query costs a few
// microseconds of host time on every call otherwise, and both the workspace
// plan and each launch ask for it.
template <typename T>
int ctas_per_sm(int D, bool gate, const DeviceInfo &di) {
    struct Entry {
        int dev, D, gate, cps;
    };
    constexpr int kEntries = 64;
    static Entry cache[kEntries];
    static int used = 0, next = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].dev == dev && cache[i].D == D && cache[i].gate == (int)gate)
                return cache[i].cps;
    }
    const int cps = ctas_per_sm_uncached<T>(D, gate, di);
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = Entry{dev, D, (int)gate, cps};
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return cps;
}

template <typename T, int K, int R>
cudaError_t bwd_ring_launch(const void *x, const float *mean, const float *rstd,
                            const void *scale, const void *dy, void *dx, float *partial,
                            int *status, const Segments &sg, const Chunking &ch, int D,
                            const void *gate, const RingGeom &g, int grid, cudaStream_t s) {
    auto kern = gate != nullptr ? adaln_bwd_ring_kernel<T, K, R, true, false>
                : mean == nullptr ? adaln_bwd_ring_kernel<T, K, R, false, true>
                                  : adaln_bwd_ring_kernel<T, K, R, false, false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)g.lay.total);
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, dim3(grid), dim3(32 + g.consumers), g.lay.total, s, (const T *)x, mean,
                     rstd, (const T *)scale, (const T *)dy, (T *)dx, partial, status, sg.rows, D,
                     sg.seg_rows, sg.offsets, sg.nseg, sg.mod_index, ch.L, ch.nchunks, g.stages,
                     g.split,
                     (const T *)gate);
    count_launch();
    return err;
}

template <typename T, int K, int R>
cudaError_t bwd_ring_tp_launch(const void *x, const float *mean, const float *rstd,
                               const void *scale, const void *dy, void *dx, float *partial,
                               int *status, const Segments &sg, const Chunking &ch, int D,
                               const void *gate, const RingGeom &g, int grid, cudaStream_t s) {
    auto kern = gate != nullptr ? adaln_bwd_ring_tp_kernel<T, K, R, true, false>
                : mean == nullptr ? adaln_bwd_ring_tp_kernel<T, K, R, false, true>
                                  : adaln_bwd_ring_tp_kernel<T, K, R, false, false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)g.lay.total);
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, dim3(grid), dim3(32 + g.consumers), g.lay.total, s, (const T *)x, mean,
                     rstd, (const T *)scale, (const T *)dy, (T *)dx, partial, status, sg.rows, D,
                     sg.seg_rows, sg.offsets, sg.nseg, sg.mod_index, ch.L, ch.nchunks, g.stages,
                     (const T *)gate);
    count_launch();
    return err;
}

template <typename T>
cudaError_t bwd_dispatch(const void *x, const float *mean, const float *rstd, const void *scale,
                         const void *dy, void *dx, float *partial, int *status,
                         const Segments &sg, const Chunking &ch, int D, const void *gate,
                         cudaStream_t s) {
    constexpr int VEC = IO<T>::VEC;
    DeviceInfo di;
    cudaError_t err = device_info(di);
    if (err != cudaSuccess) return err;
    RingGeom g;
    if (!ring_geometry(D, (int)sizeof(T), VEC, di, g, true, ctas_per_sm<T>(D, false, di)))
        return cudaErrorInvalidValue;
    const int grid = ch.ctas;
#define ADALN_RING_CASE(KK, RR)                                                                 \
    if (g.K == KK && g.R == RR)                                                                 \
        return bwd_ring_launch<T, KK, RR>(x, mean, rstd, scale, dy, dx, partial, status, sg, ch, \
                                          D, gate, g, grid, s);
    ADALN_RING_CASE(1, 8)
    ADALN_RING_CASE(1, 4)
    ADALN_RING_CASE(2, 4)
    ADALN_RING_CASE(1, 3)
    ADALN_RING_CASE(2, 3)
    ADALN_RING_CASE(1, 2)
    ADALN_RING_CASE(2, 2)
    ADALN_RING_CASE(1, 1)
    ADALN_RING_CASE(2, 1)
    ADALN_RING_CASE(4, 1)
#undef ADALN_RING_CASE
    if (g.tp && g.K == 6 && g.R == 1)
        return bwd_ring_tp_launch<T, 6, 1>(x, mean, rstd, scale, dy, dx, partial, status, sg, ch,
                                           D, gate, g, grid, s);
    return cudaErrorInvalidValue;
}

template <typename T, int K, int R>
cudaError_t gate_bwd_ring_launch(const void *dout, const void *z, const void *gate, void *dz,
                                 float *partial, int *status, const Segments &sg,
                                 const Chunking &ch, int D, const RingGeom &g, int grid,
                                 cudaStream_t s) {
    auto kern = gate_bwd_ring_kernel<T, K, R>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)g.lay.total);
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, dim3(grid), dim3(32 + g.consumers), g.lay.total, s, (const T *)dout,
                     (const T *)z, (const T *)gate, (T *)dz, partial, status, sg.rows, D,
                     sg.seg_rows, sg.offsets, sg.nseg, sg.mod_index, ch.L, ch.nchunks, g.stages);
    count_launch();
    return err;
}

template <typename T>
cudaError_t gate_bwd_dispatch(const void *dout, const void *z, const void *gate, void *dz,
                              float *partial, int *status, const Segments &sg,
                              const Chunking &ch, int D, cudaStream_t s) {
    constexpr int VEC = IO<T>::VEC;
    DeviceInfo di;
    cudaError_t err = device_info(di);
    if (err != cudaSuccess) return err;
    RingGeom g;
    if (!ring_geometry(D, (int)sizeof(T), VEC, di, g, false, ctas_per_sm<T>(D, true, di)))
        return cudaErrorInvalidValue;
    const int grid = ch.ctas;
#define ADALN_GRING_CASE(KK, RR)                                                              \
    if (g.K == KK && g.R == RR)                                                               \
        return gate_bwd_ring_launch<T, KK, RR>(dout, z, gate, dz, partial, status, sg, ch, D, g, \
                                               grid, s);
    ADALN_GRING_CASE(1, 4)
    ADALN_GRING_CASE(2, 4)
    ADALN_GRING_CASE(1, 3)
    ADALN_GRING_CASE(2, 3)
    ADALN_GRING_CASE(1, 2)
    ADALN_GRING_CASE(2, 2)
    ADALN_GRING_CASE(1, 1)
    ADALN_GRING_CASE(2, 1)
    ADALN_GRING_CASE(4, 1)
#undef ADALN_GRING_CASE
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace adaln
