// api.cpp -- the extern "C" entry points declared in include/adaln.h.
//
// Host side only: argument validation (before anything is launched), segment
// and chunk bookkeeping, workspace carving, and dispatch to the kernels.
#include "adaln.h"
#include "launch.h"

#include <cmath>
#include <cstdint>

using adaln::Chunking;
using adaln::DType;
using adaln::Segments;

namespace {

constexpr size_t kAlign = 16;

bool aligned(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % kAlign) == 0; }

// mean and rstd are read and written one float at a time
bool aligned4(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % 4) == 0; }

bool dtype_ok(adaln_dtype dt) { return dt == ADALN_F32 || dt == ADALN_BF16; }

DType to_dt(adaln_dtype dt) { return dt == ADALN_BF16 ? DType::BF16 : DType::F32; }

int vec_elems(adaln_dtype dt) { return dt == ADALN_BF16 ? 8 : 4; }

adaln_status check_dim(int64_t D, adaln_dtype dt) {
    if (!dtype_ok(dt)) return ADALN_ERR_INVALID_ARG;
    if (D <= 0 || D % vec_elems(dt) != 0) return ADALN_ERR_INVALID_ARG;
    if (D > adaln::max_dim(to_dt(dt))) return ADALN_ERR_UNSUPPORTED;
    return ADALN_OK;
}

adaln_status check_dense(int64_t B, int64_t N, int64_t D, adaln_dtype dt) {
    if (B < 0 || N < 0) return ADALN_ERR_INVALID_ARG;
    adaln_status st = check_dim(D, dt);
    if (st != ADALN_OK) return st;
    // rows * D elements must be addressable with int64 byte offsets
    if (B > 0 && N > INT64_MAX / B) return ADALN_ERR_INVALID_ARG;
    if (B * N > (INT64_MAX / 16) / D) return ADALN_ERR_INVALID_ARG;
    if (B > 0 && B > (int64_t)INT32_MAX) return ADALN_ERR_UNSUPPORTED;
    return ADALN_OK;
}

adaln_status check_offsets(const int64_t *offsets_host, const int64_t *offsets_dev, int64_t nseg,
                           int64_t D, adaln_dtype dt) {
    if (offsets_host == nullptr || offsets_dev == nullptr) return ADALN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(offsets_dev) % alignof(int64_t) != 0) return ADALN_ERR_INVALID_ARG;
    if (nseg < 0) return ADALN_ERR_INVALID_ARG;
    if (nseg > (int64_t)INT32_MAX) return ADALN_ERR_UNSUPPORTED;
    adaln_status st = check_dim(D, dt);
    if (st != ADALN_OK) return st;
    if (offsets_host[0] != 0) return ADALN_ERR_INVALID_ARG;
    for (int64_t k = 0; k < nseg; ++k)
        if (offsets_host[k + 1] < offsets_host[k]) return ADALN_ERR_INVALID_ARG;
    if (offsets_host[nseg] > (INT64_MAX / 16) / D) return ADALN_ERR_INVALID_ARG;
    return ADALN_OK;
}

Segments dense_segments(int64_t B, int64_t N) {
    Segments s;
    s.rows = B * N;
    s.nseg = B;
    s.seg_rows = N;
    s.offsets = nullptr;
    s.nmod = B;
    return s;
}

Segments ragged_segments(const int64_t *offsets_host, const int64_t *offsets_dev, int64_t nseg) {
    Segments s;
    s.rows = offsets_host[nseg];
    s.nseg = nseg;
    s.seg_rows = 0;
    s.offsets = offsets_dev;
    s.nmod = nseg;
    return s;
}

// The modulation-row index of the *_indexed calls: int32 [num_segments] on the
// host (validated) and on the device (read by the kernels), every entry in
// [0, num_mod_rows).
adaln_status check_mod_index(const int32_t *mod_index_host, const int32_t *mod_index_dev,
                             int64_t nseg, int64_t nmod) {
    if (nmod < 0) return ADALN_ERR_INVALID_ARG;
    if (nmod > (int64_t)INT32_MAX) return ADALN_ERR_UNSUPPORTED;
    if (nseg == 0) return ADALN_OK;
    if (mod_index_host == nullptr || mod_index_dev == nullptr) return ADALN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(mod_index_dev) % alignof(int32_t) != 0)
        return ADALN_ERR_INVALID_ARG;
    for (int64_t k = 0; k < nseg; ++k)
        if (mod_index_host[k] < 0 || (int64_t)mod_index_host[k] >= nmod) return ADALN_ERR_INVALID_ARG;
    return ADALN_OK;
}

Segments indexed_segments(const int64_t *offsets_host, const int64_t *offsets_dev,
                          const int32_t *mod_index_dev, int64_t nseg, int64_t nmod) {
    Segments s = ragged_segments(offsets_host, offsets_dev, nseg);
    s.mod_index = nseg > 0 ? mod_index_dev : nullptr;
    s.nmod = nmod;
    // with no segments there is no index to read, but the nmod gradient rows are
    // still written (as zeros): the column sums then see an empty index
    return s;
}

adaln_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ADALN_OK : ADALN_ERR_CUDA; }

// Chunking and workspace layout of the column reductions:
//   [ header word (16 bytes) ][ per-CTA status words, padded to 16 bytes ]
//   [ partials: npart * nq * D floats ]
//   [ LayerNorm backward on rows too wide for the pipelined kernel only:
//     4 floats of row coefficients per row ]
struct Plan {
    Chunking ch;
    size_t header_bytes = kAlign;
    size_t status_bytes = 0;
    size_t partial_bytes = 0;
    size_t coef_bytes = 0;
    size_t total() const { return header_bytes + status_bytes + partial_bytes + coef_bytes; }
    float *rowcoef(void *ws) const {
        if (coef_bytes == 0) return nullptr;
        return reinterpret_cast<float *>(static_cast<char *>(ws) + header_bytes + status_bytes +
                                         partial_bytes);
    }
    int *header(void *ws) const { return static_cast<int *>(ws); }
    int *cta_status(void *ws) const {
        return reinterpret_cast<int *>(static_cast<char *>(ws) + header_bytes);
    }
    float *partials(void *ws) const {
        return reinterpret_cast<float *>(static_cast<char *>(ws) + header_bytes + status_bytes);
    }
};

// nq = 2: the LayerNorm (or RMSNorm) backward; nq = 1: the gated-residual backward
adaln_status make_plan(const Segments &sg, int64_t D, int nq, adaln_dtype dt, Plan &plan) {
    adaln::DeviceInfo di;
    if (adaln::device_info(di) != cudaSuccess) return ADALN_ERR_CUDA;
    // one chunk per CTA of the pipelined kernel (several CTAs per SM on narrow rows)
    const bool ring = adaln::bwd_ring_fits(to_dt(dt), D, nq == 1);
    const int64_t ctas =
        (int64_t)di.sms * (ring ? adaln::bwd_ring_ctas_per_sm(to_dt(dt), D, nq == 1) : 1);
    plan.ch.L = adaln::choose_chunk_rows(sg.rows, (int)ctas);
    plan.ch.nchunks = sg.rows > 0 ? (sg.rows + plan.ch.L - 1) / plan.ch.L : 0;
    plan.ch.npart = plan.ch.nchunks > 0 ? plan.ch.nchunks + sg.nseg - 1 : 0;
    if (plan.ch.npart > (int64_t)INT32_MAX) return ADALN_ERR_UNSUPPORTED;
    plan.ch.ctas = (int)(plan.ch.nchunks < ctas ? plan.ch.nchunks : ctas);
    plan.status_bytes = ((size_t)plan.ch.ctas * sizeof(int) + kAlign - 1) / kAlign * kAlign;
    plan.partial_bytes = (size_t)plan.ch.npart * (size_t)nq * (size_t)D * sizeof(float);
    if (nq == 2 && sg.rows > 0 && !ring)
        plan.coef_bytes = (size_t)sg.rows * 4 * sizeof(float);
    return ADALN_OK;
}

adaln_status bind_workspace(const Plan &plan, void *ws, size_t ws_bytes) {
    if (ws_bytes < plan.total()) return ADALN_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(ws)) return ADALN_ERR_INVALID_ARG;
    return ADALN_OK;
}

// ------------------------------------------------------------------ shared bodies

// rms: the RMSNorm statistics; mean is then not used (pass nullptr)
adaln_status fwd_impl(const void *x, const void *shift, const void *scale, void *y, float *mean,
                      float *rstd, const Segments &sg, int64_t D, float eps, adaln_dtype dt,
                      cudaStream_t stream, bool rms = false) {
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return ADALN_ERR_INVALID_ARG;
    if (sg.nmod > 0 && (!aligned(shift) || !aligned(scale))) return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0) {
        if (!aligned(x) || !aligned(y) || !aligned4(rstd)) return ADALN_ERR_INVALID_ARG;
        if (!rms && !aligned4(mean)) return ADALN_ERR_INVALID_ARG;
        if (x == y) return ADALN_ERR_INVALID_ARG;
    }
    return cuda_status(adaln::launch_fwd(to_dt(dt), x, shift, scale, y, rms ? nullptr : mean, rstd,
                                         sg, D, eps, stream, adaln::GateEpilogue(), rms));
}

adaln_status gate_impl(const void *r, const void *z, const void *gate, void *out,
                       const Segments &sg, int64_t D, adaln_dtype dt, cudaStream_t stream) {
    if (sg.nmod > 0 && !aligned(gate)) return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0 && (!aligned(r) || !aligned(z) || !aligned(out))) return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0 && (out == r || out == z)) return ADALN_ERR_INVALID_ARG;
    return cuda_status(adaln::launch_gate(to_dt(dt), r, z, gate, out, sg, D, stream));
}

// rms: the RMSNorm backward (mean is nullptr; the kernels take that as the switch)
adaln_status bwd_impl(const void *x, const float *mean, const float *rstd, const void *scale,
                      const void *dy, void *dx, float *d_scale, float *d_shift, void *ws,
                      size_t ws_bytes, const Segments &sg, int64_t D, adaln_dtype dt,
                      cudaStream_t stream, bool rms = false) {
    if (sg.nmod > 0 && (!aligned(scale) || !aligned(d_scale) || !aligned(d_shift)))
        return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0 && (!aligned(x) || !aligned(dy) || !aligned(dx) || !aligned4(rstd)))
        return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0 && !rms && !aligned4(mean)) return ADALN_ERR_INVALID_ARG;
    if (rms) mean = nullptr;
    if (sg.rows > 0 && (dx == x || dx == dy)) return ADALN_ERR_INVALID_ARG;
    Plan plan;
    adaln_status st = make_plan(sg, D, 2, dt, plan);
    if (st != ADALN_OK) return st;
    st = bind_workspace(plan, ws, ws_bytes);
    if (st != ADALN_OK) return st;
    return cuda_status(adaln::launch_bwd(to_dt(dt), x, mean, rstd, scale, dy, dx, d_scale, d_shift,
                                         plan.partials(ws), plan.header(ws), plan.cta_status(ws),
                                         plan.rowcoef(ws), sg, plan.ch, D, stream));
}

adaln_status gate_bwd_impl(const void *dout, const void *z, const void *gate, void *dz,
                           float *d_gate, void *ws, size_t ws_bytes, const Segments &sg,
                           int64_t D, adaln_dtype dt, cudaStream_t stream) {
    if (sg.nmod > 0 && (!aligned(gate) || !aligned(d_gate))) return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0 && (!aligned(dout) || !aligned(z) || !aligned(dz))) return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0 && (dz == dout || dz == z)) return ADALN_ERR_INVALID_ARG;
    Plan plan;
    adaln_status st = make_plan(sg, D, 1, dt, plan);
    if (st != ADALN_OK) return st;
    st = bind_workspace(plan, ws, ws_bytes);
    if (st != ADALN_OK) return st;
    return cuda_status(adaln::launch_gate_bwd(to_dt(dt), dout, z, gate, dz, d_gate,
                                              plan.partials(ws), plan.header(ws),
                                              plan.cta_status(ws), sg, plan.ch, D, stream));
}

// Fused gated chain: out = r + gate * y (y optional)
adaln_status fwd_gated_impl(const void *x, const void *shift, const void *scale, const void *gate,
                            const void *r, void *out, void *y, float *mean, float *rstd,
                            const Segments &sg, int64_t D, float eps, adaln_dtype dt,
                            cudaStream_t stream) {
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return ADALN_ERR_INVALID_ARG;
    if (sg.nmod > 0 && (!aligned(shift) || !aligned(scale) || !aligned(gate)))
        return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0) {
        if (!aligned(x) || !aligned(r) || !aligned(out) || !aligned4(mean) || !aligned4(rstd))
            return ADALN_ERR_INVALID_ARG;
        if (y != nullptr && !aligned(y)) return ADALN_ERR_INVALID_ARG;
        if (out == x || out == r || out == y) return ADALN_ERR_INVALID_ARG;
        if (y != nullptr && (y == x || y == r)) return ADALN_ERR_INVALID_ARG;
    }
    adaln::GateEpilogue ge;
    ge.gate = gate;
    ge.r = r;
    ge.out = out;
    return cuda_status(
        adaln::launch_fwd(to_dt(dt), x, shift, scale, y, mean, rstd, sg, D, eps, stream, ge));
}

adaln_status bwd_gated_impl(const void *x, const float *mean, const float *rstd,
                            const void *shift, const void *scale, const void *gate,
                            const void *dout, void *dx, float *d_scale, float *d_shift,
                            float *d_gate, void *ws, size_t ws_bytes, const Segments &sg,
                            int64_t D, adaln_dtype dt, cudaStream_t stream) {
    if (sg.nmod > 0 && (!aligned(shift) || !aligned(scale) || !aligned(gate) ||
                        !aligned(d_scale) || !aligned(d_shift) || !aligned(d_gate)))
        return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0 && (!aligned(x) || !aligned(dout) || !aligned(dx) || !aligned4(mean) ||
                        !aligned4(rstd)))
        return ADALN_ERR_INVALID_ARG;
    if (sg.rows > 0 && (dx == x || dx == dout)) return ADALN_ERR_INVALID_ARG;
    Plan plan;
    adaln_status st = make_plan(sg, D, 2, dt, plan);
    if (st != ADALN_OK) return st;
    st = bind_workspace(plan, ws, ws_bytes);
    if (st != ADALN_OK) return st;
    adaln::BwdGate bg;
    bg.shift = shift;
    bg.gate = gate;
    bg.d_gate = d_gate;
    return cuda_status(adaln::launch_bwd(to_dt(dt), x, mean, rstd, scale, dout, dx, d_scale,
                                         d_shift, plan.partials(ws), plan.header(ws),
                                         plan.cta_status(ws), plan.rowcoef(ws), sg, plan.ch, D,
                                         stream, bg));
}

size_t workspace_size(const Segments &sg, int64_t D, int nq, adaln_dtype dt) {
    Plan plan;
    if (make_plan(sg, D, nq, dt, plan) != ADALN_OK) return 0;
    return plan.total();
}

}  // namespace

extern "C" {

const char *adaln_status_string(adaln_status status) {
    switch (status) {
        case ADALN_OK:
            return "ADALN_OK";
        case ADALN_ERR_INVALID_ARG:
            return "ADALN_ERR_INVALID_ARG: null or misaligned pointer, bad size, dtype or offsets";
        case ADALN_ERR_UNSUPPORTED:
            return "ADALN_ERR_UNSUPPORTED: valid arguments outside the supported range";
        case ADALN_ERR_WORKSPACE_TOO_SMALL:
            return "ADALN_ERR_WORKSPACE_TOO_SMALL: workspace smaller than the size query returned";
        case ADALN_ERR_CUDA:
            return "ADALN_ERR_CUDA: the CUDA runtime reported an error";
    }
    return "unknown adaln_status";
}

int64_t adaln_max_dim(adaln_dtype dtype) {
    if (!dtype_ok(dtype)) return 0;
    return adaln::max_dim(to_dt(dtype));
}

uint64_t adaln_launch_count(void) { return adaln::launch_count(); }

int adaln_pipeline_status(void) {
    const int fwd = adaln::pipeline_status();
    const int noalloc = adaln::noalloc_status();
    if (fwd < 0 || noalloc < 0) return -1;
    return fwd | noalloc;
}

adaln_status adaln_fwd(const void *x, const void *shift, const void *scale, void *y, float *mean,
                       float *rstd, int64_t B, int64_t N, int64_t D, float eps, adaln_dtype dtype,
                       cudaStream_t stream) {
    adaln_status st = check_dense(B, N, D, dtype);
    if (st != ADALN_OK) return st;
    return fwd_impl(x, shift, scale, y, mean, rstd, dense_segments(B, N), D, eps, dtype, stream);
}

adaln_status adaln_gate_residual(const void *r, const void *z, const void *gate, void *out,
                                 int64_t B, int64_t N, int64_t D, adaln_dtype dtype,
                                 cudaStream_t stream) {
    adaln_status st = check_dense(B, N, D, dtype);
    if (st != ADALN_OK) return st;
    return gate_impl(r, z, gate, out, dense_segments(B, N), D, dtype, stream);
}

size_t adaln_bwd_workspace_size(int64_t B, int64_t N, int64_t D, adaln_dtype dtype) {
    if (check_dense(B, N, D, dtype) != ADALN_OK) return 0;
    return workspace_size(dense_segments(B, N), D, 2, dtype);
}

adaln_status adaln_bwd(const void *x, const float *mean, const float *rstd, const void *scale,
                       const void *dy, void *dx, float *d_scale, float *d_shift, void *workspace,
                       size_t workspace_bytes, int64_t B, int64_t N, int64_t D,
                       adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_dense(B, N, D, dtype);
    if (st != ADALN_OK) return st;
    return bwd_impl(x, mean, rstd, scale, dy, dx, d_scale, d_shift, workspace, workspace_bytes,
                    dense_segments(B, N), D, dtype, stream);
}

size_t adaln_gate_residual_bwd_workspace_size(int64_t B, int64_t N, int64_t D,
                                              adaln_dtype dtype) {
    if (check_dense(B, N, D, dtype) != ADALN_OK) return 0;
    return workspace_size(dense_segments(B, N), D, 1, dtype);
}

adaln_status adaln_gate_residual_bwd(const void *dout, const void *z, const void *gate, void *dz,
                                     float *d_gate, void *workspace, size_t workspace_bytes,
                                     int64_t B, int64_t N, int64_t D, adaln_dtype dtype,
                                     cudaStream_t stream) {
    adaln_status st = check_dense(B, N, D, dtype);
    if (st != ADALN_OK) return st;
    return gate_bwd_impl(dout, z, gate, dz, d_gate, workspace, workspace_bytes,
                         dense_segments(B, N), D, dtype, stream);
}

adaln_status adaln_fwd_ragged(const void *x, const void *shift, const void *scale, void *y,
                              float *mean, float *rstd, const int64_t *offsets_host,
                              const int64_t *offsets_dev, int64_t num_segments, int64_t D,
                              float eps, adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    return fwd_impl(x, shift, scale, y, mean, rstd,
                    ragged_segments(offsets_host, offsets_dev, num_segments), D, eps, dtype,
                    stream);
}

adaln_status adaln_gate_residual_ragged(const void *r, const void *z, const void *gate,
                                        void *out, const int64_t *offsets_host,
                                        const int64_t *offsets_dev, int64_t num_segments,
                                        int64_t D, adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    return gate_impl(r, z, gate, out, ragged_segments(offsets_host, offsets_dev, num_segments), D,
                     dtype, stream);
}

size_t adaln_bwd_ragged_workspace_size(const int64_t *offsets_host, int64_t num_segments,
                                       int64_t D, adaln_dtype dtype) {
    if (offsets_host == nullptr || num_segments < 0) return 0;
    // the device pointer is not needed for the size; validate the host offsets only
    if (check_offsets(offsets_host, offsets_host, num_segments, D, dtype) != ADALN_OK) return 0;
    return workspace_size(ragged_segments(offsets_host, nullptr, num_segments), D, 2, dtype);
}

adaln_status adaln_bwd_ragged(const void *x, const float *mean, const float *rstd,
                              const void *scale, const void *dy, void *dx, float *d_scale,
                              float *d_shift, void *workspace, size_t workspace_bytes,
                              const int64_t *offsets_host, const int64_t *offsets_dev,
                              int64_t num_segments, int64_t D, adaln_dtype dtype,
                              cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    return bwd_impl(x, mean, rstd, scale, dy, dx, d_scale, d_shift, workspace, workspace_bytes,
                    ragged_segments(offsets_host, offsets_dev, num_segments), D, dtype,
                    stream);
}

size_t adaln_gate_residual_bwd_ragged_workspace_size(const int64_t *offsets_host,
                                                     int64_t num_segments, int64_t D,
                                                     adaln_dtype dtype) {
    if (offsets_host == nullptr || num_segments < 0) return 0;
    if (check_offsets(offsets_host, offsets_host, num_segments, D, dtype) != ADALN_OK) return 0;
    return workspace_size(ragged_segments(offsets_host, nullptr, num_segments), D, 1, dtype);
}

adaln_status adaln_gate_residual_bwd_ragged(const void *dout, const void *z, const void *gate,
                                            void *dz, float *d_gate, void *workspace,
                                            size_t workspace_bytes, const int64_t *offsets_host,
                                            const int64_t *offsets_dev, int64_t num_segments,
                                            int64_t D, adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    return gate_bwd_impl(dout, z, gate, dz, d_gate, workspace, workspace_bytes,
                         ragged_segments(offsets_host, offsets_dev, num_segments), D,
                         dtype, stream);
}

adaln_status adaln_fwd_ragged_indexed(const void *x, const void *shift, const void *scale,
                                      void *y, float *mean, float *rstd,
                                      const int64_t *offsets_host, const int64_t *offsets_dev,
                                      const int32_t *mod_index_host, const int32_t *mod_index_dev,
                                      int64_t num_segments, int64_t num_mod_rows, int64_t D,
                                      float eps, adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    st = check_mod_index(mod_index_host, mod_index_dev, num_segments, num_mod_rows);
    if (st != ADALN_OK) return st;
    return fwd_impl(x, shift, scale, y, mean, rstd,
                    indexed_segments(offsets_host, offsets_dev, mod_index_dev, num_segments,
                                     num_mod_rows),
                    D, eps, dtype, stream);
}

adaln_status adaln_gate_residual_ragged_indexed(const void *r, const void *z, const void *gate,
                                                void *out, const int64_t *offsets_host,
                                                const int64_t *offsets_dev,
                                                const int32_t *mod_index_host,
                                                const int32_t *mod_index_dev,
                                                int64_t num_segments, int64_t num_mod_rows,
                                                int64_t D, adaln_dtype dtype,
                                                cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    st = check_mod_index(mod_index_host, mod_index_dev, num_segments, num_mod_rows);
    if (st != ADALN_OK) return st;
    return gate_impl(r, z, gate, out,
                     indexed_segments(offsets_host, offsets_dev, mod_index_dev, num_segments,
                                      num_mod_rows),
                     D, dtype, stream);
}

adaln_status adaln_bwd_ragged_indexed(const void *x, const float *mean, const float *rstd,
                                      const void *scale, const void *dy, void *dx, float *d_scale,
                                      float *d_shift, void *workspace, size_t workspace_bytes,
                                      const int64_t *offsets_host, const int64_t *offsets_dev,
                                      const int32_t *mod_index_host, const int32_t *mod_index_dev,
                                      int64_t num_segments, int64_t num_mod_rows, int64_t D,
                                      adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    st = check_mod_index(mod_index_host, mod_index_dev, num_segments, num_mod_rows);
    if (st != ADALN_OK) return st;
    return bwd_impl(x, mean, rstd, scale, dy, dx, d_scale, d_shift, workspace, workspace_bytes,
                    indexed_segments(offsets_host, offsets_dev, mod_index_dev, num_segments,
                                     num_mod_rows),
                    D, dtype, stream);
}

adaln_status adaln_gate_residual_bwd_ragged_indexed(
    const void *dout, const void *z, const void *gate, void *dz, float *d_gate, void *workspace,
    size_t workspace_bytes, const int64_t *offsets_host, const int64_t *offsets_dev,
    const int32_t *mod_index_host, const int32_t *mod_index_dev, int64_t num_segments,
    int64_t num_mod_rows, int64_t D, adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    st = check_mod_index(mod_index_host, mod_index_dev, num_segments, num_mod_rows);
    if (st != ADALN_OK) return st;
    return gate_bwd_impl(dout, z, gate, dz, d_gate, workspace, workspace_bytes,
                         indexed_segments(offsets_host, offsets_dev, mod_index_dev, num_segments,
                                          num_mod_rows),
                         D, dtype, stream);
}

adaln_status adaln_fwd_gated(const void *x, const void *shift, const void *scale, const void *gate,
                             const void *r, void *out, void *y, float *mean, float *rstd,
                             int64_t B, int64_t N, int64_t D, float eps, adaln_dtype dtype,
                             cudaStream_t stream) {
    adaln_status st = check_dense(B, N, D, dtype);
    if (st != ADALN_OK) return st;
    return fwd_gated_impl(x, shift, scale, gate, r, out, y, mean, rstd, dense_segments(B, N), D,
                          eps, dtype, stream);
}

adaln_status adaln_fwd_gated_ragged(const void *x, const void *shift, const void *scale,
                                    const void *gate, const void *r, void *out, void *y,
                                    float *mean, float *rstd, const int64_t *offsets_host,
                                    const int64_t *offsets_dev, int64_t num_segments, int64_t D,
                                    float eps, adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    return fwd_gated_impl(x, shift, scale, gate, r, out, y, mean, rstd,
                          ragged_segments(offsets_host, offsets_dev, num_segments), D, eps, dtype,
                          stream);
}

size_t adaln_bwd_gated_workspace_size(int64_t B, int64_t N, int64_t D, adaln_dtype dtype) {
    if (check_dense(B, N, D, dtype) != ADALN_OK) return 0;
    return workspace_size(dense_segments(B, N), D, 2, dtype);
}

adaln_status adaln_bwd_gated(const void *x, const float *mean, const float *rstd,
                             const void *shift, const void *scale, const void *gate,
                             const void *dout, void *dx, float *d_scale, float *d_shift,
                             float *d_gate, void *workspace, size_t workspace_bytes, int64_t B,
                             int64_t N, int64_t D, adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_dense(B, N, D, dtype);
    if (st != ADALN_OK) return st;
    return bwd_gated_impl(x, mean, rstd, shift, scale, gate, dout, dx, d_scale, d_shift, d_gate,
                          workspace, workspace_bytes, dense_segments(B, N), D, dtype, stream);
}

size_t adaln_bwd_gated_ragged_workspace_size(const int64_t *offsets_host, int64_t num_segments,
                                             int64_t D, adaln_dtype dtype) {
    if (offsets_host == nullptr || num_segments < 0) return 0;
    if (check_offsets(offsets_host, offsets_host, num_segments, D, dtype) != ADALN_OK) return 0;
    return workspace_size(ragged_segments(offsets_host, nullptr, num_segments), D, 2, dtype);
}

adaln_status adaln_bwd_gated_ragged(const void *x, const float *mean, const float *rstd,
                                    const void *shift, const void *scale, const void *gate,
                                    const void *dout, void *dx, float *d_scale, float *d_shift,
                                    float *d_gate, void *workspace, size_t workspace_bytes,
                                    const int64_t *offsets_host, const int64_t *offsets_dev,
                                    int64_t num_segments, int64_t D, adaln_dtype dtype,
                                    cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    return bwd_gated_impl(x, mean, rstd, shift, scale, gate, dout, dx, d_scale, d_shift, d_gate,
                          workspace, workspace_bytes,
                          ragged_segments(offsets_host, offsets_dev, num_segments), D, dtype,
                          stream);
}

adaln_status adaln_fwd_rms(const void *x, const void *shift, const void *scale, void *y,
                           float *rstd, int64_t B, int64_t N, int64_t D, float eps,
                           adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_dense(B, N, D, dtype);
    if (st != ADALN_OK) return st;
    return fwd_impl(x, shift, scale, y, nullptr, rstd, dense_segments(B, N), D, eps, dtype,
                    stream, true);
}

adaln_status adaln_fwd_rms_ragged(const void *x, const void *shift, const void *scale, void *y,
                                  float *rstd, const int64_t *offsets_host,
                                  const int64_t *offsets_dev, int64_t num_segments, int64_t D,
                                  float eps, adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    return fwd_impl(x, shift, scale, y, nullptr, rstd,
                    ragged_segments(offsets_host, offsets_dev, num_segments), D, eps, dtype,
                    stream, true);
}

adaln_status adaln_bwd_rms(const void *x, const float *rstd, const void *scale, const void *dy,
                           void *dx, float *d_scale, float *d_shift, void *workspace,
                           size_t workspace_bytes, int64_t B, int64_t N, int64_t D,
                           adaln_dtype dtype, cudaStream_t stream) {
    adaln_status st = check_dense(B, N, D, dtype);
    if (st != ADALN_OK) return st;
    return bwd_impl(x, nullptr, rstd, scale, dy, dx, d_scale, d_shift, workspace, workspace_bytes,
                    dense_segments(B, N), D, dtype, stream, true);
}

adaln_status adaln_bwd_rms_ragged(const void *x, const float *rstd, const void *scale,
                                  const void *dy, void *dx, float *d_scale, float *d_shift,
                                  void *workspace, size_t workspace_bytes,
                                  const int64_t *offsets_host, const int64_t *offsets_dev,
                                  int64_t num_segments, int64_t D, adaln_dtype dtype,
                                  cudaStream_t stream) {
    adaln_status st = check_offsets(offsets_host, offsets_dev, num_segments, D, dtype);
    if (st != ADALN_OK) return st;
    return bwd_impl(x, nullptr, rstd, scale, dy, dx, d_scale, d_shift, workspace, workspace_bytes,
                    ragged_segments(offsets_host, offsets_dev, num_segments), D, dtype, stream,
                    true);
}

}  // extern "C"
