/*
 * adaln.h -- C ABI of the GB300 (sm_103a) AdaLN modulation library.
 *
 * The operator is the adaptive LayerNorm ("AdaLN") of a diffusion-transformer
 * block, as described in the "AdaptiveLoad" technical summary (gist.science
 * paper 2605.17923):
 *   - section 1, second bullet: AdaLN is invoked hundreds of times per step in
 *     (MM)DiT blocks; unfused kernels round-trip intermediates through HBM and
 *     the backward reduction of the modulation-parameter gradients runs along
 *     the sequence dimension N;
 *   - section 2.B, "Paso Adelante": one launch computes the row statistics over
 *     the feature dimension D (warp-level then block-level reductions) and
 *     applies the modulation during a further traversal of D;
 *   - section 2.B, "Paso Atras": the (d_tile, n_tile) coalesced reduction of
 *     the parameter gradients, threads pinned to a feature d and accumulating
 *     down the sequence;
 *   - section 2.B, "Simplificacion de Grafos": the chain collapses to one node
 *     per call and only the row statistics are kept for the backward.
 * The summary prints no formula for AdaLN; the one implemented is the DiT
 * adaptive LayerNorm (no affine, biased variance, eps inside the root):
 *     y    = xhat * (1 + scale[k]) + shift[k],  xhat = (x - mean) * rstd,
 *     rstd = 1 / sqrt(var + eps),               var  = mean_d (x - mean)^2,
 *     out  = r + gate[k] * z                    (gated residual),
 * where k is the segment (a sample of a dense batch, or a packed sequence)
 * the row belongs to.
 *
 * Conventions shared by every entry point
 *   - Returns adaln_status; nothing else signals errors.  All arguments are
 *     validated on the host before anything is launched; a failed validation
 *     launches nothing and leaves every output untouched.
 *   - Every device pointer is owned by the caller and must stay valid until
 *     the work queued on `stream` has finished.  Pointers to activations,
 *     modulation rows, parameter gradients and workspaces must be 16-byte
 *     aligned; mean and rstd need only float (4-byte) alignment.
 *     The library never allocates, never synchronises, keeps no per-call
 *     state and is safe to call from several host threads.  The first call
 *     of a shape on a device queries device attributes, sets kernel
 *     attributes and asks the occupancy calculator (host-side calls, which a
 *     stream capture allows); the answers are kept per device and reused.
 *     Every call can be captured into a CUDA graph and replayed.
 *   - Launches are asynchronous on `stream` (0 = the legacy default stream).
 *     A launch failure reported by the CUDA runtime returns ADALN_ERR_CUDA.
 *   - dtype selects the element type of every activation-sized tensor and of
 *     shift/scale/gate: ADALN_F32 (float) or ADALN_BF16 (bfloat16).  Row
 *     statistics (mean, rstd) and parameter gradients (d_scale, d_shift,
 *     d_gate) are always float.  Arithmetic is fp32; bf16 outputs are rounded
 *     to nearest-even once.
 *   - D must be a positive multiple of 8 (bf16) or 4 (fp32) and at most
 *     adaln_max_dim(dtype) = 16384; larger D returns ADALN_ERR_UNSUPPORTED.
 *     Wide rows take other kernels, with the same results: the bf16 forward
 *     spreads rows of 8192, 12288 and 16384 elements over four warps each, and
 *     other rows of more than 6144 (bf16) or 3072 (fp32) elements over a CTA;
 *     the backward keeps its column partials in tensor memory for bf16 rows
 *     above 11264 and fp32 rows above 5632 elements, and for fp32 rows above
 *     8448 elements computes per-row coefficients first and then goes by
 *     column slabs (x and dy are then read twice).
 *   - Layouts are row-major with D contiguous: activations are [rows, D]
 *     (dense: [B, N, D], rows = B*N); modulation rows and parameter gradients
 *     are [num_segments, D] (dense: [B, D]); mean and rstd are [rows].
 *   - Zero rows is valid: nothing is launched except the kernels that write
 *     the parameter gradients, which then hold zeros (an empty sum).
 *   - Parameter gradients are reduced deterministically (fixed order, no
 *     floating-point atomics): on one device and one workspace size the
 *     results are bitwise reproducible.
 *
 * Ragged (packed) variants: rows of all segments are packed back to back;
 * segment k holds rows [offsets[k], offsets[k+1]) and uses modulation row k.
 * The same offsets are passed twice: offsets_host (read on the host for
 * validation and launch sizing) and offsets_dev (read by the kernels).  They
 * must hold identical values; offsets[0] == 0, non-decreasing, and
 * offsets[num_segments] is the total row count.  Empty segments are allowed.
 */
#ifndef ADALN_H
#define ADALN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum adaln_status {
    ADALN_OK = 0,
    ADALN_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad size or offsets */
    ADALN_ERR_UNSUPPORTED = 2,        /* valid but outside what the kernels handle */
    ADALN_ERR_WORKSPACE_TOO_SMALL = 3,
    ADALN_ERR_CUDA = 4                /* the CUDA runtime reported an error */
} adaln_status;

typedef enum adaln_dtype { ADALN_F32 = 0, ADALN_BF16 = 1 } adaln_dtype;

/* Human-readable name of a status (static string, never NULL). */
const char *adaln_status_string(adaln_status status);

/* Largest supported feature dimension D for a dtype. */
int64_t adaln_max_dim(adaln_dtype dtype);

/* Number of kernel launches this library has issued since it was loaded
 * (diagnostic counter, process-wide). */
uint64_t adaln_launch_count(void);

/* Diagnostic: 0 unless a bounded wait inside a pipelined kernel gave up (which
 * would mean a bug; that call's outputs are then incomplete), as seen on the
 * current device:
 *   - the pipelined forward kernel, at any time since the library was loaded
 *     (a sticky word);
 *   - the last adaln_bwd_noalloc call that launched work, whose status lives in
 *     the library's built-in scratch rather than in a caller workspace.
 * Reads device words, so it synchronises with the device; -1 if a read fails.
 * The other backward calls report the same condition in the first word of
 * their workspace. */
int adaln_pipeline_status(void);

/* ---------------------------------------------------------------- forward
 * adaln_fwd: y = LN(x) * (1 + scale[b]) + shift[b] for x [B, N, D]
 * (summary section 2.B, "Paso Adelante").
 *   x      [B*N, D]  dtype   input
 *   shift  [B, D]    dtype   modulation shift, broadcast over N
 *   scale  [B, D]    dtype   modulation scale, broadcast over N
 *   y      [B*N, D]  dtype   output (may not alias x)
 *   mean   [B*N]     float   output: row mean
 *   rstd   [B*N]     float   output: 1 / sqrt(var + eps)
 * mean and rstd are the row statistics rounded once to float: they are
 * computed with error-free (compensated) fp32 arithmetic so that they equal
 * the exactly rounded fp64 values except where the exact value lies within
 * about 2^-36 (relative) of a float rounding boundary.
 * eps >= 0 and finite, else ADALN_ERR_INVALID_ARG.
 * Any finite x is handled: rows whose largest |x| reaches 2^59 take scaled
 * two-pass statistics, and rows with |mean| * rstd > 4 modulate as
 * (x - mean) * rstd.
 */
adaln_status adaln_fwd(const void *x, const void *shift, const void *scale, void *y,
                       float *mean, float *rstd, int64_t B, int64_t N, int64_t D,
                       float eps, adaln_dtype dtype, cudaStream_t stream);

/* adaln_gate_residual: out = r + gate[b] * z (the gated-residual epilogue).
 *   r, z [B*N, D] dtype inputs; gate [B, D] dtype; out [B*N, D] dtype output
 *   (out must not alias r or z: inputs are read through the read-only path). */
adaln_status adaln_gate_residual(const void *r, const void *z, const void *gate, void *out,
                                 int64_t B, int64_t N, int64_t D, adaln_dtype dtype,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------- backward
 * adaln_bwd: gradients of y = LN(x) * (1 + scale) + shift given dy
 * (summary section 1 and section 2.B, "Paso Atras"):
 *   g            = dy * (1 + scale[b])
 *   dx           = rstd * (g - mean_d(g) - xhat * mean_d(g * xhat))
 *   d_scale[b,d] = sum_n dy * xhat,   d_shift[b,d] = sum_n dy
 *   x, dy    [B*N, D] dtype inputs;  mean, rstd [B*N] float from adaln_fwd;
 *   scale    [B, D] dtype;           dx [B*N, D] dtype output (no aliasing);
 *   d_scale, d_shift [B, D] float outputs (overwritten, not accumulated).
 *   xhat is formed as x * rstd - mean * rstd (one fused multiply-add), so its
 *   absolute error is about |mean| * rstd * 2^-24: rows must have |mean| * rstd
 *   well inside the float range (nearly constant rows of values beyond about
 *   1e35 at eps = 1e-6 give NaN gradients; the forward handles them).
 *   workspace: device scratch of at least adaln_bwd_workspace_size() bytes,
 *   16-byte aligned, not shared with a concurrent call.  Its size depends on
 *   the current device (its multiprocessor count and shared memory); query it
 *   there.  For fp32 rows of more than 8448 elements it includes 16 bytes per
 *   row of coefficients.
 */
size_t adaln_bwd_workspace_size(int64_t B, int64_t N, int64_t D, adaln_dtype dtype);
adaln_status adaln_bwd(const void *x, const float *mean, const float *rstd, const void *scale,
                       const void *dy, void *dx, float *d_scale, float *d_shift,
                       void *workspace, size_t workspace_bytes, int64_t B, int64_t N,
                       int64_t D, adaln_dtype dtype, cudaStream_t stream);

/* adaln_gate_residual_bwd: dz = gate[b] * dout; d_gate[b,d] = sum_n dout * z.
 * dr = dout is the identity and is not written.
 *   dout, z [B*N, D] dtype; gate [B, D] dtype; dz [B*N, D] dtype output
 *   (dz must not alias dout or z);
 *   d_gate [B, D] float output; workspace as for adaln_bwd. */
size_t adaln_gate_residual_bwd_workspace_size(int64_t B, int64_t N, int64_t D,
                                              adaln_dtype dtype);
adaln_status adaln_gate_residual_bwd(const void *dout, const void *z, const void *gate,
                                     void *dz, float *d_gate, void *workspace,
                                     size_t workspace_bytes, int64_t B, int64_t N, int64_t D,
                                     adaln_dtype dtype, cudaStream_t stream);

/* ---------------------------------------------------------------- ragged
 * Same operations over packed sequences (segment k = rows
 * [offsets[k], offsets[k+1]), modulation row k).  Shapes as above with
 * rows = offsets[num_segments] and B replaced by num_segments.  One call
 * covers every segment in one launch per kernel (e.g. both streams of an
 * MMDiT block, or one bucket of mixed-length sequences). */
adaln_status adaln_fwd_ragged(const void *x, const void *shift, const void *scale, void *y,
                              float *mean, float *rstd, const int64_t *offsets_host,
                              const int64_t *offsets_dev, int64_t num_segments, int64_t D,
                              float eps, adaln_dtype dtype, cudaStream_t stream);

adaln_status adaln_gate_residual_ragged(const void *r, const void *z, const void *gate,
                                        void *out, const int64_t *offsets_host,
                                        const int64_t *offsets_dev, int64_t num_segments,
                                        int64_t D, adaln_dtype dtype, cudaStream_t stream);

size_t adaln_bwd_ragged_workspace_size(const int64_t *offsets_host, int64_t num_segments,
                                       int64_t D, adaln_dtype dtype);
adaln_status adaln_bwd_ragged(const void *x, const float *mean, const float *rstd,
                              const void *scale, const void *dy, void *dx, float *d_scale,
                              float *d_shift, void *workspace, size_t workspace_bytes,
                              const int64_t *offsets_host, const int64_t *offsets_dev,
                              int64_t num_segments, int64_t D, adaln_dtype dtype,
                              cudaStream_t stream);

size_t adaln_gate_residual_bwd_ragged_workspace_size(const int64_t *offsets_host,
                                                     int64_t num_segments, int64_t D,
                                                     adaln_dtype dtype);
adaln_status adaln_gate_residual_bwd_ragged(const void *dout, const void *z, const void *gate,
                                            void *dz, float *d_gate, void *workspace,
                                            size_t workspace_bytes,
                                            const int64_t *offsets_host,
                                            const int64_t *offsets_dev, int64_t num_segments,
                                            int64_t D, adaln_dtype dtype, cudaStream_t stream);

/* ---------------------------------------------------------------- ragged, indexed modulation
 * As the ragged calls, but segment k uses modulation row mod_index[k] of
 * [num_mod_rows, D] tables, so several segments may share one row (samples
 * that share a conditioning vector, or segments of one sample cut at bucket
 * boundaries) and rows no segment uses are allowed.
 *   mod_index_host, mod_index_dev: int32 [num_segments], the same values on
 *     the host (validated: every entry in [0, num_mod_rows), else
 *     ADALN_ERR_INVALID_ARG) and on the device (read by the kernels; 4-byte
 *     aligned).  Both may be NULL when num_segments == 0.
 *   shift, scale, gate [num_mod_rows, D] dtype.
 *   d_scale, d_shift, d_gate [num_mod_rows, D] float outputs: row m is the sum
 *     over every segment k with mod_index[k] == m (in ascending k, each segment's
 *     row chunks in order: a fixed order, so results are reproducible), and zero
 *     for a row no segment uses.
 *   workspace: adaln_bwd_ragged_workspace_size() /
 *     adaln_gate_residual_bwd_ragged_workspace_size() bytes for the same
 *     offsets (the workspace does not depend on the index). */
adaln_status adaln_fwd_ragged_indexed(const void *x, const void *shift, const void *scale,
                                      void *y, float *mean, float *rstd,
                                      const int64_t *offsets_host, const int64_t *offsets_dev,
                                      const int32_t *mod_index_host, const int32_t *mod_index_dev,
                                      int64_t num_segments, int64_t num_mod_rows, int64_t D,
                                      float eps, adaln_dtype dtype, cudaStream_t stream);

adaln_status adaln_gate_residual_ragged_indexed(const void *r, const void *z, const void *gate,
                                                void *out, const int64_t *offsets_host,
                                                const int64_t *offsets_dev,
                                                const int32_t *mod_index_host,
                                                const int32_t *mod_index_dev,
                                                int64_t num_segments, int64_t num_mod_rows,
                                                int64_t D, adaln_dtype dtype,
                                                cudaStream_t stream);

adaln_status adaln_bwd_ragged_indexed(const void *x, const float *mean, const float *rstd,
                                      const void *scale, const void *dy, void *dx, float *d_scale,
                                      float *d_shift, void *workspace, size_t workspace_bytes,
                                      const int64_t *offsets_host, const int64_t *offsets_dev,
                                      const int32_t *mod_index_host, const int32_t *mod_index_dev,
                                      int64_t num_segments, int64_t num_mod_rows, int64_t D,
                                      adaln_dtype dtype, cudaStream_t stream);

adaln_status adaln_gate_residual_bwd_ragged_indexed(
    const void *dout, const void *z, const void *gate, void *dz, float *d_gate, void *workspace,
    size_t workspace_bytes, const int64_t *offsets_host, const int64_t *offsets_dev,
    const int32_t *mod_index_host, const int32_t *mod_index_dev, int64_t num_segments,
    int64_t num_mod_rows, int64_t D, adaln_dtype dtype, cudaStream_t stream);

/* ---------------------------------------------------------------- fused gated chain
 * The block chain in one node per direction (summary section 2.B,
 * "Simplificacion de Grafos": the operator chain collapses to a single node):
 * the gated residual is applied to the modulated output itself (z := y), so y
 * never round-trips through HBM between the two steps:
 *     y   = LN(x) * (1 + scale[k]) + shift[k]
 *     out = r + gate[k] * y        (y kept in fp32, not rounded to dtype first)
 *
 * adaln_fwd_gated:
 *   x, r             [rows, D] dtype inputs
 *   shift, scale, gate [segments, D] dtype modulation rows
 *   out              [rows, D] dtype output
 *   y                [rows, D] dtype optional output (NULL: not written)
 *   mean, rstd       [rows] float outputs, as adaln_fwd
 *   out and y must not alias x, r or each other.
 *
 * adaln_bwd_gated: gradients of out given dout = dL/dout, with y reaching L
 * only through out (a further gradient into y adds linearly: apply adaln_bwd
 * to it and sum):
 *   dx, d_scale, d_shift  as adaln_bwd with dy = gate[k] * dout
 *   d_gate[k, d]          = sum_n dout * y   (y recomputed from x, mean, rstd)
 *   dr = dout is the identity and is not written.
 *   x, dout [rows, D] dtype; mean, rstd [rows] float from adaln_fwd_gated;
 *   shift, scale, gate [segments, D] dtype; dx [rows, D] dtype output (no
 *   aliasing); d_scale, d_shift, d_gate [segments, D] float outputs;
 *   workspace of adaln_bwd_gated_workspace_size() bytes, as for adaln_bwd.
 * Dense ([B, N, D], segments = B) and ragged (offsets, as above) variants.
 */
adaln_status adaln_fwd_gated(const void *x, const void *shift, const void *scale,
                             const void *gate, const void *r, void *out, void *y, float *mean,
                             float *rstd, int64_t B, int64_t N, int64_t D, float eps,
                             adaln_dtype dtype, cudaStream_t stream);
adaln_status adaln_fwd_gated_ragged(const void *x, const void *shift, const void *scale,
                                    const void *gate, const void *r, void *out, void *y,
                                    float *mean, float *rstd, const int64_t *offsets_host,
                                    const int64_t *offsets_dev, int64_t num_segments, int64_t D,
                                    float eps, adaln_dtype dtype, cudaStream_t stream);
size_t adaln_bwd_gated_workspace_size(int64_t B, int64_t N, int64_t D, adaln_dtype dtype);
adaln_status adaln_bwd_gated(const void *x, const float *mean, const float *rstd,
                             const void *shift, const void *scale, const void *gate,
                             const void *dout, void *dx, float *d_scale, float *d_shift,
                             float *d_gate, void *workspace, size_t workspace_bytes, int64_t B,
                             int64_t N, int64_t D, adaln_dtype dtype, cudaStream_t stream);
size_t adaln_bwd_gated_ragged_workspace_size(const int64_t *offsets_host, int64_t num_segments,
                                             int64_t D, adaln_dtype dtype);
adaln_status adaln_bwd_gated_ragged(const void *x, const float *mean, const float *rstd,
                                    const void *shift, const void *scale, const void *gate,
                                    const void *dout, void *dx, float *d_scale, float *d_shift,
                                    float *d_gate, void *workspace, size_t workspace_bytes,
                                    const int64_t *offsets_host, const int64_t *offsets_dev,
                                    int64_t num_segments, int64_t D, adaln_dtype dtype,
                                    cudaStream_t stream);

/* ---------------------------------------------------------------- RMSNorm modulation
 * The same modulation on RMS-normalised rows (the norm the Wan TPU training
 * pull request recomputes; no mean subtraction):
 *     rstd = 1 / sqrt(mean_d x^2 + eps),   xhat = x * rstd,
 *     y    = xhat * (1 + scale[k]) + shift[k].
 * adaln_fwd_rms: as adaln_fwd without the mean output; rstd [rows] float is
 *   rounded once from the exact value (same contract as adaln_fwd).
 * adaln_bwd_rms: given dy, with g = dy * (1 + scale[k]):
 *     dx = rstd * (g - xhat * mean_d(g * xhat)),
 *     d_scale[k, d] = sum_n dy * xhat,   d_shift[k, d] = sum_n dy;
 *   workspace as for adaln_bwd (adaln_bwd_workspace_size /
 *   adaln_bwd_ragged_workspace_size give its size). */
adaln_status adaln_fwd_rms(const void *x, const void *shift, const void *scale, void *y,
                           float *rstd, int64_t B, int64_t N, int64_t D, float eps,
                           adaln_dtype dtype, cudaStream_t stream);
adaln_status adaln_fwd_rms_ragged(const void *x, const void *shift, const void *scale, void *y,
                                  float *rstd, const int64_t *offsets_host,
                                  const int64_t *offsets_dev, int64_t num_segments, int64_t D,
                                  float eps, adaln_dtype dtype, cudaStream_t stream);
adaln_status adaln_bwd_rms(const void *x, const float *rstd, const void *scale, const void *dy,
                           void *dx, float *d_scale, float *d_shift, void *workspace,
                           size_t workspace_bytes, int64_t B, int64_t N, int64_t D,
                           adaln_dtype dtype, cudaStream_t stream);
adaln_status adaln_bwd_rms_ragged(const void *x, const float *rstd, const void *scale,
                                  const void *dy, void *dx, float *d_scale, float *d_shift,
                                  void *workspace, size_t workspace_bytes,
                                  const int64_t *offsets_host, const int64_t *offsets_dev,
                                  int64_t num_segments, int64_t D, adaln_dtype dtype,
                                  cudaStream_t stream);

/* ---------------------------------------------------------------- no-allocation backward
 * The paper has no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory: a plugin inside a host framework that owns
 * all device memory and exposes no allocator, or a latency-critical path that
 * must not call cudaMalloc (which can synchronise the device).
 *
 * adaln_bwd_noalloc computes exactly what adaln_bwd computes (same arguments
 * minus the workspace) but runs on a fixed scratch buffer that the library
 * keeps in device memory: adaln_noalloc_scratch_bytes() bytes (16 MiB), held
 * on every GPU that loads the library until the process exits.  It allocates
 * nothing and calls no allocating routine.
 *   - Shapes whose adaln_bwd_workspace_size() exceeds the scratch size return
 *     ADALN_ERR_WORKSPACE_TOO_SMALL before anything is launched (dense shapes
 *     up to D = 6144 fit when the rows give at most about 2 chunks per SM;
 *     many short samples can exceed it).
 *   - The first call on a device looks up the scratch address on that device
 *     (cudaGetSymbolAddress) and remembers it with the identity of the
 *     device's current context; a call made in another context of the device
 *     (after cudaDeviceReset, for example) looks it up again.  Make such a
 *     set-up call before any stream capture.
 *   - Every call shares the one buffer, which keeps the previous call's
 *     contents (the status word is cleared and every partial is rewritten on
 *     each call).  Calls whose work overlaps on the GPU (other streams, other
 *     host threads) race on it: serialise them.
 *   - A timed-out wait inside its kernels (a bug, as for adaln_bwd) is reported
 *     by adaln_pipeline_status(), which reads the scratch's status word; the
 *     parameter gradients are then NaN.  Calls with B = 0 launch nothing and
 *     leave that word as the previous call wrote it.
 */
size_t adaln_noalloc_scratch_bytes(void);
adaln_status adaln_bwd_noalloc(const void *x, const float *mean, const float *rstd,
                               const void *scale, const void *dy, void *dx, float *d_scale,
                               float *d_shift, int64_t B, int64_t N, int64_t D,
                               adaln_dtype dtype, cudaStream_t stream);

/* ---------------------------------------------------------------- planner
 * Dual-constraint bucket planner of the summary, section 2.A (host only,
 * integer arithmetic, no CUDA):
 *   adaln_bucket_batch: B_shape = max(1, min(floor(M_mem/S), floor(M_comp/S^p)))
 *   for S >= 1, M_mem >= 1, M_comp >= 1, p >= 1 (returns -1 on bad input;
 *   S^p is evaluated without overflow).
 *   adaln_plan_buckets: sorts the n lengths by (length, index) and walks them
 *   ascending, adding each sequence to the open bucket while the bucket's
 *   size plus one stays within B_shape of that sequence's length, otherwise
 *   opening a new bucket.  Outputs (caller-allocated host arrays):
 *     order[n]          sequence indices in packing order;
 *     bucket_start[n+1] bucket b = order[bucket_start[b] .. bucket_start[b+1]);
 *     bucket_of_seq[n]  bucket of each sequence;
 *     *num_buckets      number of buckets.
 *   Lengths must be >= 1.
 */
int64_t adaln_bucket_batch(int64_t S, int64_t M_mem, int64_t M_comp, int32_t p);
adaln_status adaln_plan_buckets(const int64_t *lengths, int64_t n, int64_t M_mem,
                                int64_t M_comp, int32_t p, int64_t *bucket_of_seq,
                                int64_t *order, int64_t *bucket_start,
                                int64_t *num_buckets);

/* Load balance of a bucket plan over data-parallel ranks (summary section 4,
 * "Eficiencia del Equilibrio de Carga", which reports the coefficient of
 * variation of the per-rank compute load; host only).  The plan is
 * adaln_plan_buckets' (order, bucket_start, num_buckets); an equal-tokens plan
 * is the same call with M_comp so large that only B*S <= M_mem binds.
 * Buckets are dealt in the order deal[0..num_buckets) (a permutation, e.g. a
 * seeded shuffle), one bucket per rank per step, for floor(num_buckets/ranks)
 * full steps.  A bucket's compute load is the sum over its sequences of S^p.
 * Outputs: *mean_cv = mean over the steps of (population std / mean) of the
 * ranks' loads; *mean_max_over_mean = mean over the steps of max / mean;
 * *steps = the number of full steps (both means are 0 when it is 0).
 * Returns ADALN_ERR_INVALID_ARG for a plan that is not a partition of the
 * sequences, a deal that is not a permutation, ranks < 1 or p < 1. */
adaln_status adaln_balance_cv(const int64_t *lengths, int64_t n, const int64_t *order,
                              const int64_t *bucket_start, int64_t num_buckets,
                              const int64_t *deal, int64_t ranks, int32_t p, double *mean_cv,
                              double *mean_max_over_mean, int64_t *steps);

/* Least-squares fit of the step-time model t = a + b * B * S^p over n >= 3
 * measured (B[i], S[i], t[i]) shapes (summary section 2.A: the cost-fitting
 * system that calibrates p and M_comp from shape benchmarks; host only).  For
 * each p the model is linear in (a, b) and solved in closed form; p minimises
 * the residual sum of squares over [p_lo, p_hi]: the best point of a 65-point
 * grid, refined by golden-section search between its grid neighbours (the
 * residual need not be unimodal in p).
 * Outputs a, b, p and (if rss is not NULL) the residual sum of squares.
 * ADALN_ERR_INVALID_ARG for n < 3, B or S < 1, a non-finite t, or a bad range. */
adaln_status adaln_fit_cost(const int64_t *B, const int64_t *S, const double *t, int64_t n,
                            double p_lo, double p_hi, double *a, double *b, double *p,
                            double *rss);

#ifdef __cplusplus
}
#endif

#endif /* ADALN_H */
