/*
 * adaln_oracle.c -- fp64 CPU oracle for the AdaLN modulation operator.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the operator computes.  It exists so that tests, the
 * smoke check and the CPU-baseline leg of the benchmark can check the CUDA
 * library against it.  The product path never links, loads or calls it, and it
 * shares no code, header or constant with the CUDA library.
 *
 * What it follows ("AdaptiveLoad" technical summary, gist.science paper
 * 2605.17923):
 *   - section 1, second bullet: AdaLN normalisation + modulation in a DiT/MMDiT
 *     block, and the backward reduction of the modulation-parameter gradients
 *     along the sequence dimension N;
 *   - section 2.B, "Paso Adelante": mean and variance of each row over the
 *     feature dimension D, then the linear modulation over D;
 *   - section 2.B, "Paso Atras": per-feature (column) sums over N.
 * The summary prints no formula for AdaLN itself; the operator used here is
 * the standard DiT adaptive LayerNorm (LayerNorm without affine, biased
 * variance, eps inside the square root):
 *     y   = xhat * (1 + scale[k]) + shift[k],  xhat = (x - mu) * rstd,
 *     rstd = 1 / sqrt(var + eps),  var = mean_d (x - mu)^2,
 * with the gated residual out = r + gate[k] * z, where k is the segment
 * (sample or packed sequence) a row belongs to.
 *
 * Layout: every [rows, D] array is row-major; the rows of segment k are
 * [offsets[k], offsets[k+1]); shift/scale/gate and the parameter gradients
 * are [nseg, D] with row k belonging to segment k.
 *
 * Arithmetic: IEEE double throughout, sums in ascending index order, no
 * blocking, no reordering, no fusion beyond what the formulas state.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Row statistics: two-pass mean then biased variance (Paso Adelante). */
static void row_stats(const double *x, int64_t D, double eps, double *mu_out,
                      double *rstd_out) {
    double s = 0.0;
    for (int64_t d = 0; d < D; ++d) s += x[d];
    const double mu = s / (double)D;
    double v = 0.0;
    for (int64_t d = 0; d < D; ++d) {
        const double t = x[d] - mu;
        v += t * t;
    }
    v = v / (double)D;
    *mu_out = mu;
    *rstd_out = 1.0 / sqrt(v + eps);
}

/* Forward: y = LN(x) * (1 + scale[k]) + shift[k]; mean and rstd per row. */
void oracle_adaln_fwd(const double *x, const double *shift, const double *scale,
                      const int64_t *offsets, int64_t nseg, int64_t D, double eps,
                      double *y, double *mean, double *rstd) {
    for (int64_t k = 0; k < nseg; ++k) {
        const double *sh = shift + k * D;
        const double *sc = scale + k * D;
        for (int64_t row = offsets[k]; row < offsets[k + 1]; ++row) {
            const double *xr = x + row * D;
            double *yr = y + row * D;
            double mu, rs;
            row_stats(xr, D, eps, &mu, &rs);
            mean[row] = mu;
            rstd[row] = rs;
            for (int64_t d = 0; d < D; ++d) {
                const double xhat = (xr[d] - mu) * rs;
                yr[d] = xhat * (1.0 + sc[d]) + sh[d];
            }
        }
    }
}

/* Gated residual: out = r + gate[k] * z. */
void oracle_gate_residual(const double *r, const double *z, const double *gate,
                          const int64_t *offsets, int64_t nseg, int64_t D,
                          double *out) {
    for (int64_t k = 0; k < nseg; ++k) {
        const double *g = gate + k * D;
        for (int64_t row = offsets[k]; row < offsets[k + 1]; ++row)
            for (int64_t d = 0; d < D; ++d)
                out[row * D + d] = r[row * D + d] + g[d] * z[row * D + d];
    }
}

/*
 * Backward of y = LN(x) * (1 + scale) + shift, given dy = dL/dy.
 *   g         = dy * (1 + scale[k])                      (dL/dxhat)
 *   dx        = rstd * (g - mean_d(g) - xhat * mean_d(g * xhat))
 *   d_scale[k,d] = sum over the rows n of segment k of dy * xhat
 *   d_shift[k,d] = sum over the rows n of segment k of dy
 * The statistics are recomputed here from x (the definition), not taken from
 * any forward output.  Column sums run over rows in ascending order.
 */
void oracle_adaln_bwd(const double *x, const double *scale, const double *dy,
                      const int64_t *offsets, int64_t nseg, int64_t D, double eps,
                      double *dx, double *d_scale, double *d_shift) {
    memset(d_scale, 0, sizeof(double) * (size_t)(nseg * D));
    memset(d_shift, 0, sizeof(double) * (size_t)(nseg * D));
    for (int64_t k = 0; k < nseg; ++k) {
        const double *sc = scale + k * D;
        double *ds = d_scale + k * D;
        double *db = d_shift + k * D;
        for (int64_t row = offsets[k]; row < offsets[k + 1]; ++row) {
            const double *xr = x + row * D;
            const double *dyr = dy + row * D;
            double *dxr = dx + row * D;
            double mu, rs;
            row_stats(xr, D, eps, &mu, &rs);
            double sum_g = 0.0, sum_gx = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                const double xhat = (xr[d] - mu) * rs;
                const double g = dyr[d] * (1.0 + sc[d]);
                sum_g += g;
                sum_gx += g * xhat;
            }
            const double mean_g = sum_g / (double)D;
            const double mean_gx = sum_gx / (double)D;
            for (int64_t d = 0; d < D; ++d) {
                const double xhat = (xr[d] - mu) * rs;
                const double g = dyr[d] * (1.0 + sc[d]);
                dxr[d] = rs * (g - mean_g - xhat * mean_gx);
                ds[d] += dyr[d] * xhat;
                db[d] += dyr[d];
            }
        }
    }
}

/*
 * Backward of out = r + gate * z, given dout = dL/dout:
 *   dz = gate[k] * dout,   d_gate[k,d] = sum over rows of segment k of dout * z
 *   (dr = dout is the identity and is not materialised).
 */
void oracle_gate_residual_bwd(const double *dout, const double *z,
                              const double *gate, const int64_t *offsets,
                              int64_t nseg, int64_t D, double *dz,
                              double *d_gate) {
    memset(d_gate, 0, sizeof(double) * (size_t)(nseg * D));
    for (int64_t k = 0; k < nseg; ++k) {
        const double *g = gate + k * D;
        double *dg = d_gate + k * D;
        for (int64_t row = offsets[k]; row < offsets[k + 1]; ++row)
            for (int64_t d = 0; d < D; ++d) {
                dz[row * D + d] = g[d] * dout[row * D + d];
                dg[d] += dout[row * D + d] * z[row * D + d];
            }
    }
}

/*
 * Fused gated chain (section 2.B, "Simplificacion de Grafos": the chain as one
 * node): the gated residual applied to the modulated output itself,
 *     y = LN(x) * (1 + scale[k]) + shift[k],   out = r + gate[k] * y.
 * Written as that composition of the two definitions above.
 */
void oracle_adaln_fwd_gated(const double *x, const double *shift, const double *scale,
                            const double *gate, const double *r, const int64_t *offsets,
                            int64_t nseg, int64_t D, double eps, double *out, double *y,
                            double *mean, double *rstd) {
    oracle_adaln_fwd(x, shift, scale, offsets, nseg, D, eps, y, mean, rstd);
    oracle_gate_residual(r, y, gate, offsets, nseg, D, out);
}

/*
 * Backward of the fused chain given dout = dL/dout, y reaching L only through
 * out (chain rule):
 *   dL/dy  = gate[k] * dout                  (the gate backward's dz)
 *   dx, d_scale, d_shift = the LayerNorm-modulation backward of that dL/dy
 *   d_gate[k,d] = sum over the rows of segment k of dout * y
 *   (dr = dout is the identity and is not materialised).
 * Returns 0, or -1 if the temporaries cannot be allocated.
 */
int oracle_adaln_bwd_gated(const double *x, const double *shift, const double *scale,
                           const double *gate, const double *dout, const int64_t *offsets,
                           int64_t nseg, int64_t D, double eps, double *dx, double *d_scale,
                           double *d_shift, double *d_gate) {
    const int64_t rows = offsets[nseg];
    const size_t n = (size_t)(rows * D) + 1;
    double *y = malloc(sizeof(double) * n);
    double *dy = malloc(sizeof(double) * n);
    double *mean = malloc(sizeof(double) * ((size_t)rows + 1));
    double *rstd = malloc(sizeof(double) * ((size_t)rows + 1));
    if (!y || !dy || !mean || !rstd) {
        free(y);
        free(dy);
        free(mean);
        free(rstd);
        return -1;
    }
    oracle_adaln_fwd(x, shift, scale, offsets, nseg, D, eps, y, mean, rstd);
    oracle_gate_residual_bwd(dout, y, gate, offsets, nseg, D, dy, d_gate);
    oracle_adaln_bwd(x, scale, dy, offsets, nseg, D, eps, dx, d_scale, d_shift);
    free(y);
    free(dy);
    free(mean);
    free(rstd);
    return 0;
}

/*
 * RMSNorm modulation (the norm of the Wan TPU training page; no mean):
 *     rstd = 1 / sqrt(mean_d x^2 + eps),  xhat = x * rstd,
 *     y    = xhat * (1 + scale[k]) + shift[k].
 */
void oracle_rms_fwd(const double *x, const double *shift, const double *scale,
                    const int64_t *offsets, int64_t nseg, int64_t D, double eps, double *y,
                    double *rstd) {
    for (int64_t k = 0; k < nseg; ++k) {
        const double *sh = shift + k * D;
        const double *sc = scale + k * D;
        for (int64_t row = offsets[k]; row < offsets[k + 1]; ++row) {
            const double *xr = x + row * D;
            double q = 0.0;
            for (int64_t d = 0; d < D; ++d) q += xr[d] * xr[d];
            const double rs = 1.0 / sqrt(q / (double)D + eps);
            rstd[row] = rs;
            for (int64_t d = 0; d < D; ++d) y[row * D + d] = xr[d] * rs * (1.0 + sc[d]) + sh[d];
        }
    }
}

/*
 * Backward of the RMSNorm modulation given dy (statistics recomputed from x):
 *   g  = dy * (1 + scale[k]),  dx = rstd * (g - xhat * mean_d(g * xhat)),
 *   d_scale[k,d] = sum_n dy * xhat,  d_shift[k,d] = sum_n dy.
 */
void oracle_rms_bwd(const double *x, const double *scale, const double *dy,
                    const int64_t *offsets, int64_t nseg, int64_t D, double eps, double *dx,
                    double *d_scale, double *d_shift) {
    memset(d_scale, 0, sizeof(double) * (size_t)(nseg * D));
    memset(d_shift, 0, sizeof(double) * (size_t)(nseg * D));
    for (int64_t k = 0; k < nseg; ++k) {
        const double *sc = scale + k * D;
        for (int64_t row = offsets[k]; row < offsets[k + 1]; ++row) {
            const double *xr = x + row * D;
            const double *dyr = dy + row * D;
            double q = 0.0;
            for (int64_t d = 0; d < D; ++d) q += xr[d] * xr[d];
            const double rs = 1.0 / sqrt(q / (double)D + eps);
            double sum_gx = 0.0;
            for (int64_t d = 0; d < D; ++d) sum_gx += dyr[d] * (1.0 + sc[d]) * (xr[d] * rs);
            const double mean_gx = sum_gx / (double)D;
            for (int64_t d = 0; d < D; ++d) {
                const double xhat = xr[d] * rs;
                const double g = dyr[d] * (1.0 + sc[d]);
                dx[row * D + d] = rs * (g - xhat * mean_gx);
                d_scale[k * D + d] += dyr[d] * xhat;
                d_shift[k * D + d] += dyr[d];
            }
        }
    }
}
