// planner.cpp -- dual-constraint bucket planner (host only, integer arithmetic).
//
// "AdaptiveLoad" technical summary (gist.science paper 2605.17923), section
// 2.A: a group of sequences of length S gets the batch size allowed by both the
// linear memory constraint B*S <= M_mem and the polynomial compute constraint
// B*S^p <= M_comp,
//     B_shape(S) = max(1, min(floor(M_mem / S), floor(M_comp / S^p))).
// The summary does not say how sequences are grouped; the grouping here sorts
// by (S, index) and walks ascending, adding a sequence to the open bucket while
// the bucket's size plus one stays within B_shape of its length.
#include "adaln.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <numeric>
#include <vector>

namespace {

// floor(M / S^p) without overflow: stop multiplying once S^p exceeds M.
int64_t floor_div_pow(int64_t M, int64_t S, int32_t p) {
    int64_t q = M;
    for (int32_t i = 0; i < p; ++i) {
        q /= S;  // floor(floor(M / S^i) / S) == floor(M / S^(i+1))
        if (q == 0) break;
    }
    return q;
}

}  // namespace

extern "C" int64_t adaln_bucket_batch(int64_t S, int64_t M_mem, int64_t M_comp, int32_t p) {
    if (S < 1 || M_mem < 1 || M_comp < 1 || p < 1) return -1;
    const int64_t mem = M_mem / S;
    const int64_t comp = floor_div_pow(M_comp, S, p);
    return std::max<int64_t>(1, std::min(mem, comp));
}

extern "C" adaln_status adaln_plan_buckets(const int64_t *lengths, int64_t n, int64_t M_mem,
                                           int64_t M_comp, int32_t p, int64_t *bucket_of_seq,
                                           int64_t *order, int64_t *bucket_start,
                                           int64_t *num_buckets) {
    if (n < 0 || M_mem < 1 || M_comp < 1 || p < 1 || num_buckets == nullptr)
        return ADALN_ERR_INVALID_ARG;
    if (n > 0 && (lengths == nullptr || bucket_of_seq == nullptr || order == nullptr))
        return ADALN_ERR_INVALID_ARG;
    if (bucket_start == nullptr) return ADALN_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (lengths[i] < 1) return ADALN_ERR_INVALID_ARG;

    std::vector<int64_t> idx((size_t)n);
    std::iota(idx.begin(), idx.end(), int64_t{0});
    std::sort(idx.begin(), idx.end(), [lengths](int64_t a, int64_t b) {
        return lengths[a] != lengths[b] ? lengths[a] < lengths[b] : a < b;
    });

    int64_t nb = 0, count = 0;
    for (int64_t pos = 0; pos < n; ++pos) {
        const int64_t i = idx[(size_t)pos];
        const int64_t cap = adaln_bucket_batch(lengths[i], M_mem, M_comp, p);
        if (count == 0 || count + 1 > cap) {
            bucket_start[nb++] = pos;
            count = 1;
        } else {
            ++count;
        }
        order[pos] = i;
        bucket_of_seq[i] = nb - 1;
    }
    bucket_start[nb] = n;
    *num_buckets = nb;
    return ADALN_OK;
}

// Load balance of a bucket plan over data-parallel ranks (summary section 4,
// "Eficiencia del Equilibrio de Carga": the coefficient of variation of the
// per-rank compute load).  Buckets are dealt in the caller's order `deal`, one
// per rank per step; a bucket's compute load is the sum over its sequences of
// S^p (the polynomial cost of section 2.A).  Per full step: CV = population
// standard deviation / mean of the ranks' loads, and max / mean; both are
// averaged over the steps.  Loads are exact in double for S^p * n < 2^53.
extern "C" adaln_status adaln_balance_cv(const int64_t *lengths, int64_t n, const int64_t *order,
                                         const int64_t *bucket_start, int64_t num_buckets,
                                         const int64_t *deal, int64_t ranks, int32_t p,
                                         double *mean_cv, double *mean_max_over_mean,
                                         int64_t *steps) {
    if (n < 0 || num_buckets < 0 || ranks < 1 || p < 1 || bucket_start == nullptr ||
        mean_cv == nullptr || mean_max_over_mean == nullptr || steps == nullptr)
        return ADALN_ERR_INVALID_ARG;
    if (n > 0 && (lengths == nullptr || order == nullptr)) return ADALN_ERR_INVALID_ARG;
    if (num_buckets > 0 && deal == nullptr) return ADALN_ERR_INVALID_ARG;
    if (bucket_start[0] != 0 || bucket_start[num_buckets] != n) return ADALN_ERR_INVALID_ARG;
    for (int64_t b = 0; b < num_buckets; ++b)
        if (bucket_start[b + 1] < bucket_start[b]) return ADALN_ERR_INVALID_ARG;
    std::vector<char> seen((size_t)num_buckets, 0);
    for (int64_t b = 0; b < num_buckets; ++b) {
        const int64_t d = deal[b];
        if (d < 0 || d >= num_buckets || seen[(size_t)d]) return ADALN_ERR_INVALID_ARG;
        seen[(size_t)d] = 1;
    }
    std::vector<double> load((size_t)num_buckets, 0.0);
    for (int64_t b = 0; b < num_buckets; ++b) {
        double sum = 0.0;
        for (int64_t pos = bucket_start[b]; pos < bucket_start[b + 1]; ++pos) {
            const int64_t i = order[pos];
            if (i < 0 || i >= n || lengths[i] < 1) return ADALN_ERR_INVALID_ARG;
            double c = 1.0;
            for (int32_t e = 0; e < p; ++e) c *= (double)lengths[i];
            sum += c;
        }
        load[(size_t)b] = sum;
    }
    const int64_t T = num_buckets / ranks;
    double cv_sum = 0.0, mm_sum = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        double tot = 0.0, mx = 0.0;
        for (int64_t r = 0; r < ranks; ++r) {
            const double l = load[(size_t)deal[t * ranks + r]];
            tot += l;
            mx = std::max(mx, l);
        }
        const double mean = tot / (double)ranks;
        double var = 0.0;
        for (int64_t r = 0; r < ranks; ++r) {
            const double dl = load[(size_t)deal[t * ranks + r]] - mean;
            var += dl * dl;
        }
        var /= (double)ranks;
        cv_sum += mean > 0.0 ? std::sqrt(var) / mean : 0.0;
        mm_sum += mean > 0.0 ? mx / mean : 0.0;
    }
    *steps = T;
    *mean_cv = T > 0 ? cv_sum / (double)T : 0.0;
    *mean_max_over_mean = T > 0 ? mm_sum / (double)T : 0.0;
    return ADALN_OK;
}

// ------------------------------------------------------------------ cost model
// Fit of the step-time model t = a + b * B * S^p (summary section 2.A, the
// cost-fitting system that sets p and M_comp from shape benchmarks) by least
// squares.  For a fixed p the model is linear in (a, b), so the residual sum of
// squares RSS(p) of that linear fit is minimised over p in [p_lo, p_hi]: the
// best of a 65-point grid, refined by golden-section search between its
// neighbours (a variable-projection fit).

namespace {

// closed-form least squares of t = a + b * u; returns the residual sum of squares
double fit_linear(const double *u, const double *t, int64_t n, double &a, double &b) {
    double su = 0.0, st = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        su += u[i];
        st += t[i];
    }
    const double mu = su / (double)n, mt = st / (double)n;
    double suu = 0.0, sut = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        suu += (u[i] - mu) * (u[i] - mu);
        sut += (u[i] - mu) * (t[i] - mt);
    }
    b = suu > 0.0 ? sut / suu : 0.0;
    a = mt - b * mu;
    double rss = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double e = t[i] - a - b * u[i];
        rss += e * e;
    }
    return rss;
}

double profile_rss(const int64_t *B, const int64_t *S, const double *t, int64_t n, double p,
                   std::vector<double> &u, double &a, double &b) {
    for (int64_t i = 0; i < n; ++i) u[(size_t)i] = (double)B[i] * std::pow((double)S[i], p);
    return fit_linear(u.data(), t, n, a, b);
}

}  // namespace

extern "C" adaln_status adaln_fit_cost(const int64_t *B, const int64_t *S, const double *t,
                                       int64_t n, double p_lo, double p_hi, double *a,
                                       double *b, double *p, double *rss) {
    if (n < 3 || B == nullptr || S == nullptr || t == nullptr || a == nullptr || b == nullptr ||
        p == nullptr || !(p_lo > 0.0) || !(p_hi > p_lo) || !std::isfinite(p_hi))
        return ADALN_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (B[i] < 1 || S[i] < 1 || !std::isfinite(t[i])) return ADALN_ERR_INVALID_ARG;
    std::vector<double> u((size_t)n);
    const double g = 0.5 * (std::sqrt(5.0) - 1.0);  // 1 / golden ratio
    double aa, bb;
    // RSS(p) need not be unimodal (at large p a few shapes dominate and the fit
    // flattens to a constant): scan a grid, then refine around its best point
    constexpr int kGrid = 64;
    int best = 0;
    double fbest = 0.0;
    for (int j = 0; j <= kGrid; ++j) {
        const double pj = p_lo + (p_hi - p_lo) * j / kGrid;
        const double f = profile_rss(B, S, t, n, pj, u, aa, bb);
        if (j == 0 || f < fbest) {
            fbest = f;
            best = j;
        }
    }
    double lo = p_lo + (p_hi - p_lo) * std::max(0, best - 1) / kGrid;
    double hi = p_lo + (p_hi - p_lo) * std::min(kGrid, best + 1) / kGrid;
    double x1 = hi - g * (hi - lo), x2 = lo + g * (hi - lo);
    double f1 = profile_rss(B, S, t, n, x1, u, aa, bb);
    double f2 = profile_rss(B, S, t, n, x2, u, aa, bb);
    for (int it = 0; it < 200 && hi - lo > 1e-12 * (1.0 + std::fabs(lo)); ++it) {
        if (f1 <= f2) {
            hi = x2;
            x2 = x1;
            f2 = f1;
            x1 = hi - g * (hi - lo);
            f1 = profile_rss(B, S, t, n, x1, u, aa, bb);
        } else {
            lo = x1;
            x1 = x2;
            f1 = f2;
            x2 = lo + g * (hi - lo);
            f2 = profile_rss(B, S, t, n, x2, u, aa, bb);
        }
    }
    const double pp = 0.5 * (lo + hi);
    const double r = profile_rss(B, S, t, n, pp, u, aa, bb);
    *a = aa;
    *b = bb;
    *p = pp;
    if (rss) *rss = r;
    return ADALN_OK;
}
