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
