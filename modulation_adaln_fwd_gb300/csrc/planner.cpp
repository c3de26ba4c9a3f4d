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
