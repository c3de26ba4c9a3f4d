/*
 * fastcmp.c -- test-side helpers for comparing full-size GPU results with the
 * fp64 oracle without numpy temporaries (one pass over each array).
 *
 * Test infrastructure only: none of the operator's arithmetic is here, only
 * exact widening of bf16/fp32 values to double and the largest absolute
 * difference between two arrays.  A block whose largest difference is within
 * the tolerance passes; any other block is re-checked element by element by
 * the Python check, which owns the tolerance rules.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* bf16 bit patterns -> double (exact: a bf16 is the top half of an fp32) */
void cmp_widen_bf16(const uint16_t *src, double *dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        const uint32_t u = (uint32_t)src[i] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        dst[i] = (double)f;
    }
}

void cmp_widen_f32(const float *src, double *dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = (double)src[i];
}

/* max |g - ref| with g given as bf16 bit patterns; +inf if any NaN is met */
double cmp_maxabs_bf16(const uint16_t *g, const double *ref, int64_t n) {
    double m = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const uint32_t u = (uint32_t)g[i] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        const double d = fabs((double)f - ref[i]);
        if (!(d <= m)) m = isnan(d) ? INFINITY : d;
    }
    return m;
}

double cmp_maxabs_f32(const float *g, const double *ref, int64_t n) {
    double m = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double d = fabs((double)g[i] - ref[i]);
        if (!(d <= m)) m = isnan(d) ? INFINITY : d;
    }
    return m;
}
