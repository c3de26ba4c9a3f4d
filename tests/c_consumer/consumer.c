/* A plain C program that uses the library only through include/adaln.h: the
 * boundary is a C ABI, callable without Python or C++.  Runs on a machine
 * without a GPU: it exercises the host-only entry points (status strings,
 * limits, the bucket planner) and argument validation, which rejects bad
 * calls before anything touches CUDA.  Prints one line per check and exits
 * non-zero on the first failure. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "adaln.h"

static int failures = 0;

static void check(int ok, const char *what) {
    printf("%s %s\n", ok ? "ok  " : "FAIL", what);
    if (!ok) ++failures;
}

int main(void) {
    /* status strings and limits */
    check(strncmp(adaln_status_string(ADALN_OK), "ADALN_OK", 8) == 0, "status string of ADALN_OK");
    check(strstr(adaln_status_string((adaln_status)77), "unknown") != NULL,
          "status string of an unknown code");
    check(adaln_max_dim(ADALN_BF16) == 16384 && adaln_max_dim(ADALN_F32) == 16384,
          "largest D is 16384 for both dtypes");

    /* the dual-constraint batch size: B = max(1, min(M_mem / S, M_comp / S^2)) */
    check(adaln_bucket_batch(256, 262144, 1 << 30, 2) == 1024, "B_shape(256) = 1024");
    check(adaln_bucket_batch(4096, 262144, 1 << 30, 2) == 64, "B_shape(4096) = 64");
    check(adaln_bucket_batch(32768, 262144, 1 << 30, 2) == 1, "B_shape(32768) = 1");

    /* bucket planning of six sequences: sorted by length, greedy under B_shape */
    {
        const int64_t lengths[6] = {4096, 256, 32768, 4096, 300, 20000};
        int64_t bucket_of[6], order[6], start[7], nb = -1;
        adaln_status st = adaln_plan_buckets(lengths, 6, 262144, 1 << 30, 2, bucket_of, order,
                                             start, &nb);
        check(st == ADALN_OK, "plan_buckets returns ADALN_OK");
        /* ascending length: 256, 300, 4096, 4096, 20000, 32768 */
        check(order[0] == 1 && order[1] == 4 && order[2] == 0 && order[3] == 3 &&
                  order[4] == 5 && order[5] == 2,
              "sequences sorted by (length, index)");
        /* B_shape(4096) = 64 admits the four shortest in one bucket; at S = 20000,
           B_shape = 2 < 5 sequences, so a new bucket opens; B_shape(32768) = 1
           opens a third */
        check(nb == 3 && start[0] == 0 && start[1] == 4 && start[2] == 5 && start[3] == 6,
              "three buckets: [4 shortest], [20000], [32768]");
        check(bucket_of[1] == 0 && bucket_of[5] == 1 && bucket_of[2] == 2,
              "bucket of each sequence");
    }

    /* validation before any launch: misaligned pointers, bad D, aliasing */
    {
        char *base = (char *)(uintptr_t)(1 << 20); /* never dereferenced */
        check(adaln_fwd(base, base + 64, base + 128, base + 256, (float *)(base + 512),
                        (float *)(base + 1024), 2, 4, 12, 1e-6f, ADALN_BF16, 0) ==
                  ADALN_ERR_INVALID_ARG,
              "bf16 D not a multiple of 8 is rejected");
        check(adaln_fwd(base, base + 64, base + 128, base + 256, (float *)(base + 512),
                        (float *)(base + 1024), 2, 4, 16392, 1e-6f, ADALN_BF16, 0) ==
                  ADALN_ERR_UNSUPPORTED,
              "D above the limit is unsupported");
        check(adaln_fwd(base, base + 64, base + 128, base, (float *)(base + 512),
                        (float *)(base + 1024), 2, 4, 64, 1e-6f, ADALN_BF16, 0) ==
                  ADALN_ERR_INVALID_ARG,
              "y aliasing x is rejected");
        check(adaln_fwd(base + 4, base + 64, base + 128, base + 256, (float *)(base + 512),
                        (float *)(base + 1024), 2, 4, 64, 1e-6f, ADALN_BF16, 0) ==
                  ADALN_ERR_INVALID_ARG,
              "misaligned x is rejected");
    }
    printf("%d failure(s)\n", failures);
    return failures == 0 ? 0 : 1;
}
