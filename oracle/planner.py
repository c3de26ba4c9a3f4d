"""Dual-constraint bucket planner, oracle side (exact Python integers).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the "AdaptiveLoad" technical summary (gist.science paper 2605.17923),
section 2.A: a group of sequences of length S gets the batch size that
satisfies both the linear memory constraint B*S <= M_mem and the polynomial
compute constraint B*S^p <= M_comp, floored, and at least one:

    B_shape(S) = max(1, min(floor(M_mem / S), floor(M_comp / S^p)))

The summary does not say how sequences are grouped.  Reading used here (and
stated in the design notes): sort sequences by (S, original index) ascending,
walk them in that order, and keep adding the next sequence to the open bucket
while the bucket's size plus one stays within B_shape of that sequence's
length (which, the walk being ascending, is the bucket's largest length);
otherwise close the bucket and open a new one with that sequence.
"""
from __future__ import annotations


def bucket_batch(S: int, M_mem: int, M_comp: int, p: int) -> int:
    """B_shape for one sequence length S (section 2.A of the summary)."""
    if S <= 0 or M_mem <= 0 or M_comp <= 0 or p <= 0:
        raise ValueError("S, M_mem, M_comp and p must be positive")
    return max(1, min(M_mem // S, M_comp // (S ** p)))


def plan_buckets(lengths, M_mem: int, M_comp: int, p: int):
    """Greedy ascending walk.

    Returns (bucket_of_seq, order, bucket_start):
      order        -- sequence indices in packing order (sorted by (S, index));
      bucket_start -- bucket b holds order[bucket_start[b]:bucket_start[b+1]];
      bucket_of_seq[i] -- the bucket sequence i landed in.
    """
    lengths = [int(s) for s in lengths]
    n = len(lengths)
    order = sorted(range(n), key=lambda i: (lengths[i], i))
    bucket_start = []
    count = 0
    for pos, i in enumerate(order):
        cap = bucket_batch(lengths[i], M_mem, M_comp, p)
        if count == 0 or count + 1 > cap:
            bucket_start.append(pos)
            count = 1
        else:
            count += 1
    bucket_start.append(n)
    bucket_of_seq = [0] * n
    for b in range(len(bucket_start) - 1):
        for pos in range(bucket_start[b], bucket_start[b + 1]):
            bucket_of_seq[order[pos]] = b
    return bucket_of_seq, order, bucket_start


def balance_cv(lengths, order, bucket_start, deal, ranks: int, p: int):
    """Load balance of a bucket plan over data-parallel ranks (summary section 4,
    "Eficiencia del Equilibrio de Carga": coefficient of variation of the
    per-rank compute load).  Buckets are dealt in the order `deal`, one per rank
    per step, over floor(num_buckets / ranks) full steps; a bucket's load is the
    sum of S^p over its sequences.  Returns (mean over steps of std/mean with the
    population std, mean over steps of max/mean, number of steps)."""
    nb = len(bucket_start) - 1
    load = []
    for b in range(nb):
        s = 0.0
        for pos in range(bucket_start[b], bucket_start[b + 1]):
            c = 1.0
            for _ in range(p):
                c *= float(lengths[order[pos]])
            s += c
        load.append(s)
    T = nb // ranks
    cv_sum = mm_sum = 0.0
    for t in range(T):
        ls = [load[deal[t * ranks + r]] for r in range(ranks)]
        tot = 0.0
        for v in ls:
            tot += v
        mean = tot / ranks
        var = 0.0
        for v in ls:
            var += (v - mean) * (v - mean)
        var /= ranks
        cv_sum += (var ** 0.5) / mean if mean > 0 else 0.0
        mm_sum += max(ls) / mean if mean > 0 else 0.0
    if T == 0:
        return 0.0, 0.0, 0
    return cv_sum / T, mm_sum / T, T
