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
