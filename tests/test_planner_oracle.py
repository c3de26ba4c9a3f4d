"""Pins of the oracle's dual-constraint bucket planner ("AdaptiveLoad" summary, section 2.A)."""
import itertools
import os

import pytest

from oracle.planner import bucket_batch, plan_buckets

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bucket_batch_table.txt")
M_MEM, M_COMP, P = 262_144, 1 << 30, 2


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                s, b = line.split()
                rows.append((int(s), int(b)))
    return rows


def test_bucket_batch_hand_worked_table():
    for S, B in _golden():
        assert bucket_batch(S, M_MEM, M_COMP, P) == B


def _largest_feasible(S, M_mem, M_comp, p):
    """Brute force by bisection on the two constraints themselves (no floor formula)."""
    ok = lambda B: B * S <= M_mem and B * S ** p <= M_comp
    if not ok(1):
        return 1
    lo, hi = 1, 1
    while ok(hi):
        hi *= 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if ok(mid) else (lo, mid)
    return lo


def test_bucket_batch_brute_force_1_to_40000():
    for S in range(1, 40_001):
        assert bucket_batch(S, M_MEM, M_COMP, P) == _largest_feasible(S, M_MEM, M_COMP, P), S


@pytest.mark.parametrize("p", [1, 2, 3])
def test_bucket_batch_other_exponents(p):
    for S in list(range(1, 300)) + [1023, 1024, 1025, 4095, 4096, 4097]:
        assert bucket_batch(S, 5000, 10 ** 7, p) == _largest_feasible(S, 5000, 10 ** 7, p)


def _check_walk(lengths, M_mem, M_comp, p):
    bos, order, starts = plan_buckets(lengths, M_mem, M_comp, p)
    n = len(lengths)
    # order is the stable sort by (S, index)
    assert order == sorted(range(n), key=lambda i: (lengths[i], i))
    assert starts[0] == 0 and starts[-1] == n and all(a < b for a, b in zip(starts, starts[1:]))
    for b in range(len(starts) - 1):
        members = order[starts[b]:starts[b + 1]]
        smax = max(lengths[i] for i in members)
        # every bucket obeys its dual constraint at its largest length
        assert len(members) <= bucket_batch(smax, M_mem, M_comp, p)
        assert all(bos[i] == b for i in members)
        # a bucket is closed only when the next sequence would break the constraint
        if starts[b + 1] < n:
            nxt = order[starts[b + 1]]
            assert len(members) + 1 > bucket_batch(lengths[nxt], M_mem, M_comp, p)


def test_walk_exhaustive_tiny():
    alphabet = [1, 2, 3, 5, 8]
    for n in range(1, 7):
        for L in itertools.product(alphabet, repeat=n):
            for (mm, mc, p) in [(8, 40, 2), (6, 1000, 1), (4, 9, 2), (1, 1, 2)]:
                _check_walk(list(L), mm, mc, p)


def test_walk_on_ragged_workload_lengths():
    import workloads
    L = workloads.ragged_lengths(0)
    _check_walk(L, M_MEM, M_COMP, P)
    _, order, starts = plan_buckets(L, M_MEM, M_COMP, P)
    # every bucket stays within the memory budget at its largest length
    for b in range(len(starts) - 1):
        members = order[starts[b]:starts[b + 1]]
        assert len(members) * max(L[i] for i in members) <= M_MEM or len(members) == 1
