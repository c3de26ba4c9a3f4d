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


# ----------------------------------------------------------------------------- load balance
# (summary section 4, "Eficiencia del Equilibrio de Carga": CV of the per-rank
# compute load, a bucket's load being the sum of S^p over its sequences)

def test_balance_cv_closed_forms():
    import numpy as np
    from oracle.planner import balance_cv
    # four single-sequence buckets of equal length: every step is perfectly balanced
    assert balance_cv([7, 7, 7, 7], [0, 1, 2, 3], [0, 1, 2, 3, 4], [3, 1, 0, 2], 2, 2) == \
        (0.0, 1.0, 2)
    # two ranks with loads a and b: CV = |a - b| / (a + b), max/mean = 2 max / (a + b)
    L = [3, 5]
    cv, mm, T = balance_cv(L, [0, 1], [0, 1, 2], [0, 1], 2, 2)
    a, b = 9.0, 25.0
    assert T == 1 and abs(cv - abs(a - b) / (a + b)) < 1e-15 and abs(mm - 2 * b / (a + b)) < 1e-15
    # a bucket's load sums its sequences: buckets {2, 3} and {5} with p = 1 are equal
    cv, _, _ = balance_cv([2, 3, 5], [0, 1, 2], [0, 2, 3], [0, 1], 2, 1)
    assert cv == 0.0
    # a partial last step is dropped
    assert balance_cv([2, 2, 9], [0, 1, 2], [0, 1, 2, 3], [0, 1, 2], 2, 2)[2] == 1


def test_balance_cv_matches_numpy_population_std():
    import numpy as np
    from oracle.planner import balance_cv
    rng = np.random.default_rng(3)
    L = rng.integers(1, 3000, size=60).tolist()
    _, order, starts = plan_buckets(L, 5000, 10 ** 6, 2)
    nb = len(starts) - 1
    deal = rng.permutation(nb).tolist()
    for ranks in (1, 2, 3, 8):
        cv, mm, T = balance_cv(L, order, starts, deal, ranks, 2)
        loads = np.array([sum(L[i] ** 2 for i in order[starts[b]:starts[b + 1]])
                          for b in range(nb)], dtype=float)
        steps = [loads[deal[t * ranks:(t + 1) * ranks]] for t in range(nb // ranks)]
        assert T == len(steps)
        np.testing.assert_allclose(cv, np.mean([s.std() / s.mean() for s in steps]), rtol=1e-12)
        np.testing.assert_allclose(mm, np.mean([s.max() / s.mean() for s in steps]), rtol=1e-12)


def test_dual_constraint_lowers_compute_cv_on_ragged_draws():
    """The trend the summary reports (compute-load CV 39% -> 18.9%): on
    config-5-like length draws the dual constraint balances the S^2 load far
    better than equal-tokens batching (B * S = M_mem only)."""
    import numpy as np
    import workloads
    from oracle.planner import balance_cv
    L = []
    for seed in range(8):
        L += workloads.ragged_lengths(seed)
    res = {}
    for name, m_comp in (("equal_tokens", 1 << 62), ("dual", 1 << 30)):
        _, order, starts = plan_buckets(L, M_MEM, m_comp, P)
        deal = np.random.default_rng(0).permutation(len(starts) - 1).tolist()
        res[name] = balance_cv(L, order, starts, deal, 8, 2)[0]
    assert res["dual"] < 0.5 * res["equal_tokens"], res


def test_recorded_workload_facts():
    """The synthetic inputs the results are quoted on: seed 0 gives 256 ragged
    sequences of 1,448,621 rows in all, 51 of them fixed at S = 256, planned into
    30 buckets; the Wan-scale input has ceil(1% of 75,600) = 756 outlier rows."""
    import math

    import workloads
    L = workloads.ragged_lengths(0)
    assert len(L) == 256 and sum(L) == 1_448_621
    assert sum(1 for v in L if v == 256) == 51
    _, _, starts = plan_buckets(L, workloads.RAGGED_M_MEM, workloads.RAGGED_M_COMP,
                                workloads.RAGGED_P)
    assert len(starts) - 1 == 30
    s = workloads.spec("wan")
    assert s.rows == 75_600 and math.ceil(s.outlier_frac * s.rows) == 756
