"""The C ABI on the CPU: the library loads, exports every declared entry point,
rejects bad arguments before touching CUDA, and its planner matches the
oracle's restatement bit for bit.  No kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "adaln.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(adaln_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import modulation_adaln_fwd_gb300 as m
    return m


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) == 36, names
    raw = ctypes.CDLL(lib.lib_path)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing
    # and the binding exposes the same names
    assert not [n for n in names if not hasattr(lib, n)]


def test_status_strings_and_limits(lib):
    for s in range(5):
        assert lib.adaln_status_string(s).startswith("ADALN_")
    assert "unknown" in lib.adaln_status_string(77)
    import torch
    # the boundary's row limit: D <= 16384 for both I/O types
    assert lib.adaln_max_dim(torch.bfloat16) == 16384
    assert lib.adaln_max_dim(torch.float32) == 16384


def _raw():
    import modulation_adaln_fwd_gb300 as m
    return m._lib


A16 = 1 << 20          # a fake, 16-byte aligned "device" address: never dereferenced
MIS = A16 + 4          # misaligned


@pytest.mark.parametrize("case,expect", [
    (dict(D=12), 1),            # bf16 D must be a multiple of 8
    (dict(D=0), 1),
    (dict(D=-8), 1),
    (dict(B=-1), 1),
    (dict(N=-3), 1),
    (dict(x=0), 1),             # null x with rows > 0
    (dict(x=MIS), 1),           # misaligned
    (dict(y=A16), 1),           # y aliases x
    (dict(eps=-1.0), 1),
    (dict(eps=float("nan")), 1),
    (dict(eps=float("inf")), 1),
    (dict(dt=7), 1),            # unknown dtype
    (dict(D=1 << 20), 2),       # larger than the kernels support
    (dict(D=16392), 2),         # one bf16 vector past the 16384 limit
    (dict(D=16388, dt=0), 2),   # one fp32 vector past it
])
def test_fwd_rejects_bad_arguments_before_any_launch(case, expect):
    lib = _raw()
    a = dict(x=A16, shift=A16 + 64, scale=A16 + 128, y=A16 + 256, mean=A16 + 512, rstd=A16 + 1024,
             B=2, N=4, D=64, eps=1e-6, dt=1)
    a.update(case)
    st = lib.adaln_fwd(a["x"], a["shift"], a["scale"], a["y"], a["mean"], a["rstd"], a["B"], a["N"],
                       a["D"], a["eps"], a["dt"], None)
    assert st == expect


def test_ragged_rejects_bad_offsets_before_any_launch():
    lib = _raw()

    def call(off, nseg=None, dev=A16):
        o = np.asarray(off, dtype=np.int64)
        n = len(o) - 1 if nseg is None else nseg
        return lib.adaln_fwd_ragged(A16, A16, A16, A16 + 4096, A16, A16, o.ctypes.data_as(ctypes.c_void_p),
                                    dev, n, 64, 1e-6, 1, None)
    assert call([1, 4]) == 1          # must start at 0
    assert call([0, 5, 3]) == 1       # decreasing
    assert call([0, 4], dev=0) == 1   # no device copy
    assert call([0, 4], dev=A16 + 3) == 1  # misaligned device offsets
    assert call([0, 4], nseg=-1) == 1
    assert lib.adaln_fwd_ragged(A16, A16, A16, A16, A16, A16, None, A16, 1, 64, 1e-6, 1, None) == 1


def test_indexed_calls_reject_bad_index_before_any_launch():
    lib = _raw()
    off = np.asarray([0, 4, 6], dtype=np.int64)
    offp = off.ctypes.data_as(ctypes.c_void_p)

    def fwd(idx, nmod=3, dev=A16 + 8192):
        mi = np.asarray(idx if idx is not None else [], dtype=np.int32)
        hp = mi.ctypes.data_as(ctypes.c_void_p) if idx is not None else None
        return lib.adaln_fwd_ragged_indexed(A16, A16, A16, A16 + 4096, A16, A16, offp, A16, hp,
                                            dev, 2, nmod, 64, 1e-6, 1, None)
    assert fwd([0, 3]) == 1             # row index past num_mod_rows
    assert fwd([-1, 0]) == 1            # negative
    assert fwd(None) == 1               # no host index
    assert fwd([0, 1], dev=None) == 1   # no device index
    assert fwd([0, 1], dev=A16 + 2) == 1  # misaligned device index
    assert fwd([0, 1], nmod=-1) == 1
    mi = np.asarray([2, 2], dtype=np.int32)
    mip = mi.ctypes.data_as(ctypes.c_void_p)
    assert lib.adaln_gate_residual_ragged_indexed(A16, A16 + 4096, A16, A16 + 8192, offp, A16,
                                                  mip, A16, 2, 2, 64, 1, None) == 1
    assert lib.adaln_bwd_ragged_indexed(A16, A16, A16, A16, A16, A16 + 4096, A16, A16, A16, 1 << 20,
                                        offp, A16, mip, A16, 2, 2, 64, 1, None) == 1
    assert lib.adaln_gate_residual_bwd_ragged_indexed(A16, A16, A16, A16 + 4096, A16, A16, 1 << 20,
                                                      offp, A16, mip, A16, 2, 2, 64, 1, None) == 1


def test_bwd_and_gate_reject_bad_arguments():
    lib = _raw()
    # dx aliasing dy, null mean, bad D: all before the workspace query touches CUDA
    assert lib.adaln_bwd(A16, A16, A16, A16, A16 + 64, A16 + 64, A16, A16, A16, 1 << 30,
                         1, 8, 64, 1, None) == 1
    assert lib.adaln_bwd(A16, 0, A16, A16, A16 + 64, A16 + 128, A16, A16, A16, 1 << 30,
                         1, 8, 64, 1, None) == 1
    assert lib.adaln_bwd(A16, A16, A16, A16, A16, A16, A16, A16, A16, 0, 1, 8, 60, 1, None) == 1
    assert lib.adaln_gate_residual(A16, MIS, A16, A16, 1, 8, 64, 1, None) == 1
    assert lib.adaln_gate_residual_bwd(A16, A16, 0, A16, A16, A16, 0, 1, 8, 64, 1, None) == 1
    assert lib.adaln_bwd_workspace_size(1, 8, 60, 1) == 0
    assert lib.adaln_bwd_ragged_workspace_size(None, 1, 64, 1) == 0


def test_fused_gated_calls_reject_bad_arguments():
    lib = _raw()
    X, R, OUT, Y = A16, A16 + 4096, A16 + 8192, A16 + 12288
    S, M = A16 + 16384, A16 + 20480

    def fwd(x=X, r=R, out=OUT, y=Y, gate=S, D=64):
        return lib.adaln_fwd_gated(x, S, S, gate, r, out, y, M, M, 1, 8, D, 1e-6, 1, None)
    assert fwd(out=X) == 1       # out aliases x
    assert fwd(out=R) == 1       # out aliases r
    assert fwd(y=OUT) == 1       # y aliases out
    assert fwd(y=R) == 1         # y aliases r
    assert fwd(r=0) == 1         # null r
    assert fwd(gate=0) == 1      # null gate
    assert fwd(r=MIS) == 1       # misaligned r
    assert fwd(D=60) == 1        # bf16 D not a multiple of 8

    def bwd(dx=OUT, dout=R, d_gate=S, gate=S):
        return lib.adaln_bwd_gated(X, M, M, S, S, gate, dout, dx, S, S, d_gate, A16, 1 << 30,
                                   1, 8, 64, 1, None)
    assert bwd(dx=R) == 1        # dx aliases dout
    assert bwd(dx=X) == 1        # dx aliases x
    assert bwd(d_gate=0) == 1    # null d_gate
    assert bwd(gate=MIS) == 1    # misaligned gate
    assert lib.adaln_bwd_gated_workspace_size(1, 8, 60, 1) == 0
    assert lib.adaln_bwd_gated_ragged_workspace_size(None, 1, 64, 1) == 0


def test_bucket_batch_matches_oracle(lib):
    from oracle.planner import bucket_batch
    for (mm, mc, p) in [(262_144, 1 << 30, 2), (5000, 10 ** 7, 3), (7, 7, 1), (10 ** 12, 10 ** 18, 3)]:
        for S in list(range(1, 2000)) + [4095, 4096, 4097, 32767, 32768, 10 ** 6, 2 ** 31]:
            assert lib.adaln_bucket_batch(S, mm, mc, p) == bucket_batch(S, mm, mc, p), (S, mm, mc, p)
    assert lib.adaln_bucket_batch(0, 1, 1, 1) == -1
    assert lib.adaln_bucket_batch(5, 1, 1, 0) == -1
    # S^p far beyond int64 must not overflow
    assert lib.adaln_bucket_batch(2 ** 40, 2 ** 62, 2 ** 62, 5) == 1


def test_plan_buckets_bit_exact_with_oracle_on_ragged_workload(lib):
    import workloads
    from oracle.planner import plan_buckets
    L = workloads.ragged_lengths(0)
    bos, order, starts = lib.adaln_plan_buckets(L, 262_144, 1 << 30, 2)
    obos, oorder, ostarts = plan_buckets(L, 262_144, 1 << 30, 2)
    assert bos.tolist() == obos and order.tolist() == oorder and starts.tolist() == ostarts


def test_plan_buckets_bit_exact_random_and_edge(lib):
    from oracle.planner import plan_buckets
    rng = np.random.default_rng(5)
    for trial in range(200):
        n = int(rng.integers(0, 40))
        L = rng.integers(1, 5000, size=n).tolist()
        mm, mc, p = int(rng.integers(1, 20000)), int(rng.integers(1, 10 ** 8)), int(rng.integers(1, 4))
        bos, order, starts = lib.adaln_plan_buckets(L, mm, mc, p)
        obos, oorder, ostarts = plan_buckets(L, mm, mc, p)
        assert bos.tolist() == obos and order.tolist() == oorder and starts.tolist() == ostarts
    with pytest.raises(lib.AdaLNError):
        lib.adaln_plan_buckets([3, 0, 2], 100, 100, 2)


def test_balance_cv_matches_oracle_and_rejects_bad_plans(lib):
    import workloads
    from oracle.planner import balance_cv, plan_buckets
    L = []
    for seed in range(4):
        L += workloads.ragged_lengths(seed)
    for m_comp in (1 << 62, 1 << 30):
        _, order, starts = plan_buckets(L, 262_144, m_comp, 2)
        nb = len(starts) - 1
        deal = np.random.default_rng(1).permutation(nb).tolist()
        for ranks in (1, 8, 16):
            got = lib.adaln_balance_cv(L, order, starts, deal, ranks, 2)
            ref = balance_cv(L, order, starts, deal, ranks, 2)
            assert got[2] == ref[2]
            np.testing.assert_allclose(got[:2], ref[:2], rtol=1e-12)
    _, order, starts = plan_buckets(L[:10], 262_144, 1 << 30, 2)
    nb = len(starts) - 1
    with pytest.raises(lib.AdaLNError):  # deal is not a permutation
        lib.adaln_balance_cv(L[:10], order, starts, [0] * nb, 2, 2)
    with pytest.raises(lib.AdaLNError):  # ranks < 1
        lib.adaln_balance_cv(L[:10], order, starts, list(range(nb)), 0, 2)
    with pytest.raises(lib.AdaLNError):  # buckets do not cover the sequences
        lib.adaln_balance_cv(L[:10], order, starts[:-1] + [starts[-1] - 1], list(range(nb)), 2, 2)


def test_fit_cost_recovers_exact_model_and_matches_scipy(lib):
    rng = np.random.default_rng(2)
    S = rng.integers(256, 32768, size=40)
    B = rng.integers(1, 64, size=40)  # independent of S, so a, b and p are identifiable
    for (a, b, p) in [(5e-4, 2e-12, 2.0), (1e-3, 3e-9, 1.0), (0.0, 1e-10, 1.5)]:
        t = a + b * B * S.astype(float) ** p
        fa, fb, fp, rss = lib.adaln_fit_cost(B, S, t)
        assert abs(fp - p) < 1e-6 and abs(fa - a) < 1e-9 + 1e-6 * abs(a)
        assert abs(fb - b) < 1e-5 * b and rss < 1e-18
    # with noise: the least-squares solution agrees with scipy's curve_fit
    scipy_opt = pytest.importorskip("scipy.optimize")
    t = 5e-4 + 2e-12 * B * S.astype(float) ** 2 * (1 + 0.03 * rng.standard_normal(len(S)))
    fa, fb, fp, _ = lib.adaln_fit_cost(B, S, t)
    model = lambda X, a, b, p: a + b * X[0] * X[1] ** p
    (ra, rb, rp), _ = scipy_opt.curve_fit(model, np.vstack([B, S]).astype(float), t,
                                          p0=[1e-4, 1e-12, 1.8], maxfev=20000)
    assert abs(fp - rp) < 1e-3 and abs(fb - rb) < 1e-2 * rb and abs(fa - ra) < 1e-5


def test_fit_cost_rejects_bad_input(lib):
    with pytest.raises(lib.AdaLNError):
        lib.adaln_fit_cost([1, 2], [3, 4], [1.0, 2.0])            # fewer than 3 points
    with pytest.raises(lib.AdaLNError):
        lib.adaln_fit_cost([1, 0, 2], [3, 4, 5], [1.0, 2.0, 3.0])  # B < 1
    with pytest.raises(lib.AdaLNError):
        lib.adaln_fit_cost([1, 1, 2], [3, 4, 5], [1.0, float("nan"), 3.0])
    with pytest.raises(lib.AdaLNError):
        lib.adaln_fit_cost([1, 1, 2], [3, 4, 5], [1.0, 2.0, 3.0], p_lo=2.0, p_hi=1.0)


def test_fit_cost_finds_global_minimum_on_bucket_shapes(lib):
    """Bucket shapes of the ragged workload, where B * S^p for large p is dominated
    by a few long buckets and the residual is not unimodal in p: a linear cost
    must still come back with p = 1."""
    import workloads
    from oracle.planner import plan_buckets
    L = workloads.ragged_lengths(0)
    _, order, starts = plan_buckets(L, 262_144, 1 << 30, 2)
    B, S = [], []
    for b in range(len(starts) - 1):
        lens = [L[i] for i in order[starts[b]:starts[b + 1]]]
        B.append(len(lens))
        S.append(int(round(sum(lens) / len(lens))))
    t = 0.05 + 7e-6 * np.asarray(B, float) * np.asarray(S, float)
    _, _, p, _ = lib.adaln_fit_cost(B, S, t)
    assert abs(p - 1.0) < 1e-6, p
