"""GPU parity for rows wider than the single-warp and pipelined kernels hold:
bf16 rows of more than 6,144 elements and fp32 rows of more than 3,072, up to
the 16,384 limit.  These take the CTA-per-row forward.  The LayerNorm backward
keeps its column partials in registers up to bf16 11,264 / fp32 5,632 and in
tensor memory above (up to bf16 16,384 / fp32 8,192; the widths on either side
check the switch); wider fp32 rows take the two-kernel backward (per-row
coefficients, then column slabs), and the gated-residual backward takes the
column slabs above the register limit.  Every expected value comes from the
fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from chain_util import (compare_all, compare_fused, compare_rms, oracle_chain, oracle_fused,
                        oracle_rms, run_dense, run_fused, run_ragged, run_rms, to64)

pytestmark = pytest.mark.gpu

SEGS = [1, 0, 7, 130, 3, 0, 1, 33]  # empty, one-row and multi-row segments


@pytest.fixture(scope="module")
def A():
    import modulation_adaln_fwd_gb300 as m
    return m


def _inputs(seg, D, dtype, seed=5, name="wide"):
    s = workloads.Spec(name, dtype, D, 1e-6, tuple(seg))
    return s, workloads.make_inputs(s, seed=seed, device="cuda")


def _tdt(dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def _check_chain(seg, D, dtype, xmod=None):
    s, inp = _inputs(seg, D, dtype)
    if xmod is not None:
        inp["x"] = xmod(inp["x"].float()).to(inp["x"].dtype)
    o = run_ragged(inp, s.offsets(), s.eps)
    ref = oracle_chain(to64(inp), s.offsets(), s.eps)
    return compare_all(o, ref, oracle.to_f64(inp["x"]), _tdt(dtype))


@pytest.mark.parametrize("dtype,D", [("bf16", 6152), ("bf16", 8192), ("bf16", 11264),
                                     ("bf16", 11272), ("bf16", 16384), ("f32", 3076),
                                     ("f32", 5632), ("f32", 5636), ("f32", 8192),
                                     ("f32", 8196), ("f32", 16384)])
def test_wide_chain_ragged(A, dtype, D):
    rep = _check_chain(SEGS, D, dtype)
    assert rep["mean_ties"] + rep["rstd_ties"] <= 1


def test_wide_chain_dense_bf16(A):
    B, N, D = 2, 96, 16384
    s, inp = _inputs([N] * B, D, "bf16")
    o = run_dense(inp, B, N, s.eps)
    ref = oracle_chain(to64(inp), s.offsets(), s.eps)
    compare_all(o, ref, oracle.to_f64(inp["x"]), torch.bfloat16)


@pytest.mark.parametrize("dtype,D", [("bf16", 12288), ("f32", 8192)])
def test_wide_many_short_segments(A, dtype, D):
    """Hundreds of segments of 0-6 rows: every chunk of the column slabs holds
    pieces of many segments."""
    g = np.random.default_rng(11)
    seg = [int(v) for v in g.integers(0, 7, size=300)]
    seg[0] = 0
    _check_chain(seg, D, dtype)


@pytest.mark.parametrize("dtype,D", [("bf16", 16384), ("f32", 8192)])
def test_wide_fused_chain(A, dtype, D):
    for write_y in (True, False):
        s, inp = _inputs([40, 0, 1, 90], D, dtype)
        o = run_fused(inp, s.offsets(), s.eps, write_y=write_y)
        ref = oracle_fused(to64(inp), s.offsets(), s.eps)
        compare_fused(o, ref, oracle.to_f64(inp["x"]), _tdt(dtype), write_y)


@pytest.mark.parametrize("dtype,D", [("bf16", 16384), ("f32", 16384), ("bf16", 7000)])
def test_wide_rms(A, dtype, D):
    s = workloads.Spec("rms", dtype, D, 1e-6, (60, 1, 0, 33))
    inp = workloads.make_inputs(s, seed=4, device="cuda")
    o = run_rms(inp, s.offsets(), s.eps)
    ref = oracle_rms(to64(inp), s.offsets(), s.eps)
    compare_rms(o, ref, _tdt(dtype))


@pytest.mark.parametrize("dtype,D", [("bf16", 16384), ("f32", 12288)])
def test_wide_statistics_edge_rows(A, dtype, D):
    """The cross-warp merges of the row statistics (a group of four warps per row
    in the pipelined bf16 forward, the whole CTA in the fp32 CTA-per-row
    forward) on every path they have: the two-pass fallback (|mean| >> std),
    rows whose x^2 leaves the float range (scaled statistics, with the maximum
    exponent merged across the warps), tiny rows and a zero row."""
    def xmod(x):
        x = x.clone()
        x[0] = x[0] * 1e-3 + 300.0
        x[1] *= 1e12
        x[2] *= 1e-12
        x[3] *= 1e-25
        x[4] *= 1e20
        x[5] *= 1e35
        x[6] = 0.0
        return x
    s, inp = _inputs([8], D, dtype)
    inp["x"] = xmod(inp["x"].float()).to(inp["x"].dtype)
    o = torch.empty_like(inp["x"])
    mean = torch.empty(8, device="cuda")
    rstd = torch.empty(8, device="cuda")
    A.adaln_fwd(inp["x"].view(1, 8, D), inp["shift"], inp["scale"], o.view(1, 8, D), mean, rstd,
                1e-6)
    torch.cuda.synchronize()
    x64 = oracle.to_f64(inp["x"])
    y, m, r = oracle.adaln_fwd(x64, oracle.to_f64(inp["shift"]), oracle.to_f64(inp["scale"]),
                               [0, 8], float(np.float32(1e-6)))
    from chain_util import check_elementwise, check_stats
    check_elementwise("y", o, y, _tdt(dtype))
    ties = check_stats("mean", mean, m, np.maximum(np.mean(np.abs(x64), axis=1), 1e-300))
    ties += check_stats("rstd", rstd, r, np.abs(r))
    assert ties <= 1


def test_wide_workspace_row_coefficients(A):
    """bf16 rows of up to 16,384 elements and fp32 rows of up to 8,192 take the
    single-pass backward (column partials in tensor memory), which needs no
    per-row coefficients; wider fp32 rows take the two-kernel backward, whose
    workspace holds 16 bytes of coefficients per row.  The gated-residual
    backward never needs them."""
    # fewer rows than any plan's chunks: every plan then makes a chunk per row, so
    # the partials of the two backward passes differ by exactly their count of
    # reduced quantities
    rows = 8
    for dt, D, coef in ((torch.bfloat16, 16384, False), (torch.float32, 8192, False),
                        (torch.float32, 16384, True)):
        ws_ln = A.adaln_bwd_workspace_size(1, rows, D, dt)
        ws_gate = A.adaln_gate_residual_bwd_workspace_size(1, rows, D, dt)
        # both hold a 16-byte header, the status words S and their partials (twice as
        # many for the LayerNorm backward): ln - 2 gate = coefficients - 16 - S
        if coef:
            assert 0 < ws_ln - 2 * ws_gate <= 16 * rows - 16, (dt, D)
        else:
            assert ws_ln - 2 * ws_gate < 0, (dt, D)


def test_wide_forward_more_rows_than_ctas(A):
    """More rows than the forward's CTA cap (2^20): CTAs loop over rows.  Checked
    on sampled rows (the first and last of each CTA's sweep and random ones)."""
    rows, D = (1 << 20) + 37, 6152
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    x = torch.randn(1, rows, D, device="cuda", generator=g).to(torch.bfloat16)
    shift = (0.1 * torch.randn(1, D, device="cuda", generator=g)).to(torch.bfloat16)
    scale = (0.1 * torch.randn(1, D, device="cuda", generator=g)).to(torch.bfloat16)
    y = torch.empty_like(x)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    A.adaln_fwd(x, shift, scale, y, mean, rstd, 1e-6)
    torch.cuda.synchronize()
    pick = sorted({0, 1, (1 << 20) - 1, 1 << 20, rows - 1} |
                  set(np.random.default_rng(0).integers(0, rows, 24).tolist()))
    xs = oracle.to_f64(x[0, pick])
    ys, ms, rs = oracle.adaln_fwd(xs, oracle.to_f64(shift), oracle.to_f64(scale), [0, len(pick)],
                                  float(np.float32(1e-6)))
    from chain_util import check_elementwise, check_stats
    check_elementwise("y", y[0, pick], ys, torch.bfloat16)
    ties = check_stats("mean", mean[pick], ms, np.maximum(np.mean(np.abs(xs), axis=1), 1e-300))
    ties += check_stats("rstd", rstd[pick], rs, np.abs(rs))
    assert ties <= 1
    del x, y
    torch.cuda.empty_cache()
