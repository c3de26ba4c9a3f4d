"""GPU parity of the fused gated chain (out = r + gate * y in one forward launch,
and its backward in one pipelined launch plus the column sums) against the
fp64 oracle on the same seeded inputs.  Shapes cover the register forward
(fp32, odd D), every pipelined forward geometry that has a fused variant
(D = 1152, 3072, 5120), dense and ragged calls, empty and one-row segments,
and the forward without the optional y output."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from chain_util import compare_fused, oracle_fused, run_fused, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import modulation_adaln_fwd_gb300 as m
    return m


def _inputs(seg, D, dtype, seed=3, name="fused"):
    s = workloads.Spec(name, dtype, D, 1e-6, tuple(seg))
    return s, workloads.make_inputs(s, seed=seed, device="cuda")


def _check(seg, D, dtype, dense=None, write_y=True):
    s, inp = _inputs(seg, D, dtype)
    o = run_fused(inp, s.offsets(), s.eps, dense=dense, write_y=write_y)
    ref = oracle_fused(to64(inp), s.offsets(), s.eps)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    return compare_fused(o, ref, oracle.to_f64(inp["x"]), tdt, write_y)


def test_fused_tiny_fp32_dense(A):
    rep = _check([256, 256], 128, "f32", dense=(2, 256))
    assert rep["mean_ties"] + rep["rstd_ties"] == 0


def test_fused_dit_bf16_dense(A):
    rep = _check([1024] * 8, 1152, "bf16", dense=(8, 1024))
    assert rep["mean_ties"] + rep["rstd_ties"] == 0


def test_fused_mmdit_bf16_one_launch(A):
    s = workloads.spec("mmdit")
    inp = workloads.make_inputs(s, seed=0, device="cuda", draw_device="cuda")
    before = A.adaln_launch_count()
    o = run_fused(inp, s.offsets(), s.eps)
    # one forward launch; the backward is the pipelined kernel plus the column sums
    assert A.adaln_launch_count() - before == 3
    ref = oracle_fused(to64(inp), s.offsets(), s.eps)
    rep = compare_fused(o, ref, oracle.to_f64(inp["x"]), torch.bfloat16)
    assert rep["mean_ties"] + rep["rstd_ties"] == 0


@pytest.mark.parametrize("D", [5120, 3072])
def test_fused_wide_rows_bf16(A, D):
    """The pipelined forward with one slot per warp (5120) and two rows per unit (3072)."""
    _check([1000, 0, 3, 2093], D, "bf16")


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 1000), ("f32", 128), ("f32", 1536)])
def test_fused_odd_shapes_ragged(A, dtype, D):
    _check([1, 0, 7, 130, 3, 0, 1, 33], D, dtype)


@pytest.mark.parametrize("D", [1152, 3072])
def test_fused_without_y_output(A, D):
    _check([40, 200, 1], D, "bf16", write_y=False)


def test_fused_forward_equals_unfused_chain_within_rounding(A):
    """The fused out differs from fwd -> gate only by y's bf16 rounding before the
    gate: |out_fused - out_chain| <= |gate| * half-ulp(y) + out rounding."""
    from chain_util import run_ragged
    s, inp = _inputs([300, 500], 3072, "bf16")
    fused = run_fused(inp, s.offsets(), s.eps)
    inp2 = dict(inp)
    chain = run_ragged(inp2, s.offsets(), s.eps)
    # the chain's gated residual runs on z (not y): redo it on y
    A.adaln_gate_residual_ragged(inp["r"], chain["y"], inp["gate"], chain["out"],
                                 np.asarray(s.offsets(), dtype=np.int64),
                                 torch.tensor(s.offsets(), dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(fused["mean"], chain["mean"]) and torch.equal(fused["rstd"], chain["rstd"])
    a, b = fused["out"].float(), chain["out"].float()
    g = inp["gate"].float().abs().max().item()
    lim = (g * 2.0 ** -8 + 2.0 ** -7) * torch.maximum(a.abs(), b.abs()).clamp(min=1.0)
    assert bool(((a - b).abs() <= lim).all())
