"""GPU parity of the RMSNorm modulation (rstd = 1/sqrt(mean x^2 + eps), no mean)
against the fp64 oracle: the register forward (fp32 and odd D), every pipelined
forward geometry (D = 1152, 3072, 5120), an fp32 large-D shape, dense and ragged
calls, and empty and one-row segments."""
import pytest
import torch

import workloads
from chain_util import compare_rms, oracle_rms, run_rms, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import modulation_adaln_fwd_gb300 as m
    return m


def _check(seg, D, dtype, dense=None, xmod=None, f32_rel=False):
    s = workloads.Spec("rms", dtype, D, 1e-6, tuple(seg))
    inp = workloads.make_inputs(s, seed=4, device="cuda")
    if xmod is not None:
        inp["x"] = xmod(inp["x"].float()).to(inp["x"].dtype)
    o = run_rms(inp, s.offsets(), s.eps, dense=dense)
    ref = oracle_rms(to64(inp), s.offsets(), s.eps)
    return compare_rms(o, ref, torch.float32 if dtype == "f32" else torch.bfloat16, f32_rel)


def test_rms_tiny_fp32_dense(A):
    assert _check([256, 256], 128, "f32", dense=(2, 256))["rstd_ties"] == 0


def test_rms_dit_bf16_dense(A):
    assert _check([1024] * 8, 1152, "bf16", dense=(8, 1024))["rstd_ties"] == 0


@pytest.mark.parametrize("D", [5120, 3072])
def test_rms_wide_rows_bf16(A, D):
    _check([1000, 0, 3, 2093], D, "bf16")


def test_rms_fp32_large_d(A):
    """fp32 I/O at the largest fp32 row the kernels take (adaln_max_dim: 16,384)."""
    D = A.adaln_max_dim(torch.float32)
    _check([300, 1, 0, 129], D, "f32")


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 1000), ("f32", 128), ("f32", 1536)])
def test_rms_odd_shapes_ragged(A, dtype, D):
    _check([1, 0, 7, 130, 3, 0, 1, 33], D, dtype)


def test_rms_offset_rows(A):
    """Rows far from zero mean: the RMS statistics keep the mean in, unlike LayerNorm."""
    def xmod(x):
        x = x.clone()
        x[::2] = x[::2] * 0.01 + 5.0
        return x
    _check([40, 25, 3], 1152, "bf16", xmod=xmod)


@pytest.mark.parametrize("dtype,D", [("bf16", 3072), ("bf16", 512), ("f32", 256)])
def test_rms_extreme_magnitudes(A, dtype, D):
    def xmod(x):
        x = x.clone()
        x[0] *= 1e-25
        x[1] *= 1e20
        x[2] *= 1e35
        x[3] = 0.0
        return x
    # rows scaled by 1e-25 have rstd ~ 1e3 (eps dominates), which scales their dx
    assert _check([6, 2], D, dtype, xmod=xmod, f32_rel=True)["rstd_ties"] <= 1
