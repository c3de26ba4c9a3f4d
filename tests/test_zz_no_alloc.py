"""The no-allocation backward (adaln_bwd_noalloc) against the regular one.

adaln_bwd_noalloc is for callers that cannot allocate device memory (a plugin
whose host framework owns all device memory, or a path that must not call
cudaMalloc).  It runs the same backward on a scratch buffer the library keeps
in device memory.  This file is collected last on purpose: it must pass both
on its own in a fresh process and after every other test, and two calls in a
row must both give exactly what adaln_bwd gives with a caller workspace, with
the scratch's status word (read by adaln_pipeline_status) at 0.
"""
import ctypes

import pytest
import torch

import workloads
from chain_util import BF16_ABS, F32_ABS, RED_REL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import modulation_adaln_fwd_gb300 as m
    return m


def _case(A, name, B, N, D, dtype):
    s = workloads.Spec(name, dtype, D, 1e-6, (N,) * B)
    inp = workloads.make_inputs(s, seed=3, device="cuda", tensors=("x", "shift", "scale", "dy"))
    x = inp["x"].view(B, N, D)
    dy = inp["dy"].view(B, N, D)
    mean = torch.empty(B * N, device="cuda")
    rstd = torch.empty(B * N, device="cuda")
    A.adaln_fwd(x, inp["shift"], inp["scale"], torch.empty_like(x), mean, rstd, 1e-6)
    # reference: the regular entry point with a caller-owned workspace
    ws = A.workspace(A.adaln_bwd_workspace_size(B, N, D, x.dtype), "cuda")
    ref = dict(dx=torch.empty_like(x), d_scale=torch.empty(B, D, device="cuda"),
               d_shift=torch.empty(B, D, device="cuda"))
    A.adaln_bwd(x, mean, rstd, inp["scale"], dy, ref["dx"], ref["d_scale"], ref["d_shift"], ws)
    return x, dy, mean, rstd, inp["scale"], ref


def _close(a, b, tol_abs):
    return bool(((a.float() - b.float()).abs() <= tol_abs).all())


def _same_bits(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


@pytest.mark.parametrize("B,N,D,dtype", [(1, 4096, 5120, "bf16"), (8, 1024, 1152, "bf16"),
                                          (2, 256, 128, "f32"), (3, 77, 3072, "bf16")])
def test_noalloc_matches_workspace_backward_twice(A, B, N, D, dtype):
    """Both calls run the same deterministic kernels in the same fixed order (no
    floating-point atomics), so the results must be bit-identical to the regular
    backward's; stale partials left by an earlier call would show up here.  The
    scratch's status word must read 0 after each call."""
    x, dy, mean, rstd, scale, ref = _case(A, "noalloc", B, N, D, dtype)
    for _ in range(2):
        dx = torch.full_like(x, 9.0)
        d_scale = torch.full((B, D), 9.0, device="cuda")
        d_shift = torch.full((B, D), 9.0, device="cuda")
        A.adaln_bwd_noalloc(x, mean, rstd, scale, dy, dx, d_scale, d_shift)
        torch.cuda.synchronize()
        assert A.adaln_pipeline_status() == 0
        assert _same_bits(dx, ref["dx"])
        assert _same_bits(d_scale, ref["d_scale"]) and _same_bits(d_shift, ref["d_shift"])
    # and within the oracle-derived tolerances the parity tests use (both sides
    # being the same bits, this is the regular backward's own parity)
    tol = F32_ABS if dtype == "f32" else BF16_ABS
    assert _close(dx, ref["dx"], tol)
    for got, want in ((d_scale, ref["d_scale"]), (d_shift, ref["d_shift"])):
        err = (got - want).abs().max().item()
        assert err <= RED_REL * max(want.abs().max().item(), 1e-30)


def test_noalloc_rejects_shapes_beyond_its_scratch(A):
    cap = A.adaln_noalloc_scratch_bytes()
    assert cap == 16 << 20
    # many short samples: one column partial per chunk per sample exceeds the scratch
    B, N, D = 4096, 8, 5120
    assert A.adaln_bwd_workspace_size(B, N, D, torch.bfloat16) > cap
    t = torch.empty((B, N, D), dtype=torch.bfloat16, device="cuda")
    m = torch.empty(B * N, device="cuda")
    sc = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
    g = torch.empty((B, D), device="cuda")
    with pytest.raises(A.AdaLNError) as e:
        A.adaln_bwd_noalloc(t, m, m, sc, t, t.clone(), g, g.clone())
    assert e.value.status == 3
