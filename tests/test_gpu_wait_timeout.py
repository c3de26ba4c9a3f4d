"""The bounded waits of the pipelined kernels give up, report, and return.

Every mbarrier wait inside the pipelined forward and backward kernels is
bounded: after a fixed number of polls the waiting thread records a non-zero
status and the kernel returns, so a bug that loses a copy shows up as an error
status instead of a hung GPU.  This file checks that path on the GPU without
faulting or hanging anything: it builds the library a second time, into a
temporary folder, with two test-only macros:

* ADALN_TEST_DROP_LAST_COPY: each CTA's producer never sends its last tile (or
  unit), so the consumers that wait for it wait in vain.  Every other copy is
  sent, and the producers drain their last slots before they leave, so no copy
  is in flight when a CTA exits;
* ADALN_TEST_WAIT_LIMIT: the polls before a wait gives up, cut to 2^16 so the
  test takes milliseconds rather than seconds.

It then checks that each kind of call returns with the error visible where the
header says it is: the workspace header word and NaN gradients for a backward
with a caller workspace, adaln_pipeline_status() for the no-allocation backward
and for the forward; and that the context is still usable afterwards (the
regular library runs the same shapes cleanly).  The backward and the forward
are checked on three widths, which between them take every kind of pipelined
kernel: D = 5120 (the split-phase backward, the one-warp forward), D = 3072
(the lockstep backward with 8-row tiles, two rows per forward unit) and
D = 16,384 (the lockstep backward with its partials in tensor memory, the
forward with a row per group of four warps).
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

_P, _I64, _SZ, _F, _E = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_int
BF16 = 1


@pytest.fixture(scope="module")
def A():
    import modulation_adaln_fwd_gb300 as m
    return m


@pytest.fixture(scope="module")
def T(tmp_path_factory):
    """The test build of the library (bounded waits that run out)."""
    from modulation_adaln_fwd_gb300 import build as b
    so = b.build(out_dir=str(tmp_path_factory.mktemp("adaln_wait_timeout")),
                 defines=("ADALN_TEST_WAIT_LIMIT=65536", "ADALN_TEST_DROP_LAST_COPY"))
    lib = ctypes.CDLL(so)
    sig = {
        "adaln_pipeline_status": (ctypes.c_int, []),
        "adaln_fwd": (_E, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _E, _P]),
        "adaln_bwd_workspace_size": (_SZ, [_I64, _I64, _I64, _E]),
        "adaln_bwd": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _E, _P]),
        "adaln_gate_residual_bwd_workspace_size": (_SZ, [_I64, _I64, _I64, _E]),
        "adaln_gate_residual_bwd": (_E, [_P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _E, _P]),
        "adaln_bwd_noalloc": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _E, _P]),
    }
    for name, (res, args) in sig.items():
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


B, N, D = 1, 4096, 5120  # the shape of the long-video rows: the pipelined kernels
WIDTHS = {5120: 4096, 3072: 4096, 16384: 512}  # D -> rows, for the backward and forward checks


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.fixture(scope="module")
def case(A):
    s = workloads.Spec("timeout", "bf16", D, 1e-6, (N,) * B)
    inp = workloads.make_inputs(s, seed=11, device="cuda", tensors=("x", "shift", "scale", "dy",
                                                                    "z", "gate"))
    mean = torch.empty(B * N, device="cuda")
    rstd = torch.empty(B * N, device="cuda")
    # statistics from the regular library, so the test build's forward runs last
    A.adaln_fwd(inp["x"].view(B, N, D), inp["shift"], inp["scale"],
                torch.empty_like(inp["x"]).view(B, N, D), mean, rstd, 1e-6)
    torch.cuda.synchronize()
    return inp, mean, rstd


def _inputs(A, D, N):
    s = workloads.Spec("timeout", "bf16", D, 1e-6, (N,) * B)
    inp = workloads.make_inputs(s, seed=11, device="cuda", tensors=("x", "shift", "scale", "dy",
                                                                    "z", "gate"))
    mean = torch.empty(B * N, device="cuda")
    rstd = torch.empty(B * N, device="cuda")
    # statistics from the regular library, so the test build's forward runs last
    A.adaln_fwd(inp["x"].view(B, N, D), inp["shift"], inp["scale"],
                torch.empty_like(inp["x"]).view(B, N, D), mean, rstd, 1e-6)
    torch.cuda.synchronize()
    return inp, mean, rstd


def _regular_backward_is_clean(A, inp, mean, rstd, D=D, N=N):
    ws = A.workspace(A.adaln_bwd_workspace_size(B, N, D, torch.bfloat16), "cuda")
    dx = torch.empty_like(inp["x"])
    ds = torch.empty(B, D, device="cuda")
    db = torch.empty(B, D, device="cuda")
    A.adaln_bwd(inp["x"].view(B, N, D), mean, rstd, inp["scale"], inp["dy"].view(B, N, D),
                dx.view(B, N, D), ds, db, ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    assert torch.isfinite(ds).all() and torch.isfinite(db).all()


def test_noalloc_backward_reports_timeout(A, T, case):
    inp, mean, rstd = case
    assert T.adaln_pipeline_status() == 0
    dx = torch.empty_like(inp["x"])
    ds = torch.zeros(B, D, device="cuda")
    db = torch.zeros(B, D, device="cuda")
    st = T.adaln_bwd_noalloc(_p(inp["x"]), _p(mean), _p(rstd), _p(inp["scale"]), _p(inp["dy"]),
                             _p(dx), _p(ds), _p(db), B, N, D, BF16, _stream())
    assert st == 0  # the launch itself succeeds; the kernel reports the lost tile
    torch.cuda.synchronize()
    assert T.adaln_pipeline_status() != 0  # the scratch's status word (the forward's is 0)
    assert torch.isnan(ds).all() and torch.isnan(db).all()
    _regular_backward_is_clean(A, inp, mean, rstd)


# (the gated-residual backward of 16,384-wide rows is the column-slab kernel,
# which has no ring and no wait)
@pytest.mark.parametrize("D,gate", [(3072, False), (3072, True), (5120, False), (5120, True),
                                    (16384, False)])
def test_backward_reports_timeout_in_workspace(A, T, D, gate):
    N = WIDTHS[D]
    inp, mean, rstd = _inputs(A, D, N)
    size = (T.adaln_gate_residual_bwd_workspace_size if gate else T.adaln_bwd_workspace_size)(
        B, N, D, BF16)
    ws = torch.zeros(size // 4 + 4, dtype=torch.int32, device="cuda")
    out = torch.empty_like(inp["x"])
    g1 = torch.zeros(B, D, device="cuda")
    g2 = torch.zeros(B, D, device="cuda")
    if gate:
        st = T.adaln_gate_residual_bwd(_p(inp["dy"]), _p(inp["z"]), _p(inp["gate"]), _p(out),
                                       _p(g1), _p(ws), ws.numel() * 4, B, N, D, BF16, _stream())
    else:
        st = T.adaln_bwd(_p(inp["x"]), _p(mean), _p(rstd), _p(inp["scale"]), _p(inp["dy"]),
                         _p(out), _p(g1), _p(g2), _p(ws), ws.numel() * 4, B, N, D, BF16,
                         _stream())
    assert st == 0
    torch.cuda.synchronize()
    assert int(ws[0].item()) != 0  # the header word: OR of the CTAs' status words
    assert torch.isnan(g1).all()
    if not gate:
        assert torch.isnan(g2).all()
    _regular_backward_is_clean(A, inp, mean, rstd, D, N)


@pytest.mark.parametrize("D", sorted(WIDTHS))
def test_forward_reports_timeout(A, T, D):
    N = WIDTHS[D]
    inp, mean, rstd = _inputs(A, D, N)
    y = torch.empty_like(inp["x"])
    m2 = torch.full_like(mean, float("nan"))
    r2 = torch.full_like(rstd, float("nan"))
    st = T.adaln_fwd(_p(inp["x"]), _p(inp["shift"]), _p(inp["scale"]), _p(y), _p(m2), _p(r2),
                     B, N, D, ctypes.c_float(1e-6), BF16, _stream())
    assert st == 0
    torch.cuda.synchronize()
    assert T.adaln_pipeline_status() != 0  # the forward's sticky word
    # every row but the dropped ones (one unit per CTA: one row, or two at D = 3072)
    # got its statistics
    lost = torch.isnan(m2)
    assert torch.equal(lost, torch.isnan(r2))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 1 <= int(lost.sum()) <= 2 * sms
    assert torch.equal(m2[~lost], mean[~lost]) and torch.equal(r2[~lost], rstd[~lost])
    # the regular library's forward is untouched by the test build's status word
    assert A.adaln_pipeline_status() == 0
    _regular_backward_is_clean(A, inp, mean, rstd, D, N)
