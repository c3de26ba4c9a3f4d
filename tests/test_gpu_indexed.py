"""GPU parity of the indexed ragged calls: segment k uses modulation row
mod_index[k] of [num_mod_rows, D] tables.  The expected values are the fp64
oracle's on the gathered per-segment rows (shift[mod_index], ...), with the
parameter gradients of a shared row summed over its segments (the chain rule
for a gathered parameter; rows no segment uses get zero).  Shapes cover the
pipelined forward and backward (one and several CTAs per SM), the register
forward (fp32), the wide-row kernels, empty segments, repeated and unused
modulation rows, and a call with no segments at all."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from chain_util import check_status, compare_all, empty_outputs, oracle_chain, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import modulation_adaln_fwd_gb300 as m
    return m


def run_indexed(A, inp, mod_tables, offsets, mod_index, eps):
    x = inp["x"]
    D, dt = x.shape[1], x.dtype
    nmod = mod_tables["shift"].shape[0]
    off = np.asarray(offsets, dtype=np.int64)
    mi = np.asarray(mod_index, dtype=np.int32)
    off_dev = torch.from_numpy(off).to(x.device)
    mi_dev = torch.from_numpy(mi).to(x.device) if len(mi) else None
    o = empty_outputs(x.shape[0], nmod, D, dt, x.device)
    A.adaln_fwd_ragged_indexed(x, mod_tables["shift"], mod_tables["scale"], o["y"], o["mean"],
                               o["rstd"], off, off_dev, mi, mi_dev, eps)
    A.adaln_gate_residual_ragged_indexed(inp["r"], inp["z"], mod_tables["gate"], o["out"], off,
                                         off_dev, mi, mi_dev)
    ws = A.workspace(max(A.adaln_bwd_ragged_workspace_size(off, D, dt),
                         A.adaln_gate_residual_bwd_ragged_workspace_size(off, D, dt)), x.device)
    # poison the gradients: every row must be written, unused ones with zeros
    for k in ("d_scale", "d_shift", "d_gate"):
        o[k].fill_(float("nan"))
    A.adaln_bwd_ragged_indexed(x, o["mean"], o["rstd"], mod_tables["scale"], inp["dy"], o["dx"],
                               o["d_scale"], o["d_shift"], ws, off, off_dev, mi, mi_dev)
    check_status(ws)
    A.adaln_gate_residual_bwd_ragged_indexed(inp["dy"], inp["z"], mod_tables["gate"], o["dz"],
                                             o["d_gate"], ws, off, off_dev, mi, mi_dev)
    torch.cuda.synchronize()
    return o


def expected(inp, mod_tables, offsets, mod_index, eps):
    """The oracle on the gathered rows, gradients scattered back onto the table rows."""
    idx = np.asarray(mod_index, dtype=np.int64)
    nmod = mod_tables["shift"].shape[0]
    d = to64(inp)
    for k in ("shift", "scale", "gate"):
        d[k] = oracle.to_f64(mod_tables[k])[idx] if len(idx) else np.zeros((0, inp["x"].shape[1]))
    ref = oracle_chain(d, offsets, eps)
    for k in ("d_scale", "d_shift", "d_gate"):
        acc = np.zeros((nmod, inp["x"].shape[1]))
        np.add.at(acc, idx, ref[k])
        ref[k] = acc
    return ref


def _case(seg, nmod, mod_index, D, dtype, seed=9):
    s = workloads.Spec("indexed", dtype, D, 1e-6, tuple(seg))
    inp = workloads.make_inputs(s, seed=seed, device="cuda")
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    tdt = inp["x"].dtype
    mod_tables = {k: (0.1 * torch.randn(nmod, D, generator=g)).to(tdt).cuda()
                  for k in ("shift", "scale", "gate")}
    return s, inp, mod_tables


@pytest.mark.parametrize("dtype,D", [("bf16", 1152), ("bf16", 3072), ("f32", 256),
                                     ("bf16", 16384), ("f32", 1000)])
def test_indexed_chain(A, dtype, D):
    seg = [40, 0, 7, 130, 1, 0, 64, 33]
    # rows 0 and 3 shared by several segments, row 5 used once, rows 1, 2, 4 unused
    mod_index = [3, 0, 3, 5, 0, 3, 0, 5]
    s, inp, mt = _case(seg, 6, mod_index, D, dtype)
    o = run_indexed(A, inp, mt, s.offsets(), mod_index, s.eps)
    ref = expected(inp, mt, s.offsets(), mod_index, s.eps)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    compare_all(o, ref, oracle.to_f64(inp["x"]), tdt)
    for k in ("d_scale", "d_shift", "d_gate"):
        assert torch.all(o[k][[1, 2, 4]] == 0), k


def test_indexed_identity_equals_plain_ragged(A):
    """mod_index = 0..n-1 gives bit-identical results to the plain ragged calls."""
    from chain_util import run_ragged
    seg = [100, 3, 0, 257]
    s, inp, _ = _case(seg, 4, list(range(4)), 3072, "bf16")
    mt = {k: inp[k] for k in ("shift", "scale", "gate")}
    o1 = run_indexed(A, inp, mt, s.offsets(), list(range(4)), s.eps)
    o2 = run_ragged(inp, s.offsets(), s.eps)
    for k in o1:
        a, b = o1[k], o2[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), k


def test_indexed_no_segments_zero_gradients(A):
    """No segments and no rows: the gradient tables are still written, as zeros."""
    D, bf = 256, torch.bfloat16
    inp = {k: torch.empty((0, D), dtype=bf, device="cuda") for k in ("x", "r", "z", "dy")}
    mt = {k: torch.randn(3, D, device="cuda").to(bf) for k in ("shift", "scale", "gate")}
    o = run_indexed(A, inp, mt, [0], [], 1e-6)
    for k in ("d_scale", "d_shift", "d_gate"):
        assert torch.all(o[k] == 0), k


def test_indexed_many_segments_few_rows(A):
    """Hundreds of segments over a few modulation rows: every column-sum CTA scans
    the whole index and adds many segments' chunk partials."""
    g = np.random.default_rng(5)
    seg = [int(v) for v in g.integers(0, 9, size=400)]
    mod_index = [int(v) for v in g.integers(0, 7, size=400)]
    s, inp, mt = _case(seg, 7, mod_index, 1152, "bf16")
    o = run_indexed(A, inp, mt, s.offsets(), mod_index, s.eps)
    ref = expected(inp, mt, s.offsets(), mod_index, s.eps)
    compare_all(o, ref, oracle.to_f64(inp["x"]), torch.bfloat16)


@pytest.mark.parametrize("dtype,D", [("bf16", 3072), ("f32", 512), ("bf16", 16384)])
def test_partition_invariance(A, dtype, D):
    """The same rows as one dense segment and as many ragged segments that all use
    modulation row 0: y, mean, rstd, out, dx and dz do not depend on how the rows
    are cut into segments, chunks and tiles (bit-identical); the parameter
    gradients, summed in another order, agree within the reduction tolerance."""
    from chain_util import check_reduction, run_dense
    rows = 1000
    seg = [1, 0, 257, 3, 400, 0, 339]
    assert sum(seg) == rows
    s = workloads.Spec("part", dtype, D, 1e-6, (rows,))
    inp = workloads.make_inputs(s, seed=21, device="cuda")
    od = run_dense(inp, 1, rows, s.eps)
    od = {k: v.clone() for k, v in od.items()}
    offsets = np.concatenate([[0], np.cumsum(seg)]).tolist()
    mt = {k: inp[k] for k in ("shift", "scale", "gate")}  # one modulation row
    oi = run_indexed(A, inp, mt, offsets, [0] * len(seg), s.eps)
    for k in ("y", "mean", "rstd", "out", "dx", "dz"):
        a, b = od[k], oi[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), k
    for k in ("d_scale", "d_shift", "d_gate"):
        check_reduction(k, oi[k], oracle.to_f64(od[k]))
