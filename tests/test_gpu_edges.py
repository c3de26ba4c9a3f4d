"""GPU edge cases: odd shapes, empty and one-row segments, zero rows, the
two-pass statistics fallback, degenerate rows, determinism, guard bands,
workspace errors and non-default streams.  Every expected value comes from the
fp64 oracle on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from chain_util import (compare_all, empty_outputs, oracle_chain, run_dense, run_ragged, to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import modulation_adaln_fwd_gb300 as m
    return m


def _inputs(seg, D, dtype, seed=1, name="edge"):
    s = workloads.Spec(name, dtype, D, 1e-6, tuple(seg))
    return s, workloads.make_inputs(s, seed=seed, device="cuda")


def _check_ragged(seg, D, dtype, xmod=None, eps=1e-6, f32_rel=False):
    """f32_rel: the ill-conditioned rows of the edge tests (rstd of 100 and more
    scales dx far above 1), where fp32 output rounding alone exceeds 1e-5
    absolute: 1e-5 relative above magnitude 1 instead."""
    s, inp = _inputs(seg, D, dtype)
    if xmod is not None:
        inp["x"] = xmod(inp["x"].float()).to(inp["x"].dtype)
    o = run_ragged(inp, s.offsets(), eps)
    ref = oracle_chain(to64(inp), s.offsets(), eps)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    return compare_all(o, ref, oracle.to_f64(inp["x"]), tdt, f32_rel=f32_rel)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [8, 64, 72, 1000, 1536, 2056, 3072, 4096, 5120, 6144])
def test_odd_shapes_ragged(A, dtype, D):
    """Empty, one-row and odd segments at every forward geometry: the register
    kernel, the pipelined kernel with its table in shared memory (D = 4096) and in
    tensor memory (D = 3072, 5120, 6144), whose two-row units end half empty."""
    if dtype == "f32" and D % 4:
        pytest.skip()
    _check_ragged([1, 0, 7, 130, 3, 0, 1, 33], D, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_largest_supported_D(A, dtype):
    D = A.adaln_max_dim(torch.bfloat16 if dtype == "bf16" else torch.float32)
    _check_ragged([5, 17], D, dtype)


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f32", 128), ("bf16", 3072),
                                     ("bf16", 5120), ("bf16", 8192)])
def test_many_short_segments(A, dtype, D):
    """Hundreds of segments of 0-6 rows: every row chunk of the backward holds
    pieces of many segments, and finding a chunk's first segment takes more
    than one round of the 32-way search.  In the pipelined forward every CTA
    stages a modulation table per piece, shared out among the warps of each
    tensor-memory quarter (four at D = 3072, five at D = 5120 and 8,192)."""
    g = np.random.default_rng(7)
    seg = [int(v) for v in g.integers(0, 7, size=700)]
    seg[0] = 0
    seg[-1] = 0
    _check_ragged(seg, D, dtype)


@pytest.mark.parametrize("ragged", [False, True])
def test_several_chunks_per_cta(A, ragged):
    """More rows than one chunk per SM can hold: chunks are dealt round-robin,
    several per CTA, and (ragged) run across segment boundaries."""
    seg = [350_003, 350_003] if not ragged else [1, 299_999, 0, 400_006]
    s, inp = _inputs(seg, 16, "bf16")
    o = run_dense(inp, 2, seg[0], 1e-6) if not ragged else run_ragged(inp, s.offsets(), 1e-6)
    ref = oracle_chain(to64(inp), s.offsets(), 1e-6)
    compare_all(o, ref, oracle.to_f64(inp["x"]), torch.bfloat16)


def test_dense_odd_shapes(A):
    for (B, N, D, dt) in [(3, 1, 8, "bf16"), (1, 5, 1152, "bf16"), (2, 301, 128, "f32"),
                          (5, 17, 5120, "bf16")]:
        s, inp = _inputs([N] * B, D, dt)
        o = run_dense(inp, B, N, 1e-6)
        torch.cuda.synchronize()
        ref = oracle_chain(to64(inp), s.offsets(), 1e-6)
        compare_all(o, ref, oracle.to_f64(inp["x"]), torch.float32 if dt == "f32" else torch.bfloat16)


def test_zero_rows_give_zero_gradients(A):
    D = 64
    dev = "cuda"
    sc = torch.randn(3, D, device=dev).to(torch.bfloat16)
    d_scale = torch.full((3, D), 7.0, device=dev)
    d_shift = torch.full((3, D), 7.0, device=dev)
    d_gate = torch.full((3, D), 7.0, device=dev)
    empty = torch.empty((3, 0, D), dtype=torch.bfloat16, device=dev)
    ws = A.workspace(A.adaln_bwd_workspace_size(3, 0, D, torch.bfloat16) + 64, dev)
    m = torch.empty(0, device=dev)
    A.adaln_fwd(empty, sc, sc, empty.clone(), m, m.clone(), 1e-6)
    A.adaln_bwd(empty, m, m, sc, empty, empty.clone(), d_scale, d_shift, ws)
    A.adaln_gate_residual_bwd(empty, empty, sc, empty.clone(), d_gate, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d_scale) == 0 and torch.count_nonzero(d_shift) == 0
    assert torch.count_nonzero(d_gate) == 0
    # ragged: all segments empty
    off = np.zeros(4, dtype=np.int64)
    offd = torch.from_numpy(off).cuda()
    e2 = torch.empty((0, D), dtype=torch.bfloat16, device=dev)
    d_scale.fill_(3.0)
    ws = A.workspace(A.adaln_bwd_ragged_workspace_size(off, D, torch.bfloat16), dev)
    A.adaln_bwd_ragged(e2, m, m, sc, e2, e2.clone(), d_scale, d_shift, ws, off, offd)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d_scale) == 0
    # B = 0 is a no-op
    z0 = torch.empty((0, 4, D), dtype=torch.bfloat16, device=dev)
    A.adaln_fwd(z0, sc[:0], sc[:0], z0.clone(), m, m, 1e-6)


def test_two_pass_fallback_rows(A):
    """Rows with |mean| >> std take the two-pass variance; stats stay bit-exact."""
    def xmod(x):
        x = x.clone()
        x[::3] = x[::3] * 0.01 + 37.0          # mean/std ~ 3700
        x[1::7] = x[1::7] * 1e-3 - 5.0
        return x
    rep = _check_ragged([40, 25, 3], 1152, "bf16", xmod)
    assert rep["mean_ties"] + rep["rstd_ties"] <= 1
    rep = _check_ragged([40, 25, 3], 256, "f32", xmod, f32_rel=True)
    assert rep["mean_ties"] + rep["rstd_ties"] <= 1


def test_constant_rows(A):
    def xmod(x):
        x = x.clone()
        x[0] = 0.0
        x[1] = 3.25
        x[2] = -1e-3
        return x
    _check_ragged([4, 3], 128, "bf16", xmod)          # var = 0: rstd = 1/sqrt(eps)
    _check_ragged([4, 3], 128, "f32", xmod, f32_rel=True)  # rstd = 1000 scales dx


def test_eps_zero_constant_row_gives_inf_like_oracle(A):
    s, inp = _inputs([3], 64, "bf16")
    inp["x"][1] = 2.0
    o = run_ragged(inp, s.offsets(), 0.0)
    ref = oracle_chain(to64(inp), s.offsets(), 0.0)
    assert np.isinf(ref["rstd"][1]) and torch.isinf(o["rstd"][1])
    assert o["mean"][1].item() == 2.0
    # the other rows are ordinary
    for r in (0, 2):
        assert o["rstd"][r].item() == np.float32(ref["rstd"][r])


def test_extreme_magnitudes(A):
    def xmod(x):
        x = x.clone()
        x[0] *= 1e12
        x[1] *= 1e-12
        x[2, ::2] = 0.0
        x[3] *= 1e-25  # x^2 below the smallest normal float: eps dominates var + eps
        x[4] *= 1e20   # x^2 and the variance beyond the float range: scaled statistics
        x[5] *= 1e35   # close to the largest bf16: even the row sum would overflow
        return x
    rep = _check_ragged([8], 512, "bf16", xmod)
    assert rep["mean_ties"] + rep["rstd_ties"] <= 1
    rep = _check_ragged([8], 256, "f32", xmod, f32_rel=True)
    assert rep["mean_ties"] + rep["rstd_ties"] <= 1


@pytest.mark.parametrize("dtype,D", [("bf16", 512), ("bf16", 3072), ("f32", 256)])
def test_forward_on_huge_constant_rows(A, dtype, D):
    """Constant rows of huge values: var = 0, rstd = 1/sqrt(eps), and x * rstd would
    overflow, so the forward centres first.  (The backward's x * rstd - mean * rstd
    form needs |mean| * rstd within the float range; see the header.)"""
    from chain_util import check_elementwise, check_stats
    s, inp = _inputs([5], D, dtype)
    x = inp["x"].float()
    x[0] = 3.0e36
    x[1] = -2.5e35
    x[2] *= 1e36
    inp["x"] = x.to(inp["x"].dtype)
    o = empty_outputs(5, 1, D, inp["x"].dtype, "cuda")
    A.adaln_fwd(inp["x"].view(1, 5, D), inp["shift"], inp["scale"], o["y"].view(1, 5, D),
                o["mean"], o["rstd"], 1e-6)
    torch.cuda.synchronize()
    x64 = oracle.to_f64(inp["x"])
    y, mean, rstd = oracle.adaln_fwd(x64, oracle.to_f64(inp["shift"]), oracle.to_f64(inp["scale"]),
                                     [0, 5], float(np.float32(1e-6)))
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    check_elementwise("y", o["y"], y, tdt)
    check_stats("mean", o["mean"], mean, np.maximum(np.mean(np.abs(x64), axis=1), 1e-300))
    check_stats("rstd", o["rstd"], rstd, np.abs(rstd))


def test_bitwise_deterministic(A):
    s, inp = _inputs([300, 1, 77, 1024], 3072, "bf16")
    o1 = run_ragged(inp, s.offsets(), 1e-6)
    o1 = {k: v.clone() for k, v in o1.items()}
    o2 = run_ragged(inp, s.offsets(), 1e-6)
    for k in o1:
        assert torch.equal(o1[k].view(torch.uint8) if o1[k].dtype == torch.bfloat16 else o1[k],
                           o2[k].view(torch.uint8) if o2[k].dtype == torch.bfloat16 else o2[k]), k


def test_guard_bands_untouched(A):
    """Outputs live inside larger buffers filled with a sentinel; nothing outside is written."""
    s, inp = _inputs([9, 0, 31], 136, "bf16")
    rows, D, nseg = s.rows, s.D, s.nseg
    G = 64  # guard elements on each side (a multiple of 8 keeps 16-byte alignment)

    def guarded(n, dtype):
        buf = torch.full((n + 2 * G,), -77.0, dtype=dtype, device="cuda")
        return buf, buf[G:G + n]
    outs, bufs = {}, {}
    for k, (n, dt) in {"y": (rows * D, torch.bfloat16), "out": (rows * D, torch.bfloat16),
                       "dx": (rows * D, torch.bfloat16), "dz": (rows * D, torch.bfloat16),
                       "mean": (rows, torch.float32), "rstd": (rows, torch.float32),
                       "d_scale": (nseg * D, torch.float32), "d_shift": (nseg * D, torch.float32),
                       "d_gate": (nseg * D, torch.float32)}.items():
        bufs[k], v = guarded(n, dt)
        outs[k] = v.view(rows, D) if k in ("y", "out", "dx", "dz") else (
            v.view(nseg, D) if k.startswith("d_") else v)
    run_ragged(inp, s.offsets(), 1e-6, out=outs)
    for k, b in bufs.items():
        assert torch.all(b[:G] == -77.0) and torch.all(b[-G:] == -77.0), k
    ref = oracle_chain(to64(inp), s.offsets(), 1e-6)
    compare_all(outs, ref, oracle.to_f64(inp["x"]), torch.bfloat16)


def test_workspace_too_small_and_bad_args(A):
    s, inp = _inputs([64], 256, "bf16")
    x = inp["x"].view(1, 64, 256)
    o = empty_outputs(64, 1, 256, torch.bfloat16, "cuda")
    need = A.adaln_bwd_workspace_size(1, 64, 256, torch.bfloat16)
    assert need > 0
    small = A.workspace(need - 16, "cuda")
    with pytest.raises(A.AdaLNError) as e:
        A.adaln_bwd(x, o["mean"], o["rstd"], inp["scale"], inp["dy"].view(1, 64, 256),
                    o["dx"].view(1, 64, 256), o["d_scale"], o["d_shift"], small)
    assert e.value.status == 3
    with pytest.raises(A.AdaLNError) as e:
        A.adaln_fwd(x, inp["shift"], inp["scale"], x, o["mean"], o["rstd"], 1e-6)
    assert e.value.status == 1
    wide = A.adaln_max_dim(torch.bfloat16) + 8  # one vector past the largest row
    big = torch.empty((1, 2, wide), dtype=torch.bfloat16, device="cuda")
    sc = torch.empty((1, wide), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(A.AdaLNError) as e:
        A.adaln_fwd(big, sc, sc, big.clone(), o["mean"], o["rstd"], 1e-6)
    assert e.value.status == 2


def test_side_stream(A):
    s, inp = _inputs([200, 56], 1152, "bf16")
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        o = run_ragged(inp, s.offsets(), 1e-6)
    st.synchronize()
    ref = oracle_chain(to64(inp), s.offsets(), 1e-6)
    compare_all(o, ref, oracle.to_f64(inp["x"]), torch.bfloat16)


@pytest.mark.parametrize("dtype,D", [("bf16", 1152), ("bf16", 3072), ("f32", 512), ("bf16", 16384)])
def test_workspace_size_stable_across_launches(A, dtype, D):
    """The size query gives the same answer before and after the first launches (the
    plan's CTA count must not depend on state a launch leaves behind)."""
    s, inp = _inputs([40, 0, 9], D, dtype)
    off = np.asarray(s.offsets(), dtype=np.int64)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    before = (A.adaln_bwd_ragged_workspace_size(off, D, tdt),
              A.adaln_gate_residual_bwd_ragged_workspace_size(off, D, tdt))
    o = run_ragged(inp, s.offsets(), 1e-6)
    after = (A.adaln_bwd_ragged_workspace_size(off, D, tdt),
             A.adaln_gate_residual_bwd_ragged_workspace_size(off, D, tdt))
    assert before == after
    ref = oracle_chain(to64(inp), s.offsets(), 1e-6)
    compare_all(o, ref, oracle.to_f64(inp["x"]), tdt)


@pytest.mark.parametrize("dtype,D,seg", [("bf16", 1152, [300, 0, 57]), ("f32", 256, [64, 64]),
                                         ("bf16", 16384, [9, 3])])
def test_chain_replays_from_cuda_graph(A, dtype, D, seg):
    """The library's calls can be captured into a CUDA graph (no allocation, no
    synchronisation, no host-dependent work at launch); replays give the same bits
    as direct launches."""
    s, inp = _inputs(seg, D, dtype)
    o1 = run_ragged(inp, s.offsets(), 1e-6)
    o1 = {k: v.clone() for k, v in o1.items()}
    o2 = empty_outputs(s.rows, s.nseg, D, inp["x"].dtype, "cuda")
    off = np.asarray(s.offsets(), dtype=np.int64)
    off_dev = torch.from_numpy(off).cuda()
    x = inp["x"]
    ws = A.workspace(max(A.adaln_bwd_ragged_workspace_size(off, D, x.dtype),
                         A.adaln_gate_residual_bwd_ragged_workspace_size(off, D, x.dtype)), "cuda")

    def chain():
        A.adaln_fwd_ragged(x, inp["shift"], inp["scale"], o2["y"], o2["mean"], o2["rstd"], off,
                           off_dev, 1e-6)
        A.adaln_gate_residual_ragged(inp["r"], inp["z"], inp["gate"], o2["out"], off, off_dev)
        A.adaln_bwd_ragged(x, o2["mean"], o2["rstd"], inp["scale"], inp["dy"], o2["dx"],
                           o2["d_scale"], o2["d_shift"], ws, off, off_dev)
        A.adaln_gate_residual_bwd_ragged(inp["dy"], inp["z"], inp["gate"], o2["dz"], o2["d_gate"],
                                         ws, off, off_dev)
    chain()  # first launches outside the capture (kernel attributes are set there)
    torch.cuda.synchronize()
    for t in o2.values():
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for k in o1:
        a, b = o1[k], o2[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), k
