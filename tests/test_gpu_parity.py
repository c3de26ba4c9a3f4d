"""GPU parity: the CUDA chain against the fp64 oracle on the five workloads.

Small workloads are compared element by element in full.  The long-video
workload (75,600 x 5120) is compared in full too, streaming the oracle over
row blocks.  The ragged mixed-mode workload is planned with the library's
planner (checked bit-exact against the oracle's), run bucket by bucket at
full size; three buckets (the first, the middle and the last) are compared in
full and every other bucket on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from chain_util import (check_elementwise, check_reduction, check_stats, compare_all,
                        oracle_chain, run_dense, run_ragged, to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import modulation_adaln_fwd_gb300 as m
    assert torch.cuda.is_available()
    return m


def _dense_case(A, name, draw_device="cpu"):
    s = workloads.spec(name)
    inp = workloads.make_inputs(s, seed=0, device="cuda", draw_device=draw_device)
    B, N = s.nseg, s.seg_lengths[0]
    o = run_dense(inp, B, N, s.eps)
    torch.cuda.synchronize()
    return s, inp, o


def test_tiny_fp32_full(A):
    s, inp, o = _dense_case(A, "tiny")
    ref = oracle_chain(to64(inp), s.offsets(), s.eps)
    rep = compare_all(o, ref, oracle.to_f64(inp["x"]), torch.float32)
    print("tiny", rep)
    assert rep["mean_ties"] == 0 and rep["rstd_ties"] <= 1


def test_dit_bf16_full(A):
    s, inp, o = _dense_case(A, "dit")
    ref = oracle_chain(to64(inp), s.offsets(), s.eps)
    rep = compare_all(o, ref, oracle.to_f64(inp["x"]), torch.bfloat16)
    print("dit", rep)
    assert rep["mean_ties"] + rep["rstd_ties"] <= 2


def test_mmdit_bf16_one_launch_full(A):
    s = workloads.spec("mmdit")
    inp = workloads.make_inputs(s, seed=0, device="cuda", draw_device="cuda")
    before = A.adaln_launch_count()
    o = run_ragged(inp, s.offsets(), s.eps)
    # one launch for fwd, one for the gated residual, a main + column-sum launch
    # for each backward: both streams of the block in the same launches
    assert A.adaln_launch_count() - before == 6
    ref = oracle_chain(to64(inp), s.offsets(), s.eps)
    rep = compare_all(o, ref, oracle.to_f64(inp["x"]), torch.bfloat16)
    print("mmdit", rep)
    assert rep["mean_ties"] + rep["rstd_ties"] <= 4


def test_wan_bf16_full_size_streamed_oracle(A):
    s, inp, o = _dense_case(A, "wan", draw_device="cuda")
    rows, D = s.rows, s.D
    blk = 4096
    sums = {k: np.zeros((1, D)) for k in ("d_scale", "d_shift", "d_gate")}
    ties = 0
    worst = {}
    for a in range(0, rows, blk):
        b = min(rows, a + blk)
        sl = slice(a, b)
        i64 = to64(inp, rows=sl)
        ref = oracle_chain(i64, [0, b - a], s.eps)
        for k in ("y", "out", "dx", "dz"):
            worst[k] = max(worst.get(k, 0.0), check_elementwise(k, o[k][sl], ref[k], torch.bfloat16))
        l1 = np.mean(np.abs(i64["x"]), axis=1)
        ties += check_stats("mean", o["mean"][sl], ref["mean"], l1)
        ties += check_stats("rstd", o["rstd"][sl], ref["rstd"], np.abs(ref["rstd"]))
        for k in sums:
            sums[k] += ref[k]
    for k in sums:
        worst[k] = check_reduction(k, o[k], sums[k])
    print("wan", worst, "ties", ties)
    assert ties <= 8


def _ragged_plan(A):
    L = workloads.ragged_lengths(0)
    bos, order, starts = A.adaln_plan_buckets(L, workloads.RAGGED_M_MEM, workloads.RAGGED_M_COMP,
                                              workloads.RAGGED_P)
    from oracle.planner import plan_buckets
    obos, oorder, ostarts = plan_buckets(L, workloads.RAGGED_M_MEM, workloads.RAGGED_M_COMP,
                                         workloads.RAGGED_P)
    assert bos.tolist() == obos and order.tolist() == oorder and starts.tolist() == ostarts
    return L, order.tolist(), starts.tolist()


def test_ragged_mixed_mode_bucketed(A):
    L, order, starts = _ragged_plan(A)
    D = workloads.RAGGED_D
    inp = workloads.make_packed_inputs(L, order, D, "bf16", seed=0, device="cuda",
                                       draw_device="cuda")
    total = inp["x"].shape[0]
    assert total == sum(L)
    from chain_util import empty_outputs
    out = empty_outputs(total, len(order), D, torch.bfloat16, "cuda")
    nb = len(starts) - 1
    row_start = [0]
    for b in range(nb):
        lens = [L[i] for i in order[starts[b]:starts[b + 1]]]
        offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        run_ragged(inp, offs, 1e-6, out=out, row0=row_start[-1], seg0=starts[b])
        row_start.append(row_start[-1] + int(offs[-1]))
    full = {0, nb // 2, nb - 1}
    rng = np.random.default_rng(0)
    ties = 0
    for b in range(nb):
        lens = [L[i] for i in order[starts[b]:starts[b + 1]]]
        offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        r0, r1 = row_start[b], row_start[b + 1]
        segs = slice(starts[b], starts[b + 1])
        if b in full:
            i64 = to64(inp, rows=slice(r0, r1), segs=segs)
            ref = oracle_chain(i64, offs, 1e-6)
            rep = compare_all(out, ref, i64["x"], torch.bfloat16, rows=slice(r0, r1), segs=segs)
            ties += rep["mean_ties"] + rep["rstd_ties"]
        else:
            # sampled rows: a row's outputs depend only on that row and its segment
            picks = sorted(set(rng.integers(r0, r1, size=16).tolist()) | {r0, r1 - 1})
            segpos = np.searchsorted(offs, np.array(picks) - r0, side="right") - 1
            for p, sp in zip(picks, segpos):
                k = starts[b] + int(sp)
                i64 = to64(inp, rows=slice(p, p + 1), segs=slice(k, k + 1))
                y, m, rs = oracle.adaln_fwd(i64["x"], i64["shift"], i64["scale"], [0, 1], 1e-6)
                ob = oracle.gate_residual(i64["r"], i64["z"], i64["gate"], [0, 1])
                dx, _, _ = oracle.adaln_bwd(i64["x"], i64["scale"], i64["dy"], [0, 1], 1e-6)
                dz, _ = oracle.gate_residual_bwd(i64["dy"], i64["z"], i64["gate"], [0, 1])
                check_elementwise("y", out["y"][p:p + 1], y, torch.bfloat16)
                check_elementwise("out", out["out"][p:p + 1], ob, torch.bfloat16)
                check_elementwise("dx", out["dx"][p:p + 1], dx, torch.bfloat16)
                check_elementwise("dz", out["dz"][p:p + 1], dz, torch.bfloat16)
                ties += check_stats("mean", out["mean"][p:p + 1], m, np.mean(np.abs(i64["x"]), axis=1))
                ties += check_stats("rstd", out["rstd"][p:p + 1], rs, rs)
            # parameter gradients of every segment: d_shift is a pure column sum of dy
            # (a property at any size); check it against the oracle's exact-order fp64 sum
            for j, ln in enumerate(lens):
                k = starts[b] + j
                a = r0 + int(offs[j])
                dy64 = oracle.to_f64(inp["dy"][a:a + ln])
                check_reduction("d_shift", out["d_shift"][k:k + 1], dy64.sum(axis=0, keepdims=True))
    print("ragged buckets", nb, "rows", total, "ties", ties)
    assert ties <= 16
