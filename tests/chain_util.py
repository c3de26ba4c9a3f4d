"""Helpers for the GPU parity tests: run the CUDA chain through the C ABI and
compare against the fp64 oracle on the same seeded inputs.

The chain is fwd -> gated residual -> bwd -> gated-residual bwd, the upstream
gradient dy serving both backward calls (dout = dy).
"""
from __future__ import annotations

import math
from typing import Dict, Sequence

import numpy as np
import torch

import oracle
import modulation_adaln_fwd_gb300 as A

# Tolerances (readings documented in the design notes):
#   fp32 I/O: max-abs 1e-5 on every element-wise output, relative 1e-5 where the
#             oracle's magnitude exceeds 1 (fp32 rounding alone is 6e-5 at 1000);
#   bf16 I/O: max-abs 2e-2 on element-wise outputs, except that where the
#             oracle's magnitude is >= 8 (bf16 half-ulp > 2e-2 there) the
#             error may be up to one bf16 ulp of the oracle value;
#   parameter gradients (fp32 outputs for both I/O types): normwise relative
#             max|gpu - oracle| / max|oracle| <= 1e-3.
F32_ABS = 1e-5
BF16_ABS = 2e-2
RED_REL = 1e-3
# mean/rstd: bitwise equal to the oracle's fp64 value rounded to fp32, except
# where that value lies within this relative distance of a float rounding
# boundary (then the neighbouring float is also accepted and counted).
STATS_TIE_REL = 2.0 ** -36


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def check_elementwise(name: str, gpu: torch.Tensor, ref: np.ndarray, dtype: torch.dtype):
    g = oracle.to_f64(gpu).reshape(ref.shape)
    err = np.abs(g - ref)
    if dtype == torch.float32:
        lim = F32_ABS * np.maximum(1.0, np.abs(ref))
        bad = ~(err <= lim) & ~(np.isnan(g) & np.isnan(ref))
        assert not bad.any(), (f"{name}: fp32 error {np.nanmax(err / lim):.3e} x tolerance "
                               f"(max-abs {np.nanmax(err):.3e})")
        return float(np.nanmax(err)) if err.size else 0.0
    big = np.abs(ref) >= 8.0
    ok = np.where(big, err <= bf16_ulp(ref), err <= BF16_ABS)
    assert ok.all(), (f"{name}: bf16 max-abs {np.max(np.where(big, 0, err)):.3e}, "
                      f"{int((~ok).sum())} elements out of tolerance")
    return float(np.max(np.where(big, 0, err))) if err.size else 0.0


def check_reduction(name: str, gpu: torch.Tensor, ref: np.ndarray):
    g = oracle.to_f64(gpu).reshape(ref.shape)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    err = np.max(np.abs(g - ref)) if ref.size else 0.0
    if scale == 0.0:
        assert err == 0.0, f"{name}: expected exact zeros, max-abs {err}"
        return 0.0
    rel = err / scale
    assert rel <= RED_REL, f"{name}: normwise relative error {rel:.3e} > {RED_REL}"
    return float(rel)


def check_stats(name: str, gpu: torch.Tensor, ref: np.ndarray, scale_ref: np.ndarray):
    """Bitwise equality with round-to-nearest fp32 of the oracle's fp64 value,
    except near a rounding boundary (within STATS_TIE_REL * scale_ref)."""
    g = gpu.detach().cpu().numpy().astype(np.float32)
    r32 = ref.astype(np.float32)  # numpy rounds float64 -> float32 to nearest-even
    same = (g == r32) | (np.isnan(g) & np.isnan(r32))
    idx = np.nonzero(~same)[0]
    ties = 0
    for i in idx:
        a, b = float(r32[i]), float(g[i])
        assert np.nextafter(np.float32(a), np.float32(b)) == np.float32(b), \
            f"{name}[{i}]: gpu {b!r} is not a float neighbour of the rounded oracle {a!r}"
        boundary = 0.5 * (a + b)
        assert abs(float(ref[i]) - boundary) <= STATS_TIE_REL * float(scale_ref[i]), \
            f"{name}[{i}]: gpu {b!r} vs rounded oracle {a!r} (oracle {float(ref[i])!r}) not a tie"
        ties += 1
    return ties


# ----------------------------------------------------------------------------- running the chain

def empty_outputs(rows: int, nseg: int, D: int, dtype, device):
    f = dict(device=device, dtype=torch.float32)
    return dict(
        y=torch.empty((rows, D), dtype=dtype, device=device),
        mean=torch.empty(rows, **f), rstd=torch.empty(rows, **f),
        out=torch.empty((rows, D), dtype=dtype, device=device),
        dx=torch.empty((rows, D), dtype=dtype, device=device),
        dz=torch.empty((rows, D), dtype=dtype, device=device),
        d_scale=torch.empty((nseg, D), **f), d_shift=torch.empty((nseg, D), **f),
        d_gate=torch.empty((nseg, D), **f))


def run_dense(inp: Dict[str, torch.Tensor], B: int, N: int, eps: float, out=None):
    x = inp["x"]
    D = x.shape[-1]
    dt = x.dtype
    o = out or empty_outputs(B * N, B, D, dt, x.device)
    v = lambda t: t.view(B, N, D)
    A.adaln_fwd(v(x), inp["shift"], inp["scale"], v(o["y"]), o["mean"], o["rstd"], eps)
    A.adaln_gate_residual(v(inp["r"]), v(inp["z"]), inp["gate"], v(o["out"]))
    ws = A.workspace(max(A.adaln_bwd_workspace_size(B, N, D, dt),
                         A.adaln_gate_residual_bwd_workspace_size(B, N, D, dt)), x.device)
    A.adaln_bwd(v(x), o["mean"], o["rstd"], inp["scale"], v(inp["dy"]), v(o["dx"]), o["d_scale"],
                o["d_shift"], ws)
    A.adaln_gate_residual_bwd(v(inp["dy"]), v(inp["z"]), inp["gate"], v(o["dz"]), o["d_gate"], ws)
    check_status(ws)
    return o


def check_status(ws: torch.Tensor):
    """The first word of a backward workspace is the pipelined kernel's status:
    non-zero only if one of its bounded waits gave up; the forward's is a
    library-wide device word."""
    torch.cuda.synchronize()
    st = int(ws[:4].view(torch.int32).item())
    assert st == 0, f"backward kernel reported a wait timeout (status {st})"
    assert A.adaln_pipeline_status() == 0, "forward kernel reported a wait timeout"


def run_ragged(inp: Dict[str, torch.Tensor], offsets: Sequence[int], eps: float, out=None,
               row0: int = 0, seg0: int = 0):
    """One ragged call per op over rows [row0, row0 + offsets[-1]) and modulation
    rows [seg0, seg0 + len(offsets) - 1) of the given (possibly larger) tensors."""
    x = inp["x"]
    D = x.shape[-1]
    dt = x.dtype
    off = np.asarray(offsets, dtype=np.int64)
    nseg = len(off) - 1
    rows = int(off[-1])
    o = out or empty_outputs(x.shape[0], inp["shift"].shape[0], D, dt, x.device)
    rs = slice(row0, row0 + rows)
    ss = slice(seg0, seg0 + nseg)
    off_dev = torch.from_numpy(off).to(x.device)
    A.adaln_fwd_ragged(x[rs], inp["shift"][ss], inp["scale"][ss], o["y"][rs], o["mean"][rs],
                       o["rstd"][rs], off, off_dev, eps)
    A.adaln_gate_residual_ragged(inp["r"][rs], inp["z"][rs], inp["gate"][ss], o["out"][rs], off,
                                 off_dev)
    ws = A.workspace(max(A.adaln_bwd_ragged_workspace_size(off, D, dt),
                         A.adaln_gate_residual_bwd_ragged_workspace_size(off, D, dt)), x.device)
    A.adaln_bwd_ragged(x[rs], o["mean"][rs], o["rstd"][rs], inp["scale"][ss], inp["dy"][rs],
                       o["dx"][rs], o["d_scale"][ss], o["d_shift"][ss], ws, off, off_dev)
    check_status(ws)
    A.adaln_gate_residual_bwd_ragged(inp["dy"][rs], inp["z"][rs], inp["gate"][ss], o["dz"][rs],
                                     o["d_gate"][ss], ws, off, off_dev)
    torch.cuda.synchronize()
    return o


# ----------------------------------------------------------------------------- oracle side

def oracle_chain(inp64: Dict[str, np.ndarray], offsets, eps: float):
    # the library takes eps as a float: the oracle uses that same value, widened exactly
    eps = float(np.float32(eps))
    y, mean, rstd = oracle.adaln_fwd(inp64["x"], inp64["shift"], inp64["scale"], offsets, eps)
    out = oracle.gate_residual(inp64["r"], inp64["z"], inp64["gate"], offsets)
    dx, dsc, dsh = oracle.adaln_bwd(inp64["x"], inp64["scale"], inp64["dy"], offsets, eps)
    dz, dg = oracle.gate_residual_bwd(inp64["dy"], inp64["z"], inp64["gate"], offsets)
    return dict(y=y, mean=mean, rstd=rstd, out=out, dx=dx, dz=dz, d_scale=dsc, d_shift=dsh,
                d_gate=dg)


def compare_all(gpu: Dict[str, torch.Tensor], ref: Dict[str, np.ndarray], x64: np.ndarray,
                dtype, rows=slice(None), segs=slice(None), report=None):
    rep = {} if report is None else report
    for k in ("y", "out", "dx", "dz"):
        rep[k] = check_elementwise(k, gpu[k][rows], ref[k], dtype)
    for k in ("d_scale", "d_shift", "d_gate"):
        rep[k] = check_reduction(k, gpu[k][segs], ref[k])
    l1 = np.mean(np.abs(x64), axis=1)
    rep["mean_ties"] = check_stats("mean", gpu["mean"][rows], ref["mean"], np.maximum(l1, 1e-300))
    rep["rstd_ties"] = check_stats("rstd", gpu["rstd"][rows], ref["rstd"], np.abs(ref["rstd"]))
    return rep


def to64(inp: Dict[str, torch.Tensor], rows=slice(None), segs=slice(None)):
    d = {}
    for k, t in inp.items():
        if k in ("shift", "scale", "gate"):
            d[k] = oracle.to_f64(t[segs])
        else:
            d[k] = oracle.to_f64(t[rows])
    return d


# ----------------------------------------------------------------------------- fused gated chain

def run_fused(inp: Dict[str, torch.Tensor], offsets: Sequence[int], eps: float,
              dense=None, write_y: bool = True):
    """Fused forward (out = r + gate * y) and its backward with dout = dy, through the
    dense API when dense = (B, N), else the ragged one."""
    x = inp["x"]
    rows, D = x.shape
    dt = x.dtype
    nseg = inp["shift"].shape[0]
    o = empty_outputs(rows, nseg, D, dt, x.device)
    y = o["y"] if write_y else None
    if dense is not None:
        B, N = dense
        v = lambda t: t.view(B, N, D) if t is not None else None
        A.adaln_fwd_gated(v(x), inp["shift"], inp["scale"], inp["gate"], v(inp["r"]),
                          v(o["out"]), v(y), o["mean"], o["rstd"], eps)
        ws = A.workspace(A.adaln_bwd_gated_workspace_size(B, N, D, dt), x.device)
        A.adaln_bwd_gated(v(x), o["mean"], o["rstd"], inp["shift"], inp["scale"], inp["gate"],
                          v(inp["dy"]), v(o["dx"]), o["d_scale"], o["d_shift"], o["d_gate"], ws)
    else:
        off = np.asarray(offsets, dtype=np.int64)
        offd = torch.from_numpy(off).to(x.device)
        A.adaln_fwd_gated_ragged(x, inp["shift"], inp["scale"], inp["gate"], inp["r"], o["out"],
                                 y, o["mean"], o["rstd"], off, offd, eps)
        ws = A.workspace(A.adaln_bwd_gated_ragged_workspace_size(off, D, dt), x.device)
        A.adaln_bwd_gated_ragged(x, o["mean"], o["rstd"], inp["shift"], inp["scale"],
                                 inp["gate"], inp["dy"], o["dx"], o["d_scale"], o["d_shift"],
                                 o["d_gate"], ws, off, offd)
    check_status(ws)
    return o


def oracle_fused(inp64: Dict[str, np.ndarray], offsets, eps: float):
    eps = float(np.float32(eps))
    out, y, mean, rstd = oracle.adaln_fwd_gated(inp64["x"], inp64["shift"], inp64["scale"],
                                                inp64["gate"], inp64["r"], offsets, eps)
    dx, dsc, dsh, dg = oracle.adaln_bwd_gated(inp64["x"], inp64["shift"], inp64["scale"],
                                              inp64["gate"], inp64["dy"], offsets, eps)
    return dict(out=out, y=y, mean=mean, rstd=rstd, dx=dx, d_scale=dsc, d_shift=dsh, d_gate=dg)


def compare_fused(gpu: Dict[str, torch.Tensor], ref: Dict[str, np.ndarray], x64: np.ndarray,
                  dtype, write_y: bool = True):
    rep = {}
    for k in (("out", "y", "dx") if write_y else ("out", "dx")):
        rep[k] = check_elementwise(k, gpu[k], ref[k], dtype)
    for k in ("d_scale", "d_shift", "d_gate"):
        rep[k] = check_reduction(k, gpu[k], ref[k])
    l1 = np.mean(np.abs(x64), axis=1)
    rep["mean_ties"] = check_stats("mean", gpu["mean"], ref["mean"], np.maximum(l1, 1e-300))
    rep["rstd_ties"] = check_stats("rstd", gpu["rstd"], ref["rstd"], np.abs(ref["rstd"]))
    return rep


# ----------------------------------------------------------------------------- RMSNorm modulation

def run_rms(inp: Dict[str, torch.Tensor], offsets: Sequence[int], eps: float, dense=None):
    """RMSNorm forward and backward (dy as the upstream gradient), dense API when
    dense = (B, N), else ragged."""
    x = inp["x"]
    rows, D = x.shape
    dt = x.dtype
    nseg = inp["shift"].shape[0]
    o = empty_outputs(rows, nseg, D, dt, x.device)
    if dense is not None:
        B, N = dense
        v = lambda t: t.view(B, N, D)
        A.adaln_fwd_rms(v(x), inp["shift"], inp["scale"], v(o["y"]), o["rstd"], eps)
        ws = A.workspace(A.adaln_bwd_workspace_size(B, N, D, dt), x.device)
        A.adaln_bwd_rms(v(x), o["rstd"], inp["scale"], v(inp["dy"]), v(o["dx"]), o["d_scale"],
                        o["d_shift"], ws)
    else:
        off = np.asarray(offsets, dtype=np.int64)
        offd = torch.from_numpy(off).to(x.device)
        A.adaln_fwd_rms_ragged(x, inp["shift"], inp["scale"], o["y"], o["rstd"], off, offd, eps)
        ws = A.workspace(A.adaln_bwd_ragged_workspace_size(off, D, dt), x.device)
        A.adaln_bwd_rms_ragged(x, o["rstd"], inp["scale"], inp["dy"], o["dx"], o["d_scale"],
                               o["d_shift"], ws, off, offd)
    check_status(ws)
    return o


def oracle_rms(inp64: Dict[str, np.ndarray], offsets, eps: float):
    eps = float(np.float32(eps))
    y, rstd = oracle.rms_fwd(inp64["x"], inp64["shift"], inp64["scale"], offsets, eps)
    dx, dsc, dsh = oracle.rms_bwd(inp64["x"], inp64["scale"], inp64["dy"], offsets, eps)
    return dict(y=y, rstd=rstd, dx=dx, d_scale=dsc, d_shift=dsh)


def compare_rms(gpu: Dict[str, torch.Tensor], ref: Dict[str, np.ndarray], dtype):
    rep = {}
    for k in ("y", "dx"):
        rep[k] = check_elementwise(k, gpu[k], ref[k], dtype)
    for k in ("d_scale", "d_shift"):
        rep[k] = check_reduction(k, gpu[k], ref[k])
    rep["rstd_ties"] = check_stats("rstd", gpu["rstd"], ref["rstd"], np.abs(ref["rstd"]))
    return rep
