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
#   fp32 I/O: max-abs 1e-5 on every element-wise output.  Only the edge tests
#             whose outputs are large because the rows are ill-conditioned
#             (constant rows, |mean| >> std, magnitudes near the float range:
#             rstd of 1e3 and beyond multiplies dx) pass f32_rel=True, which
#             allows 1e-5 relative where the oracle's magnitude exceeds 1;
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
# boundary (then the neighbouring float is also accepted and counted as a tie).
# 2^-40 covers the oracle's own fp64 error: its two-pass sums over D <= 16384
# terms are off by at most about D * 2^-53 of sum|x| (mean) and of the variance
# (rstd), which is 2^-39 at the largest D and far less in practice.
STATS_TIE_REL = 2.0 ** -40


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def check_elementwise(name: str, gpu: torch.Tensor, ref: np.ndarray, dtype: torch.dtype,
                      f32_rel: bool = False):
    g = oracle.to_f64(gpu).reshape(ref.shape)
    err = np.abs(g - ref)
    if dtype == torch.float32:
        lim = F32_ABS * np.maximum(1.0, np.abs(ref)) if f32_rel else F32_ABS
        bad = ~(err <= lim) & ~(np.isnan(g) & np.isnan(ref))
        assert not bad.any(), (f"{name}: fp32 error {np.nanmax(err / lim):.3e} x tolerance "
                               f"(max-abs {np.nanmax(err):.3e}, "
                               f"largest |oracle| among the failures "
                               f"{np.nanmax(np.abs(ref)[bad]):.3e})")
        return float(np.nanmax(err)) if err.size else 0.0
    ok = err <= BF16_ABS
    if not ok.all():
        # only elements whose oracle magnitude is >= 8 may exceed 2e-2 (by up to one ulp)
        big = np.abs(ref) >= 8.0
        ok = ok | (big & (err <= bf16_ulp(ref)))
    assert ok.all(), (f"{name}: bf16 max-abs {np.max(np.where(np.abs(ref) >= 8.0, 0, err)):.3e}, "
                      f"{int((~ok).sum())} elements out of tolerance")
    if not err.size:
        return 0.0
    small = np.abs(ref) < 8.0
    return float(np.max(err, where=small, initial=0.0))


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
                dtype, rows=slice(None), segs=slice(None), report=None, f32_rel: bool = False):
    rep = {} if report is None else report
    for k in ("y", "out", "dx", "dz"):
        rep[k] = check_elementwise(k, gpu[k][rows], ref[k], dtype, f32_rel)
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
                  dtype, write_y: bool = True, f32_rel: bool = False):
    rep = {}
    for k in (("out", "y", "dx") if write_y else ("out", "dx")):
        rep[k] = check_elementwise(k, gpu[k], ref[k], dtype, f32_rel)
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


def compare_rms(gpu: Dict[str, torch.Tensor], ref: Dict[str, np.ndarray], dtype,
                f32_rel: bool = False):
    rep = {}
    for k in ("y", "dx"):
        rep[k] = check_elementwise(k, gpu[k], ref[k], dtype, f32_rel)
    for k in ("d_scale", "d_shift"):
        rep[k] = check_reduction(k, gpu[k], ref[k])
    rep["rstd_ties"] = check_stats("rstd", gpu["rstd"], ref["rstd"], np.abs(ref["rstd"]))
    return rep


# ----------------------------------------------------------------------------- streamed oracle

_CMP = None


def _fastcmp():
    """The one-pass widening and max-abs helpers of tests/cmp/fastcmp.c (gcc)."""
    global _CMP
    if _CMP is None:
        import ctypes
        import os
        import subprocess
        here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "cmp")
        src = os.path.join(here, "fastcmp.c")
        so = os.path.join(here, "_build", "libfastcmp.so")
        if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
            os.makedirs(os.path.dirname(so), exist_ok=True)
            tmp = so + ".tmp%d" % os.getpid()
            subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-o", tmp,
                                   src, "-lm"])
            os.replace(tmp, so)
        lib = ctypes.CDLL(so)
        P, I = ctypes.c_void_p, ctypes.c_int64
        for f in ("cmp_widen_bf16", "cmp_widen_f32"):
            getattr(lib, f).argtypes = [P, P, I]
            getattr(lib, f).restype = None
        for f in ("cmp_maxabs_bf16", "cmp_maxabs_f32"):
            getattr(lib, f).argtypes = [P, P, I]
            getattr(lib, f).restype = ctypes.c_double
        _CMP = lib
    return _CMP


def _ptr(a):
    import ctypes
    return ctypes.c_void_p(a.data_ptr() if isinstance(a, torch.Tensor) else a.ctypes.data)


class _HostBufs:
    """One thread's reusable host buffers: pageable torch tensors for the copies
    off the device and float64 arrays for the oracle's inputs and outputs, so
    that streaming a workload allocates (and page-faults) nothing per block."""

    def __init__(self, rows: int, D: int, io_dtype: torch.dtype):
        self.rows, self.D, self.io = rows, D, io_dtype
        self.t = {}
        self.f = {}

    def host(self, name: str, t: torch.Tensor) -> torch.Tensor:
        """t copied into this thread's host tensor `name` (same dtype, shape)."""
        n = t.numel()
        h = self.t.get((name, t.dtype))
        if h is None or h.numel() < n:  # sized for a full block at once
            h = torch.empty(max(n, self.rows * self.D if t.shape[0] > 1 else n), dtype=t.dtype)
            self.t[(name, t.dtype)] = h
        v = h[:n].view(t.shape)
        v.copy_(t)
        return v

    def f64(self, name: str, shape) -> np.ndarray:
        n = int(np.prod(shape))
        a = self.f.get(name)
        if a is None or a.size < n:  # sized for a full block at once
            a = np.empty(max(n, self.rows * self.D if n > self.D else n))
            self.f[name] = a
        return a[:n].reshape(shape)


def _widen_into(h: torch.Tensor, out: np.ndarray) -> np.ndarray:
    """Exact fp64 widening of a host bf16/fp32 tensor into out."""
    lib = _fastcmp()
    f = lib.cmp_widen_bf16 if h.dtype == torch.bfloat16 else lib.cmp_widen_f32
    assert h.dtype in (torch.bfloat16, torch.float32) and h.is_contiguous()
    f(_ptr(h), _ptr(out), h.numel())
    return out


def _maxabs_host(h: torch.Tensor, ref: np.ndarray) -> float:
    lib = _fastcmp()
    f = lib.cmp_maxabs_bf16 if h.dtype == torch.bfloat16 else lib.cmp_maxabs_f32
    assert h.numel() == ref.size and ref.dtype == np.float64 and ref.flags.c_contiguous
    return float(f(_ptr(h), _ptr(ref), h.numel()))


def stream_compare(inp: Dict[str, torch.Tensor], out: Dict[str, torch.Tensor],
                   segments: Sequence[tuple], eps: float, dtype, block: int | None = None,
                   threads: int | None = None):
    """Compare a full-size chain run with the oracle, streaming it over row blocks.

    `segments` lists (segment, first row, rows): segment k's rows of every
    [rows, D] tensor and its modulation row k.  Every row's y, out, dx, dz, mean
    and rstd are compared element by element; every segment's d_scale, d_shift and
    d_gate are compared with the sum of the oracle's block results (in fp64, in
    block order).  The oracle runs in a pool of threads (its C calls, the copies
    and the one-pass comparisons release the interpreter lock).  A block whose
    largest absolute error is within the plain tolerance passes at once; any
    other block goes through check_elementwise, which applies the full rules.
    Returns the worst error per output and the number of statistics ties."""
    import concurrent.futures as cf
    import os
    import threading

    D = inp["x"].shape[1]
    # blocks of at most 3M elements: each fp64 array then stays under the size
    # above which the C allocator maps fresh pages for every array (page faults
    # cost more than the arithmetic)
    block = block or max(1, 3_000_000 // D)
    tol = F32_ABS if dtype == torch.float32 else BF16_ABS
    jobs = []
    for (k, a, n) in segments:
        for b in range(a, a + n, block):
            jobs.append((k, b, min(a + n, b + block) - b))
    tls = threading.local()
    io = inp["x"].dtype

    def job(item):
        k, b, n = item
        sl = slice(b, b + n)
        if not hasattr(tls, "bufs"):
            tls.bufs = _HostBufs(block, D, io)
        hb = tls.bufs
        i64 = {key: _widen_into(hb.host(key, inp[key][sl]), hb.f64(key, (n, D)))
               for key in ("x", "r", "z", "dy")}
        i64.update({key: _widen_into(hb.host(key, inp[key][k:k + 1]), hb.f64(key, (1, D)))
                    for key in ("shift", "scale", "gate")})
        e = float(np.float32(eps))  # the library takes eps as a float
        off = [0, n]
        ref = {}
        ref["y"], ref["mean"], ref["rstd"] = oracle.adaln_fwd(
            i64["x"], i64["shift"], i64["scale"], off, e,
            out=(hb.f64("y", (n, D)), hb.f64("mean", (n,)), hb.f64("rstd", (n,))))
        ref["out"] = oracle.gate_residual(i64["r"], i64["z"], i64["gate"], off,
                                          out=hb.f64("out", (n, D)))
        ref["dx"], ref["d_scale"], ref["d_shift"] = oracle.adaln_bwd(
            i64["x"], i64["scale"], i64["dy"], off, e,
            out=(hb.f64("dx", (n, D)), np.empty((1, D)), np.empty((1, D))))
        ref["dz"], ref["d_gate"] = oracle.gate_residual_bwd(
            i64["dy"], i64["z"], i64["gate"], off, out=(hb.f64("dz", (n, D)), np.empty((1, D))))
        worst = {}
        for key in ("y", "out", "dx", "dz"):
            m = _maxabs_host(hb.host("o_" + key, out[key][sl]), ref[key])
            worst[key] = m if m <= tol else check_elementwise(key, out[key][sl], ref[key], dtype)
        l1 = np.maximum(np.add.reduce(np.abs(i64["x"], out=hb.f64("abs", (n, D))), axis=1) / D,
                        1e-300)
        ties = check_stats("mean", out["mean"][sl], ref["mean"], l1)
        ties += check_stats("rstd", out["rstd"][sl], ref["rstd"], np.abs(ref["rstd"]))
        return k, worst, ties, {key: ref[key][0] for key in ("d_scale", "d_shift", "d_gate")}

    nt = threads or min(16, os.cpu_count() or 1)
    worst = {key: 0.0 for key in ("y", "out", "dx", "dz", "d_scale", "d_shift", "d_gate")}
    ties = 0
    sums: Dict[int, Dict[str, np.ndarray]] = {}
    _fastcmp()  # build once, before the threads start
    with cf.ThreadPoolExecutor(max_workers=nt) as ex:
        # results come back in submission order, so each segment's blocks add in row order
        for k, w, t, part in ex.map(job, jobs):
            for key, v in w.items():
                worst[key] = max(worst[key], v)
            ties += t
            acc = sums.setdefault(k, {key: np.zeros_like(v) for key, v in part.items()})
            for key, v in part.items():
                acc[key] += v
    for (k, a, n) in segments:
        for key in ("d_scale", "d_shift", "d_gate"):
            # an empty segment's gradients are exact zeros
            ref = sums[k][key][None, :] if k in sums else np.zeros((1, out[key].shape[1]))
            worst[key] = max(worst[key], check_reduction(f"{key}[{k}]", out[key][k:k + 1], ref))
    return worst, ties
