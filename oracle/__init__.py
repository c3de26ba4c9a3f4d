"""fp64 CPU oracle for the AdaLN modulation operator and the bucket planner.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
CPU-baseline leg of the benchmark may import this package.  The product path
(the CUDA library and its Python binding) never imports or calls it, and the
two share no code.

* ``adaln_oracle.c`` (built with gcc into ``_build/liboracle.so``) holds the
  operator: forward, gated residual and both backward passes, in IEEE double,
  following the "AdaptiveLoad" technical summary (gist.science paper
  2605.17923), section 2.B.
* ``planner.py`` holds the dual-constraint bucket planner of the same summary,
  section 2.A, in exact Python integers.

Inputs are numpy arrays.  bf16 or fp32 tensors are widened exactly to float64
by the caller (``to_f64``) so the oracle sees the same values as the GPU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .planner import bucket_batch, plan_buckets  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "adaln_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int64
    Dd = ctypes.c_double
    lib.oracle_adaln_fwd.argtypes = [P, P, P, P, I, I, Dd, P, P, P]
    lib.oracle_gate_residual.argtypes = [P, P, P, P, I, I, P]
    lib.oracle_adaln_bwd.argtypes = [P, P, P, P, I, I, Dd, P, P, P]
    lib.oracle_gate_residual_bwd.argtypes = [P, P, P, P, I, I, P, P]
    lib.oracle_adaln_fwd_gated.argtypes = [P, P, P, P, P, P, I, I, Dd, P, P, P, P]
    lib.oracle_rms_fwd.argtypes = [P, P, P, P, I, I, Dd, P, P]
    lib.oracle_rms_bwd.argtypes = [P, P, P, P, I, I, Dd, P, P, P]
    lib.oracle_adaln_bwd_gated.argtypes = [P, P, P, P, P, P, I, I, Dd, P, P, P, P]
    lib.oracle_adaln_bwd_gated.restype = ctypes.c_int
    for f in ("oracle_adaln_fwd", "oracle_gate_residual", "oracle_adaln_bwd",
              "oracle_gate_residual_bwd"):
        getattr(lib, f).restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


def to_f64(a) -> np.ndarray:
    """Widen a torch tensor (bf16/fp32, any device) or array exactly to float64."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu", torch.float64).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _c64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _offsets(offsets, rows: int | None = None) -> np.ndarray:
    o = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    assert o.ndim == 1 and o[0] == 0 and np.all(np.diff(o) >= 0)
    if rows is not None:
        assert o[-1] == rows
    return o


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def dense_offsets(B: int, N: int) -> np.ndarray:
    return np.arange(B + 1, dtype=np.int64) * N


def _outputs(out, shapes):
    """Caller-provided output arrays (C-contiguous float64 of the given shapes), or new ones."""
    if out is None:
        return tuple(np.empty(s) for s in shapes)
    assert len(out) == len(shapes)
    for a, s in zip(out, shapes):
        assert a.shape == s and a.dtype == np.float64 and a.flags.c_contiguous
    return tuple(out)


def adaln_fwd(x, shift, scale, offsets, eps, lib=None, out=None):
    """y, mean, rstd for x [rows, D] with per-segment shift/scale [nseg, D]."""
    lib = lib or _load()
    x, shift, scale = _c64(x), _c64(shift), _c64(scale)
    rows, D = x.shape
    o = _offsets(offsets, rows)
    nseg = len(o) - 1
    assert shift.shape == (nseg, D) and scale.shape == (nseg, D)
    y, mean, rstd = _outputs(out, [(rows, D), (rows,), (rows,)])
    lib.oracle_adaln_fwd(_ptr(x), _ptr(shift), _ptr(scale), _ptr(o), nseg, D,
                             float(eps), _ptr(y), _ptr(mean), _ptr(rstd))
    return y, mean, rstd


def gate_residual(r, z, gate, offsets, lib=None, out=None):
    """out = r + gate[k] * z."""
    lib = lib or _load()
    r, z, gate = _c64(r), _c64(z), _c64(gate)
    rows, D = r.shape
    o = _offsets(offsets, rows)
    nseg = len(o) - 1
    assert z.shape == r.shape and gate.shape == (nseg, D)
    (res,) = _outputs(None if out is None else (out,), [(rows, D)])
    lib.oracle_gate_residual(_ptr(r), _ptr(z), _ptr(gate), _ptr(o), nseg, D, _ptr(res))
    return res


def adaln_bwd(x, scale, dy, offsets, eps, lib=None, out=None):
    """dx, d_scale, d_shift; statistics recomputed from x."""
    lib = lib or _load()
    x, scale, dy = _c64(x), _c64(scale), _c64(dy)
    rows, D = x.shape
    o = _offsets(offsets, rows)
    nseg = len(o) - 1
    assert dy.shape == x.shape and scale.shape == (nseg, D)
    dx, d_scale, d_shift = _outputs(out, [(rows, D), (nseg, D), (nseg, D)])
    lib.oracle_adaln_bwd(_ptr(x), _ptr(scale), _ptr(dy), _ptr(o), nseg, D, float(eps),
                             _ptr(dx), _ptr(d_scale), _ptr(d_shift))
    return dx, d_scale, d_shift


def gate_residual_bwd(dout, z, gate, offsets, lib=None, out=None):
    """dz, d_gate (dr = dout is the identity)."""
    lib = lib or _load()
    dout, z, gate = _c64(dout), _c64(z), _c64(gate)
    rows, D = dout.shape
    o = _offsets(offsets, rows)
    nseg = len(o) - 1
    assert z.shape == dout.shape and gate.shape == (nseg, D)
    dz, d_gate = _outputs(out, [(rows, D), (nseg, D)])
    lib.oracle_gate_residual_bwd(_ptr(dout), _ptr(z), _ptr(gate), _ptr(o), nseg, D,
                                     _ptr(dz), _ptr(d_gate))
    return dz, d_gate


def adaln_fwd_gated(x, shift, scale, gate, r, offsets, eps, lib=None):
    """Fused chain: out = r + gate[k] * y, y = LN(x) * (1 + scale[k]) + shift[k].
    Returns out, y, mean, rstd."""
    lib = lib or _load()
    x, shift, scale, gate, r = _c64(x), _c64(shift), _c64(scale), _c64(gate), _c64(r)
    rows, D = x.shape
    o = _offsets(offsets, rows)
    nseg = len(o) - 1
    assert r.shape == x.shape and shift.shape == scale.shape == gate.shape == (nseg, D)
    out, y = np.empty_like(x), np.empty_like(x)
    mean, rstd = np.empty(rows), np.empty(rows)
    lib.oracle_adaln_fwd_gated(_ptr(x), _ptr(shift), _ptr(scale), _ptr(gate), _ptr(r), _ptr(o),
                               nseg, D, float(eps), _ptr(out), _ptr(y), _ptr(mean), _ptr(rstd))
    return out, y, mean, rstd


def adaln_bwd_gated(x, shift, scale, gate, dout, offsets, eps, lib=None):
    """Backward of the fused chain given dout: dx, d_scale, d_shift, d_gate."""
    lib = lib or _load()
    x, shift, scale, gate, dout = _c64(x), _c64(shift), _c64(scale), _c64(gate), _c64(dout)
    rows, D = x.shape
    o = _offsets(offsets, rows)
    nseg = len(o) - 1
    assert dout.shape == x.shape and shift.shape == scale.shape == gate.shape == (nseg, D)
    dx = np.empty_like(x)
    d_scale, d_shift, d_gate = np.empty((nseg, D)), np.empty((nseg, D)), np.empty((nseg, D))
    st = lib.oracle_adaln_bwd_gated(_ptr(x), _ptr(shift), _ptr(scale), _ptr(gate), _ptr(dout),
                                    _ptr(o), nseg, D, float(eps), _ptr(dx), _ptr(d_scale),
                                    _ptr(d_shift), _ptr(d_gate))
    if st != 0:
        raise MemoryError("oracle_adaln_bwd_gated: out of host memory")
    return dx, d_scale, d_shift, d_gate


def rms_fwd(x, shift, scale, offsets, eps, lib=None):
    """RMSNorm modulation: y, rstd."""
    lib = lib or _load()
    x, shift, scale = _c64(x), _c64(shift), _c64(scale)
    rows, D = x.shape
    o = _offsets(offsets, rows)
    nseg = len(o) - 1
    assert shift.shape == scale.shape == (nseg, D)
    y, rstd = np.empty_like(x), np.empty(rows)
    lib.oracle_rms_fwd(_ptr(x), _ptr(shift), _ptr(scale), _ptr(o), nseg, D, float(eps), _ptr(y),
                       _ptr(rstd))
    return y, rstd


def rms_bwd(x, scale, dy, offsets, eps, lib=None):
    """RMSNorm modulation backward: dx, d_scale, d_shift."""
    lib = lib or _load()
    x, scale, dy = _c64(x), _c64(scale), _c64(dy)
    rows, D = x.shape
    o = _offsets(offsets, rows)
    nseg = len(o) - 1
    assert dy.shape == x.shape and scale.shape == (nseg, D)
    dx, d_scale, d_shift = np.empty_like(x), np.empty((nseg, D)), np.empty((nseg, D))
    lib.oracle_rms_bwd(_ptr(x), _ptr(scale), _ptr(dy), _ptr(o), nseg, D, float(eps), _ptr(dx),
                       _ptr(d_scale), _ptr(d_shift))
    return dx, d_scale, d_shift


class Variant:
    """The same API bound to another build of the C source (used by mutation tests)."""

    def __init__(self, so_path):
        self._lib = _bind(so_path)

    def adaln_fwd(self, *a):
        return adaln_fwd(*a, lib=self._lib)

    def gate_residual(self, *a):
        return gate_residual(*a, lib=self._lib)

    def adaln_bwd(self, *a):
        return adaln_bwd(*a, lib=self._lib)

    def gate_residual_bwd(self, *a):
        return gate_residual_bwd(*a, lib=self._lib)

    def adaln_fwd_gated(self, *a):
        return adaln_fwd_gated(*a, lib=self._lib)

    def adaln_bwd_gated(self, *a):
        return adaln_bwd_gated(*a, lib=self._lib)

    def rms_fwd(self, *a):
        return rms_fwd(*a, lib=self._lib)

    def rms_bwd(self, *a):
        return rms_bwd(*a, lib=self._lib)


def compile_variant(src_text: str, out_dir: str, name: str) -> str:
    """Compile a (modified) copy of the oracle source into out_dir; return the .so path."""
    os.makedirs(out_dir, exist_ok=True)
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
                           "-fPIC", "-shared", "-o", so, c, "-lm"])
    return so


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()
