"""Python binding of the GB300 AdaLN modulation library (``include/adaln.h``).

Argument marshalling only: every function has the name of the C entry point it
calls, takes torch tensors where the C function takes device pointers (shapes
give the sizes), passes ``torch.cuda.current_stream()`` unless a stream is
given, and raises :class:`AdaLNError` on a non-zero status.  All compute runs
in the library's sm_103a kernels; there is no fallback: importing this module
fails when the compiled library is missing or cannot be loaded.

The operator ("AdaptiveLoad" technical summary, gist.science paper 2605.17923,
section 2.B) is the DiT adaptive LayerNorm
    y = LN(x) * (1 + scale[k]) + shift[k],   out = r + gate[k] * z,
with its backward (dx, and the sequence-dimension reductions d_scale, d_shift,
d_gate), plus the dual-constraint bucket planner of section 2.A.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

__all__ = [
    "AdaLNError", "lib_path", "adaln_fwd", "adaln_gate_residual", "adaln_bwd",
    "adaln_gate_residual_bwd", "adaln_fwd_ragged", "adaln_gate_residual_ragged",
    "adaln_bwd_ragged", "adaln_gate_residual_bwd_ragged", "adaln_bwd_workspace_size",
    "adaln_gate_residual_bwd_workspace_size", "adaln_bwd_ragged_workspace_size",
    "adaln_gate_residual_bwd_ragged_workspace_size", "adaln_bucket_batch", "adaln_plan_buckets",
    "adaln_max_dim", "adaln_launch_count", "adaln_status_string", "workspace",
    "adaln_bwd_noalloc", "adaln_noalloc_scratch_bytes", "adaln_pipeline_status",
    "adaln_fwd_gated", "adaln_fwd_gated_ragged", "adaln_bwd_gated", "adaln_bwd_gated_ragged",
    "adaln_bwd_gated_workspace_size", "adaln_bwd_gated_ragged_workspace_size",
    "adaln_balance_cv", "adaln_fit_cost", "adaln_fwd_rms", "adaln_fwd_rms_ragged",
    "adaln_bwd_rms", "adaln_bwd_rms_ragged", "adaln_fwd_ragged_indexed",
    "adaln_gate_residual_ragged_indexed", "adaln_bwd_ragged_indexed",
    "adaln_gate_residual_bwd_ragged_indexed",
]

ADALN_OK = 0
_DT = {torch.float32: 0, torch.bfloat16: 1}
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_I32 = ctypes.c_int32
_E = ctypes.c_int  # enums


class AdaLNError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = _lib.adaln_status_string(status).decode()
        super().__init__(f"{fn}: {msg} (status {status})")


def _load():
    path = _build.LIB
    if os.environ.get("ADALN_SKIP_BUILD") != "1":
        path = _build.build()
    if not os.path.exists(path):
        raise ImportError(f"AdaLN CUDA library not found at {path}; run the build first")
    lib = ctypes.CDLL(path)
    sig = {
        "adaln_status_string": (ctypes.c_char_p, [_E]),
        "adaln_max_dim": (_I64, [_E]),
        "adaln_launch_count": (ctypes.c_uint64, []),
        "adaln_pipeline_status": (ctypes.c_int, []),
        "adaln_fwd": (_E, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _E, _P]),
        "adaln_gate_residual": (_E, [_P, _P, _P, _P, _I64, _I64, _I64, _E, _P]),
        "adaln_bwd_workspace_size": (_SZ, [_I64, _I64, _I64, _E]),
        "adaln_bwd": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _E, _P]),
        "adaln_gate_residual_bwd_workspace_size": (_SZ, [_I64, _I64, _I64, _E]),
        "adaln_gate_residual_bwd": (_E, [_P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _E, _P]),
        "adaln_fwd_ragged": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _F, _E, _P]),
        "adaln_gate_residual_ragged": (_E, [_P, _P, _P, _P, _P, _P, _I64, _I64, _E, _P]),
        "adaln_bwd_ragged_workspace_size": (_SZ, [_P, _I64, _I64, _E]),
        "adaln_bwd_ragged": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _I64, _I64,
                                  _E, _P]),
        "adaln_gate_residual_bwd_ragged_workspace_size": (_SZ, [_P, _I64, _I64, _E]),
        "adaln_gate_residual_bwd_ragged": (_E, [_P, _P, _P, _P, _P, _P, _SZ, _P, _P, _I64, _I64,
                                                _E, _P]),
        "adaln_fwd_ragged_indexed": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                          _I64, _F, _E, _P]),
        "adaln_gate_residual_ragged_indexed": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                                    _I64, _E, _P]),
        "adaln_bwd_ragged_indexed": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _P,
                                          _P, _I64, _I64, _I64, _E, _P]),
        "adaln_gate_residual_bwd_ragged_indexed": (_E, [_P, _P, _P, _P, _P, _P, _SZ, _P, _P, _P,
                                                        _P, _I64, _I64, _I64, _E, _P]),
        "adaln_noalloc_scratch_bytes": (_SZ, []),
        "adaln_bwd_noalloc": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _E, _P]),
        "adaln_fwd_gated": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _E,
                                 _P]),
        "adaln_fwd_gated_ragged": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                        _F, _E, _P]),
        "adaln_bwd_gated_workspace_size": (_SZ, [_I64, _I64, _I64, _E]),
        "adaln_bwd_gated": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64,
                                 _I64, _E, _P]),
        "adaln_bwd_gated_ragged_workspace_size": (_SZ, [_P, _I64, _I64, _E]),
        "adaln_bwd_gated_ragged": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                        _P, _I64, _I64, _E, _P]),
        "adaln_bucket_batch": (_I64, [_I64, _I64, _I64, _I32]),
        "adaln_plan_buckets": (_E, [_P, _I64, _I64, _I64, _I32, _P, _P, _P, _P]),
        "adaln_fwd_rms": (_E, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _E, _P]),
        "adaln_fwd_rms_ragged": (_E, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _F, _E, _P]),
        "adaln_bwd_rms": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _E, _P]),
        "adaln_bwd_rms_ragged": (_E, [_P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _I64, _I64,
                                      _E, _P]),
        "adaln_balance_cv": (_E, [_P, _I64, _P, _P, _I64, _P, _I64, _I32, _P, _P, _P]),
        "adaln_fit_cost": (_E, [_P, _P, _P, _I64, ctypes.c_double, ctypes.c_double, _P, _P, _P,
                                _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib, path


_lib, lib_path = _load()


# ----------------------------------------------------------------------------- marshalling

def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("AdaLN tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}; use float32 or bfloat16") from None


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _check(fn: str, status: int):
    if status != ADALN_OK:
        raise AdaLNError(fn, status)


def _bnd(x: torch.Tensor):
    if x.dim() != 3:
        raise ValueError("dense AdaLN tensors are [B, N, D]")
    return x.shape[0], x.shape[1], x.shape[2]


def _host_offsets(offsets) -> np.ndarray:
    if isinstance(offsets, torch.Tensor):
        offsets = offsets.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))


def _hp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def adaln_status_string(status: int) -> str:
    return _lib.adaln_status_string(status).decode()


def adaln_max_dim(dtype: torch.dtype) -> int:
    return int(_lib.adaln_max_dim(_DT[dtype]))


def adaln_launch_count() -> int:
    return int(_lib.adaln_launch_count())


def adaln_pipeline_status() -> int:
    return int(_lib.adaln_pipeline_status())


def workspace(nbytes: int, device) -> torch.Tensor:
    """A caller-owned device buffer of at least nbytes (16-byte aligned)."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------- dense

def adaln_fwd(x, shift, scale, y, mean, rstd, eps: float, stream=None):
    B, N, D = _bnd(x)
    _check("adaln_fwd", _lib.adaln_fwd(_ptr(x), _ptr(shift), _ptr(scale), _ptr(y), _ptr(mean),
                                       _ptr(rstd), B, N, D, eps, _dt(x), _stream(stream)))


def adaln_gate_residual(r, z, gate, out, stream=None):
    B, N, D = _bnd(r)
    _check("adaln_gate_residual", _lib.adaln_gate_residual(
        _ptr(r), _ptr(z), _ptr(gate), _ptr(out), B, N, D, _dt(r), _stream(stream)))


def adaln_bwd_workspace_size(B: int, N: int, D: int, dtype: torch.dtype) -> int:
    return int(_lib.adaln_bwd_workspace_size(B, N, D, _DT[dtype]))


def adaln_bwd(x, mean, rstd, scale, dy, dx, d_scale, d_shift, ws, stream=None):
    B, N, D = _bnd(x)
    _check("adaln_bwd", _lib.adaln_bwd(
        _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dy), _ptr(dx), _ptr(d_scale),
        _ptr(d_shift), _ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0,
        B, N, D, _dt(x), _stream(stream)))


def adaln_gate_residual_bwd_workspace_size(B: int, N: int, D: int, dtype: torch.dtype) -> int:
    return int(_lib.adaln_gate_residual_bwd_workspace_size(B, N, D, _DT[dtype]))


def adaln_gate_residual_bwd(dout, z, gate, dz, d_gate, ws, stream=None):
    B, N, D = _bnd(dout)
    _check("adaln_gate_residual_bwd", _lib.adaln_gate_residual_bwd(
        _ptr(dout), _ptr(z), _ptr(gate), _ptr(dz), _ptr(d_gate), _ptr(ws),
        ws.numel() * ws.element_size() if ws is not None else 0, B, N, D, _dt(dout),
        _stream(stream)))


def adaln_noalloc_scratch_bytes() -> int:
    return int(_lib.adaln_noalloc_scratch_bytes())


def adaln_bwd_noalloc(x, mean, rstd, scale, dy, dx, d_scale, d_shift, stream=None):
    """adaln_bwd on the library's built-in scratch buffer: for callers that cannot
    allocate device memory.  Calls must not overlap on the GPU (they share it)."""
    B, N, D = _bnd(x)
    _check("adaln_bwd_noalloc", _lib.adaln_bwd_noalloc(
        _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dy), _ptr(dx), _ptr(d_scale),
        _ptr(d_shift), B, N, D, _dt(x), _stream(stream)))


# ----------------------------------------------------------------------------- ragged

def _rows_d(x):
    if x.dim() != 2:
        raise ValueError("packed AdaLN tensors are [rows, D]")
    return x.shape[1]


def adaln_fwd_ragged(x, shift, scale, y, mean, rstd, offsets_host, offsets_dev, eps: float,
                     stream=None):
    oh = _host_offsets(offsets_host)
    _check("adaln_fwd_ragged", _lib.adaln_fwd_ragged(
        _ptr(x), _ptr(shift), _ptr(scale), _ptr(y), _ptr(mean), _ptr(rstd), _hp(oh),
        _ptr(offsets_dev), len(oh) - 1, _rows_d(x), eps, _dt(x), _stream(stream)))


def adaln_gate_residual_ragged(r, z, gate, out, offsets_host, offsets_dev, stream=None):
    oh = _host_offsets(offsets_host)
    _check("adaln_gate_residual_ragged", _lib.adaln_gate_residual_ragged(
        _ptr(r), _ptr(z), _ptr(gate), _ptr(out), _hp(oh), _ptr(offsets_dev), len(oh) - 1,
        _rows_d(r), _dt(r), _stream(stream)))


def adaln_bwd_ragged_workspace_size(offsets_host, D: int, dtype: torch.dtype) -> int:
    oh = _host_offsets(offsets_host)
    return int(_lib.adaln_bwd_ragged_workspace_size(_hp(oh), len(oh) - 1, D, _DT[dtype]))


def adaln_bwd_ragged(x, mean, rstd, scale, dy, dx, d_scale, d_shift, ws, offsets_host,
                     offsets_dev, stream=None):
    oh = _host_offsets(offsets_host)
    _check("adaln_bwd_ragged", _lib.adaln_bwd_ragged(
        _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dy), _ptr(dx), _ptr(d_scale),
        _ptr(d_shift), _ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0,
        _hp(oh), _ptr(offsets_dev), len(oh) - 1, _rows_d(x), _dt(x), _stream(stream)))


def _host_index(mod_index) -> np.ndarray:
    if isinstance(mod_index, torch.Tensor):
        mod_index = mod_index.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(mod_index, dtype=np.int32))


def adaln_fwd_ragged_indexed(x, shift, scale, y, mean, rstd, offsets_host, offsets_dev,
                             mod_index_host, mod_index_dev, eps: float, stream=None):
    """Ragged forward where segment k uses modulation row mod_index[k] of shift/scale
    [num_mod_rows, D]."""
    oh, mi = _host_offsets(offsets_host), _host_index(mod_index_host)
    _check("adaln_fwd_ragged_indexed", _lib.adaln_fwd_ragged_indexed(
        _ptr(x), _ptr(shift), _ptr(scale), _ptr(y), _ptr(mean), _ptr(rstd), _hp(oh),
        _ptr(offsets_dev), _hp(mi), _ptr(mod_index_dev), len(oh) - 1, shift.shape[0], _rows_d(x),
        eps, _dt(x), _stream(stream)))


def adaln_gate_residual_ragged_indexed(r, z, gate, out, offsets_host, offsets_dev,
                                       mod_index_host, mod_index_dev, stream=None):
    oh, mi = _host_offsets(offsets_host), _host_index(mod_index_host)
    _check("adaln_gate_residual_ragged_indexed", _lib.adaln_gate_residual_ragged_indexed(
        _ptr(r), _ptr(z), _ptr(gate), _ptr(out), _hp(oh), _ptr(offsets_dev), _hp(mi),
        _ptr(mod_index_dev), len(oh) - 1, gate.shape[0], _rows_d(r), _dt(r), _stream(stream)))


def adaln_bwd_ragged_indexed(x, mean, rstd, scale, dy, dx, d_scale, d_shift, ws, offsets_host,
                             offsets_dev, mod_index_host, mod_index_dev, stream=None):
    """d_scale/d_shift [num_mod_rows, D]: row m sums every segment with mod_index == m."""
    oh, mi = _host_offsets(offsets_host), _host_index(mod_index_host)
    _check("adaln_bwd_ragged_indexed", _lib.adaln_bwd_ragged_indexed(
        _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dy), _ptr(dx), _ptr(d_scale),
        _ptr(d_shift), _ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0,
        _hp(oh), _ptr(offsets_dev), _hp(mi), _ptr(mod_index_dev), len(oh) - 1, scale.shape[0],
        _rows_d(x), _dt(x), _stream(stream)))


def adaln_gate_residual_bwd_ragged_indexed(dout, z, gate, dz, d_gate, ws, offsets_host,
                                           offsets_dev, mod_index_host, mod_index_dev,
                                           stream=None):
    oh, mi = _host_offsets(offsets_host), _host_index(mod_index_host)
    _check("adaln_gate_residual_bwd_ragged_indexed",
           _lib.adaln_gate_residual_bwd_ragged_indexed(
               _ptr(dout), _ptr(z), _ptr(gate), _ptr(dz), _ptr(d_gate), _ptr(ws),
               ws.numel() * ws.element_size() if ws is not None else 0, _hp(oh),
               _ptr(offsets_dev), _hp(mi), _ptr(mod_index_dev), len(oh) - 1, gate.shape[0],
               _rows_d(dout), _dt(dout), _stream(stream)))


def adaln_gate_residual_bwd_ragged_workspace_size(offsets_host, D: int,
                                                  dtype: torch.dtype) -> int:
    oh = _host_offsets(offsets_host)
    return int(_lib.adaln_gate_residual_bwd_ragged_workspace_size(_hp(oh), len(oh) - 1, D,
                                                                  _DT[dtype]))


def adaln_gate_residual_bwd_ragged(dout, z, gate, dz, d_gate, ws, offsets_host, offsets_dev,
                                   stream=None):
    oh = _host_offsets(offsets_host)
    _check("adaln_gate_residual_bwd_ragged", _lib.adaln_gate_residual_bwd_ragged(
        _ptr(dout), _ptr(z), _ptr(gate), _ptr(dz), _ptr(d_gate), _ptr(ws),
        ws.numel() * ws.element_size() if ws is not None else 0, _hp(oh), _ptr(offsets_dev),
        len(oh) - 1, _rows_d(dout), _dt(dout), _stream(stream)))


# ----------------------------------------------------------------------------- RMSNorm modulation

def adaln_fwd_rms(x, shift, scale, y, rstd, eps: float, stream=None):
    B, N, D = _bnd(x)
    _check("adaln_fwd_rms", _lib.adaln_fwd_rms(
        _ptr(x), _ptr(shift), _ptr(scale), _ptr(y), _ptr(rstd), B, N, D, eps, _dt(x),
        _stream(stream)))


def adaln_fwd_rms_ragged(x, shift, scale, y, rstd, offsets_host, offsets_dev, eps: float,
                         stream=None):
    oh = _host_offsets(offsets_host)
    _check("adaln_fwd_rms_ragged", _lib.adaln_fwd_rms_ragged(
        _ptr(x), _ptr(shift), _ptr(scale), _ptr(y), _ptr(rstd), _hp(oh), _ptr(offsets_dev),
        len(oh) - 1, _rows_d(x), eps, _dt(x), _stream(stream)))


def adaln_bwd_rms(x, rstd, scale, dy, dx, d_scale, d_shift, ws, stream=None):
    B, N, D = _bnd(x)
    _check("adaln_bwd_rms", _lib.adaln_bwd_rms(
        _ptr(x), _ptr(rstd), _ptr(scale), _ptr(dy), _ptr(dx), _ptr(d_scale), _ptr(d_shift),
        _ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0, B, N, D, _dt(x),
        _stream(stream)))


def adaln_bwd_rms_ragged(x, rstd, scale, dy, dx, d_scale, d_shift, ws, offsets_host,
                         offsets_dev, stream=None):
    oh = _host_offsets(offsets_host)
    _check("adaln_bwd_rms_ragged", _lib.adaln_bwd_rms_ragged(
        _ptr(x), _ptr(rstd), _ptr(scale), _ptr(dy), _ptr(dx), _ptr(d_scale), _ptr(d_shift),
        _ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0, _hp(oh),
        _ptr(offsets_dev), len(oh) - 1, _rows_d(x), _dt(x), _stream(stream)))


# ----------------------------------------------------------------------------- fused gated chain

def adaln_fwd_gated(x, shift, scale, gate, r, out, y, mean, rstd, eps: float, stream=None):
    """out = r + gate * y with y = LN(x) * (1 + scale) + shift; y may be None."""
    B, N, D = _bnd(x)
    _check("adaln_fwd_gated", _lib.adaln_fwd_gated(
        _ptr(x), _ptr(shift), _ptr(scale), _ptr(gate), _ptr(r), _ptr(out), _ptr(y), _ptr(mean),
        _ptr(rstd), B, N, D, eps, _dt(x), _stream(stream)))


def adaln_fwd_gated_ragged(x, shift, scale, gate, r, out, y, mean, rstd, offsets_host,
                           offsets_dev, eps: float, stream=None):
    oh = _host_offsets(offsets_host)
    _check("adaln_fwd_gated_ragged", _lib.adaln_fwd_gated_ragged(
        _ptr(x), _ptr(shift), _ptr(scale), _ptr(gate), _ptr(r), _ptr(out), _ptr(y), _ptr(mean),
        _ptr(rstd), _hp(oh), _ptr(offsets_dev), len(oh) - 1, _rows_d(x), eps, _dt(x),
        _stream(stream)))


def adaln_bwd_gated_workspace_size(B: int, N: int, D: int, dtype: torch.dtype) -> int:
    return int(_lib.adaln_bwd_gated_workspace_size(B, N, D, _DT[dtype]))


def adaln_bwd_gated(x, mean, rstd, shift, scale, gate, dout, dx, d_scale, d_shift, d_gate, ws,
                    stream=None):
    B, N, D = _bnd(x)
    _check("adaln_bwd_gated", _lib.adaln_bwd_gated(
        _ptr(x), _ptr(mean), _ptr(rstd), _ptr(shift), _ptr(scale), _ptr(gate), _ptr(dout),
        _ptr(dx), _ptr(d_scale), _ptr(d_shift), _ptr(d_gate), _ptr(ws),
        ws.numel() * ws.element_size() if ws is not None else 0, B, N, D, _dt(x),
        _stream(stream)))


def adaln_bwd_gated_ragged_workspace_size(offsets_host, D: int, dtype: torch.dtype) -> int:
    oh = _host_offsets(offsets_host)
    return int(_lib.adaln_bwd_gated_ragged_workspace_size(_hp(oh), len(oh) - 1, D, _DT[dtype]))


def adaln_bwd_gated_ragged(x, mean, rstd, shift, scale, gate, dout, dx, d_scale, d_shift, d_gate,
                           ws, offsets_host, offsets_dev, stream=None):
    oh = _host_offsets(offsets_host)
    _check("adaln_bwd_gated_ragged", _lib.adaln_bwd_gated_ragged(
        _ptr(x), _ptr(mean), _ptr(rstd), _ptr(shift), _ptr(scale), _ptr(gate), _ptr(dout),
        _ptr(dx), _ptr(d_scale), _ptr(d_shift), _ptr(d_gate), _ptr(ws),
        ws.numel() * ws.element_size() if ws is not None else 0, _hp(oh), _ptr(offsets_dev),
        len(oh) - 1, _rows_d(x), _dt(x), _stream(stream)))


# ----------------------------------------------------------------------------- planner

def adaln_bucket_batch(S: int, M_mem: int, M_comp: int, p: int) -> int:
    return int(_lib.adaln_bucket_batch(S, M_mem, M_comp, p))


def adaln_plan_buckets(lengths: Sequence[int], M_mem: int, M_comp: int, p: int):
    """Returns (bucket_of_seq, order, bucket_start) as int64 numpy arrays."""
    L = np.ascontiguousarray(np.asarray(lengths, dtype=np.int64))
    n = len(L)
    bos = np.empty(n, dtype=np.int64)
    order = np.empty(n, dtype=np.int64)
    starts = np.empty(n + 1, dtype=np.int64)
    nb = np.zeros(1, dtype=np.int64)
    _check("adaln_plan_buckets", _lib.adaln_plan_buckets(
        _hp(L), n, M_mem, M_comp, p, _hp(bos), _hp(order), _hp(starts), _hp(nb)))
    return bos, order, starts[: int(nb[0]) + 1].copy()


def adaln_balance_cv(lengths: Sequence[int], order, bucket_start, deal, ranks: int, p: int):
    """(mean CV, mean max/mean, full steps) of the per-rank compute load of a bucket
    plan dealt to `ranks` ranks in the order `deal`."""
    L = np.ascontiguousarray(np.asarray(lengths, dtype=np.int64))
    o = np.ascontiguousarray(np.asarray(order, dtype=np.int64))
    bs = np.ascontiguousarray(np.asarray(bucket_start, dtype=np.int64))
    d = np.ascontiguousarray(np.asarray(deal, dtype=np.int64))
    cv, mm, steps = ctypes.c_double(), ctypes.c_double(), ctypes.c_int64()
    _check("adaln_balance_cv", _lib.adaln_balance_cv(
        _hp(L), len(L), _hp(o), _hp(bs), len(bs) - 1, _hp(d), ranks, p, ctypes.byref(cv),
        ctypes.byref(mm), ctypes.byref(steps)))
    return cv.value, mm.value, steps.value


def adaln_fit_cost(B, S, t, p_lo: float = 0.25, p_hi: float = 4.0):
    """Least-squares (a, b, p, rss) of t = a + b * B * S^p."""
    Bv = np.ascontiguousarray(np.asarray(B, dtype=np.int64))
    Sv = np.ascontiguousarray(np.asarray(S, dtype=np.int64))
    tv = np.ascontiguousarray(np.asarray(t, dtype=np.float64))
    a, b, p, rss = (ctypes.c_double() for _ in range(4))
    _check("adaln_fit_cost", _lib.adaln_fit_cost(
        _hp(Bv), _hp(Sv), tv.ctypes.data_as(ctypes.c_void_p), len(tv), p_lo, p_hi,
        ctypes.byref(a), ctypes.byref(b), ctypes.byref(p), ctypes.byref(rss)))
    return a.value, b.value, p.value, rss.value
