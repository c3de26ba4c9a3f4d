"""Seeded synthetic inputs for the AdaLN modulation operator.

This module only draws random numbers and lays them out; it holds none of the
operator's arithmetic and none of the planner's.  Both the CUDA path and the
fp64 oracle are fed from it.

Recipe (all draws seeded; nothing is read from disk):

* Every tensor is drawn by its own ``torch.Generator`` seeded from
  (seed, tensor name[, sequence index]) through SHA-256, so a tensor's
  contents do not depend on the order tensors are drawn in.  ``device="cpu"``
  gives the same bytes on every machine; large workloads are drawn on the GPU
  (Philox), which is deterministic on a given device/torch build.
* Values are drawn in fp32 N(0, std) and rounded once (round-to-nearest-even)
  to the I/O dtype.  Activations (x, residual r, sublayer output z, upstream
  gradient dy) have std 1; the modulation rows shift/scale/gate have std 0.1.
* Outlier tokens (the long-video workload): ceil(1% of the rows), picked by a
  seeded permutation, multiplied by 20 in fp32 before rounding.
* Ragged lengths: floor(20%) of the sequences fixed at the minimum length
  (image-like), picked by a seeded permutation; the rest
  floor(exp(U(ln lo, ln hi))) clamped to [lo, hi].
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, List, Optional, Sequence

import torch

__all__ = ["Spec", "SPECS", "spec", "randn", "ragged_lengths", "make_inputs",
           "make_packed_inputs", "DTYPES"]

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Spec:
    """One workload: segment lengths (rows per segment), D, I/O dtype, eps."""
    name: str
    dtype: str
    D: int
    eps: float
    seg_lengths: tuple
    outlier_frac: float = 0.0
    outlier_mult: float = 20.0
    description: str = ""

    @property
    def rows(self) -> int:
        return int(sum(self.seg_lengths))

    @property
    def nseg(self) -> int:
        return len(self.seg_lengths)

    def offsets(self) -> List[int]:
        o = [0]
        for s in self.seg_lengths:
            o.append(o[-1] + int(s))
        return o


# Planner constants of the ragged mixed-mode workload.
RAGGED_M_MEM = 262_144
RAGGED_M_COMP = 1 << 30
RAGGED_P = 2
RAGGED_NSEQ = 256
RAGGED_LO, RAGGED_HI = 256, 32_768
RAGGED_D = 3072

SPECS: Dict[str, Spec] = {
    "tiny": Spec("tiny", "f32", 128, 1e-6, (256, 256),
                 description="B=2, N=256, D=128, fp32 I/O"),
    "dit": Spec("dit", "bf16", 1152, 1e-6, (1024,) * 8,
                description="DiT-XL-like block norm: B=8, N=1024 (32x32 patches), D=1152, bf16 I/O"),
    "wan": Spec("wan", "bf16", 5120, 1e-6, (75_600,), outlier_frac=0.01,
                description="Wan-14B-scale video sequence: B=1, N=75,600, D=5120, bf16 I/O, "
                            "1% outlier rows x20"),
    "mmdit": Spec("mmdit", "bf16", 3072, 1e-6, (512,) * 4 + (4096,) * 4,
                  description="MMDiT joint block: B=4, text N=512 + video N=4096, D=3072, "
                              "both streams packed into one launch (8 segments)"),
    # not one of the five configurations: rows at the boundary's D limit, which take
    # the wide-row kernels
    "wide": Spec("wide", "bf16", 16384, 1e-6, (8192,),
                 description="rows at the D limit: B=1, N=8192, D=16384, bf16 I/O"),
}


def spec(name: str) -> Spec:
    return SPECS[name]


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def randn(shape, seed: int, tag: str, device="cpu", std: float = 1.0) -> torch.Tensor:
    """fp32 N(0, std) draw from a generator private to (seed, tag)."""
    t = torch.randn(tuple(shape), generator=_gen(device, seed, tag), device=device,
                    dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def ragged_lengths(seed: int = 0, n: int = RAGGED_NSEQ, lo: int = RAGGED_LO,
                   hi: int = RAGGED_HI, fixed_frac: float = 0.2) -> List[int]:
    """Sequence lengths of the ragged mixed-mode workload (drawn on the CPU)."""
    g = _gen("cpu", seed, "ragged-lengths")
    u = torch.rand(n, generator=g, dtype=torch.float64)
    logs = math.log(lo) + u * (math.log(hi) - math.log(lo))
    L = [min(hi, max(lo, int(math.floor(math.exp(float(v)))))) for v in logs]
    nfix = int(math.floor(fixed_frac * n))
    pick = torch.randperm(n, generator=_gen("cpu", seed, "ragged-fixed"))[:nfix]
    for i in pick.tolist():
        L[i] = lo
    return L


def _outlier_rows(spec_: Spec, seed: int) -> torch.Tensor:
    rows = spec_.rows
    k = int(math.ceil(spec_.outlier_frac * rows))
    return torch.randperm(rows, generator=_gen("cpu", seed, spec_.name, "outliers"))[:k]


def make_inputs(spec_: Spec, seed: int = 0, device="cpu", draw_device=None,
                tensors: Sequence[str] = ("x", "shift", "scale", "gate", "r", "z", "dy")
                ) -> Dict[str, torch.Tensor]:
    """Dense/packed inputs of a Spec: activations [rows, D], modulation [nseg, D].

    ``draw_device`` is where the random numbers are drawn (default: ``device``);
    drawing on the CPU and moving gives bytes identical on every machine.
    """
    draw = draw_device if draw_device is not None else device
    dt = DTYPES[spec_.dtype]
    out = {}
    for name in tensors:
        if name in ("shift", "scale", "gate"):
            t = randn((spec_.nseg, spec_.D), seed, f"{spec_.name}/{name}", draw, 0.1)
        else:
            t = randn((spec_.rows, spec_.D), seed, f"{spec_.name}/{name}", draw)
            if name == "x" and spec_.outlier_frac > 0:
                idx = _outlier_rows(spec_, seed).to(t.device)
                t[idx] *= spec_.outlier_mult
        out[name] = t.to(dt).to(device)
        del t
    return out


def make_packed_inputs(lengths: Sequence[int], order: Sequence[int], D: int, dtype: str,
                       seed: int = 0, device="cpu", draw_device=None,
                       tensors: Sequence[str] = ("x", "shift", "scale", "gate", "r", "z", "dy"),
                       tag: str = "ragged") -> Dict[str, torch.Tensor]:
    """Per-sequence inputs packed in ``order`` (e.g. a planner's packing order).

    Sequence i's rows and modulation rows are drawn from generators private to
    (seed, tag, tensor, i), so its values do not depend on where it is packed.
    Activations come back as [sum(lengths), D]; modulation as [len(order), D]
    with row j belonging to sequence order[j].
    """
    draw = draw_device if draw_device is not None else device
    dt = DTYPES[dtype]
    total = int(sum(int(lengths[i]) for i in order))
    out = {}
    for name in tensors:
        if name in ("shift", "scale", "gate"):
            t = torch.empty((len(order), D), dtype=dt, device=device)
            for j, i in enumerate(order):
                t[j] = randn((D,), seed, f"{tag}/{name}/{i}", draw, 0.1).to(dt).to(device)
        else:
            t = torch.empty((total, D), dtype=dt, device=device)
            pos = 0
            for i in order:
                S = int(lengths[i])
                t[pos:pos + S] = randn((S, D), seed, f"{tag}/{name}/{i}", draw).to(dt).to(device)
                pos += S
        out[name] = t
    return out
