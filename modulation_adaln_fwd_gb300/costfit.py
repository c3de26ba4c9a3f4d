"""Cost-model fit on measured per-bucket step times.

The "AdaptiveLoad" summary, section 2.A, calibrates the exponent p and the
compute budget M_comp of its dual constraint by fitting t = a + b * B * S^p
to step times measured on benchmark shapes.  This tool measures a synthetic
stand-in step on the GPU for every bucket that the planner makes of the ragged
workload's lengths, and fits the model with adaln_fit_cost:

  adaln   the fused AdaLN chain of the bucket (one forward and one backward
          call): its cost is linear in the tokens B * S, so p comes out near 1;
  scores  the same plus a B x S x S attention-score product per bucket
          (batched bf16 matmul with a 64-wide head, via torch): the stand-in
          for the quadratic attention term, so p comes out above 1.
A bucket's shape is (B, S) = (its sequence count, its mean length).

    python -m modulation_adaln_fwd_gb300.costfit [--reps 5]

Prints one JSON line.  Needs a GPU; run from the repository root.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import (adaln_bwd_gated_ragged, adaln_bwd_gated_ragged_workspace_size,
               adaln_fit_cost, adaln_fwd_gated_ragged, adaln_plan_buckets, workspace)

HEAD = 64


def _bucket_inputs(lengths, D, dev, gen):
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    rows, nseg = int(off[-1]), len(lengths)
    bf = torch.bfloat16
    t = lambda *shape: torch.randn(*shape, device=dev, generator=gen).to(bf)
    inp = dict(x=t(rows, D), r=t(rows, D), dy=t(rows, D), shift=0.1 * t(nseg, D),
               scale=0.1 * t(nseg, D), gate=0.1 * t(nseg, D))
    out = dict(out=torch.empty(rows, D, dtype=bf, device=dev),
               dx=torch.empty(rows, D, dtype=bf, device=dev),
               mean=torch.empty(rows, device=dev), rstd=torch.empty(rows, device=dev),
               d_scale=torch.empty(nseg, D, device=dev), d_shift=torch.empty(nseg, D, device=dev),
               d_gate=torch.empty(nseg, D, device=dev))
    ws = workspace(adaln_bwd_gated_ragged_workspace_size(off, D, bf), dev)
    return off, torch.from_numpy(off).to(dev), inp, out, ws


def measure(lengths_all, M_mem, M_comp, p, D=3072, reps=5, seed=0):
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    _, order, starts = adaln_plan_buckets(lengths_all, M_mem, M_comp, p)
    rows = []
    for b in range(len(starts) - 1):
        lens = [int(lengths_all[i]) for i in order[starts[b]:starts[b + 1]]]
        # a bucket mixes lengths: its shape is (count, mean length), so that B * S is
        # the bucket's token count
        B = len(lens)
        S = int(round(sum(lens) / B))
        off, offd, i, o, ws = _bucket_inputs(lens, D, dev, gen)
        q = torch.randn(B, S, HEAD, device=dev, generator=gen).to(torch.bfloat16)
        k = torch.randn(B, HEAD, S, device=dev, generator=gen).to(torch.bfloat16)

        def adaln():
            adaln_fwd_gated_ragged(i["x"], i["shift"], i["scale"], i["gate"], i["r"], o["out"],
                                   None, o["mean"], o["rstd"], off, offd, 1e-6)
            adaln_bwd_gated_ragged(i["x"], o["mean"], o["rstd"], i["shift"], i["scale"],
                                   i["gate"], i["dy"], o["dx"], o["d_scale"], o["d_shift"],
                                   o["d_gate"], ws, off, offd)
        times = {}
        for name, fn in (("adaln", adaln), ("scores", lambda: (adaln(), torch.bmm(q, k)))):
            fn()
            ts = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                ts.append((e0, e1))
            torch.cuda.synchronize()
            times[name] = sorted(a.elapsed_time(c) for a, c in ts)[reps // 2]
        rows.append((B, S, times["adaln"], times["scores"]))
        del i, o, ws, q, k
    return rows


def main():
    import workloads
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=5)
    args = ap.parse_args()
    L = workloads.ragged_lengths(0)
    rows = measure(L, workloads.RAGGED_M_MEM, workloads.RAGGED_M_COMP, workloads.RAGGED_P,
                   reps=args.reps)
    B = [r[0] for r in rows]
    S = [r[1] for r in rows]
    res = {"buckets": len(rows), "model": "t_ms = a + b * B * S^p", "fits": {}}
    for j, name in ((2, "adaln"), (3, "scores")):
        a, b, p, rss = adaln_fit_cost(B, S, [r[j] for r in rows])
        t = np.array([r[j] for r in rows])
        res["fits"][name] = {"a_ms": a, "b_ms": b, "p": round(p, 4),
                             "rel_rms_residual": float(np.sqrt(rss / len(t)) / np.mean(t))}
    res["per_bucket"] = [{"B": r[0], "S": r[1], "adaln_ms": round(r[2], 4),
                          "scores_ms": round(r[3], 4)} for r in rows]
    print(json.dumps(res))


if __name__ == "__main__":
    main()
