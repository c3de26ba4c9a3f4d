"""Load-balance simulation of the bucket planner (host only).

Compares equal-tokens batching (only B * S <= M_mem binds) with the dual
constraint of the "AdaptiveLoad" summary, section 2.A, on ragged length
draws shaped like the mixed image/video workload: both plans come from
adaln_plan_buckets, are dealt to R data-parallel ranks in a seeded shuffled
order, and adaln_balance_cv reports the coefficient of variation of the
per-rank compute load (sum of S^p per bucket) the summary's section 4
measures ("Eficiencia del Equilibrio de Carga").

    python -m modulation_adaln_fwd_gb300.balance [--draws 16] [--ranks 8 16]

Prints one JSON line.  Run from the repository root (the length draws come
from the workloads module there).
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import adaln_balance_cv, adaln_plan_buckets

EQUAL_TOKENS_M_COMP = 1 << 62  # so large that only the memory constraint binds


def simulate(lengths, M_mem: int, M_comp: int, p: int, ranks: int, seed: int = 0):
    _, order, starts = adaln_plan_buckets(lengths, M_mem, M_comp, p)
    nb = len(starts) - 1
    deal = np.random.default_rng(seed).permutation(nb)
    cv, max_over_mean, steps = adaln_balance_cv(lengths, order, starts, deal, ranks, p)
    tokens = [int(np.sum(np.asarray(lengths)[order[starts[b]:starts[b + 1]]])) for b in range(nb)]
    return {"buckets": nb, "steps": steps, "compute_cv": round(cv, 4),
            "compute_max_over_mean": round(max_over_mean, 4),
            "mean_tokens_per_bucket": round(float(np.mean(tokens)), 1)}


def main():
    import workloads
    ap = argparse.ArgumentParser()
    ap.add_argument("--draws", type=int, default=16, help="seeded draws of 256 lengths each")
    ap.add_argument("--ranks", type=int, nargs="+", default=[8, 16])
    ap.add_argument("--seed", type=int, default=0, help="seed of the dealing order")
    args = ap.parse_args()
    L = []
    for s in range(args.draws):
        L += workloads.ragged_lengths(s)
    res = {"sequences": len(L), "M_mem": workloads.RAGGED_M_MEM, "M_comp": workloads.RAGGED_M_COMP,
           "p": workloads.RAGGED_P, "ranks": {}}
    for R in args.ranks:
        res["ranks"][R] = {
            "equal_tokens": simulate(L, workloads.RAGGED_M_MEM, EQUAL_TOKENS_M_COMP,
                                     workloads.RAGGED_P, R, args.seed),
            "dual_constraint": simulate(L, workloads.RAGGED_M_MEM, workloads.RAGGED_M_COMP,
                                        workloads.RAGGED_P, R, args.seed)}
    print(json.dumps(res))


if __name__ == "__main__":
    main()
