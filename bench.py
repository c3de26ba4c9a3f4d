"""Benchmark of the AdaLN modulation chain on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
    adaln_fwd -> adaln_gate_residual -> adaln_bwd -> adaln_gate_residual_bwd
(the ragged workload also runs the host bucket planner and one call per op and
bucket).  Inputs are resident in HBM when the timed region starts; the
end-to-end leg ("e2e") instead copies every input from pinned host memory and
every output back inside the timed region, with uploads, kernels and downloads
pipelined on three streams.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload wan]
    python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent
replica of the workload (the path has no cross-rank exchange); the job value
is the tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "AdaLN fwd+bwd tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"

WORKLOADS = {
    "wan": "Wan-14B-scale long video sequence: B=1, N=75,600, D=5120, bf16 I/O, fp32 stats",
    "dit": "DiT-XL-like block norm: B=8, N=1024, D=1152, bf16 I/O, fp32 stats",
    "mmdit": "MMDiT joint block: B=4, text N=512 + video N=4096, D=3072, bf16, one launch",
    "ragged": "Ragged mixed-mode packing: 256 sequences, log-uniform [256, 32768], D=3072, "
              "bucketed by B_shape (M_mem=262144, M_comp=2^30, p=2)",
    "tiny": "Tiny fp32: B=2, N=256, D=128",
    "wide": "Rows at the D limit (not one of the five configurations): B=1, N=8192, D=16384, "
            "bf16; the wide-row kernels",
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="wan", choices=sorted(WORKLOADS))
    p.add_argument("--chain", default="split", choices=["split", "fused", "rms"],
                   help="split: fwd -> gate -> bwd -> gate_bwd (z an input); fused: the gated "
                        "residual applied to y itself, one forward and one backward call; rms: "
                        "the RMSNorm modulation forward and backward")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--rows", type=int, default=None,
                   help="dense workloads only: a smaller N per sample (for profiler captures)")
    p.add_argument("--no-ragged", action="store_true",
                   help="with the default Wan workload, skip the ragged mixed-mode workload "
                        "that is otherwise measured after it and reported under 'ragged'")
    p.add_argument("--no-graph", action="store_true",
                   help="launch every op from the host in each timed step instead of "
                        "replaying the step's launches from a CUDA graph")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mp = json.load(f)
        return float(mp["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def job_value(local_ms, tokens_per_step, steps, world, dist=None, device=None):
    """Whole-job throughput of `world` replicas: every rank processes
    tokens_per_step per step; the job time is the slowest rank's (barrier, then a
    max-reduction).  Returns (tokens/s, job ms)."""
    import torch
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    if dist is not None:
        dist.barrier()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    job_ms = float(t.item())
    return world * tokens_per_step * steps / (job_ms / 1e3), job_ms


# ----------------------------------------------------------------------------- workload setup

class Work:
    """Device tensors of one workload and the list of ragged groups to run."""

    def __init__(self, name, device, seed=0, rows=None, chain="split"):
        import torch
        import workloads
        import modulation_adaln_fwd_gb300 as A
        self.name = name
        self.chain = chain
        self.ops = {"split": OPS, "fused": FUSED_OPS, "rms": RMS_OPS}[chain]
        self.A = A
        self.device = device
        if name == "ragged":
            L = workloads.ragged_lengths(seed)
            self.lengths = L
            bos, order, starts = A.adaln_plan_buckets(L, workloads.RAGGED_M_MEM,
                                                      workloads.RAGGED_M_COMP, workloads.RAGGED_P)
            self.order, self.starts = order.tolist(), starts.tolist()
            D = workloads.RAGGED_D
            inp = workloads.make_packed_inputs(L, self.order, D, "bf16", seed=seed, device=device,
                                               draw_device=device)
            self.dtype_name, self.eps = "bf16", 1e-6
            groups = []
            row = 0
            for b in range(len(self.starts) - 1):
                lens = [L[i] for i in self.order[self.starts[b]:self.starts[b + 1]]]
                off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
                groups.append((row, self.starts[b], off))
                row += int(off[-1])
            self.groups = groups
            self.dense = None
        else:
            s = workloads.spec(name)
            if rows is not None and name != "mmdit":
                import dataclasses
                s = dataclasses.replace(s, seg_lengths=(int(rows),) * s.nseg)
            inp = workloads.make_inputs(s, seed=seed, device=device,
                                        draw_device="cpu" if s.rows * s.D < 50_000_000 else device)
            self.dtype_name, self.eps = s.dtype, s.eps
            if name == "mmdit":
                self.groups = [(0, 0, np.asarray(s.offsets(), dtype=np.int64))]
                self.dense = None
            else:
                self.groups = None
                self.dense = (s.nseg, s.seg_lengths[0])
        self.inp = inp
        x = inp["x"]
        self.rows, self.D = x.shape
        self.nseg = inp["shift"].shape[0]
        self.E = x.element_size()
        dt = x.dtype
        self.out = dict(
            y=torch.empty_like(x), out=torch.empty_like(x), dx=torch.empty_like(x),
            dz=torch.empty_like(x),
            mean=torch.empty(self.rows, device=device), rstd=torch.empty(self.rows, device=device),
            d_scale=torch.empty((self.nseg, self.D), device=device),
            d_shift=torch.empty((self.nseg, self.D), device=device),
            d_gate=torch.empty((self.nseg, self.D), device=device))
        if self.dense:
            B, N = self.dense
            ws = max(A.adaln_bwd_workspace_size(B, N, self.D, dt),
                     A.adaln_gate_residual_bwd_workspace_size(B, N, self.D, dt))
        else:
            ws = 16
            self.offdev = []
            for (_, _, off) in self.groups:
                ws = max(ws, A.adaln_bwd_ragged_workspace_size(off, self.D, dt),
                         A.adaln_gate_residual_bwd_ragged_workspace_size(off, self.D, dt))
                self.offdev.append(torch.from_numpy(off).to(device))
        self.ws = A.workspace(ws, device)

    # bytes each op must move per launch (what the method reads and writes once)
    def algorithmic_bytes(self):
        R, D, E, S = self.rows, self.D, self.E, self.nseg
        return dict(
            fwd=R * (2 * D * E + 8) + S * 2 * D * E,
            gate=R * 3 * D * E + S * D * E,
            bwd=R * (3 * D * E + 8) + S * D * (E + 8),
            gate_bwd=R * 3 * D * E + S * D * (E + 4),
            # fused chain (y not written): read x, r, write out; read x, dout, write dx
            fwd_gated=R * (3 * D * E + 8) + S * 3 * D * E,
            bwd_gated=R * (3 * D * E + 8) + S * D * (3 * E + 12),
            # RMSNorm: rstd only
            fwd_rms=R * (2 * D * E + 4) + S * 2 * D * E,
            bwd_rms=R * (3 * D * E + 4) + S * D * (E + 8))

    def run_op(self, op, inp=None, out=None):
        A, i, o = self.A, inp or self.inp, out or self.out
        if self.dense:
            B, N = self.dense
            D = self.D
            v = lambda t: t.view(B, N, D)
            if op == "fwd":
                A.adaln_fwd(v(i["x"]), i["shift"], i["scale"], v(o["y"]), o["mean"], o["rstd"],
                            self.eps)
            elif op == "gate":
                A.adaln_gate_residual(v(i["r"]), v(i["z"]), i["gate"], v(o["out"]))
            elif op == "bwd":
                A.adaln_bwd(v(i["x"]), o["mean"], o["rstd"], i["scale"], v(i["dy"]), v(o["dx"]),
                            o["d_scale"], o["d_shift"], self.ws)
            elif op == "gate_bwd":
                A.adaln_gate_residual_bwd(v(i["dy"]), v(i["z"]), i["gate"], v(o["dz"]),
                                          o["d_gate"], self.ws)
            elif op == "fwd_rms":
                A.adaln_fwd_rms(v(i["x"]), i["shift"], i["scale"], v(o["y"]), o["rstd"], self.eps)
            elif op == "bwd_rms":
                A.adaln_bwd_rms(v(i["x"]), o["rstd"], i["scale"], v(i["dy"]), v(o["dx"]),
                                o["d_scale"], o["d_shift"], self.ws)
            elif op == "fwd_gated":
                A.adaln_fwd_gated(v(i["x"]), i["shift"], i["scale"], i["gate"], v(i["r"]),
                                  v(o["out"]), None, o["mean"], o["rstd"], self.eps)
            else:
                A.adaln_bwd_gated(v(i["x"]), o["mean"], o["rstd"], i["shift"], i["scale"],
                                  i["gate"], v(i["dy"]), v(o["dx"]), o["d_scale"], o["d_shift"],
                                  o["d_gate"], self.ws)
            return
        for (row0, seg0, off), offd in zip(self.groups, self.offdev):
            rs = slice(row0, row0 + int(off[-1]))
            ss = slice(seg0, seg0 + len(off) - 1)
            if op == "fwd":
                A.adaln_fwd_ragged(i["x"][rs], i["shift"][ss], i["scale"][ss], o["y"][rs],
                                   o["mean"][rs], o["rstd"][rs], off, offd, self.eps)
            elif op == "gate":
                A.adaln_gate_residual_ragged(i["r"][rs], i["z"][rs], i["gate"][ss], o["out"][rs],
                                             off, offd)
            elif op == "bwd":
                A.adaln_bwd_ragged(i["x"][rs], o["mean"][rs], o["rstd"][rs], i["scale"][ss],
                                   i["dy"][rs], o["dx"][rs], o["d_scale"][ss], o["d_shift"][ss],
                                   self.ws, off, offd)
            elif op == "gate_bwd":
                A.adaln_gate_residual_bwd_ragged(i["dy"][rs], i["z"][rs], i["gate"][ss],
                                                 o["dz"][rs], o["d_gate"][ss], self.ws, off, offd)
            elif op == "fwd_rms":
                A.adaln_fwd_rms_ragged(i["x"][rs], i["shift"][ss], i["scale"][ss], o["y"][rs],
                                       o["rstd"][rs], off, offd, self.eps)
            elif op == "bwd_rms":
                A.adaln_bwd_rms_ragged(i["x"][rs], o["rstd"][rs], i["scale"][ss], i["dy"][rs],
                                       o["dx"][rs], o["d_scale"][ss], o["d_shift"][ss], self.ws,
                                       off, offd)
            elif op == "fwd_gated":
                A.adaln_fwd_gated_ragged(i["x"][rs], i["shift"][ss], i["scale"][ss],
                                         i["gate"][ss], i["r"][rs], o["out"][rs], None,
                                         o["mean"][rs], o["rstd"][rs], off, offd, self.eps)
            else:
                A.adaln_bwd_gated_ragged(i["x"][rs], o["mean"][rs], o["rstd"][rs],
                                         i["shift"][ss], i["scale"][ss], i["gate"][ss],
                                         i["dy"][rs], o["dx"][rs], o["d_scale"][ss],
                                         o["d_shift"][ss], o["d_gate"][ss], self.ws, off, offd)

    def plan(self):
        """The host planner step of the ragged workload (part of every step)."""
        if self.name == "ragged":
            import workloads
            self.A.adaln_plan_buckets(self.lengths, workloads.RAGGED_M_MEM,
                                      workloads.RAGGED_M_COMP, workloads.RAGGED_P)


OPS = ("fwd", "gate", "bwd", "gate_bwd")
FUSED_OPS = ("fwd_gated", "bwd_gated")
RMS_OPS = ("fwd_rms", "bwd_rms")
CHAIN_NAME = {"split": "4-op chain", "fused": "fused gated chain", "rms": "RMSNorm fwd+bwd"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        load = [v for v in sm if v > 0.5 * (mx or max(sm))] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- timing

def time_device(work, steps, warmup, flush, graph=True):
    """Device time of `steps` chain steps (CUDA events on the launching stream).

    The timed steps carry events only around each whole step, so that the chain's
    launches follow each other as they would in use (programmatic dependent
    launch lets each kernel's prologue overlap the previous one's tail).  With
    `graph`, the step's library calls are captured once into a CUDA graph and each
    timed step replays it (the host planner still runs every step): on the small
    workloads the host needs longer to issue a step's calls than the GPU needs to
    run them.  A second pass of `steps` steps with events around every op,
    launched from the host, gives the per-kernel times (the roofline's and the
    breakdown's); it is not part of the step time."""
    import torch
    A = work.A
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        work.plan()
        for op in work.ops:
            work.run_op(op)
    torch.cuda.synchronize()
    g = None
    per_step = None
    if graph:
        g = torch.cuda.CUDAGraph()
        c0 = A.adaln_launch_count()
        with torch.cuda.graph(g):
            for op in work.ops:
                work.run_op(op)
        per_step = A.adaln_launch_count() - c0  # kernel nodes in the graph
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
    step_ev = []
    launches0 = A.adaln_launch_count()
    for _ in range(steps):
        if flush is not None:
            flush.add_(1)  # write > L2 between steps (outside the step's events)
        s0 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        work.plan()
        if g is not None:
            g.replay()
        else:
            for op in work.ops:
                work.run_op(op)
        s1 = torch.cuda.Event(enable_timing=True)
        s1.record(stream)
        step_ev.append((s0, s1))
    torch.cuda.synchronize()
    launches = per_step * steps if g is not None else A.adaln_launch_count() - launches0
    del g
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    # per-op pass
    ev = {op: [] for op in work.ops}
    for _ in range(steps):
        if flush is not None:
            flush.add_(1)
        work.plan()
        for op in work.ops:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            work.run_op(op)
            b.record(stream)
            ev[op].append((a, b))
    torch.cuda.synchronize()
    op_ms = {op: statistics.mean(a.elapsed_time(b) for a, b in ev[op]) for op in work.ops}
    return sum(step_ms), step_ms, op_ms, launches


# which inputs each op needs first, and which outputs it finishes
E2E_IN = {"fwd": ("x", "shift", "scale"), "gate": ("r", "z", "gate"), "bwd": ("dy",),
          "gate_bwd": (), "fwd_gated": ("x", "shift", "scale", "gate", "r"),
          "bwd_gated": ("dy",), "fwd_rms": ("x", "shift", "scale"), "bwd_rms": ("dy",)}
E2E_OUT = {"fwd": ("y", "mean", "rstd"), "gate": ("out",), "bwd": ("dx", "d_scale", "d_shift"),
           "gate_bwd": ("dz", "d_gate"), "fwd_gated": ("out", "mean", "rstd"),
           "bwd_gated": ("dx", "d_scale", "d_shift", "d_gate"), "fwd_rms": ("y", "rstd"),
           "bwd_rms": ("dx", "d_scale", "d_shift")}


def time_e2e(work, steps, windows=5):
    """Same chain through the public API from pinned host buffers: every step copies
    its inputs host->device and its outputs device->host inside the timed region.
    Returns the wall time of each of `windows` back-to-back windows of `steps`
    steps; the caller reports the median window.  (On the GPU machine the host link
    runs, for stretches of some hundred milliseconds, at about half its rate in
    both directions at once; one window of ten steps then carries the stretch.)

    Copies and kernels are pipelined on three streams: an op starts as soon as
    its own inputs have landed, its outputs go back while the next op runs, and
    device buffers alternate between steps so that step i+1's uploads overlap
    step i's downloads."""
    import torch
    ins = [k for op in work.ops for k in E2E_IN[op]]
    outs = [k for op in work.ops for k in E2E_OUT[op]]
    host_in = {k: torch.empty(work.inp[k].shape, dtype=work.inp[k].dtype,
                              pin_memory=True).copy_(work.inp[k]) for k in ins}
    host_out = {k: torch.empty(work.out[k].shape, dtype=work.out[k].dtype, pin_memory=True)
                for k in outs}
    dev_in = [{k: torch.empty_like(v) for k, v in work.inp.items()} for _ in range(2)]
    dev_out = [work.out, {k: torch.empty_like(v) for k, v in work.out.items()}]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    s_up, s_run, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    run_done = [None, None]   # last kernel of the step that used buffer set b
    down_done = [None, None]  # last download of the step that used buffer set b
    torch.cuda.synchronize()

    def one(i):
        b = i % 2
        ev_in, ev_out = {}, {}
        with torch.cuda.stream(s_up):
            if run_done[b] is not None:
                s_up.wait_event(run_done[b])
            for op in work.ops:
                for k in E2E_IN[op]:
                    dev_in[b][k].copy_(host_in[k], non_blocking=True)
                ev_in[op] = torch.cuda.Event()
                ev_in[op].record(s_up)
        with torch.cuda.stream(s_run):
            if down_done[b] is not None:
                s_run.wait_event(down_done[b])
            work.plan()
            for op in work.ops:
                s_run.wait_event(ev_in[op])
                work.run_op(op, inp=dev_in[b], out=dev_out[b])
                ev_out[op] = torch.cuda.Event()
                ev_out[op].record(s_run)
            run_done[b] = ev_out[work.ops[-1]]
        with torch.cuda.stream(s_down):
            for op in work.ops:
                s_down.wait_event(ev_out[op])
                for k in E2E_OUT[op]:
                    host_out[k].copy_(dev_out[b][k], non_blocking=True)
            down_done[b] = torch.cuda.Event()
            down_done[b].record(s_down)

    one(0)
    one(1)
    torch.cuda.synchronize()
    dts = []
    for _ in range(windows):
        t0 = time.perf_counter()
        for i in range(steps):
            one(i)
        torch.cuda.synchronize()
        dts.append(time.perf_counter() - t0)
    del dev_in, dev_out
    return dts, h2d, d2h


def oracle_sample(work_name):
    """A bounded sample of the workload, widened to fp64 for the oracle."""
    import oracle
    import workloads
    oracle.build()
    if work_name == "ragged":
        L = workloads.ragged_lengths(0)
        seq = int(np.argmin(np.abs(np.array(L) - 4096)))
        inp = workloads.make_packed_inputs(L, [seq], workloads.RAGGED_D, "bf16", seed=0,
                                           device="cpu")
        rows = min(2048, inp["x"].shape[0])
        desc = f"first {rows} rows of ragged sequence {seq} (S={L[seq]}), D=3072"
    else:
        s = workloads.spec(work_name)
        rows = min(s.rows, 2048 if s.D >= 3072 else 4096)
        sub = workloads.Spec(s.name, s.dtype, s.D, s.eps, (rows,))
        inp = workloads.make_inputs(sub, seed=0, device="cpu")
        desc = f"{rows} rows x D={s.D} of the {work_name} workload"
    x = {k: oracle.to_f64(v[:rows] if k not in ("shift", "scale", "gate") else v[:1])
         for k, v in inp.items()}
    return x, rows, desc


def oracle_chain_once(x, rows, chain="split", r0=0, r1=None):
    """One pass of the chain's oracle over rows [r0, r1) of the sample."""
    import oracle
    r1 = rows if r1 is None else r1
    x = {k: (v if k in ("shift", "scale", "gate") else v[r0:r1]) for k, v in x.items()}
    off = [0, r1 - r0]
    eps = float(np.float32(1e-6))
    if chain == "fused":
        oracle.adaln_fwd_gated(x["x"], x["shift"], x["scale"], x["gate"], x["r"], off, eps)
        oracle.adaln_bwd_gated(x["x"], x["shift"], x["scale"], x["gate"], x["dy"], off, eps)
        return
    if chain == "rms":
        oracle.rms_fwd(x["x"], x["shift"], x["scale"], off, eps)
        oracle.rms_bwd(x["x"], x["scale"], x["dy"], off, eps)
        return
    oracle.adaln_fwd(x["x"], x["shift"], x["scale"], off, eps)
    oracle.gate_residual(x["r"], x["z"], x["gate"], off)
    oracle.adaln_bwd(x["x"], x["scale"], x["dy"], off, eps)
    oracle.gate_residual_bwd(x["dy"], x["z"], x["gate"], off)


def host_cpu():
    """Host core count and CPU model (lscpu), for the CPU-baseline record."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"nproc": os.cpu_count(), "model": model}


class OracleRunner:
    """The oracle's chain over a bounded sample, one pass per step, with the rows
    cut into `threads` contiguous blocks that run in a thread pool (the oracle's C
    calls release the interpreter lock).  threads = 1 is the plain single-threaded
    oracle."""

    def __init__(self, x, rows, chain, threads):
        import concurrent.futures as cf
        self.x, self.rows, self.chain = x, rows, chain
        self.threads = max(1, min(threads, rows))
        b = [self.rows * i // self.threads for i in range(self.threads + 1)]
        self.blocks = list(zip(b[:-1], b[1:]))
        self.pool = cf.ThreadPoolExecutor(self.threads) if self.threads > 1 else None

    def step(self):
        if self.pool is None:
            oracle_chain_once(self.x, self.rows, self.chain)
            return
        futs = [self.pool.submit(oracle_chain_once, self.x, self.rows, self.chain, a, b)
                for a, b in self.blocks]
        for f in futs:
            f.result()

    def rate(self, seconds):
        """(tokens/s, steps, seconds) of repeated steps for about `seconds`."""
        self.step()  # untimed: page in the arrays and the library
        reps, t0 = 0, time.perf_counter()
        while True:
            self.step()
            reps += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return reps * self.rows / el, reps, el

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def cpu_oracle_rate(work_name, seconds, chain="split"):
    """The fp64 oracle, as it stands, timed on the host cores (bounded sample):
    on all cores (threads over row blocks) and on one core."""
    x, rows, desc = oracle_sample(work_name)
    host = host_cpu()
    nthr = host["nproc"] or 1
    multi = OracleRunner(x, rows, chain, nthr)
    v_all, reps_all, el_all = multi.rate(seconds)
    multi.close()
    single = OracleRunner(x, rows, chain, 1)
    v_one, reps_one, el_one = single.rate(seconds)
    return {"value": v_all, "unit": "tokens/s", "cores": multi.threads, "kind": "oracle",
            "sample": f"{desc}; {reps_all} passes of the {CHAIN_NAME[chain]} in {el_all:.1f} s, "
                      f"fp64 C, the rows cut into {multi.threads} blocks run on "
                      f"{multi.threads} threads",
            "single_core": {"value": v_one, "unit": "tokens/s", "cores": 1,
                            "sample": f"{desc}; {reps_one} passes in {el_one:.1f} s, "
                                      f"single-threaded"},
            "host": host}


def traffic_for(kernel_src_hash):
    """dram bytes per launch of the dominant kernel from the committed ncu summary,
    valid only while the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    k, v = line.strip().split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("csrc_sha256") != kernel_src_hash:
            return None
        return float(kv["dram_bytes_per_launch_full"])
    except Exception:
        return None


# the sources the dominant kernel (the bf16 backward ring kernel) is built from
DOMINANT_KERNEL_SOURCES = ("bwd_ring.cuh", "bwd_bf16.cu", "common.cuh", "launch.h", "tmem.cuh")


def csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "modulation_adaln_fwd_gb300", "csrc")
    for n in DOMINANT_KERNEL_SOURCES:
        with open(os.path.join(d, n), "rb") as f:
            h.update(n.encode())
            h.update(f.read())
    return h.hexdigest()


# ----------------------------------------------------------------------------- main

def measure(work, args, world, dist, device):
    """Device-timed steps of one workload: the step time, the job value and the
    per-kernel roofline record (the kernel with the largest event time)."""
    import torch
    flush = None
    per_tensor = work.rows * work.D * work.E
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    if per_tensor < 2 * l2:
        flush = torch.empty(int(2 * l2) // 4 + 1024, dtype=torch.float32, device=device)
        l2_note = f"L2 flushed between steps ({flush.numel() * 4 >> 20} MiB write)"
    else:
        l2_note = f"inputs larger than L2 ({per_tensor >> 20} MiB per activation tensor)"
    clk = ClockSampler(torch.cuda.current_device() if world == 1 else int(device.index or 0))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clk.start()
    total_ms, step_ms, op_ms, launches = time_device(work, args.steps, args.warmup, flush,
                                                     graph=not args.no_graph)
    clocks = clk.stop()
    del flush
    value, total_ms = job_value(total_ms, work.rows, args.steps, world, dist, device)
    ab = work.algorithmic_bytes()
    peak, peak_src = peaks()
    dom = max(work.ops, key=lambda k: op_ms[k])
    achieved = ab[dom] / (op_ms[dom] / 1e3) / 1e9
    chain_bytes = sum(ab[op] for op in work.ops)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": None, "kernel": dom,
                "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs, copy)"}
    kernels = {op: {"ms": round(op_ms[op], 4),
                    "GB_s": round(ab[op] / (op_ms[op] / 1e3) / 1e9, 1),
                    "algorithmic_bytes": ab[op]} for op in work.ops}
    chain_gbs = chain_bytes * args.steps / (total_ms / 1e3) / 1e9
    return dict(value=value, total_ms=total_ms, launches=launches, clocks=clocks,
                roofline=roofline, kernels=kernels, l2_note=l2_note,
                chain_GB_s=round(chain_gbs, 1), chain_frac_of_peak=round(chain_gbs / peak, 4),
                chain_frac_of_nominal_8tbs=round(chain_gbs / 8000.0, 4))


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl_desc = WORKLOADS[args.workload]
    if args.impl == "reference":
        # the fp64 oracle stands in for the reference: W untimed and K timed steps, each
        # one pass of the chain over a bounded sample of the workload, on rank 0 only
        if rank != 0:
            return
        x, rows, desc = oracle_sample(args.workload)
        host = host_cpu()
        runner = OracleRunner(x, rows, args.chain, host["nproc"] or 1)
        for _ in range(args.warmup):
            runner.step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            runner.step()
        el = time.perf_counter() - t0
        runner.close()
        v = args.steps * rows / el
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": wl_desc, "name": args.workload, "chain": args.chain,
                           "rows_per_step": rows},
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": runner.threads,
                                 "kind": "oracle",
                                 "sample": f"{desc}; one {CHAIN_NAME[args.chain]} per step, "
                                           f"fp64 C, the rows cut into {runner.threads} blocks "
                                           f"run on {runner.threads} threads",
                                 "host": host},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    work = Work(args.workload, device, rows=args.rows, chain=args.chain)
    m = measure(work, args, world, dist, device)
    tokens_per_step = work.rows
    if m["roofline"]["kernel"] == "bwd" and args.workload == "wan" and args.chain == "split" \
            and args.rows is None:
        m["roofline"]["traffic"] = traffic_for(csrc_hash())

    e2e = None
    pinned = 2 * sum(t.numel() * t.element_size() for t in list(work.inp.values()) + list(work.out.values()))
    if not args.no_e2e and pinned > 48 * 2 ** 30:
        e2e = {"value": None, "unit": "tokens/s", "skipped": f"needs {pinned >> 30} GiB pinned host memory"}
    elif not args.no_e2e:
        k = args.e2e_steps or max(3, min(args.steps, 10))
        dts, h2d, d2h = time_e2e(work, k)
        tt = torch.tensor(dts, dtype=torch.float64, device=device)
        if dist:
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        dts = sorted(tt.tolist())
        dt = dts[len(dts) // 2]
        e2e = {"value": world * tokens_per_step * k / dt, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k,
               "statistic": f"median of {len(dts)} back-to-back windows of {k} steps",
               "window_ms_per_step": [round(t / k * 1e3, 3) for t in dts]}
    config = {"workload": wl_desc, "name": args.workload, "chain": args.chain,
              "rows_per_step": work.rows, "D": work.D, "segments": work.nseg,
              "reduced_rows_for_profiling": args.rows,
              "buckets": len(work.groups) if work.groups else None,
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
              "l2": m["l2_note"],
              "launch": "host" if args.no_graph else
                        "CUDA graph of the step's library calls, replayed per step"}
    dtype_name = work.dtype_name
    del work
    torch.cuda.empty_cache()

    # the second 75%-of-peak workload: ragged mixed-mode packing, same chain and timing
    ragged = None
    if args.workload == "wan" and args.rows is None and not args.no_ragged:
        rw = Work("ragged", device, chain=args.chain)
        r = measure(rw, args, world, dist, device)
        ragged = {"workload": WORKLOADS["ragged"], "value": r["value"], "unit": "tokens/s",
                  "ms_per_step": r["total_ms"] / args.steps, "rows_per_step": rw.rows,
                  "buckets": len(rw.groups), "D": rw.D, "l2": r["l2_note"],
                  "chain_GB_s": r["chain_GB_s"], "chain_frac_of_peak": r["chain_frac_of_peak"],
                  "chain_frac_of_nominal_8tbs": r["chain_frac_of_nominal_8tbs"],
                  "roofline": r["roofline"], "kernels": r["kernels"],
                  "gpu_launches": r["launches"], "clocks": r["clocks"]}
        del rw
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_rate(args.workload, args.cpu_seconds, args.chain)

    if rank == 0:
        line = {
            "metric": METRIC, "value": m["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": m["total_ms"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_name,
            "data": "synthetic", "config": config,
            "chain_GB_s": m["chain_GB_s"], "chain_frac_of_peak": m["chain_frac_of_peak"],
            "chain_frac_of_nominal_8tbs": m["chain_frac_of_nominal_8tbs"],
            "roofline": m["roofline"], "kernels": m["kernels"], "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": m["launches"], "clocks": m["clocks"],
        }
        if ragged is not None:
            line["ragged"] = ragged
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
