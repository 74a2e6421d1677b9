#!/usr/bin/env python
"""Benchmark: batched speculative-decoding verification rounds/s and HBM GB/s on GB300.

One step = one verification round = one ``spec_verify`` call over a whole
batch (plan -> row sweep -> final pass).  Default workload: B=128 requests,
k=16 draft positions, V=151936, bf16 logits, half the requests with low and
half with high draft noise (see speculative_decoding_verification_58_gb300/synth.py).

Prints one JSON line.  ``value`` is verification rounds per second over all
ranks (each rank verifies its own batch: weak scaling, no collective on the
data path), with inputs resident in HBM.  The logits (1.28 GB at the default
workload) are far larger than L2, so no flush is needed between steps; the
rounds rotate over ``--copies`` (default 3) resident copies of them, so that
no round reads rows the round before left in L2 (real rounds get fresh
logits).

``--impl reference`` times the plain CPU oracle (the reference this library
is checked against) on the host cores on the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verify rounds/s & achieved HBM GB/s at B=128,k=16,V=151936 bf16 (1 GB300)"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000  # GB300 L2 (126 MiB)
COPIES = 3  # default resident copies of the batch's logits, used in turn by successive rounds


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=None, help="a name from synth.WORKLOADS")
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-full-sweep", action="store_true")
    ap.add_argument("--no-packed", action="store_true")
    ap.add_argument("--no-opd", action="store_true")
    ap.add_argument("--no-d3d", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' measurements (per_workload)")
    ap.add_argument("--copies", type=int, default=COPIES,
                    help="resident copies of the logits that successive rounds read in turn "
                         "(1 for small profiler captures)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# Small helpers
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def replica_seed(base: int, rank: int) -> int:
    """Each replica verifies its own batch: same workload recipe, its own seed."""
    return base + 1000 * rank


def aggregate_value(world: int, ms_max: float) -> float:
    """Rounds/s of the whole job: every rank completes one round per step, and the
    step time is the slowest rank's."""
    return world * 1000.0 / ms_max


class Ranks:
    """Process-group plumbing for N replicas: a barrier and a max over ranks.

    Used for timing only; no data crosses ranks (requests are independent).
    NCCL with CUDA tensors on GPUs, gloo with CPU tensors in the CPU tests.
    """

    def __init__(self, world: int, device=None, backend: str = "nccl"):
        self.world = world
        self.device = device
        if world > 1:
            import torch.distributed as dist
            if not dist.is_initialized():
                if backend == "nccl":
                    dist.init_process_group("nccl", device_id=device)
                else:
                    dist.init_process_group(backend)

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return x
        import torch
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def csrc_digest() -> str:
    """Digest of the code the sweep kernel is built from (its code, the shared
    helpers and the plan kernel that lays out its work).  Line comments and
    blank lines are left out, so that editing a comment keeps a recorded
    capture valid; any change to the code itself does not."""
    csrc = os.path.join(ROOT, "speculative_decoding_verification_58_gb300", "csrc")
    texts = []
    for name in ("common.cuh", "plan.cuh", "sweep.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as fh:
            texts.append((name, fh.read()))
    return code_digest(texts)


def code_digest(texts) -> str:
    """Digest of (name, source text) pairs with line comments and blank lines
    left out."""
    h = hashlib.sha256()
    for name, text in texts:
        code = [line.split("//", 1)[0].rstrip() for line in text.splitlines()]
        h.update(name.encode())
        h.update("\n".join(line for line in code if line).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per sweep launch from the committed ncu summary, if it matches the sources."""
    path = os.path.join(ROOT, "profiles", f"sweep_kernel_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("- traffic_bytes_per_launch", "- csrc_digest")):
            key, val = line.strip()[2:].split(":", 1)
            vals[key.strip()] = val.strip().strip("`")
    if vals.get("csrc_digest") != csrc_digest():
        return None
    try:
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            return
        self.first = threading.Event()
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # nvidia-smi's start-up (NVML initialisation) disturbs a running GPU
        # for a moment: let it finish before anything is timed.
        self.first.wait(timeout=5.0)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.samples.append(parts)
                self.first.set()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        for p in self.samples:
            try:
                sm.append(float(p[0]))
                smax.append(float(p[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, p[3:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def model_bytes(inp, o, esize):
    """M1: rows i < L_b (2 per sampling position) + the final row(s); M2: only up to n_b."""
    V = inp.V
    m1 = m2 = 0
    for b in range(inp.B):
        n = int(o.num_accepted[b])
        L = int(inp.lengths[b])
        greedy = inp.temperature[b] == 0
        per = 1 if greedy else 2
        final = 0 if (greedy and n < L) else (2 if n < L else 1)
        m1 += (per * L + final) * V * esize
        m2 += (per * (min(n + 1, L)) + final) * V * esize
    return m1, m2


def logit_bytes_of(name: str) -> int:
    """Bytes of a workload's padded target + draft logits."""
    from speculative_decoding_verification_58_gb300 import synth
    cfg = synth.WORKLOADS[name]
    esize = 2 if cfg["dtype"] == "bf16" else 4
    return cfg["B"] * (2 * cfg["k"] + 1) * cfg["V"] * esize


def flushes_l2(name: str) -> bool:
    """Inputs that fit in L2 are timed with L2 overwritten before every round."""
    return logit_bytes_of(name) < 2 * L2_BYTES


def run_config(name: str, seed: int, world: int, copies: int) -> dict:
    """The ``config`` object both arms print for a workload."""
    from speculative_decoding_verification_58_gb300 import synth
    cfg = synth.WORKLOADS[name]
    lb = logit_bytes_of(name)
    l2 = (f"L2 flushed before every round ({lb / 1e6:.1f} MB of logits)" if flushes_l2(name) else
          f"inputs larger than L2: {lb / 1e9:.2f} GB of logits, {max(1, copies)} resident copies "
          "used in turn, no flush between steps")
    return {"workload": name, "B": cfg["B"], "k": cfg["k"], "V": cfg["V"], "logits": cfg["dtype"],
            "seed": seed, "parallelism": f"replicas x{world}", "l2": l2, "early_exit": True}


def parity_counts(inp, gpu_out, gpu_n, o) -> dict:
    """The parity rule's counts for one comparison: requests that differ outside
    the 1e-6 near-tie band must be 0; near-ties are counted, and the ones that
    flipped (excused) are reported with the largest distance from their
    threshold; rows = logit rows the oracle evaluated."""
    near = (o.margin < 1e-6) & (inp.temperature != 0) & (o.num_accepted >= 0)
    same = (gpu_n == o.num_accepted) & np.all(gpu_out == o.out_tokens, axis=1)
    flips = ~same & near
    rows = 0
    for b, n in enumerate(o.num_accepted):
        if n >= 0:
            rows += (1 if inp.temperature[b] == 0 else 2) * (int(n) + 1)
    return {"requests": int(inp.B), "rows": int(rows), "mismatches": int((~same).sum()),
            "outside_near_tie_band": int((~same & ~near).sum()), "near_ties": int(near.sum()),
            "excused": int(flips.sum()),
            "max_flip_margin": float(o.margin[flips].max()) if flips.any() else 0.0}


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------

REFERENCE_BUDGET_S = 60.0  # about this long for --warmup + --steps reference steps


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    from speculative_decoding_verification_58_gb300 import synth

    name = args.workload or synth.HEADLINE
    cfg = synth.WORKLOADS[name]
    seed = replica_seed(args.seed if args.seed is not None else cfg["seed"], rank)
    inp = synth.make_workload(name, seed=seed)
    oracle.build()
    B = inp.B

    def run(idx):
        oracle.verify(inp.target[idx], inp.draft[idx], inp.tokens[idx], inp.lengths[idx],
                      inp.uniforms[idx], inp.temperature[idx])

    # A step verifies a rotating sample of the batch's requests, sized from a
    # timed single request so that all the steps take about the budget.
    run(np.arange(1))
    t0 = time.perf_counter()
    run(np.arange(1))
    t_req = max(1e-6, time.perf_counter() - t0)
    sample_b = int(min(B, max(1, REFERENCE_BUDGET_S / ((args.steps + args.warmup) * t_req))))

    def step(j):
        run((j * sample_b + np.arange(sample_b)) % B)

    for j in range(args.warmup):
        step(j)
    t0 = time.perf_counter()
    for j in range(args.steps):
        step(args.warmup + j)
    sec_per_step = (time.perf_counter() - t0) / args.steps
    value = (sample_b / B) / sec_per_step  # full rounds per second
    sample = (f"each step verifies {sample_b} of the {B} requests (rotating); value = "
              f"{sample_b}/{B} round per step time; single-threaded fp64 C++ oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rounds/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(name, seed, world, args.copies),
        "cpu_baseline": {"value": value, "unit": "rounds/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def _event_pair():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


class Workload:
    """One named workload resident on the device: its inputs (and, when they are
    larger than L2, further copies that successive rounds read in turn), a
    workspace, output buffers and bound calls."""

    def __init__(self, torch, sv, synth, name, seed, dev, stream, copies):
        self.torch, self.sv, self.name, self.seed = torch, sv, name, seed
        self.dev, self.stream = dev, stream
        self.inp = inp = synth.make_workload(name, seed=seed)
        self.esize = 2 if inp.dtype == "bf16" else 4
        self.d = sv.to_device(inp, dev)
        self.flush = flushes_l2(name)
        n_copies = 1 if self.flush else max(1, copies)
        self.ds = [self.d] + [dict(self.d, target_logits=self.d["target_logits"].clone(),
                                   draft_logits=self.d["draft_logits"].clone())
                              for _ in range(n_copies - 1)]
        self.turn = 0
        self.ws = sv.alloc_workspace(inp.B, inp.k, inp.V, dev)
        self.out = torch.empty((inp.B, inp.k + 1), dtype=torch.int32, device=dev)
        self.nacc = torch.empty(inp.B, dtype=torch.int32, device=dev)
        self.bound = {fs: [sv.Verifier(**dc, workspace=self.ws, out_tokens=self.out,
                                       num_accepted=self.nacc, stream=stream, full_sweep=fs)
                           for dc in self.ds]
                      for fs in (False, True)}
        self.logit_bytes = inp.target.nbytes + inp.draft.nbytes
        self.scrub = None

    def step(self, full_sweep=False, events=None):
        c = self.turn % len(self.ds)
        self.turn += 1
        if events is None:
            self.bound[full_sweep][c]()
        else:
            self.sv.spec_verify(**self.ds[c], workspace=self.ws, out_tokens=self.out,
                                num_accepted=self.nacc, stream=self.stream,
                                full_sweep=full_sweep, events=events)

    def sync(self):
        self.torch.cuda.synchronize(self.dev)

    def timed(self, steps, flush):
        """Mean ms per round over ``steps`` rounds on the stream.  flush: L2
        overwritten before every round (an event pair around each round);
        otherwise back to back, one event pair around all."""
        torch = self.torch
        if flush:
            if self.scrub is None:
                self.scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=self.dev)
            pairs = [_event_pair() for _ in range(steps)]
            for a, b in pairs:
                self.scrub.fill_(1)
                a.record(self.stream)
                self.step()
                b.record(self.stream)
            self.sync()
            return sum(a.elapsed_time(b) for a, b in pairs) / steps
        e0, e1 = _event_pair()
        e0.record(self.stream)
        for _ in range(steps):
            self.step()
        e1.record(self.stream)
        self.sync()
        return e0.elapsed_time(e1) / steps

    def kernel_times(self, reps, full_sweep=False):
        """Mean durations of plan, sweep and final: rounds with events between them."""
        evs = [[self.torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
        for row in evs:
            for e in row:
                e.record(self.stream)  # creates the handles
        self.sync()
        for row in evs:
            self.step(full_sweep=full_sweep, events=row)
        self.sync()
        return tuple(statistics.mean(r[j].elapsed_time(r[j + 1]) for r in evs) for j in range(3))

    def outputs(self):
        return self.out.cpu().numpy(), self.nacc.cpu().numpy()

    def release(self):
        self.d = self.ds = self.bound = self.scrub = None


class OurArm:
    """This library's side of the benchmark: one verification round per step,
    then the extra legs (every other workload, early exit off, packed batch,
    OPD statistics, D3D selection, end to end, CPU baseline) on the same inputs."""

    def __init__(self, args, world, rank, local):
        import torch

        import speculative_decoding_verification_58_gb300 as sv
        from speculative_decoding_verification_58_gb300 import synth

        self.torch, self.sv, self.synth = torch, sv, synth
        self.args, self.world, self.rank = args, world, rank
        torch.cuda.set_device(local)
        self.dev = dev = torch.device("cuda", local)
        self.ranks = Ranks(world, dev, "nccl")
        sv.lib()
        self.stream = torch.cuda.current_stream(dev)
        self.name = args.workload or synth.HEADLINE
        cfg = synth.WORKLOADS[self.name]
        self.seed = replica_seed(args.seed if args.seed is not None else cfg["seed"], rank)
        self.w = Workload(torch, sv, synth, self.name, self.seed, dev, self.stream, args.copies)
        self.inp, self.esize = self.w.inp, self.w.esize
        self.d, self.ws, self.out, self.nacc = self.w.d, self.w.ws, self.w.out, self.w.nacc
        self.logit_bytes = self.w.logit_bytes
        self.reps = max(10, min(args.steps, 200))
        self.others = []  # per-workload results kept for the CPU-baseline leg's parity

    def step(self, full_sweep=False, events=None):
        self.w.step(full_sweep, events)

    def sync(self):
        self.torch.cuda.synchronize(self.dev)

    # -- the timed region ---------------------------------------------------
    def timed_rounds(self):
        """K rounds after W warm-up rounds, device-timed with events on the stream."""
        args = self.args
        for _ in range(max(3, args.warmup)):
            self.step()
        self.sync()
        self.ranks.barrier()
        self.sync()
        self.flush = self.w.flush
        total_ms = self.w.timed(args.steps, self.flush) * args.steps
        self.ranks.barrier()
        self.ms = self.ranks.max(total_ms / args.steps)
        self.rep = self.sv.spec_verify_report(self.ws, self.stream)
        self.gpu_out, self.gpu_n = self.w.outputs()

    # -- measurements around the timed region --------------------------------
    def round_percentiles(self):
        """An event pair around each round (the events sit between rounds, so a
        round cannot start under the previous one's tail)."""
        rev = [_event_pair() for _ in range(self.reps)]
        for a, b in rev:
            a.record(self.stream)
            self.step()
            b.record(self.stream)
        self.sync()
        rts = sorted(a.elapsed_time(b) for a, b in rev)
        n = self.reps
        return {"p10": rts[int(0.1 * (n - 1))], "p50": rts[(n - 1) // 2],
                "p90": rts[int(0.9 * (n - 1))], "rounds": n, "unit": "ms"}

    def kernel_times(self, full_sweep=False):
        return self.w.kernel_times(self.reps, full_sweep)

    def full_sweep_leg(self):
        """The same workload with early exit switched off (every row i < L_b is swept)."""
        for _ in range(3):
            self.step(full_sweep=True)
        f0, f1 = _event_pair()
        f0.record(self.stream)
        for _ in range(self.reps):
            self.step(full_sweep=True)
        f1.record(self.stream)
        self.sync()
        frep = self.sv.spec_verify_report(self.ws, self.stream)
        fsweep = self.kernel_times(full_sweep=True)[1]
        return {"ms_per_step": f0.elapsed_time(f1) / self.reps, "sweep_ms": fsweep,
                "sweep_bytes": frep.sweep_bytes,
                "sweep_gbs": frep.sweep_bytes / (fsweep * 1e-3) / 1e9}

    def workload_legs(self, hbm_peak):
        """Every other workload: rounds/s with its L2 regime (L2-resident inputs
        timed both flushed and hot), the kernels' times, bytes moved and the
        fraction of the measured copy bandwidth.  Parity against the oracle is
        added by the CPU-baseline leg."""
        torch, sv, synth = self.torch, self.sv, self.synth
        out = {}
        steps = max(50, min(self.args.steps, 500))
        for name, cfg in synth.WORKLOADS.items():
            if name == self.name:
                continue
            w = Workload(torch, sv, synth, name, cfg["seed"], self.dev, self.stream,
                         self.args.copies)
            for _ in range(5):
                w.step()
            w.sync()
            ms = w.timed(steps, w.flush)
            entry = {"B": w.inp.B, "k": w.inp.k, "V": w.inp.V, "logits": w.inp.dtype,
                     "seed": cfg["seed"], "rounds_per_s": 1000.0 / ms, "ms_per_step": ms,
                     "steps": steps,
                     "l2": "flushed before every round" if w.flush else
                           f"{len(w.ds)} resident copies used in turn"}
            if w.flush:
                hot = w.timed(steps, False)
                entry["hot"] = {"rounds_per_s": 1000.0 / hot, "ms_per_step": hot,
                                "l2": "inputs left in L2 (back-to-back rounds)"}
            rep = sv.spec_verify_report(w.ws, self.stream)
            k_plan, k_sweep, k_final = w.kernel_times(max(20, min(steps, 100)))
            moved = rep.sweep_bytes + rep.final_bytes
            entry.update({
                "kernels_ms": {"plan": k_plan, "sweep": k_sweep, "final": k_final},
                "moved_bytes": int(moved), "moved_gbs": moved / (ms * 1e-3) / 1e9,
                "moved_frac": moved / (ms * 1e-3) / 1e9 / hbm_peak,
                "sweep_bytes": int(rep.sweep_bytes),
                "sweep_gbs": rep.sweep_bytes / (k_sweep * 1e-3) / 1e9,
                "sweep_frac": rep.sweep_bytes / (k_sweep * 1e-3) / 1e9 / hbm_peak})
            gpu_out, gpu_n = w.outputs()
            self.others.append((name, w.inp, gpu_out, gpu_n))
            w.release()
            del w
            torch.cuda.empty_cache()
            out[name] = entry
        return out

    def packed_leg(self):
        """The same batch packed (AdaFlash Section 3.3: total length sum_b L_b rows
        instead of B x k): same outputs, a smaller resident footprint."""
        sv, d = self.sv, self.d
        pk = self.synth.pack_rows(self.inp)
        rows = sv.to_device_packed(pk, self.dev)
        pargs = [dict(**{key: (t if c == 0 else t.clone()) for key, t in rows.items()},
                      draft_tokens=d["draft_tokens"], lengths=d["lengths"],
                      uniforms=d["uniforms"], temperature=d["temperature"], workspace=self.ws,
                      out_tokens=self.out, num_accepted=self.nacc, stream=self.stream)
                 for c in range(len(self.w.ds))]
        for j in range(3):
            sv.spec_verify_packed(**pargs[j % len(pargs)])
        self.sync()
        p0, p1 = _event_pair()
        p0.record(self.stream)
        for j in range(self.reps):
            sv.spec_verify_packed(**pargs[j % len(pargs)])
        p1.record(self.stream)
        self.sync()
        same = bool(np.array_equal(self.out.cpu().numpy(), self.gpu_out) and
                    np.array_equal(self.nacc.cpu().numpy(), self.gpu_n))
        pms = p0.elapsed_time(p1) / self.reps
        del rows, pargs
        self.torch.cuda.empty_cache()
        return {"ms_per_step": pms, "value": 1000.0 / pms, "unit": "rounds/s",
                "logit_bytes": int(pk.target_rows.nbytes + pk.draft_rows.nbytes),
                "padded_logit_bytes": int(self.logit_bytes), "same_outputs_as_padded": same}

    def opd_leg(self):
        """OPD supervision statistics (AdaFlash Section 3.1) on the same buffers:
        both rows of every verified position."""
        sv, d, inp = self.sv, self.d, self.inp
        st = sv.spec_opd_stats(d["target_logits"], d["draft_logits"], d["lengths"],
                               stream=self.stream)

        def call(j):
            dc = self.w.ds[j % len(self.w.ds)]
            sv.spec_opd_stats(dc["target_logits"], dc["draft_logits"], dc["lengths"], out=st,
                              stream=self.stream)
        for j in range(3):
            call(j)
        self.sync()
        o0, o1 = _event_pair()
        oreps = max(10, min(self.args.steps, 100))
        o0.record(self.stream)
        for j in range(oreps):
            call(j)
        o1.record(self.stream)
        self.sync()
        oms = o0.elapsed_time(o1) / oreps
        positions = int(inp.lengths.sum())
        obytes = positions * 2 * inp.V * self.esize
        return {"ms_per_call": oms, "positions": positions,
                "positions_per_s": positions / (oms * 1e-3), "bytes_per_call": obytes,
                "gbs": obytes / (oms * 1e-3) / 1e9,
                "loss_mean": float(st.loss.float().mean().item())}

    def opd_fused_leg(self):
        """Verification and OPD statistics in one pass (spec_verify_opd): every
        verified row pair read once for both; compared with the round and the
        statistics run separately."""
        sv, inp = self.sv, self.inp
        st = None

        def call(j):
            nonlocal st
            dc = self.w.ds[j % len(self.w.ds)]
            _, _, st = sv.spec_verify_opd(**dc, workspace=self.ws, out_tokens=self.out,
                                          num_accepted=self.nacc, out=st, stream=self.stream)
        for j in range(3):
            call(j)
        self.sync()
        reps = max(10, min(self.args.steps, 100))
        f0, f1 = _event_pair()
        f0.record(self.stream)
        for j in range(reps):
            call(j)
        f1.record(self.stream)
        self.sync()
        fms = f0.elapsed_time(f1) / reps
        out, n = self.out.cpu().numpy(), self.nacc.cpu().numpy()
        positions = int(inp.lengths.sum())
        obytes = positions * 2 * inp.V * self.esize
        return {"ms_per_call": fms, "positions": positions, "bytes_per_call": obytes,
                "gbs": obytes / (fms * 1e-3) / 1e9,
                "same_verification_outputs": bool(np.array_equal(out, self.gpu_out) and
                                                  np.array_equal(n, self.gpu_n)),
                "requests_differing": int(np.sum(np.any(out != self.gpu_out, axis=1) |
                                                 (n != self.gpu_n)))}

    def d3d_leg(self):
        """D3D branch selection on this round's outcome: the paper's main budget
        (block 16, coverage C = 12, fan-out F = 2, 24 branches per request)."""
        sv, inp = self.sv, self.inp
        br = self.synth.make_d3d_branches(inp.lengths, inp.V, C=12, F=2, blk=16,
                                          seed=self.seed + 7)
        tb = {key: self.torch.from_numpy(getattr(br, key)).to(self.dev)
              for key in ("pos", "tok", "block")}
        hit, nxt, hits = sv.spec_d3d_select(self.nacc, self.out, tb["pos"], tb["tok"],
                                            tb["block"], stream=self.stream)
        call = lambda: sv.spec_d3d_select(self.nacc, self.out, tb["pos"], tb["tok"], tb["block"],
                                          hit=hit, next_block=nxt, hits=hits, stream=self.stream)
        for _ in range(3):
            call()
        self.sync()
        g0, g1 = _event_pair()
        g0.record(self.stream)
        for _ in range(self.reps):
            call()
        g1.record(self.stream)
        self.sync()
        # The same call captured in a CUDA graph, 20 calls per graph: device time
        # per call without the binding's per-call checks on the host.
        torch = self.torch
        gs = torch.cuda.Stream(self.dev)
        per_graph, replays = 20, 20
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(per_graph):
                sv.spec_d3d_select(self.nacc, self.out, tb["pos"], tb["tok"], tb["block"],
                                   hit=hit, next_block=nxt, hits=hits, stream=gs)
        self.sync()
        with torch.cuda.stream(gs):
            graph.replay()
            gs.synchronize()
            r0, r1 = _event_pair()
            r0.record(gs)
            for _ in range(replays):
                graph.replay()
            r1.record(gs)
        self.sync()
        graph_us = r0.elapsed_time(r1) / (replays * per_graph) * 1000
        return {"us_per_call": g0.elapsed_time(g1) / self.reps * 1000,
                "us_per_call_graph": graph_us, "requests": inp.B,
                "branches_per_request": int(br.pos.shape[1]), "block": 16,
                "hit_rate": int(hits.item()) / inp.B,
                "note": "branch tokens are uniform draws, so hits are rare; latency-bound"}

    def e2e_legs(self):
        """End to end through the public API: pinned host inputs in, results out,
        every step; the padded buffers, then the packed batch (AdaFlash Section
        3.3: only the rows a round can read, rows 0..L_b of each request)."""
        torch, sv, d = self.torch, self.sv, self.d
        host = {}
        for key, t in d.items():
            host[key] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            host[key].copy_(t.cpu())
        h_out = torch.empty(self.out.shape, dtype=torch.int32, pin_memory=True)
        h_n = torch.empty(self.nacc.shape, dtype=torch.int32, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = h_out.numel() * 4 + h_n.numel() * 4
        steps = self.args.e2e_steps or max(5, min(50, self.args.steps))

        def timed(step_fn):
            for _ in range(2):
                step_fn()
            self.ranks.barrier()
            t0 = time.perf_counter()
            for _ in range(steps):
                step_fn()
            return self.ranks.max((time.perf_counter() - t0) / steps)

        def padded_step():
            for key, t in host.items():
                d[key].copy_(t, non_blocking=True)
            self.step()
            h_out.copy_(self.out, non_blocking=True)
            h_n.copy_(self.nacc, non_blocking=True)
            self.stream.synchronize()

        padded_s = timed(padded_step)

        pk = self.synth.pack_rows(self.inp)
        hp = {key: torch.from_numpy(np.ascontiguousarray(v)).pin_memory()
              for key, v in (("target_row_start", pk.target_row_start),
                             ("draft_row_start", pk.draft_row_start))}
        for key, v in (("target_rows", pk.target_rows), ("draft_rows", pk.draft_rows)):
            t = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) \
                if v.dtype == np.uint16 else torch.from_numpy(v)
            hp[key] = t.pin_memory()
        for key in ("draft_tokens", "lengths", "uniforms", "temperature"):
            hp[key] = host[key]
        dp = {key: torch.empty(t.shape, dtype=t.dtype, device=self.dev) for key, t in hp.items()}
        h2d_packed = sum(t.numel() * t.element_size() for t in hp.values())

        def packed_step():
            for key, t in hp.items():
                dp[key].copy_(t, non_blocking=True)
            sv.spec_verify_packed(**dp, workspace=self.ws, out_tokens=self.out,
                                  num_accepted=self.nacc, stream=self.stream)
            h_out.copy_(self.out, non_blocking=True)
            h_n.copy_(self.nacc, non_blocking=True)
            self.stream.synchronize()

        packed_step()
        same = bool(np.array_equal(h_out.numpy(), self.gpu_out) and
                    np.array_equal(h_n.numpy(), self.gpu_n))
        packed_s = timed(packed_step)

        # The packed rows stay in pinned host memory and the kernels read them
        # over the CPU-GPU link themselves: only the rows the round reads
        # cross it (early exit spares the rest); the small per-request arrays
        # are copied as before.
        small = ("target_row_start", "draft_row_start", "draft_tokens", "lengths", "uniforms",
                 "temperature")

        def direct_step():
            for key in small:
                dp[key].copy_(hp[key], non_blocking=True)
            sv.spec_verify_packed(target_rows=hp["target_rows"], draft_rows=hp["draft_rows"],
                                  **{key: dp[key] for key in small}, workspace=self.ws,
                                  out_tokens=self.out, num_accepted=self.nacc, stream=self.stream)
            h_out.copy_(self.out, non_blocking=True)
            h_n.copy_(self.nacc, non_blocking=True)
            self.stream.synchronize()

        direct_step()
        same_direct = bool(np.array_equal(h_out.numpy(), self.gpu_out) and
                           np.array_equal(h_n.numpy(), self.gpu_n))
        rep = sv.spec_verify_report(self.ws, stream=self.stream)
        read = int(rep.sweep_bytes) + int(rep.final_bytes)
        h2d_direct = read + sum(hp[key].numel() * hp[key].element_size() for key in small)
        direct_s = timed(direct_step)
        del dp
        copy_leg = {"value": self.world / packed_s, "unit": "rounds/s",
                    "h2d_bytes_per_step": h2d_packed, "d2h_bytes_per_step": d2h,
                    "layout": "packed (rows 0..L_b of each request) copied to the device",
                    "same_outputs": same}
        direct_leg = {"value": self.world / direct_s, "unit": "rounds/s",
                      "h2d_bytes_per_step": h2d_direct, "d2h_bytes_per_step": d2h,
                      "layout": "packed rows in pinned host memory, read by the kernels over "
                                "the CPU-GPU link (only the rows the round reads)",
                      "logit_bytes_read": read, "same_outputs": same_direct}
        padded_leg = {"value": self.world / padded_s, "unit": "rounds/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "layout": "padded [B, k+1, V] / [B, k, V]"}

        # The padded buffers left in pinned host memory, read in place.
        psmall = ("draft_tokens", "lengths", "uniforms", "temperature")

        def padded_direct_step():
            for key in psmall:
                d[key].copy_(host[key], non_blocking=True)
            sv.spec_verify(host["target_logits"], host["draft_logits"],
                           **{key: d[key] for key in psmall}, workspace=self.ws,
                           out_tokens=self.out, num_accepted=self.nacc, stream=self.stream)
            h_out.copy_(self.out, non_blocking=True)
            h_n.copy_(self.nacc, non_blocking=True)
            self.stream.synchronize()

        padded_direct_step()
        same_pd = bool(np.array_equal(h_out.numpy(), self.gpu_out) and
                       np.array_equal(h_n.numpy(), self.gpu_n))
        rep = sv.spec_verify_report(self.ws, stream=self.stream)
        read_pd = int(rep.sweep_bytes) + int(rep.final_bytes)
        pd_s = timed(padded_direct_step)
        padded_leg["direct"] = {
            "value": self.world / pd_s, "unit": "rounds/s",
            "h2d_bytes_per_step": read_pd + sum(host[key].numel() * host[key].element_size()
                                                for key in psmall),
            "d2h_bytes_per_step": d2h, "logit_bytes_read": read_pd, "same_outputs": same_pd,
            "layout": "padded buffers in pinned host memory, read in place over the link"}
        return direct_leg, copy_leg, padded_leg

    def cpu_baseline(self, result, round_bytes):
        """The oracle on one host core for about ten seconds of full rounds, and the
        parity of the timed run against it; then the parity of every other
        workload's last round (the oracle over host threads, one request per
        call, only as a checker)."""
        import oracle
        from concurrent.futures import ThreadPoolExecutor
        inp = self.inp
        oracle.build()
        reps, spent = 0, 0.0
        t0 = time.perf_counter()
        o = None
        while reps < 1 or (spent < 10.0 and reps < 30):
            o = oracle.verify(inp.target, inp.draft, inp.tokens, inp.lengths, inp.uniforms,
                              inp.temperature)
            reps += 1
            spent = time.perf_counter() - t0
        result["cpu_baseline"] = {
            "value": reps / spent, "unit": "rounds/s", "cores": 1, "kind": "oracle",
            "sample": f"the full {inp.B}-request round, {reps} time(s), single-threaded fp64 oracle"}
        m1, m2 = model_bytes(inp, o, self.esize)
        result["parity"] = parity_counts(inp, self.gpu_out, self.gpu_n, o)
        result["parity"]["rule"] = ("no request may differ outside the 1e-6 near-tie band; "
                                    "near-ties are counted and the flipped ones reported")
        result["byte_models"] = {
            "M1_all_rows": m1, "M2_rows_to_first_reject": m2, "moved": round_bytes,
            "M1_effective_gbs": m1 / (self.ms * 1e-3) / 1e9,
            "M1_effective_note": ("M1 bytes over the round time: what a sweep of every row i < L_b "
                                  "would need to reach the same round time; not a bandwidth "
                                  "(early exit skips most of those rows)"),
            "mean_accepted": float(o.num_accepted.mean())}

        def threaded(w):
            with ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as pool:
                parts = list(pool.map(
                    lambda b: oracle.verify(w.target[b:b + 1], w.draft[b:b + 1],
                                            w.tokens[b:b + 1], w.lengths[b:b + 1],
                                            w.uniforms[b:b + 1], w.temperature[b:b + 1]),
                    range(w.B)))
            return oracle.OracleResult(*(np.concatenate([getattr(q, f) for q in parts])
                                         for f in ("out_tokens", "num_accepted", "margin",
                                                   "final_mass", "residual_zero")),
                                       sum(q.bad_requests for q in parts))

        for name, w_inp, gpu_out, gpu_n in self.others:
            if name in result.get("per_workload", {}):
                result["per_workload"][name]["parity"] = parity_counts(
                    w_inp, gpu_out, gpu_n, threaded(w_inp))
        self.others = []

    def run(self):
        args, inp = self.args, self.inp
        props = self.torch.cuda.get_device_properties(self.dev)
        peaks, peak_kind = measured_peaks()
        hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
        sampler = ClockSampler(f"GPU-{props.uuid}" if getattr(props, "uuid", None)
                               else str(self.dev.index))
        self.timed_rounds()
        round_pct = self.round_percentiles()
        k_plan, k_sweep, k_final = self.kernel_times()
        full = None if args.no_full_sweep else self.full_sweep_leg()
        packed = None if args.no_packed else self.packed_leg()
        opd = None if args.no_opd else self.opd_leg()
        opd_fused = None if args.no_opd else self.opd_fused_leg()
        d3d = None if args.no_d3d else self.d3d_leg()
        e2e_direct, e2e_copy, e2e_padded = self.e2e_legs()
        # The end-to-end figure is the library's path for host-resident logits:
        # the kernels read the pinned rows over the link (the copy-first
        # path is reported beside it; a direct run whose outputs differed
        # from the device run would not count).
        e2e = e2e_direct if e2e_direct["same_outputs"] else e2e_copy
        clocks = sampler.stop()
        per_workload = (self.workload_legs(hbm_peak)
                        if self.world == 1 and not args.no_workloads else None)
        self.ranks.barrier()
        if self.rank != 0:
            return

        rep, ms, world = self.rep, self.ms, self.world
        sweep_gbs = rep.sweep_bytes / (k_sweep * 1e-3) / 1e9
        round_bytes = rep.sweep_bytes + rep.final_bytes
        result = {
            "metric": METRIC, "value": aggregate_value(world, ms), "unit": "rounds/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": run_config(self.name, self.seed, world, args.copies),
            "hbm_gbs": round_bytes / (ms * 1e-3) / 1e9,
            "hbm_gbs_frac": round_bytes / (ms * 1e-3) / 1e9 / hbm_peak,
            "roofline": {"bound": "hbm", "kernel": "sweep_kernel", "achieved": sweep_gbs,
                         "peak": hbm_peak, "unit": "GB/s", "frac": sweep_gbs / hbm_peak,
                         "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "traffic": ncu_traffic(self.name),
                         "bytes_per_launch": rep.sweep_bytes},
            "kernels_ms": {"plan": k_plan, "sweep": k_sweep, "final": k_final},
            "round_ms_percentiles": round_pct,
            "round_bytes": {"sweep": rep.sweep_bytes, "final": rep.final_bytes},
            "e2e": e2e,
            "e2e_padded": e2e_padded,
            "e2e_direct": e2e_direct,
            "e2e_copy": e2e_copy,
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
        }
        if full is not None:
            full["sweep_frac"] = full["sweep_gbs"] / hbm_peak
            result["full_sweep"] = full
        if packed is not None:
            result["packed"] = packed
        if opd is not None:
            opd["frac"] = opd["gbs"] / hbm_peak
            result["opd"] = opd
        if opd_fused is not None:
            opd_fused["frac"] = opd_fused["gbs"] / hbm_peak
            opd_fused["separate_ms"] = ms + (opd["ms_per_call"] if opd else 0.0)
            result["opd_fused"] = opd_fused
        if d3d is not None:
            result["d3d"] = d3d
        if per_workload is not None:
            result["per_workload"] = per_workload
        if world == 1 and not args.no_cpu_baseline:
            self.cpu_baseline(result, round_bytes)
        print(json.dumps(result), flush=True)


def run_ours(args, world, rank, local):
    OurArm(args, world, rank, local).run()


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
