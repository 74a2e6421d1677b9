#!/usr/bin/env python
"""Benchmark: batched speculative-decoding verification rounds/s and HBM GB/s on GB300.

One step = one verification round = one ``spec_verify`` call over a whole
batch (plan -> row sweep -> final pass).  Default workload: B=128 requests,
k=16 draft positions, V=151936, bf16 logits, half the requests with low and
half with high draft noise (see speculative_decoding_verification_58_gb300/synth.py).

Prints one JSON line.  ``value`` is verification rounds per second over all
ranks (each rank verifies its own batch: weak scaling, no collective on the
data path), with inputs resident in HBM.  The logits (1.28 GB at the default
workload) are far larger than L2, so no flush is needed between steps.

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
    """Digest of the sources the sweep kernel is built from (its code, the
    shared helpers and the plan kernel that lays out its work)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_58_gb300", "csrc")
    files = [os.path.join(csrc, name) for name in ("common.cuh", "plan.cuh", "sweep.cuh")]
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
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


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    from speculative_decoding_verification_58_gb300 import synth

    name = args.workload or synth.HEADLINE
    cfg = synth.WORKLOADS[name]
    inp = synth.make_workload(name, seed=args.seed)
    oracle.build()
    sample_b = max(1, inp.B // 16)

    def step(j):
        lo = (j * sample_b) % inp.B
        sl = slice(lo, lo + sample_b)
        oracle.verify(inp.target[sl], inp.draft[sl], inp.tokens[sl], inp.lengths[sl],
                      inp.uniforms[sl], inp.temperature[sl])

    for j in range(args.warmup):
        step(j)
    t0 = time.perf_counter()
    for j in range(args.steps):
        step(args.warmup + j)
    dt = time.perf_counter() - t0
    sec_per_round = dt / args.steps * (inp.B / sample_b)
    value = 1.0 / sec_per_round
    sample = (f"{sample_b} of the {inp.B} requests per step (rotating), scaled to a full "
              f"{inp.B}-request round; single-threaded fp64 C++ oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rounds/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec_per_round * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "B": cfg["B"], "k": cfg["k"], "V": cfg["V"],
                   "logits": cfg["dtype"]},
        "cpu_baseline": {"value": value, "unit": "rounds/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def run_ours(args, world, rank, local):
    import torch

    import speculative_decoding_verification_58_gb300 as sv
    from speculative_decoding_verification_58_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks(world, dev, "nccl")
    sv.lib()

    name = args.workload or synth.HEADLINE
    cfg = synth.WORKLOADS[name]
    seed = replica_seed(args.seed if args.seed is not None else cfg["seed"], rank)
    inp = synth.make_workload(name, seed=seed)
    esize = 2 if inp.dtype == "bf16" else 4
    d = sv.to_device(inp, dev)
    ws = sv.alloc_workspace(inp.B, inp.k, inp.V, dev)
    out = torch.empty((inp.B, inp.k + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty(inp.B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # Bound calls: buffers checked once, one C call per round.
    bound = {fs: sv.Verifier(**d, workspace=ws, out_tokens=out, num_accepted=nacc, stream=stream,
                             full_sweep=fs) for fs in (False, True)}

    def step(full_sweep=False, events=None):
        if events is None:
            bound[full_sweep]()
        else:
            sv.spec_verify(**d, workspace=ws, out_tokens=out, num_accepted=nacc, stream=stream,
                           full_sweep=full_sweep, events=events)

    barrier, max_over_ranks = ranks.barrier, ranks.max

    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local))

    # Warm-up, then the timed region: K rounds, device-timed with events on the launch stream.
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    logit_bytes = inp.target.nbytes + inp.draft.nbytes
    flush = logit_bytes < 2 * L2_BYTES
    if not flush:
        # Inputs larger than L2: back-to-back rounds, one pair of events around all.
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = e0.elapsed_time(e1)
    else:
        # Inputs that fit in L2: overwrite a buffer larger than L2 before every
        # round and time each round alone.
        scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        for a, b in pairs:
            scrub.fill_(1)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = sum(a.elapsed_time(b) for a, b in pairs)
    barrier()
    ms = max_over_ranks(total_ms / args.steps)
    rep = sv.spec_verify_report(ws, stream)
    gpu_out, gpu_n = out.cpu().numpy(), nacc.cpu().numpy()

    # Round-time distribution: an event pair around each round (the events sit
    # between rounds, so a round cannot start under the previous one's tail).
    preps = max(10, min(args.steps, 200))
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(preps)]
    for a_, b_ in rev:
        a_.record(stream)
        step()
        b_.record(stream)
    torch.cuda.synchronize(dev)
    rts = sorted(a_.elapsed_time(b_) for a_, b_ in rev)
    round_pct = {"p10": rts[int(0.1 * (preps - 1))], "p50": rts[(preps - 1) // 2],
                 "p90": rts[int(0.9 * (preps - 1))], "rounds": preps, "unit": "ms"}

    # Per-kernel durations: the same rounds with events between the kernels.
    kreps = max(10, min(args.steps, 200))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(kreps)]
    for row in evs:
        for e in row:
            e.record(stream)  # creates the handles
    torch.cuda.synchronize(dev)
    for row in evs:
        step(events=row)
    torch.cuda.synchronize(dev)
    k_plan = statistics.mean(r[0].elapsed_time(r[1]) for r in evs)
    k_sweep = statistics.mean(r[1].elapsed_time(r[2]) for r in evs)
    k_final = statistics.mean(r[2].elapsed_time(r[3]) for r in evs)

    # Same workload with early exit switched off (every row i < L_b is swept).
    full = None
    if not args.no_full_sweep:
        for _ in range(3):
            step(full_sweep=True)
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(kreps)]
        for row in fev:
            for e in row:
                e.record(stream)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(kreps):
            step(full_sweep=True)
        f1.record(stream)
        torch.cuda.synchronize(dev)
        frep = sv.spec_verify_report(ws, stream)
        for row in fev:
            step(full_sweep=True, events=row)
        torch.cuda.synchronize(dev)
        fsweep = statistics.mean(r[1].elapsed_time(r[2]) for r in fev)
        full = {"ms_per_step": f0.elapsed_time(f1) / kreps, "sweep_ms": fsweep,
                "sweep_bytes": frep.sweep_bytes,
                "sweep_gbs": frep.sweep_bytes / (fsweep * 1e-3) / 1e9}

    # The same batch packed (AdaFlash Section 3.3: total length sum_b L_b rows
    # instead of B x k): same outputs, a smaller resident footprint.
    packed = None
    if not args.no_packed:
        pk = synth.pack_rows(inp)
        rows = sv.to_device_packed(pk, dev)
        pargs = dict(**rows, draft_tokens=d["draft_tokens"], lengths=d["lengths"],
                     uniforms=d["uniforms"], temperature=d["temperature"], workspace=ws,
                     out_tokens=out, num_accepted=nacc, stream=stream)
        for _ in range(3):
            sv.spec_verify_packed(**pargs)
        torch.cuda.synchronize(dev)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(kreps):
            sv.spec_verify_packed(**pargs)
        p1.record(stream)
        torch.cuda.synchronize(dev)
        same = bool(np.array_equal(out.cpu().numpy(), gpu_out) and
                    np.array_equal(nacc.cpu().numpy(), gpu_n))
        pms = p0.elapsed_time(p1) / kreps
        packed = {"ms_per_step": pms, "value": 1000.0 / pms, "unit": "rounds/s",
                  "logit_bytes": int(pk.target_rows.nbytes + pk.draft_rows.nbytes),
                  "padded_logit_bytes": int(logit_bytes), "same_outputs_as_padded": same}
        del rows, pargs
        torch.cuda.empty_cache()

    # OPD supervision statistics (AdaFlash Section 3.1) on the same buffers:
    # both rows of every verified position read once.
    opd = None
    if not args.no_opd:
        st = sv.spec_opd_stats(d["target_logits"], d["draft_logits"], d["lengths"], stream=stream)
        for _ in range(3):
            sv.spec_opd_stats(d["target_logits"], d["draft_logits"], d["lengths"], out=st,
                              stream=stream)
        torch.cuda.synchronize(dev)
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        oreps = max(10, min(args.steps, 100))
        o0.record(stream)
        for _ in range(oreps):
            sv.spec_opd_stats(d["target_logits"], d["draft_logits"], d["lengths"], out=st,
                              stream=stream)
        o1.record(stream)
        torch.cuda.synchronize(dev)
        oms = o0.elapsed_time(o1) / oreps
        positions = int(inp.lengths.sum())
        obytes = positions * 2 * inp.V * esize
        opd = {"ms_per_call": oms, "positions": positions, "positions_per_s": positions / (oms * 1e-3),
               "bytes_per_call": obytes, "gbs": obytes / (oms * 1e-3) / 1e9,
               "loss_mean": float(st.loss.float().mean().item())}

    # D3D branch selection on this round's outcome: the paper's main budget
    # (block 16, coverage C = 12, fan-out F = 2, 24 branches per request).
    d3d = None
    if not args.no_d3d:
        br = synth.make_d3d_branches(inp.lengths, inp.V, C=12, F=2, blk=16, seed=seed + 7)
        tb = {key: torch.from_numpy(getattr(br, key)).to(dev) for key in ("pos", "tok", "block")}
        hit, nxt, hits = sv.spec_d3d_select(nacc, out, tb["pos"], tb["tok"], tb["block"],
                                            stream=stream)
        for _ in range(3):
            sv.spec_d3d_select(nacc, out, tb["pos"], tb["tok"], tb["block"], hit=hit,
                               next_block=nxt, hits=hits, stream=stream)
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(kreps):
            sv.spec_d3d_select(nacc, out, tb["pos"], tb["tok"], tb["block"], hit=hit,
                               next_block=nxt, hits=hits, stream=stream)
        g1.record(stream)
        torch.cuda.synchronize(dev)
        d3d = {"us_per_call": g0.elapsed_time(g1) / kreps * 1000, "requests": inp.B,
               "branches_per_request": int(br.pos.shape[1]), "block": 16,
               "hit_rate": int(hits.item()) / inp.B,
               "note": "branch tokens are uniform draws, so hits are rare; latency-bound"}

    # End to end through the public API: pinned host inputs in, results out, every step.
    import numpy as _np
    host = {}
    for key, t in d.items():
        host[key] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        host[key].copy_(t.cpu())
    h_out = torch.empty(out.shape, dtype=torch.int32, pin_memory=True)
    h_n = torch.empty(nacc.shape, dtype=torch.int32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = h_out.numel() * 4 + h_n.numel() * 4
    e2e_steps = args.e2e_steps or max(5, min(50, args.steps))

    def e2e_step():
        for key, t in host.items():
            d[key].copy_(t, non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        h_n.copy_(nacc, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_padded_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps)

    # The same, with the batch packed (AdaFlash Section 3.3): the host sends
    # only the rows a round can read (rows 0..L_b), which is what a serving
    # engine's packed verification batch holds.
    pk_host = synth.pack_rows(inp)
    hp = {key: torch.from_numpy(np.ascontiguousarray(v)).pin_memory()
          for key, v in (("target_row_start", pk_host.target_row_start),
                         ("draft_row_start", pk_host.draft_row_start))}
    for key, v in (("target_rows", pk_host.target_rows), ("draft_rows", pk_host.draft_rows)):
        t = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16 \
            else torch.from_numpy(v)
        hp[key] = t.pin_memory()
    for key in ("draft_tokens", "lengths", "uniforms", "temperature"):
        hp[key] = host[key]
    dp = {key: torch.empty(t.shape, dtype=t.dtype, device=dev) for key, t in hp.items()}
    h2d_packed = sum(t.numel() * t.element_size() for t in hp.values())

    def e2e_packed_step():
        for key, t in hp.items():
            dp[key].copy_(t, non_blocking=True)
        sv.spec_verify_packed(**dp, workspace=ws, out_tokens=out, num_accepted=nacc,
                              stream=stream)
        h_out.copy_(out, non_blocking=True)
        h_n.copy_(nacc, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        e2e_packed_step()
    e2e_same = bool(np.array_equal(h_out.numpy(), gpu_out) and np.array_equal(h_n.numpy(), gpu_n))
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_packed_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps)
    del dp
    clocks = sampler.stop()
    barrier()

    if rank != 0:
        return

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    sweep_gbs = rep.sweep_bytes / (k_sweep * 1e-3) / 1e9
    round_bytes = rep.sweep_bytes + rep.final_bytes
    value = aggregate_value(world, ms)

    result = {
        "metric": METRIC, "value": value, "unit": "rounds/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": name, "B": inp.B, "k": inp.k, "V": inp.V, "logits": inp.dtype,
                   "seed": seed, "parallelism": f"replicas x{world}",
                   "l2": (f"L2 flushed before every round ({logit_bytes / 1e6:.1f} MB of logits)"
                          if flush else
                          f"inputs larger than L2: {logit_bytes / 1e9:.2f} GB of logits resident, "
                          "no flush between steps"),
                   "early_exit": True},
        "hbm_gbs": round_bytes / (ms * 1e-3) / 1e9,
        "hbm_gbs_frac": round_bytes / (ms * 1e-3) / 1e9 / hbm_peak,
        "roofline": {"bound": "hbm", "kernel": "sweep_kernel", "achieved": sweep_gbs,
                     "peak": hbm_peak, "unit": "GB/s", "frac": sweep_gbs / hbm_peak,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind ==
                     "measured" else "fallback 6.8 TB/s",
                     "traffic": ncu_traffic(name),
                     "bytes_per_launch": rep.sweep_bytes},
        "kernels_ms": {"plan": k_plan, "sweep": k_sweep, "final": k_final},
        "round_ms_percentiles": round_pct,
        "round_bytes": {"sweep": rep.sweep_bytes, "final": rep.final_bytes},
        "e2e": {"value": world / e2e_s, "unit": "rounds/s", "h2d_bytes_per_step": h2d_packed,
                "d2h_bytes_per_step": d2h, "layout": "packed (rows 0..L_b of each request)",
                "same_outputs": e2e_same},
        "e2e_padded": {"value": world / e2e_padded_s, "unit": "rounds/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "layout": "padded [B, k+1, V] / [B, k, V]"},
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
    if d3d is not None:
        result["d3d"] = d3d

    if world == 1 and not args.no_cpu_baseline:
        import oracle
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
        same = (gpu_n == o.num_accepted) & _np.all(gpu_out == o.out_tokens, axis=1)
        near = o.margin < 1e-6
        m1, m2 = model_bytes(inp, o, esize)
        result["parity"] = {"requests": int(inp.B), "mismatches": int((~same).sum()),
                            "outside_near_tie_band": int((~same & ~near).sum()),
                            "near_ties": int(near.sum())}
        result["byte_models"] = {"M1_all_rows": m1, "M2_rows_to_first_reject": m2,
                                 "moved": round_bytes,
                                 "M1_gbs": m1 / (ms * 1e-3) / 1e9,
                                 "mean_accepted": float(o.num_accepted.mean())}
    print(json.dumps(result), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
