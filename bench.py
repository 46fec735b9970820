"""Benchmark: soft-capped attention forward + backward on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl capattn|reference]
                    [--workload 2] [--no-cpu-baseline] [--no-e2e] [--no-per-workload]

A step is one forward (capattn_fwd) and one backward (capattn_bwd_ex, reusing
the spans and visit maps the forward left in the shared workspace) over the
workload's batch of synthetic seeded inputs.  The default workload is
causal_tanh: B=2, Hq=Hkv=16, L=2048, D=128, bf16, causal, tanh cap 50.

Metric: mask-aware TFLOP/s of forward + backward, 14 * D * N FLOPs per step
(N = unmasked (query, key) pairs summed over batch and heads, counted by the
oracle from the seeded masks and stored in tests/golden/pair_counts.json).

Timing: inputs resident in HBM; an L2 flush (a 512 MB write) runs before every
timed step, outside the events; each step is bracketed by CUDA events on the
stream the kernels run on; exactly K steps are timed.  `value` = total FLOPs /
summed step time.  Clock samples (nvidia-smi) cover an untimed soak of about a
second of the same step right before the timed steps, and the timed steps.
`e2e` repeats the step through the same C ABI with pinned host buffers:
host-to-device copies of Q, K, V, dO (+ temperature, segments, bounds), the
forward, the backward and device-to-host copies of O, LSE, dQ, dK, dV, all
inside the timed region (dO's copy overlaps the forward and O / LSE leave
during the backward, on a second stream).

`per_workload` (single process only) measures every workload of the table the
same way (fwd / bwd split from a pass with every kernel bracketed by events),
with the fp64 oracle's forward and backward seconds on one (batch, KV head)
plane of each on the host cores.

Multi-GPU: each rank runs an independent replica of the workload (the path
shards over (batch, KV head) without any exchange), timing is the max over
ranks and `value` sums all ranks' FLOPs ("scaling": "weak").

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (whole (batch, head) planes, forward + backward) on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from soft_capped_attention_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

PAIR_COUNTS = os.path.join(ROOT, "tests", "golden", "pair_counts.json")
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "capped-attention fwd+bwd TFLOP/s (mask-aware) and % of GB300 BF16 peak"
# Algorithmic FLOPs per unmasked pair and head dim, per kernel: the forward
# does Q K^T and P V; the dK/dV kernel recomputes S and does dP, dV, dK; the dQ
# kernel's own product is dQ (its S and dP recomputations are not counted).
KERNEL_FLOPS_PER_PAIR_D = {"fwd": 4, "dkv": 8, "dq": 2}
SOAK_SECONDS = 1.0  # default of --soak-seconds


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over all ranks (the slowest rank's
    times), or the list itself in a single process."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return [float(x) for x in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def pairs_of(idx: int) -> int:
    with open(PAIR_COUNTS) as f:
        return int(json.load(f)[str(idx)]["pairs"])


def read_peak():
    try:
        with open(PEAKS) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def config_of(w, idx: int, world: int, dtemp: bool = False) -> dict:
    """The workload's description, identical in both arms."""
    N = pairs_of(idx)
    return {"workload": w.name, "B": w.B, "L": w.L, "Lk": w.key_len, "Hq": w.Hq, "Hkv": w.Hkv,
            "D": w.D, "causal": w.causal, "window_len": w.window_len,
            "cap": [w.cap_method, w.cap, w.alpha, w.beta], "z_loss_weight": w.z_loss_weight,
            "temperature": None if w.temp_range is None else list(w.temp_range),
            "packed_documents": None if w.doc_len_range is None else list(w.doc_len_range),
            "ranker_bounds": None if w.ranker_hu_range is None else
            {"hu": list(w.ranker_hu_range), "candidates": list(w.ranker_cand_range)},
            "unmasked_pairs": N, "flops_per_step": 14.0 * w.D * N, "dtemp": dtemp,
            "parallelism": f"replicas x{world}"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index),
                                      f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits"],
                                     capture_output=True, text=True, timeout=5).stdout.strip()
                if out:
                    self.samples.append([x.strip() for x in out.split(",")])
            except Exception:
                pass
            self._stop.wait(0.02)

    def __enter__(self):
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        pw = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for n, v in zip(names, s[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.samples), "power_w_max": max(pw) if pw else None,
                "window": "an untimed soak of the same step (--soak-seconds), then the timed steps"}


_C_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def kernel_source_hash(csrc: str = None) -> str:
    """Hash of the kernel sources' code: C / C++ / CUDA files without their
    comments and with whitespace collapsed (a comment edit keeps the hash),
    other files as they are."""
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "soft_capped_attention_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        path = os.path.join(csrc, f)
        if not os.path.isfile(path):
            continue
        with open(path, "rb") as fh:
            data = fh.read()
        if f.endswith((".cu", ".cuh", ".h", ".cpp", ".c")):
            data = " ".join(_C_COMMENT.sub(" ", data.decode()).split()).encode()
        h.update(f.encode() + data)
    return h.hexdigest()[:16]


_INCLUDE = re.compile(r'#include\s+"([^"]+)"')


def kernel_files(source: str, csrc: str = None) -> list:
    """A kernel's translation unit, the csrc headers it includes (transitively)
    and the host layer that sizes its launches and workspace."""
    csrc = csrc or os.path.join(ROOT, "soft_capped_attention_gb300", "csrc")
    seen, todo = set(), [source, "capattn_api.cu"]
    while todo:
        f = os.path.normpath(todo.pop())
        if f in seen or not os.path.isfile(os.path.join(csrc, f)):
            continue  # (system headers)
        seen.add(f)
        with open(os.path.join(csrc, f)) as fh:
            base = os.path.dirname(f)
            todo.extend(os.path.join(base, i) for i in _INCLUDE.findall(fh.read()))
    return sorted(seen)


def files_hash(files, csrc: str = None) -> str:
    """kernel_source_hash over the given csrc files only."""
    csrc = csrc or os.path.join(ROOT, "soft_capped_attention_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(csrc, f), "rb") as fh:
            data = fh.read()
        if f.endswith((".cu", ".cuh", ".h", ".cpp", ".c")):
            data = " ".join(_C_COMMENT.sub(" ", data.decode()).split()).encode()
        h.update(f.encode() + data)
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """ncu DRAM bytes per launch of `kernel` on `workload`, if taken on this
    kernel's code (its source file with the headers it includes, when the
    capture names it; otherwise all kernel sources)."""
    try:
        with open(TRAFFIC) as f:
            t = json.load(f)
        e = t[workload][kernel]
        src = e.get("source_file")
        now = files_hash(kernel_files(src)) if src else kernel_source_hash()
        if e.get("source_hash") != now:
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# capattn arm
# ---------------------------------------------------------------------------

class Run:
    """One workload's inputs resident on the device and its forward + backward step."""

    def __init__(self, idx: int, dev, dtemp: bool = False):
        from soft_capped_attention_gb300 import capattn as ca
        self.ca = ca
        self.idx = idx
        self.w = w = WORKLOADS[idx]
        self.inp = inp = make_inputs(w, seed=idx)
        self.dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.ap = ca.params_from_workload(w)
        self.host = {n: torch.from_numpy(inp[n]).to(self.dtype).contiguous() for n in ("q", "k", "v", "do")}
        self.aux = {n: (None if inp[n] is None else torch.from_numpy(inp[n]).contiguous())
                    for n in ("temp", "seg", "bounds")}
        self.d = {n: t.to(dev) for n, t in self.host.items()}
        self.da = {n: (None if t is None else t.to(dev)) for n, t in self.aux.items()}
        self.cfg = ca.make_config(self.ap, w.B, w.L, w.Hq, w.Hkv, w.D, self.dtype, Lk=w.key_len)
        self.ws = ca.new_workspace(self.cfg, dev)
        self.dev = dev
        self.dtemp = dtemp and self.aux["temp"] is not None
        if dtemp and not self.dtemp:
            raise SystemExit("--dtemp needs a workload with a temperature")
        self.N = pairs_of(idx)
        self.flops = 14.0 * w.D * self.N

    def bwd(self, q, k, v, o, lse, do, temp, seg, bounds):
        """The backward of the forward just run on self.ws with the same inputs:
        it reuses that forward's spans and visit maps."""
        return self.ca.capattn_bwd_ex(q, k, v, o, lse, do, self.ap, temp, seg, bounds,
                                      want_dtemp=self.dtemp, workspace=self.ws,
                                      reuse_fwd_maps=True)[:3]

    def step(self, stream=None, split=False):
        d, da = self.d, self.da
        o, lse, _, _ = self.ca.capattn_fwd(d["q"], d["k"], d["v"], self.ap, da["temp"], da["seg"],
                                           da["bounds"], workspace=self.ws)
        ev_mid = None
        if split:
            ev_mid = torch.cuda.Event(enable_timing=True)
            ev_mid.record(stream)
        self.bwd(d["q"], d["k"], d["v"], o, lse, d["do"], da["temp"], da["seg"], da["bounds"])
        return ev_mid


def breakdown_pass(run: Run, steps: int, flush, stream):
    """Every library kernel bracketed by events and a mark between forward and
    backward: per-kernel milliseconds and launches, and the fwd / bwd split."""
    ca = run.ca
    ca.capattn_profile_select(None)
    ca.capattn_profile_enable(True)
    ca.capattn_profile_read(reset=True)
    split = []
    for _ in range(steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e1 = run.step(stream, split=True)
        e2.record(stream)
        split.append((e0, e1, e2))
    torch.cuda.synchronize()
    prof = ca.capattn_profile_read(reset=True)
    ca.capattn_profile_enable(False)
    fw = sum(a.elapsed_time(b) for a, b, _ in split)
    bw = sum(b.elapsed_time(c) for _, b, c in split)
    kern_ms = {k: v[0] for k, v in prof.items() if v[1] > 0}
    launches = {k: v[1] for k, v in prof.items()}
    dom = max(KERNEL_FLOPS_PER_PAIR_D, key=lambda k: kern_ms.get(k, 0.0))
    return fw, bw, kern_ms, launches, dom


def timed_steps(run: Run, steps: int, flush, stream):
    """Exactly `steps` steps, each bracketed by events; returns summed milliseconds."""
    times = []
    for _ in range(steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run.step(stream)
        e2.record(stream)
        times.append((e0, e2))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in times)


def check_status(run: Run):
    st, bits = run.ca.capattn_device_status(run.ws)
    if st != 0:
        raise RuntimeError(f"{run.w.name}: device status {st} (bits {bits})")


def e2e_measure(run: Run, args, world, dev, stream, flush):
    """The step from pinned host buffers: inputs copied in and results copied out
    inside the timed region (dO's copy overlaps the forward on a second
    stream; O and LSE leave during the backward)."""
    ca, w = run.ca, run.w
    ph = {n: t.pin_memory() for n, t in run.host.items()}
    pa = {n: (None if t is None else t.pin_memory()) for n, t in run.aux.items()}
    out_h = {"o": torch.empty_like(ph["q"]).pin_memory(),
             "lse": torch.empty(w.B, w.Hq, w.L, dtype=torch.float32).pin_memory(),
             "dq": torch.empty_like(ph["q"]).pin_memory(),
             "dk": torch.empty_like(ph["k"]).pin_memory(),
             "dv": torch.empty_like(ph["v"]).pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in ph.values()) + \
        sum(t.numel() * t.element_size() for t in pa.values() if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in out_h.values())
    dbuf = {n: torch.empty_like(t, device=dev) for n, t in ph.items()}
    dabuf = {n: (None if t is None else torch.empty_like(t, device=dev)) for n, t in pa.items()}
    side = torch.cuda.Stream(dev)

    def e2e_step():
        start = torch.cuda.Event()
        start.record(stream)
        side.wait_event(start)
        with torch.cuda.stream(side):
            dbuf["do"].copy_(ph["do"], non_blocking=True)
        ev_do = torch.cuda.Event()
        ev_do.record(side)
        for n in ("q", "k", "v"):
            dbuf[n].copy_(ph[n], non_blocking=True)
        for n in pa:
            if pa[n] is not None:
                dabuf[n].copy_(pa[n], non_blocking=True)
        o, lse, _, _ = ca.capattn_fwd(dbuf["q"], dbuf["k"], dbuf["v"], run.ap, dabuf["temp"],
                                      dabuf["seg"], dabuf["bounds"], workspace=run.ws)
        ev_fwd = torch.cuda.Event()
        ev_fwd.record(stream)
        side.wait_event(ev_fwd)
        with torch.cuda.stream(side):
            out_h["o"].copy_(o, non_blocking=True)
            out_h["lse"].copy_(lse, non_blocking=True)
        stream.wait_event(ev_do)
        dq, dk, dv = run.bwd(dbuf["q"], dbuf["k"], dbuf["v"], o, lse, dbuf["do"], dabuf["temp"],
                             dabuf["seg"], dabuf["bounds"])
        out_h["dq"].copy_(dq, non_blocking=True)
        out_h["dk"].copy_(dk, non_blocking=True)
        out_h["dv"].copy_(dv, non_blocking=True)
        ev_side = torch.cuda.Event()
        ev_side.record(side)
        stream.wait_event(ev_side)
        o.record_stream(side)
        lse.record_stream(side)

    for _ in range(max(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    etot = 0.0
    for _ in range(args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b_ = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b_.record(stream)
        b_.synchronize()
        etot += a.elapsed_time(b_)
    if world > 1:
        etot = max_over_ranks([etot], dev)[0]
    check_status(run)
    return {"value": round(run.flops * args.steps * world / (etot * 1e-3) / 1e12, 3),
            "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(etot / args.steps, 4),
            "overlap": "dO's copy overlaps the forward and O / LSE leave during the backward (second stream)"}


def per_workload_measure(args, dev, stream, flush, headline: dict):
    """Every workload of the table, the headline's numbers reused."""
    peak, _ = read_peak()
    out = {}
    for idx in sorted(WORKLOADS):
        if idx == args.workload:
            out[WORKLOADS[idx].name] = headline
            continue
        run = Run(idx, dev)
        steps = max(3, args.per_workload_steps)
        for _ in range(3):
            flush.zero_()
            run.step(stream)
        torch.cuda.synchronize()
        check_status(run)
        fw, bw, kern_ms, launches, dom = breakdown_pass(run, steps, flush, stream)
        tot = timed_steps(run, steps, flush, stream)
        check_status(run)
        D, N = run.w.D, run.N
        value = run.flops * steps / (tot * 1e-3) / 1e12
        out[run.w.name] = {
            "workload": idx, "dtype": run.w.dtype, "unmasked_pairs": N, "steps": steps,
            "fwd_bwd_tflops": round(value, 3), "frac_of_peak": round(value / peak, 4),
            "fwd_tflops": round(4.0 * D * N * steps / (fw * 1e-3) / 1e12, 3),
            "bwd_tflops": round(10.0 * D * N * steps / (bw * 1e-3) / 1e12, 3),
            "ms_per_step": round(tot / steps, 4), "dominant_kernel": dom,
            "kernel_ms_per_launch": {k: round(kern_ms[k] / max(launches[k], 1), 4) for k in kern_ms}}
        del run
        torch.cuda.empty_cache()
    return out


def run_capattn(args, rank, world, local_rank):
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    run = Run(args.workload, dev, dtemp=args.dtemp)
    ca, w = run.ca, run.w
    use_dtemp = run.dtemp
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        flush.zero_()
        run.step(stream)
    torch.cuda.synchronize()
    check_status(run)

    D, N = w.D, run.N
    flops_step = run.flops

    # Breakdown pass (not the headline): every kernel bracketed by events and a
    # mark between forward and backward.  Each recorded event costs the stream a
    # few microseconds, so the headline run below records only the events of the
    # kernel its roofline names.
    fw, bw, kern_ms_all, launches_all, dom = breakdown_pass(run, args.steps, flush, stream)
    total_kernel_ms = sum(kern_ms_all.values())

    # Headline run: step events plus the events of the roofline kernel only,
    # after an untimed soak of the same step under the clock sampler.
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    step_ms_est = (fw + bw) / max(args.steps, 1)
    soak = int(args.soak_seconds / max(step_ms_est * 1e-3 + 1e-4, 1e-6)) if args.soak_seconds > 0 else 0
    with ClockSampler(local_rank) as clk:
        for _ in range(soak):
            flush.zero_()
            run.step(stream)
        ca.capattn_profile_select([dom])
        ca.capattn_profile_enable(True)
        ca.capattn_profile_read(reset=True)
        tot = timed_steps(run, args.steps, flush, stream)
        prof = ca.capattn_profile_read(reset=True)
        ca.capattn_profile_enable(False)
        ca.capattn_profile_select(None)
    check_status(run)
    if world > 1:
        torch.distributed.barrier()
    ms_step = tot / args.steps
    if world > 1:
        tot, fw, bw = max_over_ranks([tot, fw, bw], dev)
        ms_step = tot / args.steps

    value = flops_step * args.steps * world / (tot * 1e-3) / 1e12
    fwd_tf = 4.0 * D * N * args.steps * world / (fw * 1e-3) / 1e12
    bwd_tf = 10.0 * D * N * args.steps * world / (bw * 1e-3) / 1e12
    peak, peak_src = read_peak()

    # roofline: the kernel with the largest share of device time, its duration
    # taken in the headline run
    launches = {k: v[1] for k, v in prof.items()}
    gpu_launches = int(sum(launches.values()))
    per_launch_ms = prof[dom][0] / max(launches[dom], 1)
    ach = KERNEL_FLOPS_PER_PAIR_D[dom] * D * N / (per_launch_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(ach, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(ach / peak, 4), "peak_source": peak_src,
                "traffic": traffic_for(dom, w.name),
                "kernel_ms_per_launch_headline": round(per_launch_ms, 4),
                "kernel_ms_per_launch": {k: round(kern_ms_all[k] / max(launches_all[k], 1), 4)
                                         for k in kern_ms_all},
                "kernel_share": {k: round(kern_ms_all[k] / total_kernel_ms, 4) for k in kern_ms_all},
                "breakdown": "kernel_ms_per_launch / kernel_share from a separate pass with every "
                             "kernel bracketed by events"}

    e2e = None if args.no_e2e else e2e_measure(run, args, world, dev, stream, flush)

    headline = {"workload": args.workload, "dtype": w.dtype, "unmasked_pairs": N,
                "steps": args.steps, "fwd_bwd_tflops": round(value / world, 3),
                "frac_of_peak": round(value / world / peak, 4), "fwd_tflops": round(fwd_tf / world, 3),
                "bwd_tflops": round(bwd_tf / world, 3), "ms_per_step": round(ms_step, 4),
                "dominant_kernel": dom, "kernel_ms_per_launch": roofline["kernel_ms_per_launch"]}
    per_wl = None
    if world == 1 and not args.no_per_workload:
        del run
        torch.cuda.empty_cache()
        per_wl = per_workload_measure(args, dev, stream, flush, headline)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(WORKLOADS[args.workload], args.workload, args.cpu_seconds)
        if per_wl is not None:
            for idx in sorted(WORKLOADS):
                per_wl[WORKLOADS[idx].name]["cpu_oracle"] = oracle_fwd_bwd_plane(idx)

    clocks = clk.summary()
    line = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded normal Q, K, V, dO; seeded masks)",
            "config": config_of(w, args.workload, world, use_dtemp),
            "l2": "flushed before every timed step",
            "fwd_tflops": round(fwd_tf, 3), "bwd_tflops": round(bwd_tf, 3),
            "fwd_bwd_split": "from the breakdown pass (events around every kernel)",
            "frac_of_peak": round(value / peak, 4), "peak_tflops": peak, "peak_source": peak_src,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
            "clocks": clocks, "per_workload": per_wl}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

_ORACLE_INPUTS = {}


def _oracle_inputs(w, idx):
    if idx not in _ORACLE_INPUTS:
        _ORACLE_INPUTS.clear()
        _ORACLE_INPUTS[idx] = make_inputs(w, seed=idx)
    return _ORACLE_INPUTS[idx]


def _plane_pairs(w, inp, cfg, b):
    from oracle import capattn_oracle as orc
    return orc.pair_count(w.L, cfg, None if inp["seg"] is None else inp["seg"][b:b + 1],
                          None if inp["bounds"] is None else inp["bounds"][b:b + 1], B=1,
                          Lk=w.key_len)


def oracle_sample(w, idx, seconds: float, start: int = 0):
    """Runs the oracle forward + backward on whole (batch, KV head) planes of the
    workload, starting at plane `start`, until `seconds` elapse (at least one
    plane); returns (FLOPs counted mask-aware, seconds, planes)."""
    from oracle import capattn_oracle as orc
    inp = _oracle_inputs(w, idx)
    cfg = orc.config_from_workload(w)
    flops = 0.0
    t0 = time.perf_counter()
    planes = 0
    nplanes = w.B * w.Hkv
    for pidx in range(start, start + nplanes):
        b, g = divmod(pidx % nplanes, w.Hkv)
        orc.backward_kv_head(inp["q"], inp["k"], inp["v"], inp["temp"], inp["seg"],
                             inp["bounds"], inp["do"], cfg, b, g)
        flops += 14.0 * w.D * _plane_pairs(w, inp, cfg, b) * w.G
        planes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return flops, time.perf_counter() - t0, planes


def oracle_fwd_bwd_plane(idx):
    """The oracle's forward and backward seconds, timed apart, on plane (b=0,
    KV head 0) of workload idx (its G query heads), and the TFLOP/s they give."""
    from oracle import capattn_oracle as orc
    w = WORKLOADS[idx]
    inp = _oracle_inputs(w, idx)
    cfg = orc.config_from_workload(w)
    G = w.G
    sl = lambda x: None if x is None else x[0:1]
    q, do = inp["q"][0:1, :, 0:G], inp["do"][0:1, :, 0:G]
    k, v = inp["k"][0:1, :, 0:1], inp["v"][0:1, :, 0:1]
    t0 = time.perf_counter()
    O, LSE, _, _ = orc.forward(q, k, v, sl(inp["temp"]), sl(inp["seg"]), sl(inp["bounds"]), cfg)
    t1 = time.perf_counter()
    orc.backward(q, k, v, sl(inp["temp"]), sl(inp["seg"]), sl(inp["bounds"]), O, LSE, do, cfg)
    t2 = time.perf_counter()
    n = _plane_pairs(w, inp, cfg, 0) * G
    return {"fwd_s": round(t1 - t0, 4), "bwd_s": round(t2 - t1, 4),
            "fwd_tflops": round(4.0 * w.D * n / (t1 - t0) / 1e12, 6),
            "bwd_tflops": round(10.0 * w.D * n / (t2 - t1) / 1e12, 6),
            "cores": len(os.sched_getaffinity(0)),
            "sample": f"plane (batch 0, KV head 0) with its {G} query head(s), fp64"}


def cpu_baseline(w, idx, seconds):
    cores = len(os.sched_getaffinity(0))
    flops, secs, planes = oracle_sample(w, idx, seconds)
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{planes} (batch, KV head) plane(s) of {w.name}, fp64 forward + backward, "
                      f"{secs:.1f} s, numpy BLAS threads on {cores} host cores"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    for i in range(args.warmup):
        oracle_sample(w, args.workload, 0.0, start=i)
    flops = secs = 0.0
    planes = 0
    for i in range(args.steps):
        f, s, p = oracle_sample(w, args.workload, 0.0, start=i)
        flops += f
        secs += s
        planes += p
    cores = len(os.sched_getaffinity(0))
    value = flops / secs / 1e12
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded normal Q, K, V, dO; seeded masks)", "impl": "reference",
            "config": config_of(w, args.workload, world, args.dtemp and w.temp_range is not None),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"each step: one (batch, KV head) plane of {w.name}, "
                                       "fp64 forward + backward"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("capattn", "reference"), default="capattn")
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--per-workload-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--soak-seconds", type=float, default=SOAK_SECONDS,
                    help="untimed run of the step under the clock sampler before the timed steps")
    ap.add_argument("--dtemp", action="store_true",
                    help="also compute the temperature gradient (workloads with a temperature)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    try:
        run_capattn(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
