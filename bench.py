"""Benchmark: soft-capped attention forward + backward on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl capattn|reference]
                    [--workload 2] [--no-cpu-baseline]

A step is one forward (capattn_fwd) and one backward (capattn_bwd) over the
workload's batch of synthetic seeded inputs.  The default workload is
causal_tanh: B=2, Hq=Hkv=16, L=2048, D=128, bf16, causal, tanh cap 50.

Metric: mask-aware TFLOP/s of forward + backward, 14 * D * N FLOPs per step
(N = unmasked (query, key) pairs summed over batch and heads, counted by the
oracle from the seeded masks and stored in tests/golden/pair_counts.json).

Timing: inputs resident in HBM; an L2 flush (a 512 MB write) runs before every
timed step, outside the events; each step is bracketed by CUDA events on the
stream the kernels run on.  `value` = total FLOPs / summed step time.  `e2e`
repeats the step through the same C ABI with pinned host buffers: host-to-
device copies of Q, K, V, dO, the forward, the backward and device-to-host
copies of O, LSE, dQ, dK, dV all inside the timed region.

Multi-GPU: each rank runs an independent replica of the workload (the path
shards over (batch, KV head) without any exchange), timing is the max over
ranks and `value` sums all ranks' FLOPs ("scaling": "weak").

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (whole (batch, head) planes, forward + backward) on the host cores.
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
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for n, v in zip(names, s[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.samples)}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "soft_capped_attention_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """ncu DRAM bytes per launch of `kernel` on `workload`, if taken on this source."""
    try:
        with open(TRAFFIC) as f:
            t = json.load(f)
        e = t[workload][kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# capattn arm
# ---------------------------------------------------------------------------

def run_capattn(args, rank, world, local_rank):
    from soft_capped_attention_gb300 import capattn as ca

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, seed=args.workload)
    dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ap = ca.params_from_workload(w)
    host = {n: torch.from_numpy(inp[n]).to(dtype).contiguous() for n in ("q", "k", "v", "do")}
    aux = {n: (None if inp[n] is None else torch.from_numpy(inp[n]).contiguous())
           for n in ("temp", "seg", "bounds")}
    d = {n: t.to(dev) for n, t in host.items()}
    da = {n: (None if t is None else t.to(dev)) for n, t in aux.items()}
    cfg = ca.make_config(ap, w.B, w.L, w.Hq, w.Hkv, w.D, dtype, Lk=w.key_len)
    ws = ca.new_workspace(cfg, dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    use_dtemp = args.dtemp and aux["temp"] is not None
    if args.dtemp and not use_dtemp:
        raise SystemExit("--dtemp needs a workload with a temperature")

    def bwd(*a, **kw):
        if use_dtemp:
            return ca.capattn_bwd_dtemp(*a, **kw)[:3]
        return ca.capattn_bwd(*a, **kw)[:3]

    def step(split=False):
        o, lse, _, _ = ca.capattn_fwd(d["q"], d["k"], d["v"], ap, da["temp"], da["seg"],
                                      da["bounds"], workspace=ws)
        ev_mid = None
        if split:
            ev_mid = torch.cuda.Event(enable_timing=True)
            ev_mid.record(stream)
        bwd(d["q"], d["k"], d["v"], o, lse, d["do"], ap, da["temp"], da["seg"],
                       da["bounds"], workspace=ws)
        return ev_mid

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st, bits = ca.capattn_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} (bits {bits}) after warm-up")

    N = pairs_of(args.workload)
    D = w.D
    flops_step = 14.0 * D * N

    # Breakdown pass (not the headline): every kernel bracketed by events and a
    # mark between forward and backward.  Each recorded event costs the stream a
    # few microseconds, so the headline run below records only the events of the
    # kernel its roofline names.
    ca.capattn_profile_select(None)
    ca.capattn_profile_enable(True)
    ca.capattn_profile_read(reset=True)
    split = []
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e1 = step(split=True)
        e2.record(stream)
        split.append((e0, e1, e2))
    torch.cuda.synchronize()
    prof_all = ca.capattn_profile_read(reset=True)
    fw = sum(a.elapsed_time(b) for a, b, _ in split)
    bw = sum(b.elapsed_time(c) for _, b, c in split)
    kern_ms_all = {k: v[0] for k, v in prof_all.items() if v[1] > 0}
    launches_all = {k: v[1] for k, v in prof_all.items()}
    dom = max(KERNEL_FLOPS_PER_PAIR_D, key=lambda k: kern_ms_all.get(k, 0.0))
    total_kernel_ms = sum(kern_ms_all.values())

    # Headline run: step events plus the events of the roofline kernel only.
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ca.capattn_profile_select([dom])
    ca.capattn_profile_read(reset=True)
    times_total = []
    with ClockSampler(local_rank) as clk:
        time.sleep(0.05)
        for _ in range(args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e2 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e2.record(stream)
            times_total.append((e0, e2))
        torch.cuda.synchronize()
        time.sleep(0.05)
    prof = ca.capattn_profile_read(reset=True)
    ca.capattn_profile_enable(False)
    ca.capattn_profile_select(None)
    if world > 1:
        torch.distributed.barrier()
    tot = sum(e0.elapsed_time(e2) for e0, e2 in times_total)
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

    # e2e through the C ABI with pinned host buffers
    e2e = None
    if not args.no_e2e:
        ph = {n: t.pin_memory() for n, t in host.items()}
        pa = {n: (None if t is None else t.pin_memory()) for n, t in aux.items()}
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

        def e2e_step():
            for n in ph:
                dbuf[n].copy_(ph[n], non_blocking=True)
            for n in pa:
                if pa[n] is not None:
                    dabuf[n].copy_(pa[n], non_blocking=True)
            o, lse, _, _ = ca.capattn_fwd(dbuf["q"], dbuf["k"], dbuf["v"], ap, dabuf["temp"],
                                          dabuf["seg"], dabuf["bounds"], workspace=ws)
            dq, dk, dv = bwd(dbuf["q"], dbuf["k"], dbuf["v"], o, lse, dbuf["do"], ap,
                                           dabuf["temp"], dabuf["seg"], dabuf["bounds"],
                                           workspace=ws)
            out_h["o"].copy_(o, non_blocking=True)
            out_h["lse"].copy_(lse, non_blocking=True)
            out_h["dq"].copy_(dq, non_blocking=True)
            out_h["dk"].copy_(dk, non_blocking=True)
            out_h["dv"].copy_(dv, non_blocking=True)

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
            t = torch.tensor([etot], dtype=torch.float64, device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            etot = float(t.item())
        e2e = {"value": round(flops_step * args.steps * world / (etot * 1e-3) / 1e12, 3),
               "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(etot / args.steps, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.workload, args.cpu_seconds)

    clocks = clk.summary()
    line = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded normal Q, K, V, dO; seeded masks)",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "Lk": w.key_len, "Hq": w.Hq, "Hkv": w.Hkv,
                       "D": w.D, "causal": w.causal, "window_len": w.window_len,
                       "cap": [w.cap_method, w.cap, w.alpha, w.beta],
                       "z_loss_weight": w.z_loss_weight, "unmasked_pairs": N,
                       "dtemp": use_dtemp,
                       "flops_per_step": flops_step, "l2": "flushed before every timed step",
                       "parallelism": f"replicas x{world}"},
            "fwd_tflops": round(fwd_tf, 3), "bwd_tflops": round(bwd_tf, 3),
            "fwd_bwd_split": "from the breakdown pass (events around every kernel)",
            "frac_of_peak": round(value / peak, 4), "peak_tflops": peak, "peak_source": peak_src,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
            "clocks": clocks}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

_ORACLE_INPUTS = {}


def oracle_sample(w, idx, seconds: float, start: int = 0):
    """Runs the oracle forward + backward on whole (batch, KV head) planes of the
    workload, starting at plane `start`, until `seconds` elapse (at least one
    plane); returns (FLOPs counted mask-aware, seconds, planes)."""
    from oracle import capattn_oracle as orc
    if idx not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[idx] = make_inputs(w, seed=idx)
    inp = _ORACLE_INPUTS[idx]
    cfg = orc.config_from_workload(w)
    flops = 0.0
    t0 = time.perf_counter()
    planes = 0
    nplanes = w.B * w.Hkv
    for pidx in range(start, start + nplanes):
        b, g = divmod(pidx % nplanes, w.Hkv)
        if True:
            orc.backward_kv_head(inp["q"], inp["k"], inp["v"], inp["temp"], inp["seg"],
                                 inp["bounds"], inp["do"], cfg, b, g)
            n_head = orc.pair_count(w.L, cfg, None if inp["seg"] is None else inp["seg"][b:b + 1],
                                    None if inp["bounds"] is None else inp["bounds"][b:b + 1], B=1,
                                    Lk=w.key_len)
            flops += 14.0 * w.D * n_head * w.G
            planes += 1
            if time.perf_counter() - t0 >= seconds:
                return flops, time.perf_counter() - t0, planes
    return flops, time.perf_counter() - t0, planes


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
            "config": {"workload": w.name, "B": w.B, "L": w.L, "Lk": w.key_len, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D},
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
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
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
