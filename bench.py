#!/usr/bin/env python
"""Benchmark of the cumulative proxy-attention KV eviction path on one GB300.

One benchmark step is one pass of the whole path over the workload: reset the
state, score and bulk-evict the prompt (tensor-core column sums + selection),
run every decode step (one kernel launch for all of them: a row's next step
starts as soon as its own previous step is done) and apply the last step's
pending compaction. Keys are seeded synthetic fp16 N(0,1) draws, RoPE-rotated
at their positions, generated on the device before the timed region.

Prints one JSON line. ``value`` = decode head-steps (batch x layers x KV heads
x decode tokens) per second of whole-pass time, inputs resident in HBM;
``e2e`` = the same metric through ``kvevict_run_host`` with the keys in pinned
host memory and the evicted-slot log copied back, every host<->device transfer
inside the timed region (the library moves page-locked buffers with its own
kernels: the prompt is staged by a copy kernel, the decode keys are read in
place over the CPU-GPU link); ``roofline`` = the decode kernel's algorithmic bytes (from the actual
eviction log) over its time, against the measured HBM copy bandwidth;
``cpu_baseline`` = the fp64 CPU oracle on a bounded sample of the same
workload on this host's cores.

``--impl reference`` times the fp64 CPU oracle itself on a bounded sample of
the workload (the pages publish no runnable reference implementation).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = ("evict head-steps/s (batch×layers×KV-heads×tokens); "
          "achieved HBM GB/s vs peak")
UNIT = "head-steps/s"
DEFAULT_WORKLOAD = "large_context"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.ALL))
    ap.add_argument("--batch", type=int, default=None, help="override the batch (profiling)")
    ap.add_argument("--decode", type=int, default=None, help="override the decode steps (profiling)")
    ap.add_argument("--decode-kernel", choices=["auto", "stream", "resident"], default="auto",
                    help="decode kernel (the library's choice by default)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    return ap.parse_args()


def workload_of(args):
    wl = workloads.ALL[args.workload]
    kw = {}
    if args.batch:
        kw["batch"] = args.batch
    if args.decode:
        kw["decode"] = args.decode
    return wl.scaled(**kw) if kw else wl


def tau_text(wl):
    """The temperature schedule as the run applies it: tau anneals over absolute
    positions 0..anneal_steps, prompt positions included, so a prompt at least
    that long leaves every decode step at tau_end."""
    if wl.tau_init == wl.tau_end or not wl.anneal_steps:
        return f"{wl.tau_init:g} (constant)"
    span = f"{wl.tau_init:g}->{wl.tau_end:g} over positions 0..{wl.anneal_steps}"
    if wl.prefill >= wl.anneal_steps:
        return span + f"; the {wl.prefill}-token prompt covers the ramp, every decode step runs at {wl.tau_end:g}"
    t0 = wl.tau_init + wl.prefill * (wl.tau_end - wl.tau_init) / wl.anneal_steps
    last = wl.prefill + wl.decode - 1
    t1 = wl.tau_init + min(last, wl.anneal_steps) * (wl.tau_end - wl.tau_init) / wl.anneal_steps
    return span + f"; decode runs from {t0:g} to {t1:g}"


def config_of(wl, budgets):
    tau = tau_text(wl)
    return {"workload": wl.name, "batch": wl.batch, "layers": wl.n_layers, "kv_heads": wl.n_kv_heads,
            "head_dim": wl.head_dim, "avg_budget": wl.avg_budget, "pyramid_beta": wl.beta,
            "budgets": f"{budgets[0]}..{budgets[-1]}", "n_sink": wl.n_sink, "tau": tau,
            "rope_theta": wl.rope_theta, "prefill_tokens": wl.prefill, "decode_steps": wl.decode,
            "late_riser": wl.late_riser}


def profiled_traffic(wl, kernel_src, bytes_per_launch):
    """DRAM bytes (read + write) of one decode launch on this workload, scaled
    from the committed small-case ncu capture (profiles/decode_step_small.md):
    that launch's DRAM bytes over its algorithmic bytes, times this launch's
    algorithmic bytes. None when decode.cu has changed since the counters were
    taken, or when the capture was of another workload."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "decode_step_small.md")) as f:
            lines = [ln.split() for ln in f if ln.startswith("traffic_ratio ")]
        with open(kernel_src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    for ln in lines:
        kv = dict(x.split("=", 1) for x in ln[1:] if "=" in x)
        if kv.get("workload") == wl.name and kv.get("decode_cu_sha256") == sha:
            return int(round(int(kv["dram_bytes"]) / int(kv["algorithmic_bytes"]) * bytes_per_launch))
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- CPU oracle
def sample_rows(wl, n):
    rows = []
    for i in range(n):
        l = (i * wl.n_layers) // n
        rows.append((i % wl.batch, l, (3 * i) % wl.n_kv_heads))
    return rows


def oracle_pass(wl, rows, threads=0):
    """Whole pass (prompt + every decode step) of the fp64 oracle over sampled rows."""
    import oracle
    budgets = oracle.budgets(wl.n_layers, wl.avg_budget, wl.n_sink, wl.beta)
    prms = [oracle.HeadParams(D=wl.head_dim, budget=budgets[l], n_sink=wl.n_sink, layer=l, head=h,
                              tau_init=wl.tau_init, tau_end=wl.tau_end,
                              anneal_steps=wl.anneal_steps, theta=wl.rope_theta,
                              seed=wl.gumbel_seed, recent=wl.recent, mode=wl.score_mode)
            for (b, l, h) in rows]
    keys = [wl.head_keys(b, l, h, 0, wl.positions) for (b, l, h) in rows]
    pk = np.stack([k[: wl.prefill] for k in keys]) if wl.prefill else None
    dk = np.stack([k[wl.prefill:] for k in keys])
    t0 = time.perf_counter()
    out = oracle.run_heads(prms, pk, dk, n_threads=threads)
    dt = time.perf_counter() - t0
    return dt, out[-1]


def cpu_sample_size(wl):
    return 2 * max(1, os.cpu_count() or 1)   # two rows per core: about 10 s on 16 Grace cores


def cpu_baseline(wl):
    rows = sample_rows(wl, cpu_sample_size(wl))
    dt, used = oracle_pass(wl, rows)
    return {"value": len(rows) * wl.decode / dt, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{len(rows)} cache rows spread over the layers, each a whole pass "
                      f"(prompt of {wl.prefill} + {wl.decode} decode steps), fp64 C oracle, "
                      f"OpenMP over rows; {dt:.1f} s"}


def cpu_single_core():
    """The oracle on one core: every row of the tiny H2O configuration and a few
    rows of the Keyformer 3B configuration, each a whole pass."""
    out = []
    for wl, n in ((workloads.TINY_H2O, None), (workloads.KEYFORMER_3B, 4)):
        rows = ([(b, l, h) for b in range(wl.batch) for l in range(wl.n_layers) for h in range(wl.n_kv_heads)]
                if n is None else sample_rows(wl, n))
        dt, used = oracle_pass(wl, rows, threads=1)
        out.append({"workload": wl.name, "value": len(rows) * wl.decode / dt, "unit": UNIT, "cores": used,
                    "rows": len(rows), "seconds": round(dt, 2)})
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = workload_of(args)
    import oracle
    budgets = oracle.budgets(wl.n_layers, wl.avg_budget, wl.n_sink, wl.beta)
    rows = sample_rows(wl, cpu_sample_size(wl))
    times = []
    used = 1
    for k in range(args.warmup + args.steps):
        dt, used = oracle_pass(wl, rows)
        if k >= args.warmup:
            times.append(dt)
    step = statistics.median(times)
    value = len(rows) * wl.decode / step
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(wl, budgets), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": f"{len(rows)} cache rows of the workload, each a whole "
                                       f"pass (prompt {wl.prefill} + {wl.decode} decode steps)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- ranks
def init_ranks(backend="nccl"):
    """(world, rank, dist or None) from the torchrun environment. One process
    per GPU; every rank runs its own replica of the workload (cache rows are
    independent, so nothing is exchanged on the data path)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)
    return world, rank, dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist, device="cuda"):
    """The slowest rank's value: the job is done when every replica is."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, seconds):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / seconds


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", device_id], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def device_id():
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        return str(torch.cuda.current_device())


# ----------------------------------------------------------------------------- GPU arm
def algorithmic_bytes(wl, budgets, ev):
    """Bytes the decode kernel must move, summed over the run's head-steps.

    Per head-step with n rows before the append and evicted slot e:
      evicting : (n+1)*2D K read + (n-e)*2D K written + 8(n+1) scores read+written
                 + 4(n+1) Gumbel read + 12(n-e) Gumbel/positions moved
      otherwise: (n+1)*2D K read + 2D new key written + 8(n+1) scores + 8 new g/pos
    """
    import torch
    T = ev.shape[0]
    D2 = 2 * wl.head_dim
    p = wl.prefill + torch.arange(T, device=ev.device, dtype=torch.int64)
    b = torch.tensor(budgets, device=ev.device, dtype=torch.int64)
    n = torch.minimum(p[:, None], b[None, :])[:, None, :, None].expand(ev.shape)
    e = ev.to(torch.int64)
    evict = e >= 0
    moved = (n - e).clamp(min=0)
    by_ev = (n + 1) * D2 + moved * D2 + 8 * (n + 1) + 4 * (n + 1) + 12 * moved
    by_no = (n + 1) * D2 + D2 + 8 * (n + 1) + 8
    return int(torch.where(evict, by_ev, by_no).sum().item())


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import kv_cache_attention_02_gb300 as kvx
    from workloads import gpu as wgpu

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    world, rank, dist = init_ranks("nccl")

    wl = workload_of(args)
    B, L, H, D, T = wl.batch, wl.n_layers, wl.n_kv_heads, wl.head_dim, wl.decode
    pre, dec = wgpu.device_inputs(wl)
    h = kvx.from_workload(wl, decode_kernel={"auto": kvx.DECODE_AUTO, "stream": kvx.DECODE_STREAM,
                                             "resident": kvx.DECODE_RESIDENT}[args.decode_kernel])
    state_bytes = h.device_bytes()   # the cache arena and prompt scratch (before any host staging)
    budgets = h.budgets
    decode_kernel = ("resident_step_kernel" if h.decode_kernel_for(T) == kvx.DECODE_RESIDENT
                     else "decode_step_kernel")
    ev = torch.empty((T, B, L, H), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    ev_marks = []

    def one_pass(mark=False):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e3 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h.reset(stream=stream)
        if pre is not None:
            h.prefill(pre, stream=stream)
        e1.record(stream)
        h.decode(dec, ev, stream=stream)
        e2.record(stream)
        h.flush(stream=stream)
        e3.record(stream)
        if mark:
            ev_marks.append((e0, e1, e2, e3))

    for _ in range(args.warmup):
        one_pass()
    torch.cuda.synchronize()
    h.check(stream=stream)
    step_bytes = algorithmic_bytes(wl, budgets, ev)

    # L2 is flushed between timed passes (outside the timed events) so every
    # pass starts cold, whatever the size of the workload's state.
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    clocks = ClockSampler(device_id())
    barrier(dist)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        flush_buf.fill_(1)
        one_pass(mark=True)
    torch.cuda.synchronize()
    barrier(dist)
    clk = clocks.stop()
    h.check(stream=stream)

    pass_ms = [a.elapsed_time(d) for a, _, _, d in ev_marks]
    ms_per_step = max_over_ranks(sum(pass_ms) / len(pass_ms), dist)
    prefill_ms = statistics.median(a.elapsed_time(b) for a, b, _, _ in ev_marks)
    decode_ms = statistics.median(b.elapsed_time(c) for _, b, c, _ in ev_marks)
    flush_ms = statistics.median(c.elapsed_time(d) for _, _, c, d in ev_marks)
    heads = B * L * H
    value = job_rate(world, heads * T, ms_per_step / 1e3)

    # decode kernel roofline: algorithmic bytes per launch over average launch time
    launch_ms = decode_ms / T
    achieved = (step_bytes / T) / (launch_ms / 1e3) / 1e9
    peak, peak_kind = peaks()
    prefill_flops = 2.0 * 2.0 * D * (wl.prefill * (wl.prefill + 1) / 2) * heads if wl.prefill else 0.0

    # end to end: keys in pinned host memory, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        pre_h = None
        if pre is not None:
            pre_h = torch.empty(pre.shape, dtype=torch.float16, pin_memory=True)
            pre_h.copy_(pre)
        dec_h = torch.empty(dec.shape, dtype=torch.float16, pin_memory=True)
        dec_h.copy_(dec)
        ev_h = torch.empty(ev.shape, dtype=torch.int32, pin_memory=True)
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            h.reset(stream=stream)
            h.run_host(pre_h, dec_h, ev_h, stream=stream)
        e2e_clocks = ClockSampler(device_id())
        e2e_ms = []
        barrier(dist)
        for _ in range(args.steps):
            t0 = time.perf_counter()
            h.reset(stream=stream)
            h.run_host(pre_h, dec_h, ev_h, stream=stream)
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
        barrier(dist)
        e2e_clk = e2e_clocks.stop()
        dt = max_over_ranks(sum(e2e_ms) / len(e2e_ms) / 1e3, dist)
        if not np.array_equal(ev_h.numpy(), ev.cpu().numpy()):
            raise SystemExit("end-to-end run disagrees with the device-resident run")
        h2d = (pre_h.numel() * 2 if pre_h is not None else 0) + dec_h.numel() * 2
        e2e = {"value": job_rate(world, heads * T, dt), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": ev_h.numel() * 4, "ms_per_step": dt * 1e3,
               "pass_ms": [round(x, 1) for x in e2e_ms], "clocks": e2e_clk}

    cpu = single = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(wl)
        single = cpu_single_core()

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {**config_of(wl, budgets), "l2": "flushed (256 MB write) before every timed pass",
                   "state_gb": round(state_bytes / 1e9, 3),
                   "input_gb": round(heads * wl.positions * D * 2 / 1e9, 3)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": (profiled_traffic(wl, os.path.join(ROOT, "kv_cache_attention_02_gb300", "csrc",
                                                                   "decode.cu"), step_bytes)
                                 if decode_kernel == "decode_step_kernel" else None),
                     "kernel": f"{decode_kernel}<{D}>",
                     "bytes_per_launch": step_bytes, "launch_us": decode_ms * 1e3,
                     "steps_per_launch": T, "us_per_step": launch_ms * 1e3,
                     "peak_kind": f"of {peak_kind}"},
        "e2e": e2e,
        "cpu_baseline": cpu,
        "cpu_single_core": single,
        # per pass: Gumbel table, scorer passes 0 and 1 (or the last-row scorer), selection;
        # one decode launch for every step; flush
        "gpu_launches": args.steps * ((4 if wl.score_mode == 0 else 3) * (1 if wl.prefill else 0) + 1 + 1),
        "clocks": clk,
        "decode_head_steps_per_s": world * heads * T / (decode_ms / 1e3),
        "prefill_ms": prefill_ms, "decode_ms": decode_ms, "flush_ms": flush_ms,
        "prefill_tflops": (prefill_flops / (prefill_ms / 1e3) / 1e12) if prefill_flops else None,
    }
    if rank == 0:
        print(json.dumps(line))
    h.close()
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
