#!/usr/bin/env python
"""Benchmark of the adapted linear layer in normal form on a mixed PEFT batch.

Workload (decode, Llama-3-8B-shaped): one step is one pass of the whole hot
path over the six projections q (4096->4096), k, v (4096->1024), gate, up
(4096->14336) and down (14336->4096) for 64 tokens whose ids are uniform over
32 adapters, method = id mod 5 (LoRA, DoRA, (IA)^3, VeRA, OFT), rank 16,
shared VeRA rank 256, OFT blocks of 32.  Inputs are seeded synthetic tensors
(``workloads.decode_mixed``, one independent input per projection), resident
in device memory before timing.  The headline step is ONE scute_linear_batch
call over the six projections (one launch).  Two other groupings of the same
work are timed beside it: the groups a transformer block's data dependencies
allow ({q, k, v}, {gate, up}, {down}: three launches) and six separate
scute_linear calls.

Metric: tokens per second through the adapted layer (one step), plus the
step's algorithmic HBM GB/s and its overhead against an all-LoRA batch of the
same size, ids and rank.  Timing: each step is a CUDA graph replay bracketed by
CUDA events; L2 is flushed (a 512 MiB write) before every step, outside the
timed interval.  The step kernel is also timed alone, in a second graph whose
event records sit on the launching stream around the launch.

`--impl reference` times the float64 CPU oracle on the same workload instead
(a bounded sample per step).  Under torchrun each rank serves its own batch of
64 tokens (weak scaling, no collective on the data path); rank 0 prints one
JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

PROJ = ("q", "k", "v", "gate", "up", "down")
METRIC = "adapted-linear tokens/s + HBM GB/s (mixed PEFT batch) vs all-LoRA overhead %"
WORKLOAD = ("decode_mixed: Llama-3-8B-shaped q,k,v,gate,up,down; n=64 tokens; 32 adapters "
            "(method = id mod 5: LoRA, DoRA, (IA)^3, VeRA, OFT); rank 16; VeRA shared rank 256; "
            "OFT block 32; ids uniform")


def captured_traffic():
    """DRAM bytes (read + write) per launch of the step kernel from the committed
    ncu summary, or None when the kernel source has changed since that capture."""
    import hashlib
    import re
    try:
        md = open(os.path.join(ROOT, "profiles", "step_kernel_decode_mixed_ncu_full.md")).read()
        src = open(os.path.join(ROOT, "lora_normal_form_gb300", "csrc", "k_step.cu"), "rb").read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes=(\d+) k_step_sha16=([0-9a-f]{16})", md)
    if not m or hashlib.sha256(src).hexdigest()[:16] != m.group(2):
        return None
    return int(m.group(1))


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="scute", choices=["scute", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true", help="skip the prefill base-GEMM leg")
    p.add_argument("--eager-steps", type=int, default=0,
                   help="only run this many untimed batched steps of the mixed workload and exit "
                        "(a fixed launch sequence for profilers); prints no JSON line")
    return p.parse_args()


def max_over_ranks(values, device):
    """Element-wise maximum of a few host floats over every rank of the
    default process group (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [ln.strip().split(", ") for ln in self.f.read().splitlines() if ln.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
            except ValueError:
                continue
            for k, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(k)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle timing (CPU)
def oracle_step_sample(w, tokens) -> float:
    """Wall time of the float64 oracle computing the whole step (six
    projections) for the given token rows."""
    from oracle import batch as BT
    t0 = time.perf_counter()
    for p in PROJ:
        BT.linear(w, p, rows=tokens)
    return time.perf_counter() - t0


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return int(max(i.get("num_threads", 1) for i in info))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_baseline(w, budget_s=20.0):
    tokens = []
    t = 0.0
    i = 0
    while t < budget_s and i < w.n:
        dt = oracle_step_sample(w, [i])
        t += dt
        tokens.append(i)
        i += 1
    value = len(tokens) / t
    return {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"float64 NumPy oracle, whole step (6 projections) for the first {len(tokens)} of "
                      f"{w.n} tokens, one token at a time ({t:.1f} s)"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = WL.decode_mixed()
    for _ in range(args.warmup):
        oracle_step_sample(w, [0])
    times = []
    for s in range(args.steps):
        times.append(oracle_step_sample(w, [s % w.n]))
    ms = 1000.0 * float(np.mean(times))
    value = 1000.0 / ms
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": "one token per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": "float64 NumPy oracle, whole step (6 projections) for one token per "
                                       "step, cycling through the 64 tokens"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def prefill_leg(scute, dev, flush, steps=8):
    """The prefill-shaped bf16 batch (16 requests of U{64..1024} tokens, 8772 in
    all, one adapter each from 32 of mixed methods) through the q and gate
    projections: the base GEMM timed by the library's event pair around its
    launch, as TFLOP/s of 2 n d_in d_out against the bf16 tensor peak, and the
    whole call (every kernel of the prefill path) beside it."""
    import torch
    _, tf_peak, peak_kind = peaks()
    w = WL.prefill_mixed(proj=("q", "gate"))
    ctx = scute.Context("bf16", max_tokens=w.n, max_adapters=w.n_adapters + 8, max_layers=3, device=dev.index)
    try:
        ctx.load_workload(w)
        ids = torch.from_numpy(w.ids.copy()).to(dev)
        st = torch.cuda.current_stream(dev)
        res = {}
        for p in ("q", "gate"):
            L = w.layer(p)
            x = torch.from_numpy(np.ascontiguousarray(L.get("x")).view(np.int16)).to(dev).view(torch.bfloat16)
            out = torch.empty(w.n, L.d_out, dtype=torch.bfloat16, device=dev)
            for _ in range(2):
                ctx.linear(x, ids, ctx.layer_ids[p], out, "bf16", stream=st)
            torch.cuda.synchronize()
            ctx.timing(True)
            ctx.timing_reset()
            call_ms = []
            for _ in range(steps):
                flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(st)
                ctx.linear(x, ids, ctx.layer_ids[p], out, "bf16", stream=st)
                e1.record(st)
                e1.synchronize()
                call_ms.append(e0.elapsed_time(e1))
            gemm_ms = ctx.timing_read()
            ctx.timing(False)
            g = float(np.median(np.array(gemm_ms[-steps:], dtype=np.float64)))
            tflops = 2.0 * w.n * L.d_in * L.d_out / (g * 1e-3) / 1e12
            res[p] = {"shape": f"{L.d_in}->{L.d_out}", "base_gemm_ms": g, "achieved": tflops,
                      "frac": tflops / tf_peak, "call_ms": float(np.median(call_ms))}
        if ctx.sync_status() != 0:
            raise RuntimeError("device status error in the prefill leg")
        return {"workload": f"prefill_mixed: {w.n} tokens, q and gate projections", "bound": "tensor",
                "unit": "TFLOP/s", "peak": tf_peak, "peak_kind": peak_kind, "per_projection": res}
    finally:
        ctx.close()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist

    import lora_normal_form_gb300 as scute

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    scute.load()
    dev = torch.device("cuda", local_rank)

    # each rank serves its own batch (weak scaling); rank 0's ids are the seed-0 ids
    w = WL.decode_mixed()
    if rank > 0:
        w.ids = WL.uniform_ids(1000 + rank, w.n, 32)
    wl = WL.all_lora_of(w)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    ctx = scute.Context("bf16", max_tokens=64, max_adapters=40, max_layers=8, device=local_rank)
    ctx.load_workload(w)
    if args.eager_steps > 0:
        xs = {p: to_dev(w.layer(p).get("x")) for p in PROJ}
        ids = torch.from_numpy(w.ids.copy()).to(dev)
        outs = {p: torch.empty(w.n, w.layer(p).d_out, dtype=torch.bfloat16, device=dev) for p in PROJ}
        for _ in range(args.eager_steps):
            ctx.linear_batch([(xs[p], ctx.layer_ids[p], outs[p]) for p in PROJ], ids, "bf16")
        torch.cuda.synchronize()
        if ctx.sync_status() != 0:
            raise RuntimeError("device status error")
        ctx.close()
        return
    ctx_l = scute.Context("bf16", max_tokens=64, max_adapters=40, max_layers=8, device=local_rank)
    ctx_l.load_workload(wl)
    xs = {p: to_dev(w.layer(p).get("x")) for p in PROJ}
    ids = torch.from_numpy(w.ids.copy()).to(dev)
    outs = {p: torch.empty(w.n, w.layer(p).d_out, dtype=torch.bfloat16, device=dev) for p in PROJ}
    outs_l = {p: torch.empty(w.n, w.layer(p).d_out, dtype=torch.bfloat16, device=dev) for p in PROJ}

    stream = torch.cuda.Stream(device=dev)

    BLOCK_GROUPS = (("q", "k", "v"), ("gate", "up"), ("down",))

    def step(c, o):
        c.linear_batch([(xs[p], c.layer_ids[p], o[p]) for p in PROJ], ids, "bf16", stream=stream)

    def step_grouped(c, o):
        for grp in BLOCK_GROUPS:
            c.linear_batch([(xs[p], c.layer_ids[p], o[p]) for p in grp], ids, "bf16", stream=stream)

    def step_calls(c, o):
        for p in PROJ:
            c.linear(xs[p], ids, c.layer_ids[p], o[p], "bf16", stream=stream)

    # eager warm-up (also builds the kernels' attributes), then graph capture
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step(ctx, outs)
            step(ctx_l, outs_l)
            step_grouped(ctx, outs)
            step_calls(ctx, outs)
    torch.cuda.synchronize()
    st = ctx.sync_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    def capture(fn, c, o):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                fn(c, o)
        return g

    n0 = ctx.launch_count()
    g_mixed = capture(step, ctx, outs)
    launches_per_step = ctx.launch_count() - n0
    g_lora = capture(step, ctx_l, outs_l)
    g_grouped = capture(step_grouped, ctx, outs)
    g_calls = capture(step_calls, ctx, outs)
    ctx.timing(True)
    ctx.timing_reset()
    g_timed = capture(step, ctx, outs)
    ctx.timing(False)

    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def timed(graph, K, read_kernel):
        t_steps, t_kernel = [], []
        for _ in range(K):
            with torch.cuda.stream(stream):
                flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            e1.synchronize()
            t_steps.append(e0.elapsed_time(e1))
            if read_kernel:
                t_kernel.append(ctx.timing_read()[:1])
        return t_steps, t_kernel

    # warm-up replays
    for g in (g_mixed, g_lora, g_grouped, g_calls):
        timed(g, args.warmup, False)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    t_mixed, _ = timed(g_mixed, args.steps, False)
    clocks = sampler.stop()
    torch.cuda.synchronize()
    t_lora, _ = timed(g_lora, args.steps, False)
    t_grouped, _ = timed(g_grouped, args.steps, False)
    t_calls, _ = timed(g_calls, args.steps, False)
    timed(g_timed, args.warmup, False)
    _, t_kernel = timed(g_timed, min(args.steps, 200), True)

    ms = float(np.mean(t_mixed))
    ms_lora = float(np.mean(t_lora))
    if world > 1:
        ms, ms_lora = max_over_ranks([ms, ms_lora], dev)

    # byte model of the step: the one launch moves every projection's bytes
    bm = {p: ctx.predict_bytes(w.ids, ctx.layer_ids[p], "bf16") for p in PROJ}
    alg_bytes = sum(bm[p]["algorithmic_bytes"] for p in PROJ)
    kernel_ms = float(np.mean(np.array(t_kernel, dtype=np.float64)))
    hbm_peak, _, peak_kind = peaks()
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9

    # end to end through the host-buffer entry point (copies inside the timed region)
    h_x = {p: torch.from_numpy(np.ascontiguousarray(w.layer(p).get("x")).view(np.int16))
           .view(torch.bfloat16).pin_memory() for p in PROJ}
    h_ids = torch.from_numpy(w.ids.copy()).pin_memory()
    h_out = {p: torch.empty(w.n, w.layer(p).d_out, dtype=torch.bfloat16).pin_memory() for p in PROJ}
    h2d = sum(w.n * w.layer(p).d_in * 2 for p in PROJ) + w.n * 4
    d2h = sum(w.n * w.layer(p).d_out * 2 for p in PROJ)
    e2e_t = []
    for i in range(args.warmup + min(args.steps, 100)):
        with torch.cuda.stream(stream):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ctx.linear_batch_host([(h_x[p], ctx.layer_ids[p], h_out[p]) for p in PROJ], h_ids, "bf16",
                                  stream=stream)
            e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            e2e_t.append(e0.elapsed_time(e1))
    e2e_ms = float(np.mean(e2e_t))
    if world > 1:
        (e2e_ms,) = max_over_ranks([e2e_ms], dev)
    if ctx.sync_status() != 0:
        raise RuntimeError("device status error after the timed region")

    tokens = w.n * world
    line = {
        "metric": METRIC,
        "value": tokens / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_gpu": w.n, "l2": "flushed (512 MiB write) before every step",
                   "timing": "CUDA graph replay per step, CUDA events", "parallelism": f"dp{world} (independent batches)"},
        "hbm_gbs": alg_bytes * world / (ms * 1e-3) / 1e9,
        "hbm_frac": alg_bytes / (ms * 1e-3) / 1e9 / hbm_peak,
        "algorithmic_bytes_per_step": alg_bytes,
        "all_lora_ms_per_step": ms_lora,
        "overhead_vs_all_lora_pct": 100.0 * (ms / ms_lora - 1.0),
        "roofline": {"kernel": "decode step (tcgen05 + TMA, one persistent launch per step)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "peak_kind": peak_kind, "traffic": captured_traffic(), "kernel_ms": kernel_ms,
                     "algorithmic_bytes_per_launch": alg_bytes},
        "block_groups_ms_per_step": float(np.mean(t_grouped)),
        "separate_calls_ms_per_step": float(np.mean(t_calls)),
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": int(launches_per_step * args.steps),
        "launches_per_step": int(launches_per_step),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_prefill:
        try:
            line["prefill"] = prefill_leg(scute, dev, flush)
        except Exception as exc:   # the headline line is printed whatever this leg does
            line["prefill"] = {"error": str(exc)[:300]}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    ctx_l.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
