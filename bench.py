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

At one GPU the line also carries, each as its own key:
  * ``prefill``: the 8772-token prefill batch through q and gate, every
    kernel of the call timed (base GEMM and VeRA GEMMs against the tensor
    roofline, the rest against HBM);
  * ``scaling``: 256 tokens, 1024 (IA)^3 / VeRA adapters with Zipf(1.0) ids,
    against the same ids as rank-64 LoRA conversions, at 4096->4096 and
    4096->14336;
  * ``stack``: the 32-layer x 7-projection stack at 128 tokens, per-step time
    of the mixed pool against its all-LoRA twin;
  * ``time_model``: the zero-parameter time model's prediction (bytes /
    measured bandwidth + launches x measured launch cost) beside each measured
    time.
The scaling and stack legs draw their tensors on the device with torch's
seeded generator (same distributions as the host generator; drawing ~30 GB of
weights and adapters with NumPy would take minutes): they feed timings only.

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
STEP_CAPTURE = os.path.join("profiles", "step_kernel_decode_mixed_ncu_full.md")


def captured_traffic():
    """DRAM bytes (read + write) per launch of the step kernel from the committed
    ncu summary, or None when the kernel source has changed since that capture."""
    import hashlib
    import re
    try:
        md = open(os.path.join(ROOT, STEP_CAPTURE)).read()
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
    p.add_argument("--no-prefill", action="store_true", help="skip the prefill leg")
    p.add_argument("--no-scaling", action="store_true", help="skip the adapter-count scaling leg")
    p.add_argument("--no-stack", action="store_true", help="skip the 32-layer stack leg")
    p.add_argument("--no-validation", action="store_true", help="skip the time-model validation leg")
    p.add_argument("--eager-steps", type=int, default=0,
                   help="only run this many untimed batched steps of the mixed workload and exit "
                        "(a fixed launch sequence for profilers); prints no JSON line")
    p.add_argument("--eager-variant", type=int, default=0, choices=[0, 1, 2, 3],
                   help="launch placement of the --eager-steps calls: 0 fused, 1 the rotation as its own "
                        "pass, 2 DoRA's and (IA)^3's s as their own pass, 3 both; the byte model's bytes "
                        "per launch of that placement go to stderr")
    p.add_argument("--prefill-eager", type=int, default=0,
                   help="only run this many untimed prefill calls (q projection) and exit (profilers)")
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
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, kind)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


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
    n = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else (os.cpu_count() or 1)


def cpu_baseline_worker(budget_s: float) -> dict:
    """The oracle timed in this process (its BLAS threads as the environment
    sets them): the inputs are drawn first, then tokens are computed one at a
    time until the budget is spent."""
    w = WL.decode_mixed()
    oracle_step_sample(w, [0])           # draws every tensor the step reads (untimed)
    tokens, t, i = [], 0.0, 0
    while t < budget_s and i < w.n:
        t += oracle_step_sample(w, [i])
        tokens.append(i)
        i += 1
    return {"value": len(tokens) / t, "tokens": len(tokens), "seconds": t, "threads": blas_threads()}


def cpu_baseline(budget_s=10.0):
    """The oracle on the host cores, once with one BLAS thread and once with
    all of them, each in a fresh process (spawned, so no CUDA state is shared)."""
    res = {}
    for label, threads in (("all_cores", None), ("one_thread", 1)):
        env = dict(os.environ)
        for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            env.pop(k, None)
            if threads:
                env[k] = str(threads)
        cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-worker", str(budget_s)]
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        if r.returncode != 0:
            res[label] = {"error": r.stderr[-300:]}
            continue
        res[label] = json.loads(r.stdout.strip().splitlines()[-1])
    a = res.get("all_cores", {})
    one = res.get("one_thread", {})
    return {"value": a.get("value"), "unit": "tokens/s", "cores": a.get("threads"), "kind": "oracle",
            "host_cpu_count": os.cpu_count(),
            "sample": (f"float64 NumPy oracle, whole step (6 projections), tokens computed one at a time "
                       f"after the inputs are drawn: {a.get('tokens')} of 64 tokens in "
                       f"{a.get('seconds', 0):.1f} s with all BLAS threads; value = tokens / second"),
            "one_thread": {"value": one.get("value"), "threads": one.get("threads"),
                           "sample": f"{one.get('tokens')} tokens in {one.get('seconds', 0):.1f} s"}}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = WL.decode_mixed()
    for _ in range(max(1, args.warmup)):
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


# ------------------------------------------------------------------ GPU helpers
def launch_cost_us(dev) -> float:
    """Per-launch cost inside a CUDA graph: a graph of 400 dependent
    one-element kernels, replayed, time / 400 (the time model's launch term)."""
    import torch
    x = torch.zeros(1, device=dev)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        x.add_(1.0)
        with torch.cuda.graph(g, stream=s):
            for _ in range(400):
                x.add_(1.0)
    ts = []
    for _ in range(12):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return 1000.0 * float(np.median(ts[2:])) / 400.0


def graph_time(graph, stream, flush, K):
    """Mean ms of K replays of a CUDA graph, L2 flushed before each."""
    import torch
    ts = []
    for _ in range(K):
        with torch.cuda.stream(stream):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return float(np.mean(ts)), ts


def capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def predicted(scute, report, hbm, tf, launch_us):
    """Predicted microseconds of a launch list: the article's bytes /
    bandwidth + launches x launch cost (pure form), and with the tensor-core
    term for launches bound by arithmetic.  A merged list is predicted part
    by part (the library takes at most 64 launches per report)."""
    parts = report.get("parts", [report])
    return (sum(scute.scute_predict_time(r, hbm, 0.0, launch_us) for r in parts),
            sum(scute.scute_predict_time(r, hbm, tf, launch_us) for r in parts))


def merge_reports(reps):
    out = {"kernels": [], "algorithmic_bytes": 0, "parts": reps}
    for r in reps:
        out["kernels"] += r["kernels"]
        out["algorithmic_bytes"] += r["algorithmic_bytes"]
    return out


def load_device_drawn(ctx, w, dev, seed=0, only_lora_rank=None):
    """Register a workload's layers and adapters with tensors drawn on the
    device (``workloads.device_*``).  ``only_lora_rank``: register every
    adapter as a LoRA of that rank instead (the comparators)."""
    import torch
    for L in w.layers:
        lid = len(ctx.layer_ids)
        ctx.layer_ids[L.name] = lid
        t = WL.device_layer_tensors(seed, L, "bf16", dev)
        ctx.add_layer(lid, L.d_in, L.d_out, t["W"])
        if L.shared_rank and only_lora_rank is None:
            ctx.set_shared(lid, L.shared_rank, t["A_sh"], t["B_sh"])
        del t
    for a in sorted(w.adapters, key=lambda a: a.id):
        if only_lora_rank is not None:
            a = WL.Adapter(id=a.id, method="lora", c=2.0, rank=only_lora_rank, layers=tuple(L.name for L in w.layers))
        tens = []
        for lname, t in WL.device_adapter_tensors(seed + 17, a, w.layers, "bf16", dev):
            d = {"layer": ctx.layer_ids[lname], "rank": a.rank, "c": a.c}
            d.update(t)
            tens.append(d)
        aid = ctx.register(a.method, tens)
        assert aid == a.id
        del tens
    torch.cuda.synchronize()


# ------------------------------------------------------------------ legs
def prefill_leg(scute, dev, flush, launch_us, steps=6):
    """The prefill-shaped bf16 batch (16 requests of U{64..1024} tokens, 8772 in
    all, one adapter each from 32 of mixed methods) through the q and gate
    projections: every kernel of the call timed by the library's event pairs
    (tensor-core GEMMs in TFLOP/s against min(peak, AI x bandwidth), the rest
    in GB/s against the HBM peak), the whole call beside them."""
    import torch
    hbm, tf_peak, _, peak_kind = peaks()
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
            # the whole call, untimed by the library (launches overlap as they do in use)
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
            # every launch timed
            ctx.timing(True)
            per = {}
            for _ in range(steps):
                ctx.timing_reset()
                flush.fill_(1)
                ctx.linear(x, ids, ctx.layer_ids[p], out, "bf16", stream=st)
                ms = ctx.timing_read()
                for k, v in zip(ctx.timing_kinds(), ms):
                    per.setdefault(k, []).append(v)
            ctx.timing(False)
            rep = ctx.predict_bytes(w.ids, ctx.layer_ids[p], "bf16")
            kb = {}
            for name, b, f in rep["kernels"]:
                kb.setdefault(name, [0, 0])
                kb[name][0] += b
                kb[name][1] += f
            kb["lowrank"] = [kb.pop("lr_shrink", [0, 0])[0] + kb.pop("lr_expand", [0, 0])[0], 0]
            kern = {}
            for k, v in per.items():
                t = float(np.median(v))
                b, f = kb.get(k, [0, 0])
                e = {"ms": t, "bytes": b, "flops": f, "gbs": b / (t * 1e-3) / 1e9}
                if f and k in ("base_gemm", "vera_shrink", "vera_expand"):
                    ai = f / max(b, 1)
                    attainable = min(tf_peak, ai * hbm / 1e3)
                    e.update(tflops=f / (t * 1e-3) / 1e12, attainable_tflops=attainable,
                             frac=f / (t * 1e-3) / 1e12 / attainable, bound="tensor" if attainable >= tf_peak else "hbm")
                else:
                    e.update(frac=e["gbs"] / hbm, bound="hbm")
                # the time model for this launch (the owned low-rank timing covers
                # the shrink and, unless the base GEMM's epilogue runs it, the expand)
                nl = sum(1 for name, _, _ in rep["kernels"] if name in ("lr_shrink", "lr_expand")) \
                    if k == "lowrank" else 1
                e["predicted_us"] = max(b / (hbm * 1e3), f / (tf_peak * 1e6)) + nl * launch_us
                e["model_error_pct"] = 100.0 * abs(1e3 * t - e["predicted_us"]) / (1e3 * t)
                kern[k] = e
            g = kern["base_gemm"]["ms"]
            pure, full = predicted(scute, rep, hbm, tf_peak, launch_us)
            res[p] = {"shape": f"{L.d_in}->{L.d_out}", "base_gemm_ms": g,
                      "achieved": 2.0 * w.n * L.d_in * L.d_out / (g * 1e-3) / 1e12,
                      "frac": 2.0 * w.n * L.d_in * L.d_out / (g * 1e-3) / 1e12 / tf_peak,
                      "call_ms": float(np.median(call_ms)), "kernels": kern,
                      "predicted_call_ms": full / 1e3, "predicted_call_ms_bytes_only": pure / 1e3}
        if ctx.sync_status() != 0:
            raise RuntimeError("device status error in the prefill leg")
        return {"workload": f"prefill_mixed: {w.n} tokens, q and gate projections", "bound": "tensor",
                "unit": "TFLOP/s", "peak": tf_peak, "peak_kind": peak_kind, "per_projection": res}
    finally:
        ctx.close()


def scaling_leg(scute, dev, flush, launch_us, steps=20):
    """Adapter-count scaling: 256 tokens, 1024 adapters (even ids (IA)^3, odd
    VeRA, shared rank 256), Zipf(1.0) ids, at 4096->4096 and 4096->14336,
    against the same ids as rank-64 LoRA conversions."""
    import torch
    hbm, tf, _, peak_kind = peaks()
    w = WL.scaling_ia3_vera()
    names = [L.name for L in w.layers]
    res = {}
    stream = torch.cuda.Stream(device=dev)
    ids = torch.from_numpy(w.ids.copy()).to(dev)
    xs = {L.name: WL.device_normal(0, f"x/{L.name}", (w.n, L.d_in), 1.0, "bf16", dev) for L in w.layers}
    for label, conv in (("scute", None), ("lora64_conversions", 64)):
        ctx = scute.Context("bf16", max_tokens=w.n, max_adapters=w.n_adapters, max_layers=len(names), device=dev.index)
        try:
            load_device_drawn(ctx, w, dev, only_lora_rank=conv)
            outs = {n: torch.empty(w.n, w.layer(n).d_out, dtype=torch.bfloat16, device=dev) for n in names}
            r = {}
            for n in names:
                def call(n=n):
                    ctx.linear(xs[n], ids, ctx.layer_ids[n], outs[n], "bf16", stream=stream)
                with torch.cuda.stream(stream):
                    call()
                torch.cuda.synchronize()
                g = capture(call, stream)
                graph_time(g, stream, flush, 3)
                ms, _ = graph_time(g, stream, flush, steps)
                rep = ctx.predict_bytes(w.ids, ctx.layer_ids[n], "bf16")
                pure, full = predicted(scute, rep, hbm, tf, launch_us)
                gbs = rep["algorithmic_bytes"] / (ms * 1e-3) / 1e9
                # every launch of the call timed on its own (event pairs)
                ctx.timing(True)
                per = {}
                for _ in range(5):
                    ctx.timing_reset()
                    with torch.cuda.stream(stream):
                        flush.fill_(1)
                    call()
                    for k, v in zip(ctx.timing_kinds(), ctx.timing_read()):
                        per.setdefault(k, []).append(v)
                ctx.timing(False)
                kernel_ms = {k: float(np.median(v)) for k, v in per.items()}
                r[n] = {"shape": f"{w.layer(n).d_in}->{w.layer(n).d_out}", "ms": ms,
                        "tokens_per_s": w.n / (ms * 1e-3), "algorithmic_bytes": rep["algorithmic_bytes"],
                        "adapter_bytes": rep["adapter_bytes"], "gbs": gbs, "frac": gbs / hbm,
                        "launches": len(rep["kernels"]), "predicted_ms": full / 1e3,
                        "predicted_ms_bytes_only": pure / 1e3, "kernel_ms": kernel_ms}
            if ctx.sync_status() != 0:
                raise RuntimeError("device status error in the scaling leg")
            res[label] = r
        finally:
            ctx.close()
    for n in names:
        res.setdefault("conversion_over_scute_time", {})[n] = (res["lora64_conversions"][n]["ms"] /
                                                               res["scute"][n]["ms"])
    return {"workload": "scaling_ia3_vera: 256 tokens, 1024 adapters half (IA)^3 half VeRA (shared rank 256), "
                        "Zipf(1.0) ids; comparator: the same ids as rank-64 LoRA conversions",
            "unit": "tokens/s", "peak_gbs": hbm, "peak_kind": peak_kind, **res}


def stack_leg(scute, dev, flush, launch_us, steps=10):
    """The 32-layer stack of all 7 projections (q, k, v, o, gate, up, down)
    per layer at 128 tokens, 128 adapters (method = id mod 5, OFT on every
    projection, (IA)^3 on k, v, up): one step = every layer once, captured in
    one CUDA graph; per-step time of the mixed pool against its all-LoRA
    twin (the same ids as rank-16 LoRA adapters).  Two launch groupings: one
    batched call per layer, and the groups a block's data dependencies allow
    ({q, k, v}, {o}, {gate, up}, {down})."""
    import torch
    hbm, tf, _, peak_kind = peaks()
    w = WL.stack_32layer()
    n_layers = 32
    P7 = ("q", "k", "v", "o", "gate", "up", "down")
    GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))
    stream = torch.cuda.Stream(device=dev)
    ids = torch.from_numpy(w.ids.copy()).to(dev)
    xs = {L.name: WL.device_normal(0, f"x/{L.name}", (w.n, L.d_in), 1.0, "bf16", dev) for L in w.layers}
    outs = {L.name: torch.empty(w.n, L.d_out, dtype=torch.bfloat16, device=dev) for L in w.layers}
    res = {}
    for label, conv in (("mixed", None), ("all_lora", 16)):
        ctx = scute.Context("bf16", max_tokens=w.n, max_adapters=w.n_adapters, max_layers=len(w.layers),
                            device=dev.index)
        try:
            t0 = time.time()
            load_device_drawn(ctx, w, dev, only_lora_rank=conv)
            load_s = time.time() - t0

            def per_layer(groups):
                def fn():
                    for li in range(n_layers):
                        for grp in groups:
                            names = [f"L{li}.{p}" for p in grp]
                            ctx.linear_batch([(xs[n], ctx.layer_ids[n], outs[n]) for n in names], ids, "bf16",
                                             stream=stream)
                return fn
            r = {"load_s": load_s}
            for gname, groups in (("one_launch_per_layer", (P7,)), ("block_groups", GROUPS)):
                fn = per_layer(groups)
                with torch.cuda.stream(stream):
                    fn()
                torch.cuda.synchronize()
                n0 = ctx.launch_count()
                g = capture(fn, stream)
                launches = ctx.launch_count() - n0
                graph_time(g, stream, flush, 2)
                ms, _ = graph_time(g, stream, flush, steps)
                reps = []
                for li in range(n_layers):
                    for grp in groups:
                        reps.append(ctx.predict_batch([ctx.layer_ids[f"L{li}.{p}"] for p in grp], w.ids, "bf16"))
                rep = merge_reports(reps)
                pure, full = predicted(scute, rep, hbm, tf, launch_us)
                gbs = rep["algorithmic_bytes"] / (ms * 1e-3) / 1e9
                r[gname] = {"ms_per_step": ms, "tokens_per_s": w.n / (ms * 1e-3), "launches_per_step": launches,
                            "algorithmic_bytes": rep["algorithmic_bytes"], "gbs": gbs, "frac": gbs / hbm,
                            "predicted_ms": full / 1e3, "predicted_ms_bytes_only": pure / 1e3}
                del g
            if ctx.sync_status() != 0:
                raise RuntimeError("device status error in the stack leg")
            res[label] = r
        finally:
            ctx.close()
            torch.cuda.empty_cache()
    for g in ("one_launch_per_layer", "block_groups"):
        res.setdefault("overhead_vs_all_lora_pct", {})[g] = 100.0 * (res["mixed"][g]["ms_per_step"] /
                                                                     res["all_lora"][g]["ms_per_step"] - 1.0)
    return {"workload": "stack_32layer: 32 layers x 7 projections (q,k,v,o,gate,up,down), 128 tokens, 128 "
                        "adapters (method = id mod 5, OFT on every projection, (IA)^3 on k, v, up), rank 16; "
                        "all-LoRA twin: same ids, rank-16 LoRA", "peak_gbs": hbm, "peak_kind": peak_kind, **res}


def validation_leg(scute, dev, flush, launch_us, steps=30):
    """The time model checked on separate-pass placements (the article's
    validation: OFT's rotation in its own pass, DoRA's s outside the expand):
    the six decode projections at 16, 32, 64 and 128 tokens, each placement's
    added time predicted (extra bytes / bandwidth + extra launches x launch
    cost) and measured (graph replays, L2 flushed), and each pass launch's own
    time beside its prediction."""
    import torch
    hbm, tf, _, peak_kind = peaks()
    w = WL.decode_mixed(n=128)
    ctx = scute.Context("bf16", max_tokens=128, max_adapters=40, max_layers=8, device=dev.index)
    rows = []
    try:
        ctx.load_workload(w)
        stream = torch.cuda.Stream(device=dev)
        xs = {p: torch.from_numpy(np.ascontiguousarray(w.layer(p).get("x")).view(np.int16)).to(dev)
              .view(torch.bfloat16) for p in PROJ}
        outs = {p: torch.empty(128, w.layer(p).d_out, dtype=torch.bfloat16, device=dev) for p in PROJ}
        ids_all = torch.from_numpy(w.ids.copy()).to(dev)
        for n in (16, 32, 64, 128):
            ids = ids_all[:n]

            def call():
                ctx.linear_batch([(xs[p][:n], ctx.layer_ids[p], outs[p][:n]) for p in PROJ], ids, "bf16",
                                 stream=stream)
            res = {}
            for v in (0, 1, 2, 3):
                ctx.set_variant(v)
                with torch.cuda.stream(stream):
                    call()
                torch.cuda.synchronize()
                g = capture(call, stream)
                graph_time(g, stream, flush, 3)
                ms, _ = graph_time(g, stream, flush, steps)
                # each launch of the call timed on its own (eager, event pairs)
                ctx.timing(True)
                per = {}
                for _ in range(5):
                    ctx.timing_reset()
                    with torch.cuda.stream(stream):
                        flush.fill_(1)
                    call()
                    for k, t in zip(ctx.timing_kinds(), ctx.timing_read()):
                        per.setdefault(k, []).append(t)
                ctx.timing(False)
                rep = ctx.predict_batch([ctx.layer_ids[p] for p in PROJ], w.ids[:n], "bf16")
                res[v] = {"ms": ms, "rep": rep, "kernel_ms": {k: float(np.median(t)) for k, t in per.items()}}
                del g
            base = res[0]
            pred0 = scute.scute_predict_time(base["rep"], hbm, 0.0, launch_us)
            for v, label in ((1, "rotation as its own pass"), (2, "DoRA / (IA)^3 s as its own pass"),
                             (3, "both passes")):
                r = res[v]
                pred = scute.scute_predict_time(r["rep"], hbm, 0.0, launch_us)
                added_meas = 1e3 * (r["ms"] - base["ms"])
                added_pred = pred - pred0
                row = {"n": n, "placement": label, "added_predicted_us": added_pred, "added_measured_us": added_meas,
                       "added_error_pct": 100.0 * abs(added_meas - added_pred) / max(abs(added_meas), 1e-9)}
                # the pass launches alone: their own predicted and measured times
                for name, b, f in r["rep"]["kernels"]:
                    if name in ("oft_pass", "s_pass"):
                        p_us = b / (hbm * 1e3) + launch_us
                        m_us = 1e3 * r["kernel_ms"].get(name, float("nan"))
                        row[name] = {"bytes": b, "predicted_us": p_us, "measured_us": m_us,
                                     "error_pct": 100.0 * abs(m_us - p_us) / m_us}
                rows.append(row)
        ctx.set_variant(0)
        if ctx.sync_status() != 0:
            raise RuntimeError("device status error in the validation leg")
    finally:
        ctx.close()
    pass_err = [r[k]["error_pct"] for r in rows for k in ("oft_pass", "s_pass") if k in r]
    added_err = [r["added_error_pct"] for r in rows]
    return {"workload": "decode_mixed projections q,k,v,gate,up,down at 16/32/64/128 tokens; placements of the "
                        "rotation and of DoRA's and (IA)^3's s in launches of their own",
            "hbm_gbs": hbm, "peak_kind": peak_kind, "launch_us": launch_us, "rows": rows,
            "median_error_pct_pass_launches": float(np.median(pass_err)) if pass_err else None,
            "median_error_pct_added_time": float(np.median(added_err)) if added_err else None}


# ------------------------------------------------------------------ GPU arm
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

    if args.prefill_eager > 0:
        wp = WL.prefill_mixed(proj=("q",))
        ctx = scute.Context("bf16", max_tokens=wp.n, max_adapters=wp.n_adapters + 8, max_layers=2,
                            device=local_rank)
        ctx.load_workload(wp)
        x = to_dev(wp.layer("q").get("x"))
        ids = torch.from_numpy(wp.ids.copy()).to(dev)
        out = torch.empty(wp.n, 4096, dtype=torch.bfloat16, device=dev)
        for _ in range(args.prefill_eager):
            ctx.linear(x, ids, ctx.layer_ids["q"], out, "bf16")
        torch.cuda.synchronize()
        if ctx.sync_status() != 0:
            raise RuntimeError("device status error")
        ctx.close()
        return

    ctx = scute.Context("bf16", max_tokens=64, max_adapters=40, max_layers=8, device=local_rank)
    ctx.load_workload(w)
    if args.eager_steps > 0:
        xs = {p: to_dev(w.layer(p).get("x")) for p in PROJ}
        ids = torch.from_numpy(w.ids.copy()).to(dev)
        outs = {p: torch.empty(w.n, w.layer(p).d_out, dtype=torch.bfloat16, device=dev) for p in PROJ}
        ctx.set_variant(args.eager_variant)
        rep = ctx.predict_batch([ctx.layer_ids[p] for p in PROJ], w.ids, "bf16")
        for name, b, _f in rep["kernels"]:
            print(f"byte model, placement {args.eager_variant}: {name} {b} bytes", file=sys.stderr)
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

    n0 = ctx.launch_count()
    g_mixed = capture(lambda: step(ctx, outs), stream)
    launches_per_step = ctx.launch_count() - n0
    g_lora = capture(lambda: step(ctx_l, outs_l), stream)
    g_grouped = capture(lambda: step_grouped(ctx, outs), stream)
    g_calls = capture(lambda: step_calls(ctx, outs), stream)
    ctx.timing(True)
    ctx.timing_reset()
    g_timed = capture(lambda: step(ctx, outs), stream)
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

    hbm_peak, tf_peak, _, peak_kind = peaks()
    launch_us = launch_cost_us(dev)
    # byte model of the step as launched: one launch moves every projection's bytes
    layer_ids = [ctx.layer_ids[p] for p in PROJ]
    rep_mixed = ctx.predict_batch(layer_ids, w.ids, "bf16")
    rep_lora = ctx_l.predict_batch([ctx_l.layer_ids[p] for p in PROJ], wl.ids, "bf16")
    rep_grouped = merge_reports([ctx.predict_batch([ctx.layer_ids[p] for p in grp], w.ids, "bf16")
                                 for grp in BLOCK_GROUPS])
    rep_calls = merge_reports([ctx.predict_batch([ctx.layer_ids[p]], w.ids, "bf16") for p in PROJ])
    alg_bytes = rep_mixed["algorithmic_bytes"]
    kernel_ms = float(np.mean(np.array(t_kernel, dtype=np.float64)))
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9

    time_model = {"hbm_gbs": hbm_peak, "launch_us": launch_us,
                  "launch_us_how": "CUDA graph of 400 dependent one-element kernels, replay time / 400",
                  "rows": []}

    def tm_row(name, rep, measured_ms):
        pure, full = predicted(scute, rep, hbm_peak, tf_peak, launch_us)
        time_model["rows"].append({"what": name, "launches": len(rep["kernels"]),
                                   "predicted_us": pure, "measured_us": 1e3 * measured_ms,
                                   "error_pct": 100.0 * (1e3 * measured_ms - pure) / (1e3 * measured_ms)})

    tm_row("decode step, mixed (1 launch)", rep_mixed, ms)
    tm_row("decode step, all-LoRA (1 launch)", rep_lora, ms_lora)
    tm_row("decode, block groups (3 launches)", rep_grouped, float(np.mean(t_grouped)))
    tm_row("decode, separate calls (6 launches)", rep_calls, float(np.mean(t_calls)))
    added_pred = (predicted(scute, rep_mixed, hbm_peak, tf_peak, launch_us)[0] -
                  predicted(scute, rep_lora, hbm_peak, tf_peak, launch_us)[0])
    time_model["added_mixed_over_all_lora"] = {"predicted_us": added_pred, "measured_us": 1e3 * (ms - ms_lora)}

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

    traffic = captured_traffic()
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
                     "peak_kind": peak_kind, "traffic": traffic,
                     "traffic_source": (f"committed ncu capture ({STEP_CAPTURE}); k_step.cu unchanged since"
                                        if traffic is not None else None),
                     "kernel_ms": kernel_ms, "algorithmic_bytes_per_launch": alg_bytes},
        "block_groups_ms_per_step": float(np.mean(t_grouped)),
        "separate_calls_ms_per_step": float(np.mean(t_calls)),
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": int(launches_per_step * args.steps),
        "launches_per_step": int(launches_per_step),
        "clocks": clocks,
        "time_model": time_model,
    }
    ctx.close()
    ctx_l.close()
    del g_mixed, g_lora, g_grouped, g_calls, g_timed
    torch.cuda.empty_cache()
    if rank == 0 and world == 1:
        for key, skip, fn in (("prefill", args.no_prefill, prefill_leg), ("adapter_scaling", args.no_scaling, scaling_leg),
                              ("stack", args.no_stack, stack_leg),
                              ("time_model_validation", args.no_validation, validation_leg)):
            if skip:
                continue
            assert key not in line, key   # a leg never replaces a key of the line's contract
            try:
                line[key] = fn(scute, dev, flush, launch_us)
            except Exception as exc:   # the headline line is printed whatever a leg does
                line[key] = {"error": f"{type(exc).__name__}: {str(exc)[:300]}"}
            torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    if len(sys.argv) == 3 and sys.argv[1] == "--cpu-baseline-worker":
        print(json.dumps(cpu_baseline_worker(float(sys.argv[2]))), flush=True)
    else:
        main()
