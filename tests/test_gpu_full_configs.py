"""GPU parity at the full sizes of the larger workloads, graded on sampled
output rows that the float64 oracle computes one by one:

* prefill: 16 requests of 64..1024 tokens (8772 in all), one adapter each from
  32 mixed adapters, Llama-3-8B-shaped q (4096->4096) and down (14336->4096);
* adapter-count scaling: 256 tokens, 1024 adapters (even ids (IA)^3, odd ids
  VeRA), Zipf(1.0) ids, 4096->4096 and 4096->14336 layers;
* layer stack: two of the 32 Llama-shaped layers, all seven projections each,
  128 tokens, 128 adapters, every layer's projections in one batched call.
"""
import numpy as np
import pytest

import workloads as WL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import gpu_harness as H  # noqa: E402


@pytest.fixture(scope="module")
def scute(gpu_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gpu_lib


def _rows(n, k=12, seed=0):
    g = np.random.default_rng(seed)
    return sorted(set([0, n - 1] + g.choice(n, size=k, replace=False).tolist()))


def test_prefill_full_shapes_sampled(scute):
    w = WL.prefill_mixed(proj=("q", "down"))
    assert w.n == 8772
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, ("q", "down"), "fp32")
    assert ctx.sync_status() == 0
    rows = _rows(w.n)
    for name in ("q", "down"):
        H.grade(w, name, outs[name], "fp32", rows=rows)
    ctx.close()


def test_scaling_ia3_vera_full_sampled(scute):
    w = WL.scaling_ia3_vera()
    ctx = H.make_ctx(scute, w)
    names = [L.name for L in w.layers]
    outs = H.run_layers(ctx, w, names, "fp32")
    assert ctx.sync_status() == 0
    rows = _rows(w.n)
    for name in names:
        H.grade(w, name, outs[name], "fp32", rows=rows)
    ctx.close()


def test_layer_stack_two_layers_batched_sampled(scute):
    w = WL.stack_32layer(n_layers=2)
    ctx = H.make_ctx(scute, w)
    ids_t = torch.from_numpy(np.ascontiguousarray(w.ids, dtype=np.int32)).cuda()
    rows = _rows(w.n)
    for li in range(2):
        names = [f"L{li}.{p}" for p in ("q", "k", "v", "o", "gate", "up", "down")]
        calls, outs = [], []
        for name in names:
            L = w.layer(name)
            out = torch.full((w.n, L.d_out), float("nan"), device="cuda", dtype=torch.float32)
            calls.append((H.dev(L.get("x")), ctx.layer_ids[name], out))
            outs.append(out)
        ctx.linear_batch(calls, ids_t, "fp32")
        torch.cuda.synchronize()
        assert ctx.sync_status() == 0
        for name, o in zip(names, outs):
            H.grade(w, name, o, "fp32", rows=rows)
        del calls
    ctx.close()
