"""GPU parity at the full sizes of the larger workloads, graded on sampled
output rows that the float64 oracle computes one by one.  Rows are picked per
method (``gpu_harness.stratified_rows``): every method in the batch has rows
graded, OFT included.

* prefill: 16 requests of 64..1024 tokens (8772 in all), one adapter each from
  32 mixed adapters, Llama-3-8B-shaped q (4096->4096) and down (14336->4096);
  the seed-0 draw of request adapters has no OFT adapter, so a second case
  gives the 16 requests adapters 0..15 (every method, OFT at d_in 4096 and
  14336);
* adapter-count scaling: 256 tokens, 1024 adapters (even ids (IA)^3, odd ids
  VeRA), Zipf(1.0) ids, 4096->4096 and 4096->14336 layers;
* layer stack: two of the 32 Llama-shaped layers, all seven projections each,
  128 tokens, 128 adapters, every layer's projections in one batched call.
Each runs with float32 and with bf16 outputs.
"""
import numpy as np
import pytest

import workloads as WL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import gpu_harness as H  # noqa: E402

ALL5 = {"lora", "dora", "ia3", "vera", "oft"}


@pytest.fixture(scope="module")
def scute(gpu_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gpu_lib


@pytest.mark.parametrize("out_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("pool", ["drawn", "every_method"])
def test_prefill_full_shapes_sampled(scute, pool, out_dtype):
    req = None if pool == "drawn" else list(range(16))
    w = WL.prefill_mixed(proj=("q", "down"), req_adapters=req)
    assert w.n == 8772
    rows = H.stratified_rows(w, per_method=3)
    if pool == "every_method":
        assert H.methods_in(w, rows) >= ALL5
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, ("q", "down"), out_dtype)
    assert ctx.sync_status() == 0
    for name in ("q", "down"):
        H.grade(w, name, outs[name], out_dtype, rows=rows)
    ctx.close()


@pytest.mark.parametrize("out_dtype", ["fp32", "bf16"])
def test_scaling_ia3_vera_full_sampled(scute, out_dtype):
    w = WL.scaling_ia3_vera()
    ctx = H.make_ctx(scute, w)
    names = [L.name for L in w.layers]
    outs = H.run_layers(ctx, w, names, out_dtype)
    assert ctx.sync_status() == 0
    rows = H.stratified_rows(w, per_method=6)
    assert H.methods_in(w, rows) >= {"ia3", "vera"}
    for name in names:
        H.grade(w, name, outs[name], out_dtype, rows=rows)
    ctx.close()


@pytest.mark.parametrize("out_dtype", ["fp32", "bf16"])
def test_layer_stack_two_layers_batched_sampled(scute, out_dtype):
    w = WL.stack_32layer(n_layers=2)
    ctx = H.make_ctx(scute, w)
    ids_t = torch.from_numpy(np.ascontiguousarray(w.ids, dtype=np.int32)).cuda()
    rows = H.stratified_rows(w, per_method=3)
    assert H.methods_in(w, rows) >= ALL5
    for li in range(2):
        names = [f"L{li}.{p}" for p in ("q", "k", "v", "o", "gate", "up", "down")]
        calls, outs = [], []
        for name in names:
            L = w.layer(name)
            out = torch.full((w.n, L.d_out), float("nan"), device="cuda",
                             dtype=torch.float32 if out_dtype == "fp32" else torch.bfloat16)
            calls.append((H.dev(L.get("x")), ctx.layer_ids[name], out))
            outs.append(out)
        ctx.linear_batch(calls, ids_t, out_dtype)
        torch.cuda.synchronize()
        assert ctx.sync_status() == 0
        for name, o in zip(names, outs):
            H.grade(w, name, o, out_dtype, rows=rows)
        del calls
    ctx.close()
