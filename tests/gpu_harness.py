"""Shared helpers of the GPU tests: move a synthetic workload onto the device,
run it through the C ABI, and grade it against the float64 oracle."""
import numpy as np
import torch

import workloads as WL
from oracle import batch as BT
import metrics as MX


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy storage array -> device tensor (uint16 bit patterns become bf16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def make_ctx(scute, w, layer_names=None, max_tokens=None, max_adapters=None):
    names = [L.name for L in w.layers] if layer_names is None else list(layer_names)
    ctx = scute.Context(dtype=w.dtype, max_tokens=max_tokens or max(w.n, 64),
                        max_adapters=max_adapters or (w.n_adapters + 8), max_layers=len(names) + 1)
    ctx.load_workload(w, names)
    return ctx


def run_layers(ctx, w, names, out_dtype, ids=None):
    ids_np = w.ids if ids is None else ids
    ids_t = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    outs = {}
    for name in names:
        L = w.layer(name)
        x = dev(L.get("x"))
        out = torch.empty(w.n, L.d_out, device="cuda",
                          dtype=torch.float32 if out_dtype == "fp32" else torch.bfloat16)
        ctx.linear(x, ids_t, ctx.layer_ids[name], out, out_dtype)
        outs[name] = out
    torch.cuda.synchronize()
    return outs


def grade(w, name, g, out_dtype, rows=None, check_effect=True):
    """Compare device output rows with the oracle; returns a small report."""
    ref = BT.linear(w, name, rows=rows)
    gg = to_f64(g) if rows is None else to_f64(g[torch.as_tensor(rows, device=g.device)])
    rep = {}
    if w.dtype == "fp32":
        rep["fp32_rel"] = MX.fp32_rel_err(gg, ref)
        assert rep["fp32_rel"] <= MX.FP32_REL_TOL, f"{name}: fp32 rel error {rep['fp32_rel']:.3g}"
    elif out_dtype == "bf16":
        MX.assert_bf16_out(gg, ref, name)
        rep["bf16"] = MX.grade_bf16_out(gg, ref)
    if check_effect and (out_dtype == "fp32"):
        base = BT.base_output(w, name, rows=rows)
        ids = np.asarray(w.ids)[np.arange(w.n) if rows is None else np.asarray(rows)]
        ee = MX.effect_errors(gg, ref, base, ids)
        rep["effect_max"] = max(ee.values()) if ee else 0.0
        bad = {a: e for a, e in ee.items() if e > MX.EFFECT_TOL}
        assert not bad, f"{name}: adapter effect errors above 1%: {bad}"
    return rep
