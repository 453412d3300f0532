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


def method_of(w, aid: int) -> str:
    """Method name of adapter id ``aid`` in workload ``w`` ("base" for -1 or an
    id that names no adapter)."""
    if aid < 0:
        return "base"
    try:
        return w.adapter(int(aid)).method
    except KeyError:
        return "base"


def stratified_rows(w, per_method: int = 2, seed: int = 0) -> list:
    """Rows to grade at full size: ``per_method`` rows of every method present
    in the batch (from different adapters where the batch has several), the
    base-only rows' first, and the first and last token."""
    g = np.random.default_rng(seed)
    ids = np.asarray(w.ids)
    picked = {0, w.n - 1}
    by_method = {}
    for aid in np.unique(ids):
        by_method.setdefault(method_of(w, int(aid)), []).append(int(aid))
    for m, aids in by_method.items():
        aids = list(g.permutation(aids))
        k = per_method if m != "base" else 1
        for j in range(k):
            a = aids[j % len(aids)]
            rows = np.nonzero(ids == a)[0]
            picked.add(int(g.choice(rows)))
    return sorted(picked)


def methods_in(w, rows) -> set:
    return {method_of(w, int(w.ids[r])) for r in rows}


def grade(w, name, g, out_dtype, rows=None, check_effect=True, ref=None, base=None):
    """Compare device output rows with the oracle; returns a small report.
    ``ref`` / ``base``: the oracle's outputs and ``x W`` for these rows when
    the caller has them already."""
    ref = BT.linear(w, name, rows=rows) if ref is None else ref
    gg = to_f64(g) if rows is None else to_f64(g[torch.as_tensor(rows, device=g.device)])
    ids = np.asarray(w.ids)[np.arange(w.n) if rows is None else np.asarray(rows)]
    rep = {}
    if w.dtype == "fp32":
        rep["fp32_rel"] = MX.fp32_rel_err(gg, ref)
        assert rep["fp32_rel"] <= MX.FP32_REL_TOL, f"{name}: fp32 rel error {rep['fp32_rel']:.3g}"
    elif out_dtype == "bf16":
        MX.assert_bf16_out(gg, ref, name)
        rep["bf16"] = MX.grade_bf16_out(gg, ref)
    if check_effect:
        base = BT.base_output(w, name, rows=rows) if base is None else base
        ee = MX.effect_errors(gg, ref, base, ids)
        rep["effect"] = ee
        rep["effect_max"] = max(ee.values()) if ee else 0.0
        per = {}
        for a, e in ee.items():
            m = method_of(w, a)
            per[m] = max(per.get(m, 0.0), e)
        rep["effect_by_method"] = per
        if out_dtype == "fp32":
            bad = {a: e for a, e in ee.items() if e > MX.EFFECT_TOL}
            assert not bad, f"{name}: adapter effect errors above 1%: {bad}"
        else:
            # a bf16 output carries its own rounding: per adapter, the error
            # may exceed the float32-output bound by what rounding the exact
            # result to bf16 costs (the oracle's own bf16 floor); twice that
            # floor leaves room for the spread of rounding errors over a
            # few hundred elements
            floor = MX.effect_errors(MX.round_bf16(ref), ref, base, ids)
            rep["bf16_floor"] = floor
            bad = {a: (e, floor.get(a, 0.0)) for a, e in ee.items()
                   if e > MX.EFFECT_TOL + 2.0 * floor.get(a, 0.0)}
            assert not bad, f"{name}: bf16-output effect errors above 1% + the bf16 floor: {bad}"
    return rep
