"""Byte model of one adapted-layer call, restated from its definition.

Test infrastructure only (see ``oracle/__init__``).

The article ("Where is the cheapest place to compute the remaining slots?")
measures adapter work in bytes moved and predicts added time as extra bytes /
bandwidth + extra launches x launch cost.  The definition restated here
counts, per kernel launch of the call, every operand read once and every
result written once, and for the call
its algorithmic bytes: W once, each distinct adapter's live tensors once, the
shared VeRA pair once when a VeRA token is present, x read, out written, ids
read.  This module computes those integers with plain Python loops.

Each adapter is described on one layer by the slots it keeps after the fold:
``{"method": str, "rank": int, "s": bool, "b": bool, "R": bool,
"vera": bool, "vera_e": bool}``; ids without an entry are base-only tokens.
"""
from __future__ import annotations


def lowrank_ks(d_in: int) -> int:
    """K splits of the owned low-rank shrink: ceil(d_in / 2048) chunks, at most
    8, each a multiple of 256 elements (the chunk count after rounding)."""
    ks = min(8, -(-d_in // 2048))
    chunk = -(-d_in // ks)
    chunk = -(-chunk // 256) * 256
    return -(-d_in // chunk)


def _layer_counts(ids, adapters: dict, d_in: int, d_out: int, shared_rank: int, dtype: str,
                  out_dtype: str) -> dict:
    """Rows, distinct adapters and live-tensor bytes of one layer's call."""
    E = 4 if dtype == "fp32" else 2
    c = {"E": E, "Eo": 4 if out_dtype == "fp32" else 2, "kd": 3 * d_in if dtype == "fp32" else d_in,
         "rv": shared_rank, "krv": 3 * shared_rank if dtype == "fp32" else shared_rank,
         "n": len(ids), "d_in": d_in, "d_out": d_out}
    seen = []
    has_base = False
    n_lr = lr_rank_rows = n_v = n_rot = 0
    for a in ids:
        a = int(a)
        if a not in adapters:
            has_base = True
            continue
        ad = adapters[a]
        if ad["rank"] > 0:
            n_lr += 1
            lr_rank_rows += ad["rank"]
        if ad["vera"]:
            n_v += 1
        if ad["R"]:
            n_rot += 1
        if a not in seen:
            seen.append(a)
    # tokens of DoRA / (IA)^3 adapters with a live s, and those adapters' distinct s bytes
    n_s = sum(1 for a in ids if int(a) in adapters and adapters[int(a)]["s"]
              and adapters[int(a)]["method"] in ("dora", "ia3"))
    s_pass_vec = 4 * d_out * sum(1 for a in seen if adapters[a]["s"] and adapters[a]["method"] in ("dora", "ia3"))
    live = R_b = sb_b = A_b = B_b = d_b = e_b = 0
    for a in seen:
        ad = adapters[a]
        if ad["s"]:
            live += 4 * d_out
            sb_b += 4 * d_out
        if ad["b"]:
            live += 4 * d_out
            sb_b += 4 * d_out
        if ad["R"]:
            live += 32 * d_in * E
            R_b += 32 * d_in * E
        if ad["rank"] > 0:
            live += ad["rank"] * (d_in + d_out) * E
            A_b += ad["rank"] * d_in * E
            B_b += ad["rank"] * d_out * E
        if ad["vera"]:
            live += 4 * shared_rank
            d_b += 4 * shared_rank
            if ad["vera_e"]:
                live += 4 * d_out
                e_b += 4 * d_out
    c.update(n_s=n_s, s_pass_vec=s_pass_vec)
    c.update(seen=seen, segments=len(seen) + (1 if has_base else 0), n_lr=n_lr, lr_rank_rows=lr_rank_rows,
             n_v=n_v, n_rot=n_rot, live=live, R_b=R_b, sb_b=sb_b, A_b=A_b, B_b=B_b, d_b=d_b, e_b=e_b)
    c["shared"] = (d_in + d_out) * shared_rank * E if n_v else 0
    c["W"] = d_in * d_out * E
    # W once, each distinct adapter's live tensors once, the shared pair once
    # when a VeRA token is present, x read, out written (ids counted by the caller)
    c["alg_no_ids"] = c["W"] + live + c["shared"] + c["n"] * d_in * E + c["n"] * d_out * c["Eo"]
    # every term of the normal form over the batch: base GEMM, rotation,
    # owned shrink and expand, VeRA shrink and expand (2 flops per multiply-add)
    c["flops"] = (2 * c["n"] * d_in * d_out + 2 * n_rot * d_in * 32 + 2 * lr_rank_rows * (d_in + d_out)
                  + 2 * n_v * shared_rank * (d_in + d_out))
    return c


def _per_kernel_plan(c, lowrank_launched: bool, vera_launched: bool, lr_fused: bool = False) -> list:
    """Launches of one layer's call on the per-kernel plan, (name, bytes, flops).

    With ``lr_fused`` (bf16 contexts, more than 256 tokens) the owned shrink
    runs before the base GEMM and the owned expand inside the GEMM's epilogue:
    the GEMM then also reads the shrink's partial v and each B', and out is
    written once.  There the VeRA shrink of a shared rank that is a multiple
    of 64 (its tensor-core form) also comes before the base GEMM."""
    n, E, Eo, kd, d_in, d_out = c["n"], c["E"], c["Eo"], c["kd"], c["d_in"], c["d_out"]
    rv, krv = c["rv"], c["krv"]
    index_out = 8 * n + 4 * (c["segments"] + 1) + 4 * c["segments"] + 88
    ks = lowrank_ks(d_in)
    shrink = ("lr_shrink", c["n_lr"] * d_in * E + c["A_b"] + ks * c["lr_rank_rows"] * 4,
              2 * c["lr_rank_rows"] * d_in)
    fused = lowrank_launched and lr_fused
    # W, x', s/b vectors, perm/ids, out (and the fused expand's v partials and B')
    gemm_b = d_out * kd * E + n * kd * E + c["sb_b"] + 8 * n + n * d_out * Eo
    gemm_f = 2 * n * kd * d_out
    if fused:
        gemm_b += ks * c["lr_rank_rows"] * 4 + c["B_b"]
        gemm_f += 2 * c["lr_rank_rows"] * d_out
    kernels = [
        # ids in; perm and sorted ids out; segment table; 22-int summary
        ("index", 4 * n + index_out, 0),
        # x in, perm/ids in, R of each distinct rotating adapter, x' out
        ("rotate", n * d_in * E + 8 * n + c["R_b"] + n * kd * E, 2 * c["n_rot"] * d_in * 32),
    ]
    n_v = c["n_v"]
    shA = rv * kd * E if n_v else 0
    shB = d_out * krv * E if n_v else 0
    vshrink = ("vera_shrink", n_v * kd * E + shA + c["d_b"] + n_v * krv * E, 2 * n_v * rv * kd)
    vs_first = vera_launched and lr_fused and rv % 64 == 0
    if fused:
        kernels.append(shrink)
    if vs_first:
        kernels.append(vshrink)
    kernels.append(("base_gemm", gemm_b, gemm_f))
    if lowrank_launched and not fused:
        kernels.append(shrink)
        kernels.append(("lr_expand", ks * c["lr_rank_rows"] * 4 + c["B_b"] + 2 * c["n_lr"] * d_out * Eo,
                        2 * c["lr_rank_rows"] * d_out))
    if vera_launched:
        if not vs_first:
            kernels.append(vshrink)
        kernels.append(("vera_expand", n_v * krv * E + shB + c["e_b"] + 2 * n_v * d_out * Eo,
                        2 * n_v * krv * d_out))
    return kernels


def batch_bytes(ids, layers: list, dtype: str, out_dtype: str, variant: int = 0) -> dict:
    """Launch list and algorithmic bytes of one batched call over ``layers``
    (each a dict with keys adapters, d_in, d_out, shared_rank,
    lowrank_launched, vera_launched) that read the same ids.

    A bf16 batch of at most 128 tokens is one launch over every layer; its
    bytes are what crosses that launch: the ids once and every layer's W, live
    adapter tensors, shared pair, x and out.  Otherwise every layer follows
    the per-kernel plan in turn."""
    n = len(ids)
    cs = [_layer_counts(ids, L["adapters"], L["d_in"], L["d_out"], L["shared_rank"], dtype, out_dtype)
          for L in layers]
    alg = 4 * n + sum(c["alg_no_ids"] for c in cs)
    if dtype != "fp32" and n <= 128:
        # separate-pass placements (variant bits 1: rotation, 2: DoRA / (IA)^3 s)
        step_bytes, step_flops = alg, sum(c["flops"] for c in cs)
        kernels = []
        if variant & 1:
            b = 4 * n + sum(2 * c["n"] * c["d_in"] * c["E"] + c["R_b"] for c in cs)
            f = sum(2 * c["n_rot"] * c["d_in"] * 32 for c in cs)
            step_bytes -= sum(c["R_b"] for c in cs)
            step_flops -= f
            kernels.append(("oft_pass", b, f))
        if variant & 2:
            sb = 4 * n + sum(2 * c["n_s"] * c["d_out"] * c["Eo"] + c["s_pass_vec"] for c in cs)
            sf = sum(c["n_s"] * c["d_out"] for c in cs)
            step_bytes -= sum(c["s_pass_vec"] for c in cs)
        kernels.append(("step", step_bytes, step_flops))
        if variant & 2:
            kernels.append(("s_pass", sb, sf))
    else:
        kernels = []
        for L, c in zip(layers, cs):
            kernels += _per_kernel_plan(c, L["lowrank_launched"], L["vera_launched"],
                                        lr_fused=dtype != "fp32" and n > 256)
    return {
        "kernels": kernels,
        "algorithmic_bytes": alg,
        "adapter_bytes": sum(c["live"] + c["shared"] for c in cs),
        "base_weight_bytes": sum(c["W"] for c in cs),
        "distinct_adapters": len(cs[0]["seen"]),
    }


def call_bytes(ids, adapters: dict, d_in: int, d_out: int, shared_rank: int, dtype: str,
               out_dtype: str, lowrank_launched: bool, vera_launched: bool) -> dict:
    """One call of one layer: a batch of one."""
    return batch_bytes(ids, [{"adapters": adapters, "d_in": d_in, "d_out": d_out, "shared_rank": shared_rank,
                              "lowrank_launched": lowrank_launched, "vera_launched": vera_launched}],
                       dtype, out_dtype)


def predict_time_us(kernels, hbm_gbs: float, tensor_tflops: float, launch_us: float) -> float:
    """The article's time model, launch by launch: bytes / bandwidth plus one
    launch cost per launch; a launch bound by arithmetic instead takes
    flops / tensor peak (dropped when tensor_tflops <= 0)."""
    t = 0.0
    for _, b, f in kernels:
        t_mem = b / (hbm_gbs * 1e3)
        t_math = f / (tensor_tflops * 1e6) if tensor_tflops > 0 else 0.0
        t += max(t_mem, t_math)
    return t + launch_us * len(kernels)


def adapter_slots_after_fold(method: str, raw_slots, rank: int) -> dict:
    """Which slots a method keeps live on a layer after the fold rule, from the
    raw tensors it has there (article, "Which slots can be merged at load?")."""
    raw = set(raw_slots)
    owned = "A" in raw
    return {
        "method": method,
        "rank": rank if owned else 0,
        "s": (method == "dora" and owned) or (method == "ia3" and "l" in raw) or (method == "nf" and "s" in raw),
        "b": method == "nf" and "b" in raw,
        "R": "R" in raw,
        "vera": method == "vera" and "d" in raw,
        "vera_e": method == "vera" and "e" in raw,
    }
