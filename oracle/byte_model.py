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
    """K splits of the owned low-rank shrink: ceil(d_in / 512) chunks, at most
    8, each a multiple of 256 elements (the chunk count after rounding)."""
    ks = min(8, -(-d_in // 512))
    chunk = -(-d_in // ks)
    chunk = -(-chunk // 256) * 256
    return -(-d_in // chunk)


def call_bytes(ids, adapters: dict, d_in: int, d_out: int, shared_rank: int, dtype: str,
               out_dtype: str, lowrank_launched: bool, vera_launched: bool) -> dict:
    E = 4 if dtype == "fp32" else 2
    Eo = 4 if out_dtype == "fp32" else 2
    kd = 3 * d_in if dtype == "fp32" else d_in
    rv = shared_rank
    krv = 3 * rv if dtype == "fp32" else rv
    n = len(ids)

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
            live += 4 * rv
            d_b += 4 * rv
            if ad["vera_e"]:
                live += 4 * d_out
                e_b += 4 * d_out
    segments = len(seen) + (1 if has_base else 0)

    # bf16 calls of at most 128 tokens follow the fused decode plan (one
    # prologue launch and one GEMM launch); others launch one kernel per step
    fused = dtype != "fp32" and n <= 128
    index_out = 8 * n + 4 * (segments + 1) + 4 * segments + 88
    if fused:
        shA = rv * d_in * E if n_v else 0
        shB = d_out * rv * E if n_v else 0
        kernels = [
            # ids; x once; R, A', shared A, d once each; x', v, U and the index out
            ("prep", 4 * n + n * d_in * E + R_b + A_b + shA + d_b + n * kd * E + lr_rank_rows * 4
             + n_v * rv * E + index_out,
             2 * n_rot * d_in * 32 + 2 * lr_rank_rows * d_in + 2 * n_v * rv * d_in),
            # W, x', s/b, B', v, shared B, U, e, perm/ids, out
            ("base_gemm", d_out * kd * E + n * kd * E + sb_b + B_b + lr_rank_rows * 4 + shB + n_v * rv * E
             + e_b + 8 * n + n * d_out * Eo,
             2 * n * kd * d_out + 2 * lr_rank_rows * d_out + 2 * n_v * rv * d_out),
        ]
    else:
        kernels = [
            # ids in; perm and sorted ids out; segment table; 22-int summary
            ("index", 4 * n + index_out, 0),
            # x in, perm/ids in, R of each distinct rotating adapter, x' out
            ("rotate", n * d_in * E + 8 * n + R_b + n * kd * E, 2 * n_rot * d_in * 32),
            # W, x', s/b vectors, perm/ids, out
            ("base_gemm", d_out * kd * E + n * kd * E + sb_b + 8 * n + n * d_out * Eo, 2 * n * kd * d_out),
        ]
        if lowrank_launched:
            ks = lowrank_ks(d_in)
            kernels.append(("lr_shrink", n_lr * d_in * E + A_b + ks * lr_rank_rows * 4, 2 * lr_rank_rows * d_in))
            kernels.append(("lr_expand", ks * lr_rank_rows * 4 + B_b + 2 * n_lr * d_out * Eo,
                            2 * lr_rank_rows * d_out))
        if vera_launched:
            shA = rv * kd * E if n_v else 0
            shB = d_out * krv * E if n_v else 0
            kernels.append(("vera_shrink", n_v * kd * E + shA + d_b + n_v * krv * E, 2 * n_v * rv * kd))
            kernels.append(("vera_expand", n_v * krv * E + shB + e_b + 2 * n_v * d_out * Eo,
                            2 * n_v * krv * d_out))
    shared = (d_in + d_out) * rv * E if n_v else 0
    W = d_in * d_out * E
    return {
        "kernels": kernels,
        "algorithmic_bytes": W + live + shared + n * d_in * E + n * d_out * Eo + 4 * n,
        "adapter_bytes": live + shared,
        "base_weight_bytes": W,
        "distinct_adapters": len(seen),
    }


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
