"""A heterogeneous batch evaluated per token (float64).

Test infrastructure only (see ``oracle/__init__``).

Every token carries its own adapter id; the article's batched layer computes,
for each token t with adapter a = ids[t], ``F_a(x_t)`` ("The big picture").
Rows are independent, so rows that share an adapter are evaluated together as
one matrix (a row subset of the same definition, no reordering of any sum).
Tokens with id -1, or with an id that names no adapter, get ``x_t W``.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from workloads import to_f64
from . import methods as M
from . import normal_form as NF


def adapter_params(w, aid: int, layer) -> Optional[dict]:
    """Raw float64 parameters of adapter ``aid`` on ``layer``, or None when it
    has no tensors there (all slots identity)."""
    a = w.adapter(aid)
    slots = a.slots(layer.name)
    if not slots:
        return None
    p = {s: to_f64(a.get(layer.name, s)) for s in slots}
    if a.method in ("lora", "dora", "nf"):
        p["c"] = float(a.c)
    if a.method == "vera":
        p["A_sh"] = to_f64(layer.get("A_sh"))
        p["B_sh"] = to_f64(layer.get("B_sh"))
    return p


def linear(w, layer_name: str, rows: Optional[Sequence[int]] = None,
           form: str = "definitional", x: Optional[np.ndarray] = None) -> np.ndarray:
    """Outputs of ``rows`` (default all tokens) of one adapted linear layer.

    ``form``: "definitional" (each method from its own definition), "normal"
    (unfolded normal form), "folded" (normal form after the fold rule) or
    "merged" (explicit per-adapter weight, tiny shapes only).
    """
    L = w.layer(layer_name)
    W = to_f64(L.get("W"))
    X = to_f64(L.get("x")) if x is None else x
    rows = np.arange(w.n) if rows is None else np.asarray(rows, dtype=np.int64)
    ids = np.asarray(w.ids)[rows]
    out = np.zeros((rows.size, L.d_out), dtype=np.float64)
    known = {a.id for a in w.adapters}
    for aid in np.unique(ids):
        sel = np.nonzero(ids == aid)[0]
        xs = X[rows[sel]]
        p = adapter_params(w, int(aid), L) if int(aid) in known else None
        if p is None:
            out[sel] = M.base(xs, W)
            continue
        method = w.adapter(int(aid)).method
        if form == "definitional":
            out[sel] = NF.definitional(method, xs, W, p)
        elif form == "normal":
            out[sel] = NF.evaluate(NF.from_method(method, W, p), xs, W)
        elif form == "folded":
            out[sel] = NF.evaluate(NF.fold(NF.from_method(method, W, p)), xs, W)
        elif form == "merged":
            out[sel] = NF.merged_apply(NF.from_method(method, W, p), xs, W)
        else:
            raise ValueError(form)
    return out


def base_output(w, layer_name: str, rows=None) -> np.ndarray:
    """``x W`` for the same rows: the reference the adapter effect is taken
    against (article, "Does it actually work better?": error as a share of how
    much the adapter changes the output)."""
    L = w.layer(layer_name)
    X = to_f64(L.get("x"))
    rows = np.arange(w.n) if rows is None else np.asarray(rows, dtype=np.int64)
    return M.base(X[rows], to_f64(L.get("W")))
