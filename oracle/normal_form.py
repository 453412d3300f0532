"""The six-slot normal form, the method -> slot mapping and the fold rule.

Test infrastructure only (see ``oracle/__init__``).

The article ("The big picture: six extra slots in the LoRA computation") writes
every adapter as

    F_a(x) = ((x R) W) * s + b + sum_k c_k (((x A_k) * d_k) B_k * e_k)

with base-path slots R (input rotation), s (per-output-column factor), b
(shift) and, per low-rank term, d (between A and B), e (after B) and the scalar
c.  An unused slot holds the identity (1, ones, 0 or I).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np

from . import methods as M


@dataclass
class Term:
    """One low-rank term: ``c (((x A) * d) B * e)``.  ``shared`` marks a term
    whose A and B all tenants share (VeRA); None in d / e means ones."""
    A: np.ndarray
    B: np.ndarray
    d: Optional[np.ndarray] = None
    e: Optional[np.ndarray] = None
    c: float = 1.0
    shared: bool = False


@dataclass
class NormalForm:
    """Slots of one adapter on one layer.  None means the identity value."""
    R: Optional[np.ndarray] = None          # [d_in, d_in] (already assembled)
    s: Optional[np.ndarray] = None          # [d_out]
    b: Optional[np.ndarray] = None          # [d_out]
    terms: List[Term] = field(default_factory=list)


def evaluate(nf: NormalForm, x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Evaluate the normal-form equation slot by slot, in its written order."""
    xr = x if nf.R is None else x @ nf.R
    y = xr @ W
    if nf.s is not None:
        y = y * nf.s
    if nf.b is not None:
        y = y + nf.b
    for t in nf.terms:
        u = x @ t.A
        if t.d is not None:
            u = u * t.d
        z = u @ t.B
        if t.e is not None:
            z = z * t.e
        y = y + t.c * z
    return y


def from_method(method: str, W: np.ndarray, p: dict) -> NormalForm:
    """Write one method's raw parameters into the slots (unfolded).

    * LoRA: one owned term (A, B, c); every other slot identity.
    * DoRA: s = m / ||col(W + cAB)|| on the base path and the same factor as e
      on the low-rank path (article, "Which slots can be merged at load?").
    * (IA)^3: s = l (only on layers that carry l).
    * VeRA: one shared term (A_sh, B_sh) with live d and e, c = 1.
    * OFT: R = blockdiag(R_1 .. R_{d_in / b}).
    * nf: raw slots as given (s, b, R blocks, one owned term with d, e, c).
    ``p`` holds float64 arrays; missing keys mean the slot is absent.
    """
    if method == "lora":
        return NormalForm(terms=[Term(A=p["A"], B=p["B"], c=p["c"])])
    if method == "dora":
        s = M.dora_scale(W, p["A"], p["B"], p["c"], p["m"])
        return NormalForm(s=s, terms=[Term(A=p["A"], B=p["B"], e=s, c=p["c"])])
    if method == "ia3":
        return NormalForm(s=p.get("l"))
    if method == "vera":
        if "d" not in p:
            return NormalForm()
        return NormalForm(terms=[Term(A=p["A_sh"], B=p["B_sh"], d=p["d"], e=p["e"],
                                      c=1.0, shared=True)])
    if method == "oft":
        return NormalForm(R=M.block_diag(p["R"]) if "R" in p else None)
    if method == "nf":
        terms = []
        if "A" in p:
            terms.append(Term(A=p["A"], B=p["B"], d=p.get("d"), e=p.get("e"), c=p["c"]))
        return NormalForm(R=M.block_diag(p["R"]) if "R" in p else None,
                          s=p.get("s"), b=p.get("b"), terms=terms)
    raise ValueError(method)


def fold(nf: NormalForm) -> NormalForm:
    """Apply the fold rule at load (article, "Which slots can be merged at
    load?").  A slot next to a tensor the adapter owns is multiplied into it:
    ``(xA) * d = x (A diag(d))`` puts d into A, the scalar c goes into A too,
    and e goes into the adapter's own B.  Slots whose neighbours are all shared
    (s, b and R next to W; VeRA's d and e next to the shared A and B) stay live.
    The folds are exact algebra, so they are applied unconditionally.
    """
    terms = []
    for t in nf.terms:
        if t.shared:
            terms.append(replace(t))
            continue
        A = t.A * t.c
        if t.d is not None:
            A = A * t.d[None, :]
        B = t.B if t.e is None else t.B * t.e[None, :]
        terms.append(Term(A=A, B=B, d=None, e=None, c=1.0, shared=False))
    return NormalForm(R=nf.R, s=nf.s, b=nf.b, terms=terms)


def merged_weight(nf: NormalForm, W: np.ndarray) -> np.ndarray:
    """The per-adapter weight an engine would need without batching:
    ``W_a = R W diag(s) + sum_k c_k A_k diag(d_k) B_k diag(e_k)``, so that
    ``F_a(x) = x W_a + b`` (brute force, tiny inputs only)."""
    d_in, d_out = W.shape
    R = np.eye(d_in) if nf.R is None else nf.R
    s = np.ones(d_out) if nf.s is None else nf.s
    Wa = (R @ W) @ np.diag(s)
    for t in nf.terms:
        r = t.A.shape[1]
        d = np.ones(r) if t.d is None else t.d
        e = np.ones(d_out) if t.e is None else t.e
        Wa = Wa + t.c * (t.A @ np.diag(d) @ t.B @ np.diag(e))
    return Wa


def merged_apply(nf: NormalForm, x: np.ndarray, W: np.ndarray) -> np.ndarray:
    y = x @ merged_weight(nf, W)
    if nf.b is not None:
        y = y + nf.b
    return y


def definitional(method: str, x, W, p: dict) -> np.ndarray:
    """Dispatch to the method's own definition (``oracle.methods``)."""
    if method == "lora":
        return M.lora(x, W, p["A"], p["B"], p["c"])
    if method == "dora":
        return M.dora(x, W, p["A"], p["B"], p["c"], p["m"])
    if method == "ia3":
        return M.ia3(x, W, p["l"]) if "l" in p else M.base(x, W)
    if method == "vera":
        return M.vera(x, W, p["A_sh"], p["B_sh"], p["d"], p["e"]) if "d" in p else M.base(x, W)
    if method == "oft":
        return M.oft(x, W, p["R"]) if "R" in p else M.base(x, W)
    if method == "nf":
        return evaluate(from_method("nf", W, p), x, W)
    raise ValueError(method)
