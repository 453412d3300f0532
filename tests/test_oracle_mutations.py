"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutation swaps one oracle function for a plausible wrong variant (a
dropped term, a transposed operand, a wrong norm axis, a wrong slot order) and
runs the pins of ``test_oracle_pins``; the test passes when some pin fails.
"""
import numpy as np
import pytest

from oracle import methods as M
from oracle import normal_form as NF
from oracle import indexing as IX
import test_oracle_pins as P


def _wrong_dora(x, W, A, B, c, m):
    Wp = W + c * (A @ B)
    n = np.sqrt(np.sum(Wp * Wp, axis=1))           # row norms instead of column norms
    return x @ (Wp * (m / n[: Wp.shape[1]])[None, :])


def _wrong_dora_scale(W, A, B, c, m):
    Wp = W + (A @ B)                                 # dropped c
    return m / np.sqrt(np.sum(Wp * Wp, axis=0))


def _wrong_oft(x, W, R):
    return (x @ M.block_diag(R).T) @ W              # transposed rotation


def _wrong_vera(x, W, A, B, d, e):
    return x @ W + (((x @ A)) @ B) * e               # dropped d


def _wrong_lora(x, W, A, B, c):
    return x @ (W + A @ B)                           # dropped c


def _wrong_evaluate(nf, x, W):
    xr = x if nf.R is None else x @ nf.R
    y = xr @ W
    if nf.s is not None:
        y = y * nf.s
    for t in nf.terms:                               # b dropped, e applied before B
        u = x @ t.A
        if t.d is not None:
            u = u * t.d
        y = y + t.c * (u @ t.B)
    return y


def _wrong_fold(nf):
    terms = []
    for t in nf.terms:
        if t.shared:
            terms.append(t)
            continue
        terms.append(NF.Term(A=t.A, B=t.B, c=1.0))     # forgets to fold c, d, e
    return NF.NormalForm(R=nf.R, s=nf.s, b=nf.b, terms=terms)


def _run_all_pins():
    failures = 0
    for case in P._load_golden():
        try:
            P.test_hand_examples_definitional_and_normal_form(case)
        except Exception:
            failures += 1
    checks = [
        lambda: [P.test_definitional_equals_normal_form(m, s) for m in
                 ["lora", "dora", "ia3", "vera", "oft", "nf"] for s in (0, 1)],
        lambda: [P.test_fold_equivalence(m, c) for m in ["lora", "dora", "nf"] for c in (0.5, 2.0)],
        P.test_fold_keeps_live_slots,
        P.test_special_cases_reduce_to_base,
        P.test_oft_rotation_is_orthogonal_and_norm_preserving,
        P.test_dora_column_norm_invariant,
        lambda: [P.test_merged_weight_brute_force(m) for m in ["lora", "dora", "ia3", "vera", "oft", "nf"]],
        P.test_lora_effect_linear_in_c_and_vera_effect_linear_in_d,
        lambda: [P.test_indexing_brute_force(s) for s in range(6)],
        P.test_indexing_edge_cases,
    ]
    for c in checks:
        try:
            c()
        except Exception:
            failures += 1
    return failures


MUTATIONS = {
    "dora_row_norm": (M, "dora", _wrong_dora),
    "dora_scale_drops_c": (M, "dora_scale", _wrong_dora_scale),
    "oft_transposed": (M, "oft", _wrong_oft),
    "vera_drops_d": (M, "vera", _wrong_vera),
    "lora_drops_c": (M, "lora", _wrong_lora),
    "normal_form_drops_b_and_e": (NF, "evaluate", _wrong_evaluate),
    "fold_forgets_slots": (NF, "fold", _wrong_fold),
}


def test_unmutated_oracle_passes_every_pin():
    assert _run_all_pins() == 0


@pytest.mark.parametrize("name", sorted(MUTATIONS) + ["block_diag_reversed", "index_reversed"])
def test_planted_mistake_is_caught(name, monkeypatch):
    if name == "block_diag_reversed":
        orig = M.block_diag
        monkeypatch.setattr(M, "block_diag", lambda b, _o=orig: _o(b[::-1]))
    elif name == "index_reversed":
        orig = IX.index_tokens

        def bad(ids, mo, A, _o=orig):
            ix = _o(ids, mo, A)
            ix.perm = ix.perm[::-1].copy()
            return ix
        monkeypatch.setattr(IX, "index_tokens", bad)
    else:
        mod, attr, fn = MUTATIONS[name]
        monkeypatch.setattr(mod, attr, fn)
    assert _run_all_pins() > 0
