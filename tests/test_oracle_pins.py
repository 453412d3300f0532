"""Pins of the float64 oracle to things other than itself (CPU only).

Each test checks the oracle against hand-derived worked examples, closed
forms, invariants, special cases that reduce to a library routine, or brute
force, so that a dropped term, a wrong sign or index, or a transposed operand
anywhere in ``oracle/`` fails at least one of them.  Citations name sections
of the article "Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA"
(paper-daily.com).
"""
import itertools
import json
import os

import numpy as np
import pytest

import workloads as WL
from oracle import methods as M
from oracle import normal_form as NF
from oracle import indexing as IX
from oracle import batch as BT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _load_golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    out = []
    for ex in g["examples"]:
        W = g[ex["W"]] if isinstance(ex["W"], str) else ex["W"]
        p = {}
        for k, v in ex.get("params", {}).items():
            p[k] = v if k == "c" else np.array(v, dtype=np.float64)
        out.append((ex, np.array(ex["x"], dtype=np.float64)[None, :], np.array(W, dtype=np.float64), p))
    return out


@pytest.mark.parametrize("case", _load_golden(), ids=lambda c: c[0]["name"])
def test_hand_examples_definitional_and_normal_form(case):
    """Worked examples (tests/golden/hand_examples.json): the definitional form,
    the unfolded and folded normal form and the merged weight all give the
    hand-derived output exactly (dyadic arithmetic, so float64 is exact)."""
    ex, x, W, p = case
    y = np.array(ex["y"], dtype=np.float64)[None, :]
    m = ex["method"]
    if m == "base":
        np.testing.assert_array_equal(M.base(x, W), y)
        return
    if m != "dora":  # DoRA's norms are exact here too, but go through sqrt
        np.testing.assert_array_equal(NF.definitional(m, x, W, p), y)
    np.testing.assert_allclose(NF.definitional(m, x, W, p), y, rtol=0, atol=1e-14)
    nf = NF.from_method(m, W, p)
    np.testing.assert_allclose(NF.evaluate(nf, x, W), y, rtol=0, atol=1e-14)
    np.testing.assert_allclose(NF.evaluate(NF.fold(nf), x, W), y, rtol=0, atol=1e-14)
    np.testing.assert_allclose(NF.merged_apply(nf, x, W), y, rtol=0, atol=1e-14)
    if "s" in ex:
        np.testing.assert_allclose(nf.s, ex["s"], rtol=0, atol=1e-15)
    if "merged_weight" in ex:
        np.testing.assert_array_equal(NF.merged_weight(nf, W), np.array(ex["merged_weight"], float))


def _rand_case(seed, d_in=64, d_out=48, n=5, r=4, rv=8, blk=8):
    g = np.random.default_rng(seed)
    W = g.normal(0, 0.5, (d_in, d_out))
    x = g.normal(0, 1, (n, d_in))
    S = np.triu(g.normal(0, 0.3, (d_in // blk, blk, blk)), 1)
    S = S - np.transpose(S, (0, 2, 1))
    I = np.eye(blk)[None]
    Rb = np.matmul(I + S, np.linalg.inv(I - S))
    P = {
        "lora": {"A": g.normal(0, 0.5, (d_in, r)), "B": g.normal(0, 0.5, (r, d_out)), "c": 2.0},
        "dora": {"A": g.normal(0, 0.5, (d_in, r)), "B": g.normal(0, 0.5, (r, d_out)), "c": 0.5,
                 "m": np.abs(g.normal(3, 1, d_out)) + 0.1},
        "ia3": {"l": 1 + 0.3 * g.normal(size=d_out)},
        "vera": {"A_sh": g.normal(0, 0.5, (d_in, rv)), "B_sh": g.normal(0, 0.5, (rv, d_out)),
                 "d": 1 + 0.3 * g.normal(size=rv), "e": 1 + 0.3 * g.normal(size=d_out)},
        "oft": {"R": Rb},
        "nf": {"R": Rb, "s": 1 + 0.3 * g.normal(size=d_out), "b": g.normal(size=d_out),
               "A": g.normal(0, 0.5, (d_in, r)), "B": g.normal(0, 0.5, (r, d_out)),
               "d": 1 + 0.3 * g.normal(size=r), "e": 1 + 0.3 * g.normal(size=d_out), "c": 0.5},
    }
    return x, W, P


def _rel(a, b):
    return np.max(np.abs(a - b)) / np.max(np.abs(b))


@pytest.mark.parametrize("method", ["lora", "dora", "ia3", "vera", "oft", "nf"])
@pytest.mark.parametrize("seed", [0, 1])
def test_definitional_equals_normal_form(method, seed):
    """Each method from its own definition equals its normal form (article,
    "The big picture": every method written in one formula)."""
    x, W, P = _rand_case(seed)
    y_def = NF.definitional(method, x, W, P[method])
    y_nf = NF.evaluate(NF.from_method(method, W, P[method]), x, W)
    assert _rel(y_nf, y_def) <= 1e-12


@pytest.mark.parametrize("method", ["lora", "dora", "nf"])
@pytest.mark.parametrize("c", [0.5, 2.0, 0.3])
def test_fold_equivalence(method, c):
    """Folding owned slots at load (c and d into A, e into B) leaves the output
    unchanged (article, "Which slots can be merged at load?": (xA)*d = x(A diag d))."""
    x, W, P = _rand_case(7)
    p = dict(P[method])
    p["c"] = c
    nf = NF.from_method(method, W, p)
    fo = NF.fold(nf)
    assert all(t.d is None and t.e is None and t.c == 1.0 for t in fo.terms if not t.shared)
    assert _rel(NF.evaluate(fo, x, W), NF.evaluate(nf, x, W)) <= 1e-12


def test_fold_keeps_live_slots():
    """Slots next to shared tensors stay live after the fold: DoRA's s, VeRA's
    d and e, OFT's R (article, "Which slots can be merged at load?")."""
    x, W, P = _rand_case(3)
    fd = NF.fold(NF.from_method("dora", W, P["dora"]))
    assert fd.s is not None and fd.terms[0].e is None
    fv = NF.fold(NF.from_method("vera", W, P["vera"]))
    assert fv.terms[0].shared and fv.terms[0].d is not None and fv.terms[0].e is not None
    np.testing.assert_array_equal(fv.terms[0].A, P["vera"]["A_sh"])
    fo = NF.fold(NF.from_method("oft", W, P["oft"]))
    assert fo.R is not None


def test_identity_slots_reduce_to_xW_exactly():
    """All slots at identity give exactly x @ W (bit-equal): the library
    special case (article, "The big picture": unused slots hold the identity)."""
    x, W, _ = _rand_case(11)
    nf = NF.NormalForm()
    np.testing.assert_array_equal(NF.evaluate(nf, x, W), x @ W)
    # and explicit identity values give xW to rounding
    nf2 = NF.NormalForm(R=np.eye(W.shape[0]), s=np.ones(W.shape[1]), b=np.zeros(W.shape[1]),
                        terms=[NF.Term(A=np.zeros((W.shape[0], 3)), B=np.ones((3, W.shape[1])))])
    np.testing.assert_allclose(NF.evaluate(nf2, x, W), x @ W, rtol=1e-13, atol=1e-13)


def test_special_cases_reduce_to_base():
    """LoRA with B = 0, VeRA with d = 0, (IA)^3 with l = 1 and OFT with
    Cayley(0) = I each equal x @ W."""
    x, W, P = _rand_case(5)
    p = dict(P["lora"]); p["B"] = np.zeros_like(p["B"])
    np.testing.assert_allclose(M.lora(x, W, p["A"], p["B"], p["c"]), x @ W, rtol=0, atol=1e-13)
    p = dict(P["vera"]); p["d"] = np.zeros_like(p["d"])
    np.testing.assert_allclose(M.vera(x, W, p["A_sh"], p["B_sh"], p["d"], p["e"]), x @ W, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(M.ia3(x, W, np.ones(W.shape[1])), x @ W)
    blocks = np.broadcast_to(np.eye(8), (W.shape[0] // 8, 8, 8)).copy()
    np.testing.assert_allclose(M.oft(x, W, blocks), x @ W, rtol=0, atol=1e-13)
    # the generator's Cayley transform with std 0 is exactly I
    R0 = WL.draw_cayley_blocks(0, "zero", 4, "fp32", std=0.0)
    np.testing.assert_array_equal(R0, np.broadcast_to(np.eye(32, dtype=np.float32), (4, 32, 32)))


def test_oft_rotation_is_orthogonal_and_norm_preserving():
    """Cayley blocks are orthogonal (closed form: (I+S)(I-S)^-1 with S skew),
    so xR keeps every row's norm (article, "What problem is it solving?":
    OFT multiplies the input by a rotation)."""
    x, W, P = _rand_case(9)
    R = M.block_diag(P["oft"]["R"])
    assert np.max(np.abs(R.T @ R - np.eye(R.shape[0]))) <= 1e-12
    np.testing.assert_allclose(np.linalg.norm(x @ R, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)


def test_dora_column_norm_invariant():
    """After DoRA every column of the effective weight W' diag(s) has length
    m exactly (closed form of the column renormalisation; article, "What
    problem is it solving?")."""
    x, W, P = _rand_case(13, d_in=40, d_out=24)
    p = P["dora"]
    Wp = W + p["c"] * (p["A"] @ p["B"])
    s = M.dora_scale(W, p["A"], p["B"], p["c"], p["m"])
    np.testing.assert_allclose(np.linalg.norm(Wp * s[None, :], axis=0), p["m"], rtol=1e-12)
    # the norm is per output column (over d_in), not per row
    assert s.shape == (W.shape[1],)


@pytest.mark.parametrize("method", ["lora", "dora", "ia3", "vera", "oft", "nf"])
def test_merged_weight_brute_force(method):
    """The explicitly merged per-adapter weight W_a (tiny) gives the same
    output as the normal form (article, "What problem is it solving?": merging
    each tenant into its own copy of the model is exact)."""
    x, W, P = _rand_case(17, d_in=16, d_out=12, n=3, r=2, rv=4, blk=4)
    nf = NF.from_method(method, W, P[method])
    # brute force: element by element with explicit loops
    Wa = NF.merged_weight(nf, W)
    y = np.zeros((x.shape[0], W.shape[1]))
    for t in range(x.shape[0]):
        for j in range(W.shape[1]):
            y[t, j] = sum(x[t, k] * Wa[k, j] for k in range(W.shape[0]))
            if nf.b is not None:
                y[t, j] += nf.b[j]
    assert _rel(NF.evaluate(nf, x, W), y) <= 1e-12


def test_lora_effect_linear_in_c_and_vera_effect_linear_in_d():
    x, W, P = _rand_case(19)
    p = dict(P["lora"])
    e1 = M.lora(x, W, p["A"], p["B"], 1.0) - x @ W
    e3 = M.lora(x, W, p["A"], p["B"], 3.0) - x @ W
    np.testing.assert_allclose(e3, 3 * e1, rtol=1e-11, atol=1e-12)
    q = dict(P["vera"])
    v1 = M.vera(x, W, q["A_sh"], q["B_sh"], q["d"], q["e"]) - x @ W
    v2 = M.vera(x, W, q["A_sh"], q["B_sh"], 2 * q["d"], q["e"]) - x @ W
    np.testing.assert_allclose(v2, 2 * v1, rtol=1e-11, atol=1e-12)


def test_ia3_ffn_reorder():
    """act(xWg) * (xWu) * l = act(xWg) * ((xWu) * l): l becomes the s slot of
    the up projection (article, "The big picture")."""
    g = np.random.default_rng(23)
    x = g.normal(size=(4, 16)); Wg = g.normal(size=(16, 24)); Wu = g.normal(size=(16, 24))
    l = 1 + 0.3 * g.normal(size=24)
    np.testing.assert_allclose(M.ia3_ffn(x, Wg, Wu, l), M.ia3_ffn_reordered(x, Wg, Wu, l),
                               rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(M.ia3_ffn_reordered(x, Wg, Wu, l),
                               M.silu(x @ Wg) * M.ia3(x, Wu, l), rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- indexing
def _brute_force_index(ids, method_of, A):
    """The unique permutation (over all n! of them) that makes keys
    non-decreasing and keeps equal keys in token order."""
    key, valid, bad = IX.sort_keys(ids, method_of, A)
    n = len(ids)
    found = []
    for p in itertools.permutations(range(n)):
        ks = [key[i] for i in p]
        if all(ks[i] <= ks[i + 1] for i in range(n - 1)) and \
           all(p[i] < p[i + 1] for i in range(n - 1) if ks[i] == ks[i + 1]):
            found.append(p)
    assert len(found) == 1
    return np.array(found[0]), bad


@pytest.mark.parametrize("seed", range(6))
def test_indexing_brute_force(seed):
    g = np.random.default_rng(seed)
    A = 6
    method_of = {0: "lora", 1: "vera", 2: "dora", 3: "oft", 4: "ia3"}  # 5 registered
    n = int(g.integers(1, 8))
    ids = g.integers(-1, A, n).astype(np.int32)  # includes -1 and the unregistered id 5
    ix = IX.index_tokens(ids, method_of, A)
    perm, bad = _brute_force_index(ids, method_of, A)
    np.testing.assert_array_equal(ix.perm, perm)
    assert ix.bad == bad == bool(np.any(ids == 5))
    # segments are maximal runs of one adapter; counts per method add up
    assert ix.seg_start[0] == 0 and ix.seg_start[-1] == n
    for s in range(len(ix.seg_aid)):
        run = ix.aid_sorted[ix.seg_start[s]:ix.seg_start[s + 1]]
        assert np.all(run == ix.seg_aid[s])
    assert all(ix.seg_aid[s] != ix.seg_aid[s + 1] for s in range(len(ix.seg_aid) - 1))
    assert ix.count.sum() == n and ix.count[IX.BASE_RANK] == np.sum(ix.aid_sorted == -1)


def test_indexing_edge_cases():
    mo = {0: "lora", 1: "vera"}
    ix = IX.index_tokens(np.zeros(0, np.int32), mo, 4)
    assert ix.perm.size == 0 and list(ix.seg_start) == [0] and ix.seg_aid.size == 0
    ix = IX.index_tokens(np.full(5, -1, np.int32), mo, 4)
    assert list(ix.perm) == [0, 1, 2, 3, 4] and list(ix.seg_aid) == [-1] and not ix.bad
    ix = IX.index_tokens(np.array([1, 0, 1, 0, 9, -7], np.int32), mo, 4)
    assert ix.bad and list(ix.perm) == [1, 3, 0, 2, 4, 5]
    assert list(ix.seg_aid) == [0, 1, -1] and list(ix.count) == [2, 0, 0, 2, 0, 0, 2]


# ---------------------------------------------------------------- batch
def test_batch_forms_agree_and_match_per_token_loop():
    """The batch evaluator's four forms agree, and equal a per-token loop over
    the methods' definitions (pure-Python loop, small case)."""
    w = WL.with_nf_adapters(WL.tiny_fp32())
    ref = BT.linear(w, "lin", form="definitional")
    for f in ("normal", "folded", "merged"):
        assert _rel(BT.linear(w, "lin", form=f), ref) <= 1e-12
    L = w.layer("lin")
    X = WL.to_f64(L.get("x")); W = WL.to_f64(L.get("W"))
    for t in range(w.n):
        a = int(w.ids[t])
        if a < 0:
            y = X[t:t + 1] @ W
        else:
            y = NF.definitional(w.adapter(a).method, X[t:t + 1], W, BT.adapter_params(w, a, L))
        np.testing.assert_allclose(ref[t], y[0], rtol=1e-13, atol=1e-13)


def test_batch_rows_subset():
    w = WL.tiny_fp32()
    full = BT.linear(w, "lin")
    rows = [3, 0, 15, 7]
    # BLAS may block a different row count differently: equal to rounding
    np.testing.assert_allclose(BT.linear(w, "lin", rows=rows), full[rows], rtol=1e-13, atol=1e-14)


def test_bf16_storage_roundtrip():
    """Storage helper: bf16 round-to-nearest-even of representative values."""
    v = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-3, 65504.0], dtype=np.float32)
    b = WL.bf16_values(WL.bf16_bits(v))
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0); 1 + 1.5*2^-8 rounds up
    np.testing.assert_array_equal(b[:3], np.array([1.0, 1.0, 1.0078125], np.float32))
    assert b[3] == -2.5
    assert abs(b[4] - 3.0e-3) <= 3.0e-3 * 2 ** -8
