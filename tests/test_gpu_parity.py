"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.  Indexing is compared bit for bit; floating point is
graded with the tolerances in ``metrics``."""
import copy

import numpy as np
import pytest

import workloads as WL
from oracle import batch as BT
from oracle import indexing as IX
import metrics as MX

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def scute(gpu_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gpu_lib


import gpu_harness as H  # noqa: E402


# ------------------------------------------------------------------ indexing
def _index_ctx(scute, A):
    """A context with adapters of every method registered under ids 0..A-3
    (ids A-2, A-1 stay free, so they are 'unregistered')."""
    ctx = scute.Context(dtype="bf16", max_tokens=16384, max_adapters=A, max_layers=1)
    W = WL.draw_normal(0, "Widx", (64, 64), 0.02, "bf16")
    ctx.add_layer(0, 64, 64, W)
    ctx.set_shared(0, 32, WL.draw_normal(0, "Ai", (64, 32), 0.02, "bf16"),
                   WL.draw_normal(0, "Bi", (32, 64), 0.02, "bf16"))
    methods = {}
    order = ["vera", "lora", "oft", "ia3", "dora", "nf"]
    for i in range(A - 2):
        m = order[(i * 7 + 3) % 6]
        t = {"layer": 0}
        if m == "lora" or m == "dora":
            t.update(rank=1, c=2.0, A=WL.draw_normal(i, "a", (64, 1), 0.02, "bf16"),
                     B=WL.draw_normal(i, "b", (1, 64), 0.02, "bf16"))
            if m == "dora":
                t["magnitude"] = np.ones(64, np.float32)
        elif m == "ia3":
            t["l"] = np.ones(64, np.float32)
        elif m == "vera":
            t["d"] = np.ones(32, np.float32)
        elif m == "oft":
            t["R"] = WL.draw_cayley_blocks(i, "r", 2, "bf16")
        else:
            t["s"] = np.ones(64, np.float32)
        aid = ctx.register(m, [t])
        assert aid == i
        methods[i] = m
    return ctx, methods


@pytest.mark.parametrize("n,A", [(1, 8), (7, 8), (64, 40), (300, 40), (2049, 1024), (8772, 40),
                                 (16384, 1024),
                                 # the sort's pass plans: keys below 6 A + 1 take one 8-bit pass up
                                 # to A = 42, one 9-bit pass up to A = 85 (512 threads from 2048
                                 # tokens down), two 8-bit passes beyond
                                 (700, 42), (300, 64), (2048, 85), (2049, 48), (8772, 48),
                                 (16384, 85), (2048, 86)])
def test_index_bit_exact(scute, n, A):
    ctx, methods = _index_ctx(scute, A)
    g = np.random.default_rng(n * 31 + A)
    ids = g.integers(-1, A, n).astype(np.int32)  # -1 and the unregistered A-2, A-1 included
    ids_t = torch.from_numpy(ids).cuda()
    perm = torch.empty(n, dtype=torch.int32, device="cuda")
    aid = torch.empty(n, dtype=torch.int32, device="cuda")
    seg_start = torch.full((n + 1,), -7, dtype=torch.int32, device="cuda")
    seg_aid = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    counts = torch.empty(22, dtype=torch.int32, device="cuda")
    ctx.debug_index(ids_t, n, perm, aid, seg_start, seg_aid, counts)
    torch.cuda.synchronize()
    ref = IX.index_tokens(ids, methods, A)
    c = counts.cpu().numpy()
    n_seg = int(c[0])
    np.testing.assert_array_equal(perm.cpu().numpy(), ref.perm)
    np.testing.assert_array_equal(aid.cpu().numpy(), ref.aid_sorted)
    assert n_seg == len(ref.seg_aid)
    np.testing.assert_array_equal(seg_start.cpu().numpy()[:n_seg + 1], ref.seg_start)
    np.testing.assert_array_equal(seg_aid.cpu().numpy()[:n_seg], ref.seg_aid)
    np.testing.assert_array_equal(c[1:8], ref.count)
    np.testing.assert_array_equal(c[8:15], ref.offset)
    seg_rank = np.zeros(7, np.int64)
    for a in ref.seg_aid:
        seg_rank[IX.METHOD_RANK[methods[int(a)]] if a >= 0 else IX.BASE_RANK] += 1
    np.testing.assert_array_equal(c[15:22], seg_rank)
    st = ctx.sync_status()
    assert st == (5 if ref.bad else 0)
    ctx.close()


# ------------------------------------------------------------------ small shapes, several tiles + ragged tails
SMALL_NAMES = ("q", "k", "up", "down")


def _small_decode(n=50):
    return WL.with_nf_adapters(WL.decode_mixed(n=n, shapes=WL.SMALL_PROJ, proj=SMALL_NAMES))


@pytest.mark.parametrize("n", [50, 128, 200])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_small_decode_parity(scute, out_dtype, n):
    """n <= 128: fused decode path (one prologue + one GEMM launch);
    128 < n <= 256: separate kernels, tokens on the tile's N side."""
    w = _small_decode(n)
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, SMALL_NAMES, out_dtype)
    assert ctx.sync_status() == 0
    for name in SMALL_NAMES:
        H.grade(w, name, outs[name], out_dtype)
    ctx.close()


def _batch_run(ctx, w, names, out_dtype, ids=None):
    """All layers in one scute_linear_batch call (one launch for n <= 128)."""
    ids_np = w.ids if ids is None else ids
    ids_t = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    calls, outs = [], []
    for name in names:
        L = w.layer(name)
        out = torch.full((w.n, L.d_out), float("nan"), device="cuda",
                         dtype=torch.float32 if out_dtype == "fp32" else torch.bfloat16)
        calls.append((H.dev(L.get("x")), ctx.layer_ids[name], out))
        outs.append(out)
    ctx.linear_batch(calls, ids_t, out_dtype)
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("n", [2, 50, 128, 200])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_small_decode_batch_parity(scute, out_dtype, n):
    """Every layer in one batched call; the same layer twice gets its own slot.
    n <= 128 runs as one persistent launch, n = 200 as consecutive calls."""
    w = _small_decode(n)
    ctx = H.make_ctx(scute, w)
    names = list(SMALL_NAMES) + ["q"]
    outs = _batch_run(ctx, w, names, out_dtype)
    assert ctx.sync_status() == 0
    for name, o in zip(names, outs):
        H.grade(w, name, o, out_dtype)
    # the two copies of q are split differently over the CTAs (other K ranges,
    # other summation order), so they agree to rounding, not bit for bit
    d = (outs[0].double() - outs[-1].double()).abs().max().item()
    assert d <= 2e-2
    ctx.close()


@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_separate_pass_variants(scute, variant, out_dtype):
    """The rotation (1) and DoRA's / (IA)^3's s (2) placed in launches of their
    own around the decode step: one extra launch each, results still the
    oracle's (the raw normal-form adapter with R and an owned term checks that
    the low-rank shrink keeps reading x, not the rotated copy)."""
    w = _small_decode(50)
    ctx = H.make_ctx(scute, w)
    ctx.set_variant(variant)
    names = list(SMALL_NAMES)
    n0 = ctx.launch_count()
    outs = _batch_run(ctx, w, names, out_dtype)
    assert ctx.launch_count() - n0 == 1 + (variant & 1) + (variant >> 1)
    assert ctx.sync_status() == 0
    for name, o in zip(names, outs):
        H.grade(w, name, o, out_dtype)
    ctx.close()


def _plan_check(ctx, w, names, n):
    """The library's recorded plan of its last decode launch equals the host
    restatement (tests/step_plan.py), whose range check then covers it."""
    import step_plan as SP
    from lora_normal_form_gb300 import scute_debug_step_plan
    rec = SP.parse(scute_debug_step_plan(ctx.handle))
    shapes = SP.layer_shapes(w, names)
    all_shapes = SP.layer_shapes(w, [L.name for L in w.layers if L.name in ctx.layer_ids])
    ws = SP.workspace(all_shapes, ctx.max_tokens, rec.head["grid"])
    mine = SP.plan(shapes, n, torch.cuda.get_device_properties(0).multi_processor_count, ws,
                   smem_optin=rec.head["smem_optin"])
    assert rec.head == mine.head
    assert rec.calls == [{key: k[key] for key in SP.CALL_KEYS} for k in mine.calls]
    assert rec.start == mine.start
    SP.audit(rec, SP.seg_lr_counts(w, names, w.ids[:n]))


def test_step_plan_matches_restatement(decode_full, scute):
    """The bench launch's plan (six Llama-3-8B projections, 64 tokens) and a
    small-shape batch with a repeated layer: recorded plan == restated plan,
    and every plan-derived index of the kernel in range."""
    w, ctx, _, _ = decode_full
    _batch_run(ctx, w, FULL, "bf16")
    assert ctx.sync_status() == 0
    _plan_check(ctx, w, list(FULL), w.n)
    ws = _small_decode(50)
    c2 = H.make_ctx(scute, ws)
    names = list(SMALL_NAMES) + ["q"]
    _batch_run(c2, ws, names, "bf16")
    assert c2.sync_status() == 0
    _plan_check(c2, ws, names, ws.n)
    c2.close()


def _without_rotation_on(w, layers):
    """The same workload with every R slot of the given layers removed: those
    layers then have no rotation adapter (an OFT adapter is the identity there)."""
    ads = []
    for a in w.adapters:
        b = copy.copy(a)
        b._gen = {k: g for k, g in a._gen.items() if not (k[1] == "R" and k[0] in layers)}
        b._cache = {}
        b.layers = tuple(name for name in a.layers if b.slots(name))
        ads.append(b)
    return WL.Workload(w.name + "_norot", w.dtype, w.n, w.ids, w.layers, ads, recipe=w.recipe)


@pytest.mark.parametrize("norot", [("k", "down"), tuple(SMALL_NAMES)])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_batch_layers_without_rotation(scute, norot, out_dtype):
    """A layer with no rotation adapter reads x itself as the token operand
    (no copy, no wait); in one batch with layers that do rotate, every call is
    still the oracle's."""
    w = _without_rotation_on(_small_decode(50), set(norot))
    ctx = H.make_ctx(scute, w)
    names = list(SMALL_NAMES)
    outs = _batch_run(ctx, w, names, out_dtype)
    assert ctx.sync_status() == 0
    for name, o in zip(names, outs):
        H.grade(w, name, o, out_dtype)
    ctx.close()


def test_batch_repeats_bit_for_bit(scute):
    """Partial tiles are summed in a fixed order, whichever CTA finishes a tile,
    so repeated calls give identical bits."""
    w = _small_decode(64)
    ctx = H.make_ctx(scute, w)
    first = _batch_run(ctx, w, SMALL_NAMES, "bf16")
    for _ in range(4):
        again = _batch_run(ctx, w, SMALL_NAMES, "bf16")
        for name, a, b in zip(SMALL_NAMES, first, again):
            assert torch.equal(a, b), name
    ctx.close()


FULL = ("q", "k", "v", "gate", "up", "down")


@pytest.fixture(scope="module")
def decode_full(scute):
    """The Llama-3-8B-shaped decode workload (64 tokens, q, k, v, gate, up,
    down, 32 adapters of all five methods) and the oracle's outputs for every
    row, computed once for both output types."""
    w = WL.decode_mixed()
    ctx = H.make_ctx(scute, w, layer_names=FULL)
    refs = {name: BT.linear(w, name) for name in FULL}
    bases = {name: BT.base_output(w, name) for name in FULL}
    yield w, ctx, refs, bases
    ctx.close()


@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_decode_full_shapes_all_rows(decode_full, out_dtype):
    """The bench's workload in one batched call, every row of every projection
    graded: LoRA, DoRA, (IA)^3, VeRA and OFT rows at d_in 4096 and 14336.
    bf16 output: max abs error 3e-2 (one bf16 spacing where rounding alone
    exceeds it) and the per-adapter effect error within 1% plus the oracle's
    own bf16-rounding floor; fp32 output: effect error <= 1% per adapter."""
    w, ctx, refs, bases = decode_full
    assert H.methods_in(w, range(w.n)) >= {"lora", "dora", "ia3", "vera", "oft"}
    outs = _batch_run(ctx, w, FULL, out_dtype)
    assert ctx.sync_status() == 0
    worst = {}
    for name, o in zip(FULL, outs):
        rep = H.grade(w, name, o, out_dtype, ref=refs[name], base=bases[name])
        for m, e in rep["effect_by_method"].items():
            worst[m] = max(worst.get(m, 0.0), e)
        # every method with an effect on this layer was graded
        present = {H.method_of(w, a) for a in rep["effect"]}
        expect = {"lora", "dora", "vera", "oft"} | ({"ia3"} if name in ("k", "v", "up") else set())
        assert present >= expect, (name, present)
    print(f"decode_mixed full size, {out_dtype} out: worst effect error per method "
          + ", ".join(f"{m} {e:.2e}" for m, e in sorted(worst.items())))


@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_small_prefill_parity(scute, out_dtype):
    """n > 256: tokens on the 128-row side of the tensor-core tile."""
    w = WL.with_nf_adapters(WL.prefill_mixed(n_req=6, lo=40, hi=200, shapes=WL.SMALL_PROJ, proj=SMALL_NAMES))
    assert w.n > 256
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, SMALL_NAMES, out_dtype)
    assert ctx.sync_status() == 0
    for name in SMALL_NAMES:
        H.grade(w, name, outs[name], out_dtype)
    ctx.close()


@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_prefill_more_tiles_than_sms(scute, out_dtype):
    """About 4000 tokens on the ragged small shapes: the q and up base GEMMs
    have more tiles than SMs (160 and 192 for 152), so persistent CTAs run a
    second, short wave; every row graded, with LoRA / DoRA terms on the
    tensor-core expand and NF adapters on the CUDA-core one."""
    w = WL.with_nf_adapters(WL.prefill_mixed(n_req=20, lo=150, hi=250, shapes=WL.SMALL_PROJ, proj=SMALL_NAMES))
    n = w.n
    for name in ("q", "up"):
        tiles = -(-n // 128) * -(-WL.SMALL_PROJ[name][1] // 256)
        assert tiles >= 152 and 0 < tiles % 152 <= 76, (name, tiles)
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, SMALL_NAMES, out_dtype)
    assert ctx.sync_status() == 0
    for name in SMALL_NAMES:
        H.grade(w, name, outs[name], out_dtype)
    ctx.close()


@pytest.mark.parametrize("rank", [1, 8, 24, 64])
@pytest.mark.parametrize("n", [200, 700])
def test_tensor_core_shrink_ranks(scute, rank, n):
    """Layers with no adapter that both rotates and owns a term run the owned
    shrink on the tensor cores (tiles of up to 128 sorted rows of one segment,
    A' boxes of the rank rounded up to 16 rows): ranks 1..64, segments shorter
    and longer than a tile, the ragged small shapes, both output types."""
    w = WL.prefill_mixed(n_req=max(2, n // 120), lo=20, hi=240, shapes=WL.SMALL_PROJ, proj=SMALL_NAMES,
                         rank=rank, req_adapters=list(range(max(2, n // 120))))
    assert w.n > 128
    assert all("R" not in a.slots(name) or a.method == "oft" for a in w.adapters for name in a.layers)
    ctx = H.make_ctx(scute, w)
    for out_dtype in ("bf16", "fp32"):
        outs = H.run_layers(ctx, w, SMALL_NAMES, out_dtype)
        assert ctx.sync_status() == 0
        for name in SMALL_NAMES:
            H.grade(w, name, outs[name], out_dtype)
    ctx.close()


@pytest.mark.parametrize("rv", [96, 1024])
def test_prefill_vera_shared_ranks(scute, rv):
    """Prefill-sized batches with VeRA tenants at shared rank 1024 (the largest:
    16 column tiles of the tensor-core VeRA shrink) and 96 (not a multiple of
    64: the GEMM path), both output types, ragged shapes."""
    w = WL.prefill_mixed(n_req=4, lo=60, hi=200, shapes=WL.SMALL_PROJ, proj=SMALL_NAMES, rv=rv,
                         req_adapters=[3, 8, 0, 13])   # three VeRA requests and a LoRA one
    assert w.n > 256 and H.methods_in(w, range(w.n)) >= {"vera", "lora"}
    ctx = H.make_ctx(scute, w)
    for out_dtype in ("bf16", "fp32"):
        outs = H.run_layers(ctx, w, SMALL_NAMES, out_dtype)
        assert ctx.sync_status() == 0
        for name in SMALL_NAMES:
            H.grade(w, name, outs[name], out_dtype)
    ctx.close()


def test_tiny_fp32(scute):
    """fp32 single linear, 16 tokens, one adapter per method: max rel <= 1e-4.
    Also prints the score under a 1e-3 rms(r) floor, the tighter choice of
    relative floor that was weighed against the 1e-2 one used here."""
    w = WL.tiny_fp32()
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, ["lin"], "fp32")
    assert ctx.sync_status() == 0
    rep = H.grade(w, "lin", outs["lin"], "fp32")
    assert rep["fp32_rel"] <= 1e-4
    g = H.to_f64(outs["lin"])
    r = BT.linear(w, "lin")
    print(f"tiny_fp32 max rel error: floor 1e-3 rms {MX.fp32_rel_err(g, r, 1e-3):.3e}, "
          f"floor 1e-2 rms {MX.fp32_rel_err(g, r, 1e-2):.3e}, "
          f"no floor near zero excluded: normwise {MX.normwise_err(g, r):.3e}")
    ctx.close()


@pytest.mark.parametrize("n", [1, 2, 17, 64, 65, 128, 129, 256, 257, 600])
def test_base_only_equals_xW(scute, n):
    """All ids -1: every slot is the identity and the output is x W (bf16
    inputs, float32 accumulation: normwise error at the float32 level)."""
    w = WL.decode_mixed(n=n, shapes=WL.SMALL_PROJ, proj=("q",), n_adapters=5,
                        ids=np.full(n, -1, np.int32))
    ctx = H.make_ctx(scute, w, max_tokens=max(n, 64))
    outs = H.run_layers(ctx, w, ["q"], "fp32")
    ref = BT.base_output(w, "q")
    g = H.to_f64(outs["q"])
    assert MX.normwise_err(g, ref) <= 1e-5
    ctx.close()


@pytest.mark.parametrize("method", ["lora", "dora", "ia3", "vera", "oft"])
def test_single_adapter_batch(scute, method):
    """Every token on one adapter (one segment), plus a one-token call."""
    k = WL.MOD5.index(method)
    n = 40
    w = WL.decode_mixed(n=n, shapes=WL.SMALL_PROJ, proj=SMALL_NAMES, n_adapters=5,
                        ids=np.full(n, k, np.int32))
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, SMALL_NAMES, "fp32")
    for name in SMALL_NAMES:
        H.grade(w, name, outs[name], "fp32")
    w1 = WL.decode_mixed(n=1, shapes=WL.SMALL_PROJ, proj=SMALL_NAMES, n_adapters=5,
                         ids=np.full(1, k, np.int32))
    ctx1 = H.make_ctx(scute, w1)
    outs1 = H.run_layers(ctx1, w1, SMALL_NAMES, "fp32")
    for name in SMALL_NAMES:
        H.grade(w1, name, outs1[name], "fp32")
    ctx.close()
    ctx1.close()


def test_rank1_and_rank64(scute):
    n = 48
    for rank in (1, 64):
        w = WL.decode_mixed(n=n, shapes=WL.SMALL_PROJ, proj=("q", "down"), n_adapters=4, rank=rank,
                            ids=np.random.default_rng(rank).integers(-1, 4, n).astype(np.int32))
        ctx = H.make_ctx(scute, w)
        outs = H.run_layers(ctx, w, ("q", "down"), "fp32")
        for name in ("q", "down"):
            H.grade(w, name, outs[name], "fp32")
        ctx.close()


@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_many_short_segments_rank64(scute, out_dtype):
    """200 tokens over 160 adapters with Zipf(1.0) ids, LoRA / DoRA rank 64:
    most segments hold one or two rows (the per-kernel plan's segmented
    low-rank kernels in their decode-like regime, and rank groups beyond 16)."""
    n = 200
    ids = WL.zipf_ids(5, n, 160)
    w = WL.decode_mixed(n=n, shapes=WL.SMALL_PROJ, proj=("q", "down"), n_adapters=160, rank=64, ids=ids)
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, ("q", "down"), out_dtype)
    assert ctx.sync_status() == 0
    for name in ("q", "down"):
        H.grade(w, name, outs[name], out_dtype)
    ctx.close()


def test_bad_ids_become_base_and_are_reported(scute):
    w = _small_decode(n=32)
    ids = w.ids.copy()
    ids[3] = 999
    ids[7] = -5
    ctx = H.make_ctx(scute, w, max_adapters=1024)
    outs = H.run_layers(ctx, w, ["q"], "fp32", ids=ids)
    assert ctx.sync_status() == 5  # SCUTE_ERR_BAD_ADAPTER
    assert ctx.sync_status() == 0  # cleared by the read
    ref = BT.base_output(w, "q", rows=[3, 7])
    g = H.to_f64(outs["q"][[3, 7]])
    assert MX.normwise_err(g, ref) <= 1e-5
    ctx.close()


def test_n_zero_is_a_no_op(scute):
    w = _small_decode(n=8)
    ctx = H.make_ctx(scute, w)
    before = ctx.launch_count()
    out = torch.empty(0, 1056, device="cuda", dtype=torch.bfloat16)
    x = torch.empty(0, 544, device="cuda", dtype=torch.bfloat16)
    ids = torch.empty(0, device="cuda", dtype=torch.int32)
    ctx.linear(x, ids, ctx.layer_ids["q"], out, "bf16", n=0)
    assert ctx.launch_count() == before
    ctx.close()


@pytest.mark.parametrize("pinned_out", [True, False])
def test_linear_host_matches_linear(scute, pinned_out):
    """scute_linear_host on a decode batch: a pinned output buffer is stored
    into by the step directly, a pageable one copied back; both equal the
    device-buffer call bit for bit."""
    w = _small_decode(n=24)
    ctx = H.make_ctx(scute, w)
    outs = H.run_layers(ctx, w, ["up"], "bf16")
    L = w.layer("up")
    x_host = torch.from_numpy(L.get("x").view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_host = torch.from_numpy(w.ids.copy()).pin_memory()
    out_host = torch.empty(w.n, L.d_out, dtype=torch.bfloat16)
    if pinned_out:
        out_host = out_host.pin_memory()
    ctx.linear_host(x_host, ids_host, ctx.layer_ids["up"], out_host, "bf16",
                    stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.equal(out_host, outs["up"].cpu())
    ctx.close()


@pytest.mark.parametrize("pinned", [True, "unaligned_out", False])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_linear_batch_host_matches_linear_batch(scute, pinned, out_dtype):
    """scute_linear_batch_host over several layers: pinned host buffers go
    through one gather launch before the step, which then stores the outputs
    straight into the (16-byte-aligned) pinned output buffers; pinned outputs
    that are not 16-byte aligned through one scatter launch after the step;
    pageable buffers through a copy each.  All equal the device-buffer call
    bit for bit."""
    w = _small_decode(n=40)
    names = list(SMALL_NAMES)
    ctx = H.make_ctx(scute, w)
    dt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    ids_dev = torch.from_numpy(w.ids.copy()).cuda()
    xs, outs_dev, calls_h = {}, {}, []
    for name in names:
        L = w.layer(name)
        xs[name] = torch.from_numpy(L.get("x").view(np.int16)).view(torch.bfloat16)
        outs_dev[name] = torch.empty(w.n, L.d_out, dtype=dt, device="cuda")
    ctx.linear_batch([(xs[nm].cuda(), ctx.layer_ids[nm], outs_dev[nm]) for nm in names], ids_dev, out_dtype)
    torch.cuda.synchronize()
    ids_h = torch.from_numpy(w.ids.copy())
    outs_h = {nm: torch.empty(w.n, w.layer(nm).d_out, dtype=dt) for nm in names}
    if pinned:
        ids_h = ids_h.pin_memory()
        xs = {nm: t.pin_memory() for nm, t in xs.items()}
        outs_h = {nm: t.pin_memory() for nm, t in outs_h.items()}
    if pinned == "unaligned_out":
        # each output one element into a pinned buffer of its own
        for nm in names:
            d = w.layer(nm).d_out
            big = torch.empty(w.n * d + 8, dtype=dt).pin_memory()
            outs_h[nm] = big[1:1 + w.n * d].view(w.n, d)
            assert outs_h[nm].data_ptr() % 16 != 0
    n0 = ctx.launch_count()
    ctx.linear_batch_host([(xs[nm], ctx.layer_ids[nm], outs_h[nm]) for nm in names], ids_h, out_dtype,
                          stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    # the step; pinned: plus the gather, and the scatter for unaligned outputs
    assert ctx.launch_count() - n0 == {True: 2, "unaligned_out": 3, False: 1}[pinned]
    assert ctx.sync_status() == 0
    for nm in names:
        assert torch.equal(outs_h[nm], outs_dev[nm].cpu()), nm
    ctx.close()


def test_linear_batch_host_s_pass_keeps_staged_outputs(scute):
    """With DoRA's / (IA)^3's s in a launch of its own (which reads out back),
    pinned outputs are not the step's out pointers: the batch is gather, step,
    s pass and scatter, and its outputs equal the device-buffer call with the
    same placement bit for bit."""
    w = _small_decode(n=40)
    names = list(SMALL_NAMES)
    ctx = H.make_ctx(scute, w)
    ctx.set_variant(2)
    ids_dev = torch.from_numpy(w.ids.copy()).cuda()
    xs = {nm: torch.from_numpy(w.layer(nm).get("x").view(np.int16)).view(torch.bfloat16) for nm in names}
    outs_dev = {nm: torch.empty(w.n, w.layer(nm).d_out, dtype=torch.bfloat16, device="cuda") for nm in names}
    ctx.linear_batch([(xs[nm].cuda(), ctx.layer_ids[nm], outs_dev[nm]) for nm in names], ids_dev, "bf16")
    torch.cuda.synchronize()
    ids_h = torch.from_numpy(w.ids.copy()).pin_memory()
    xs_h = {nm: t.pin_memory() for nm, t in xs.items()}
    outs_h = {nm: torch.empty(w.n, w.layer(nm).d_out, dtype=torch.bfloat16).pin_memory() for nm in names}
    n0 = ctx.launch_count()
    ctx.linear_batch_host([(xs_h[nm], ctx.layer_ids[nm], outs_h[nm]) for nm in names], ids_h, "bf16",
                          stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert ctx.launch_count() - n0 == 4
    assert ctx.sync_status() == 0
    for nm in names:
        assert torch.equal(outs_h[nm], outs_dev[nm].cpu()), nm
    ctx.close()


def test_cuda_graph_replay_matches_eager(scute):
    w = _small_decode(n=40)
    ctx = H.make_ctx(scute, w)
    eager = H.run_layers(ctx, w, SMALL_NAMES, "bf16")
    ids_t = torch.from_numpy(w.ids.copy()).cuda()
    xs = {n: H.dev(w.layer(n).get("x")) for n in SMALL_NAMES}
    outs = {n: torch.zeros(w.n, w.layer(n).d_out, device="cuda", dtype=torch.bfloat16) for n in SMALL_NAMES}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for n in SMALL_NAMES:
                ctx.linear(xs[n], ids_t, ctx.layer_ids[n], outs[n], "bf16", stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for n in SMALL_NAMES:
        assert torch.equal(outs[n], eager[n]), n
    ctx.close()
