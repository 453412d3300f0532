"""C-ABI library checks that need no GPU: it loads, exports every declared
symbol, reports missing devices as an error, and its host byte model equals
the oracle's restatement bit for bit."""
import json
import os
import re

import numpy as np
import pytest

import workloads as WL
from oracle import byte_model as OBM

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "scute.h")


@pytest.fixture(scope="module")
def lib():
    import lora_normal_form_gb300 as scute
    if not os.path.exists(scute.LIB_PATH):
        from lora_normal_form_gb300 import build as B
        B.build()
    return scute


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(scute_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    fns = _declared_functions()
    for must in ("scute_create", "scute_register_adapter", "scute_linear", "scute_sync_status",
                 "scute_byte_model", "scute_predict_bytes", "scute_linear_host", "scute_debug_index"):
        assert must in fns


def test_library_exports_every_declared_symbol(lib):
    cdll = lib.load()
    missing = [f for f in _declared_functions() if not hasattr(cdll, f)]
    assert not missing, missing
    assert lib.scute_version() == 10000


def test_create_without_device_is_an_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(lib.ScuteError) as e:
        lib.scute_create(0, lib.BF16, 64, 4, 1)
    assert e.value.code == 9  # SCUTE_ERR_NO_DEVICE


def test_create_argument_errors(lib):
    for args in [(0, 7, 64, 4, 1), (0, 0, 0, 4, 1), (0, 0, 64, 0, 1), (0, 0, 1 << 20, 4, 1)]:
        with pytest.raises(lib.ScuteError) as e:
            lib.scute_create(*args)
        assert e.value.code in (1, 3)


def _bm_inputs(w, layer_name, out_dtype):
    L = w.layer(layer_name)
    ads = {}
    for a in w.adapters:
        ads[a.id] = OBM.adapter_slots_after_fold(a.method, a.slots(layer_name), a.rank)
    lowrank = any(v["rank"] > 0 for v in ads.values())
    vera = L.shared_rank > 0 and any(v["vera"] for v in ads.values())
    return L, ads, lowrank, vera


def _c_report(lib, w, L, ads, lowrank, vera, ids, out_dtype, max_adapters):
    import ctypes
    arr = (lib.BmAdapter * max_adapters)()
    for i in range(max_adapters):
        arr[i].method = -1
    for aid, v in ads.items():
        arr[aid].method = lib.METHOD_ID[v["method"]]
        arr[aid].rank = v["rank"]
        arr[aid].has_s, arr[aid].has_b, arr[aid].has_R = int(v["s"]), int(v["b"]), int(v["R"])
        arr[aid].has_vera, arr[aid].has_vera_e = int(v["vera"]), int(v["vera_e"])
    bl = lib.BmLayer(dtype=lib.FP32 if w.dtype == "fp32" else lib.BF16,
                     out_dtype=lib.FP32 if out_dtype == "fp32" else lib.BF16,
                     d_in=L.d_in, d_out=L.d_out, shared_rank=L.shared_rank,
                     lowrank_launched=int(lowrank), vera_launched=int(vera), max_adapters=max_adapters,
                     adapters=ctypes.cast(arr, ctypes.POINTER(lib.BmAdapter)))
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    return lib.scute_byte_model(bl, ids, int(ids.size))


CASES = [
    ("tiny_fp32", lambda: WL.tiny_fp32(), "lin", "fp32"),
    ("decode_small_q", lambda: WL.decode_mixed(n=50, shapes=WL.SMALL_PROJ, proj=("q", "k", "up", "down")), "q", "bf16"),
    ("decode_small_up_fp32out", lambda: WL.decode_mixed(n=50, shapes=WL.SMALL_PROJ, proj=("q", "k", "up", "down")), "up", "fp32"),
    ("decode_small_nf", lambda: WL.with_nf_adapters(WL.decode_mixed(n=50, shapes=WL.SMALL_PROJ, proj=("q", "down"))), "down", "bf16"),
    ("decode_llama_k", lambda: WL.decode_mixed(), "k", "bf16"),
    ("scaling", lambda: WL.scaling_ia3_vera(), "up", "bf16"),
    ("prefill_small_fused_expand", lambda: WL.prefill_mixed(n_req=6, lo=40, hi=200, shapes=WL.SMALL_PROJ,
                                                            proj=("q", "k", "up", "down")), "up", "bf16"),
    ("prefill_small_rank64", lambda: WL.prefill_mixed(n_req=6, lo=40, hi=200, rank=64, shapes=WL.SMALL_PROJ,
                                                      proj=("q", "k", "up", "down")), "q", "fp32"),
]


@pytest.mark.parametrize("name,make,layer,out_dtype", CASES, ids=[c[0] for c in CASES])
def test_byte_model_matches_oracle(lib, name, make, layer, out_dtype):
    w = make()
    L, ads, lowrank, vera = _bm_inputs(w, layer, out_dtype)
    A = max(ads) + 3
    ids = w.ids.copy()
    if ids.size > 4:
        ids[1] = -1
        ids[2] = A - 1   # unregistered id: a base-only token
    got = _c_report(lib, w, L, ads, lowrank, vera, ids, out_dtype, A)
    ref = OBM.call_bytes(ids, ads, L.d_in, L.d_out, L.shared_rank, w.dtype, out_dtype, lowrank, vera)
    assert got["kernels"] == [tuple(k) for k in ref["kernels"]]
    for k in ("algorithmic_bytes", "adapter_bytes", "base_weight_bytes", "distinct_adapters"):
        assert got[k] == ref[k], k


@pytest.mark.parametrize("case", [0, 1])
def test_byte_model_hand_example(lib, case):
    """Hand-counted bytes (tests/golden/byte_model_hand.json), both launch plans."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "byte_model_hand.json")))
    ads = {int(k): v for k, v in g["adapters"].items()}
    c = g["cases"][case]
    ref = OBM.call_bytes(g["ids"], ads, c["d_in"], c["d_out"], c["shared_rank"], c["dtype"], c["out_dtype"],
                         c["lowrank_launched"], c["vera_launched"])
    exp = c["expected"]
    assert [list(k) for k in ref["kernels"]] == exp["kernels"]
    assert ref["algorithmic_bytes"] == exp["algorithmic_bytes"]
    assert ref["adapter_bytes"] == exp["adapter_bytes"]

    class W:
        dtype = c["dtype"]

    class Lr:
        d_in, d_out, shared_rank = c["d_in"], c["d_out"], c["shared_rank"]
    got = _c_report(lib, W, Lr, ads, c["lowrank_launched"], c["vera_launched"], np.array(g["ids"]),
                    c["out_dtype"], 8)
    assert [list(k) for k in got["kernels"]] == exp["kernels"]
    assert got["algorithmic_bytes"] == exp["algorithmic_bytes"]


def test_byte_model_rejects_bad_arguments(lib):
    import ctypes
    arr = (lib.BmAdapter * 1)()
    bl = lib.BmLayer(dtype=0, out_dtype=0, d_in=0, d_out=64, shared_rank=0, lowrank_launched=0,
                     vera_launched=0, max_adapters=1, adapters=ctypes.cast(arr, ctypes.POINTER(lib.BmAdapter)))
    with pytest.raises(lib.ScuteError):
        lib.scute_byte_model(bl, np.zeros(1, np.int32), 1)


def test_batch_byte_model_matches_oracle(lib):
    """A batched call over several layers (the decode workload's six
    projections, the same layer twice, and a batch above the decode step's
    token limit): the library's launch list equals the oracle's."""
    for w, names, out_dtype in [
        (WL.decode_mixed(), ("q", "k", "v", "gate", "up", "down"), "bf16"),
        (WL.decode_mixed(n=50, shapes=WL.SMALL_PROJ, proj=("q", "k", "up", "down")), ("q", "up", "q"), "fp32"),
        (WL.decode_mixed(n=200, shapes=WL.SMALL_PROJ, proj=("q", "k", "up", "down")), ("k", "down"), "bf16"),
    ]:
        import ctypes
        A = max(a.id for a in w.adapters) + 3
        keep = []
        layers, ref_layers = [], []
        for name in names:
            L, ads, lowrank, vera = _bm_inputs(w, name, out_dtype)
            arr = (lib.BmAdapter * A)()
            for i in range(A):
                arr[i].method = -1
            for aid, v in ads.items():
                arr[aid].method = lib.METHOD_ID[v["method"]]
                arr[aid].rank = v["rank"]
                arr[aid].has_s, arr[aid].has_b, arr[aid].has_R = int(v["s"]), int(v["b"]), int(v["R"])
                arr[aid].has_vera, arr[aid].has_vera_e = int(v["vera"]), int(v["vera_e"])
            keep.append(arr)
            layers.append(lib.BmLayer(dtype=lib.FP32 if w.dtype == "fp32" else lib.BF16,
                                      out_dtype=lib.FP32 if out_dtype == "fp32" else lib.BF16,
                                      d_in=L.d_in, d_out=L.d_out, shared_rank=L.shared_rank,
                                      lowrank_launched=int(lowrank), vera_launched=int(vera), max_adapters=A,
                                      adapters=ctypes.cast(arr, ctypes.POINTER(lib.BmAdapter))))
            ref_layers.append({"adapters": ads, "d_in": L.d_in, "d_out": L.d_out, "shared_rank": L.shared_rank,
                               "lowrank_launched": lowrank, "vera_launched": vera})
        ids = w.ids.copy()
        ids[1] = -1
        got = lib.scute_byte_model_batch(layers, np.ascontiguousarray(ids, np.int32), int(ids.size))
        ref = OBM.batch_bytes(ids, ref_layers, w.dtype, out_dtype)
        assert got["kernels"] == [tuple(k) for k in ref["kernels"]]
        for k in ("algorithmic_bytes", "adapter_bytes", "base_weight_bytes", "distinct_adapters"):
            assert got[k] == ref[k], k
        if w.dtype != "fp32" and w.n <= 128:
            # one launch, whose bytes are the call's algorithmic bytes
            assert len(got["kernels"]) == 1 and got["kernels"][0][1] == got["algorithmic_bytes"]
        # the time model: library and oracle agree
        for bw, tf, lc in [(6794.5, 0.0, 2.0), (6794.5, 1846.4, 1.3)]:
            t = lib.scute_predict_time(got, bw, tf, lc)
            assert abs(t - OBM.predict_time_us(ref["kernels"], bw, tf, lc)) <= 1e-9 * max(1.0, t)


def test_fused_expand_plan_moves_only_the_out_rewrite():
    """bf16 batches above 256 tokens run the owned expand inside the base
    GEMM's epilogue.  Against the separate expand the launch list loses
    lr_expand, the shrink comes before the GEMM (and the tensor-core VeRA
    shrink, for a shared rank that is a multiple of 64, right after it), the
    GEMM gains the expand's v partials, B' and flops, and the total bytes drop
    by exactly the owned rows of out read and written once more; the flops are
    unchanged."""
    w = WL.prefill_mixed(n_req=6, lo=40, hi=200, shapes=WL.SMALL_PROJ, proj=("q", "k", "up", "down"))
    assert w.n > 256
    for layer in ("q", "up"):
        L, ads, lowrank, vera = _bm_inputs(w, layer, "bf16")
        assert lowrank
        c = OBM._layer_counts(w.ids, ads, L.d_in, L.d_out, L.shared_rank, "bf16", "bf16")
        sep = OBM._per_kernel_plan(c, lowrank, vera, lr_fused=False)
        fus = OBM._per_kernel_plan(c, lowrank, vera, lr_fused=True)
        names_sep, names_fus = [k[0] for k in sep], [k[0] for k in fus]
        vs_first = vera and L.shared_rank % 64 == 0
        assert names_sep[:5] == ["index", "rotate", "base_gemm", "lr_shrink", "lr_expand"]
        head = ["index", "rotate", "lr_shrink"] + (["vera_shrink"] if vs_first else []) + ["base_gemm"]
        assert names_fus[:len(head)] == head
        rest_sep = [k for k in names_sep[5:] if not (vs_first and k == "vera_shrink")]
        assert "lr_expand" not in names_fus and names_fus[len(head):] == rest_sep
        if vera:
            assert dict((k[0], k) for k in sep)["vera_shrink"] == dict((k[0], k) for k in fus)["vera_shrink"]
        ks = OBM.lowrank_ks(L.d_in)
        g_sep, g_fus = dict((k[0], k) for k in sep)["base_gemm"], dict((k[0], k) for k in fus)["base_gemm"]
        assert g_fus[1] - g_sep[1] == ks * c["lr_rank_rows"] * 4 + c["B_b"]
        assert g_fus[2] - g_sep[2] == 2 * c["lr_rank_rows"] * L.d_out
        assert sum(k[1] for k in sep) - sum(k[1] for k in fus) == 2 * c["n_lr"] * L.d_out * 2
        assert sum(k[2] for k in sep) == sum(k[2] for k in fus)
        # the public entry takes the fused plan for bf16 above 256 tokens only
        ref = OBM.call_bytes(w.ids, ads, L.d_in, L.d_out, L.shared_rank, "bf16", "bf16", lowrank, vera)
        assert [k[0] for k in ref["kernels"]] == names_fus
        ref = OBM.call_bytes(w.ids[:256], ads, L.d_in, L.d_out, L.shared_rank, "bf16", "bf16", lowrank, vera)
        assert "lr_expand" in [k[0] for k in ref["kernels"]]


def test_time_model_hand_example(lib):
    """Two launches counted by hand: 1e6 bytes at 1000 GB/s is 1 us; 2e9 flops
    at 1000 TFLOP/s is 2 us, so the first launch takes max(1, 2) = 2 us; the
    second moves 3e6 bytes (3 us) and does no arithmetic; plus 2 launches of
    0.5 us: 2 + 3 + 1 = 6 us.  Without the flops term (the article's form):
    1 + 3 + 1 = 5 us."""
    rep = {"kernels": [("a", 1_000_000, 2_000_000_000), ("b", 3_000_000, 0)]}
    assert abs(lib.scute_predict_time(rep, 1000.0, 1000.0, 0.5) - 6.0) <= 1e-12
    assert abs(lib.scute_predict_time(rep, 1000.0, 0.0, 0.5) - 5.0) <= 1e-12
    assert abs(OBM.predict_time_us(rep["kernels"], 1000.0, 1000.0, 0.5) - 6.0) <= 1e-12
    assert abs(OBM.predict_time_us(rep["kernels"], 1000.0, 0.0, 0.5) - 5.0) <= 1e-12
    with pytest.raises(lib.ScuteError):
        lib.scute_predict_time(rep, 0.0, 0.0, 0.5)


def _bm_layer_struct(lib, ads, dtype, out_dtype, d_in, d_out, shared_rank, lowrank, vera, A, variant, keep):
    import ctypes
    arr = (lib.BmAdapter * A)()
    for i in range(A):
        arr[i].method = -1
    for aid, v in ads.items():
        arr[aid].method = lib.METHOD_ID[v["method"]]
        arr[aid].rank = v["rank"]
        arr[aid].has_s, arr[aid].has_b, arr[aid].has_R = int(v["s"]), int(v["b"]), int(v["R"])
        arr[aid].has_vera, arr[aid].has_vera_e = int(v["vera"]), int(v["vera_e"])
    keep.append(arr)
    return lib.BmLayer(dtype=lib.FP32 if dtype == "fp32" else lib.BF16,
                       out_dtype=lib.FP32 if out_dtype == "fp32" else lib.BF16, d_in=d_in, d_out=d_out,
                       shared_rank=shared_rank, lowrank_launched=int(lowrank), vera_launched=int(vera),
                       max_adapters=A, adapters=ctypes.cast(arr, ctypes.POINTER(lib.BmAdapter)), variant=variant)


def test_variant_byte_model_hand_example(lib):
    """The separate-pass placements counted by hand (tests/golden/byte_model_hand.json)."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "byte_model_hand.json")))
    for c in g["variant_cases"]:
        ads = {int(k): v for k, v in c["adapters"].items()}
        L = {"adapters": ads, "d_in": c["d_in"], "d_out": c["d_out"], "shared_rank": c["shared_rank"],
             "lowrank_launched": c["lowrank_launched"], "vera_launched": c["vera_launched"]}
        ref = OBM.batch_bytes(c["ids"], [L], c["dtype"], c["out_dtype"], c["variant"])
        exp = c["expected"]
        assert [list(k) for k in ref["kernels"]] == exp["kernels"]
        assert ref["algorithmic_bytes"] == exp["algorithmic_bytes"]
        assert ref["adapter_bytes"] == exp["adapter_bytes"]
        keep = []
        bl = _bm_layer_struct(lib, ads, c["dtype"], c["out_dtype"], c["d_in"], c["d_out"], c["shared_rank"],
                              c["lowrank_launched"], c["vera_launched"], 8, c["variant"], keep)
        got = lib.scute_byte_model_batch([bl], np.array(c["ids"], np.int32), len(c["ids"]))
        assert [list(k) for k in got["kernels"]] == exp["kernels"]
        assert got["algorithmic_bytes"] == exp["algorithmic_bytes"]


@pytest.mark.parametrize("variant", [1, 2, 3])
def test_variant_byte_model_matches_oracle(lib, variant):
    """The decode workload's six projections with each placement: the
    library's launch list equals the oracle's, and the per-launch bytes add up
    to the algorithmic bytes plus what the passes move again."""
    w = WL.decode_mixed()
    names = ("q", "k", "v", "gate", "up", "down")
    A = max(a.id for a in w.adapters) + 3
    keep, layers, ref_layers = [], [], []
    for name in names:
        L, ads, lowrank, vera = _bm_inputs(w, name, "bf16")
        layers.append(_bm_layer_struct(lib, ads, "bf16", "bf16", L.d_in, L.d_out, L.shared_rank, lowrank, vera, A,
                                       variant, keep))
        ref_layers.append({"adapters": ads, "d_in": L.d_in, "d_out": L.d_out, "shared_rank": L.shared_rank,
                           "lowrank_launched": lowrank, "vera_launched": vera})
    ids = np.ascontiguousarray(w.ids, np.int32)
    got = lib.scute_byte_model_batch(layers, ids, int(ids.size))
    ref = OBM.batch_bytes(ids, ref_layers, "bf16", "bf16", variant)
    assert got["kernels"] == [tuple(k) for k in ref["kernels"]]
    names_got = [k[0] for k in got["kernels"]]
    assert names_got == (["oft_pass"] if variant & 1 else []) + ["step"] + (["s_pass"] if variant & 2 else [])
