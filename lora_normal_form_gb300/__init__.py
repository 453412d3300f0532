"""Python binding of libscute.so: the adapted linear layer in normal form.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  The functions below carry the C ABI's names (``include/scute.h``) and
take torch tensors (device pointers), numpy arrays (host pointers) or ints.
Loading fails loudly when ``libscute.so`` is missing; there is no fallback.

Citations name sections of the article "Scute: Exact Batched Serving for PEFT
Adapters Beyond LoRA" (paper-daily.com).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libscute.so")

LORA, DORA, IA3, VERA, OFT, NF = range(6)
METHOD_ID = {"lora": LORA, "dora": DORA, "ia3": IA3, "vera": VERA, "oft": OFT, "nf": NF}
BF16, FP32 = 0, 1
STATUS = {0: "OK", 1: "ERR_ARG", 2: "ERR_SHAPE", 3: "ERR_DTYPE", 4: "ERR_OOM", 5: "ERR_BAD_ADAPTER",
          6: "ERR_CUDA", 7: "ERR_TIMEOUT", 8: "ERR_UNSUPPORTED", 9: "ERR_NO_DEVICE"}
MAX_TOKENS = 16384
TIMING_SLOTS = 256
BM_MAX_KERNELS = 64


class ScuteError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class LayerTensors(ctypes.Structure):
    _fields_ = [("layer", ctypes.c_int), ("rank", ctypes.c_int), ("c", ctypes.c_float),
                ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("d", ctypes.c_void_p),
                ("e", ctypes.c_void_p), ("s", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("R", ctypes.c_void_p), ("magnitude", ctypes.c_void_p), ("l", ctypes.c_void_p)]


class ByteReport(ctypes.Structure):
    _fields_ = [("n_kernels", ctypes.c_int), ("name", (ctypes.c_char * 24) * BM_MAX_KERNELS),
                ("bytes", ctypes.c_int64 * BM_MAX_KERNELS), ("flops", ctypes.c_int64 * BM_MAX_KERNELS),
                ("algorithmic_bytes", ctypes.c_int64), ("adapter_bytes", ctypes.c_int64),
                ("base_weight_bytes", ctypes.c_int64), ("distinct_adapters", ctypes.c_int32)]

    def as_dict(self) -> dict:
        k = self.n_kernels
        return {"kernels": [(self.name[i].value.decode(), int(self.bytes[i]), int(self.flops[i]))
                            for i in range(k)],
                "algorithmic_bytes": int(self.algorithmic_bytes),
                "adapter_bytes": int(self.adapter_bytes),
                "base_weight_bytes": int(self.base_weight_bytes),
                "distinct_adapters": int(self.distinct_adapters)}


class BmAdapter(ctypes.Structure):
    _fields_ = [("method", ctypes.c_int), ("rank", ctypes.c_int), ("has_s", ctypes.c_int),
                ("has_b", ctypes.c_int), ("has_R", ctypes.c_int), ("has_vera", ctypes.c_int),
                ("has_vera_e", ctypes.c_int)]


class BmLayer(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("d_in", ctypes.c_int),
                ("d_out", ctypes.c_int), ("shared_rank", ctypes.c_int),
                ("lowrank_launched", ctypes.c_int), ("vera_launched", ctypes.c_int),
                ("max_adapters", ctypes.c_int), ("adapters", ctypes.POINTER(BmAdapter)), ("variant", ctypes.c_int)]


class Call(ctypes.Structure):
    """One entry of a batched call (scute_call)."""
    _fields_ = [("x", ctypes.c_void_p), ("layer", ctypes.c_int), ("out", ctypes.c_void_p)]


MAX_CALLS = 8

_lib: Optional[ctypes.CDLL] = None

_SIGS = {
    "scute_version": (ctypes.c_int, []),
    "scute_create": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "scute_destroy": (None, [ctypes.c_void_p]),
    "scute_last_error": (ctypes.c_char_p, [ctypes.c_void_p]),
    "scute_add_layer": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p]),
    "scute_set_shared": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_void_p]),
    "scute_register_adapter": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(LayerTensors),
                                              ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]),
    "scute_unregister_adapter": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "scute_linear": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    "scute_linear_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    "scute_linear_batch": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(Call), ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]),
    "scute_linear_batch_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(Call), ctypes.c_int,
                                               ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]),
    "scute_sync_status": (ctypes.c_int, [ctypes.c_void_p]),
    "scute_debug_index": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64] +
                          [ctypes.c_void_p] * 5 + [ctypes.c_void_p]),
    "scute_index_tokens_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                  ctypes.c_int64] + [ctypes.c_void_p] * 7),
    "scute_byte_model": (ctypes.c_int, [ctypes.POINTER(BmLayer), ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.POINTER(ByteReport)]),
    "scute_predict_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_int, ctypes.POINTER(ByteReport)]),
    "scute_byte_model_batch": (ctypes.c_int, [ctypes.POINTER(BmLayer), ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.POINTER(ByteReport)]),
    "scute_predict_batch": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(Call), ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ByteReport)]),
    "scute_predict_time": (ctypes.c_int, [ctypes.POINTER(ByteReport), ctypes.c_double, ctypes.c_double,
                                          ctypes.c_double, ctypes.POINTER(ctypes.c_double)]),
    "scute_launch_count": (ctypes.c_int64, [ctypes.c_void_p]),
    "scute_timing_enable": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "scute_timing_reset": (ctypes.c_int, [ctypes.c_void_p]),
    "scute_debug_inject": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "scute_debug_fail_alloc": (None, [ctypes.c_int]),
    "scute_set_variant": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "scute_debug_step_plan": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int)]),
    "scute_timing_read": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_float), ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int)]),
    "scute_timing_kinds": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int)]),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libscute.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; "
                           "g.build()'` (the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def ptr(x) -> Optional[int]:
    """Address of a torch tensor, numpy array, int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("numpy array must be C-contiguous")
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream_handle(stream) -> Optional[int]:
    """The cudaStream_t to pass: an int as given, a torch stream's handle, or,
    for None, torch's current stream on the current device (so that calls
    made under ``torch.cuda.stream(s)`` are ordered with that stream's work)."""
    if stream is None:
        import sys
        torch = sys.modules.get("torch")
        if torch is not None and torch.cuda.is_available() and torch.cuda.is_initialized():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(ctx, code: int):
    if code != 0:
        msg = _lib.scute_last_error(ctx).decode() if ctx else ""
        raise ScuteError(code, msg)


# ------------------------------------------------------------------ C ABI names
def scute_version() -> int:
    return load().scute_version()


def scute_create(device: int, dtype: int, max_tokens: int, max_adapters: int, max_layers: int) -> int:
    lib = load()
    h = ctypes.c_void_p()
    code = lib.scute_create(ctypes.byref(h), device, dtype, max_tokens, max_adapters, max_layers)
    if code != 0:
        raise ScuteError(code, "scute_create failed")
    return h.value


def scute_destroy(ctx: int) -> None:
    load().scute_destroy(ctx)


def scute_add_layer(ctx, layer, d_in, d_out, W):
    _check(ctx, load().scute_add_layer(ctx, layer, d_in, d_out, ptr(W)))


def scute_set_shared(ctx, layer, rank, A_sh, B_sh):
    _check(ctx, load().scute_set_shared(ctx, layer, rank, ptr(A_sh), ptr(B_sh)))


def scute_register_adapter(ctx, method: int, tensors: list) -> int:
    """tensors: list of dicts with keys layer, rank, c, A, B, d, e, s, b, R, magnitude, l."""
    arr = (LayerTensors * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i].layer = t["layer"]
        arr[i].rank = int(t.get("rank", 0))
        arr[i].c = float(t.get("c", 1.0))
        for k in ("A", "B", "d", "e", "s", "b", "R", "magnitude", "l"):
            setattr(arr[i], k, ptr(t.get(k)))
    out = ctypes.c_int32()
    _check(ctx, load().scute_register_adapter(ctx, method, arr, len(tensors), ctypes.byref(out)))
    return out.value


def scute_unregister_adapter(ctx, adapter_id: int):
    _check(ctx, load().scute_unregister_adapter(ctx, adapter_id))


def scute_linear(ctx, x, adapter_ids, n, layer, out, out_dtype, stream=None):
    _check(ctx, load().scute_linear(ctx, ptr(x), ptr(adapter_ids), n, layer, ptr(out), out_dtype,
                                    _stream_handle(stream)))


def scute_linear_host(ctx, x_host, ids_host, n, layer, out_host, out_dtype, stream=None):
    _check(ctx, load().scute_linear_host(ctx, ptr(x_host), ptr(ids_host), n, layer, ptr(out_host),
                                         out_dtype, _stream_handle(stream)))


def _calls(calls):
    arr = (Call * max(1, len(calls)))()
    for i, (x, layer, out) in enumerate(calls):
        arr[i].x = ptr(x)
        arr[i].layer = layer
        arr[i].out = ptr(out)
    return arr


def scute_linear_batch(ctx, calls, adapter_ids, n, out_dtype, stream=None):
    """``calls``: sequence of (x, layer, out) with device tensors."""
    _check(ctx, load().scute_linear_batch(ctx, _calls(calls), len(calls), ptr(adapter_ids), n, out_dtype,
                                          _stream_handle(stream)))


def scute_linear_batch_host(ctx, calls, ids_host, n, out_dtype, stream=None):
    """``calls``: sequence of (x_host, layer, out_host) with host arrays."""
    _check(ctx, load().scute_linear_batch_host(ctx, _calls(calls), len(calls), ptr(ids_host), n, out_dtype,
                                               _stream_handle(stream)))


def scute_sync_status(ctx) -> int:
    return load().scute_sync_status(ctx)


def scute_debug_index(ctx, ids, n, perm, aid_sorted, seg_start, seg_aid, counts, stream=None):
    _check(ctx, load().scute_debug_index(ctx, ptr(ids), n, ptr(perm), ptr(aid_sorted), ptr(seg_start),
                                         ptr(seg_aid), ptr(counts), _stream_handle(stream)))


NOALLOC_MAX_ADAPTERS = 8192


def scute_index_tokens_noalloc(method_of_adapter, ids, n, perm, aid_sorted, seg_start, seg_aid, counts,
                               flags=None, stream=None):
    """Context-free indexing on the current device; ``method_of_adapter`` is a
    host int8 numpy array (method code per adapter id, -1 = none)."""
    import numpy as np
    tab = np.ascontiguousarray(method_of_adapter, dtype=np.int8)
    code = load().scute_index_tokens_noalloc(ptr(tab), int(tab.size), ptr(ids), n, ptr(perm), ptr(aid_sorted),
                                             ptr(seg_start), ptr(seg_aid), ptr(counts), ptr(flags),
                                             _stream_handle(stream))
    if code != 0:
        why = {1: "null output, n < 0, no adapters or a method code outside -1..5",
               8: f"n above {MAX_TOKENS} tokens or more than {NOALLOC_MAX_ADAPTERS} adapters "
                  "(size of the static method table)",
               9: "the current device is not sm_103", 6: "a CUDA call failed"}.get(code, "")
        raise ScuteError(code, why)


def scute_byte_model(layer: BmLayer, ids_host, n) -> dict:
    rep = ByteReport()
    code = load().scute_byte_model(ctypes.byref(layer), ptr(ids_host), n, ctypes.byref(rep))
    if code != 0:
        raise ScuteError(code, "scute_byte_model failed")
    return rep.as_dict()


def scute_predict_bytes(ctx, ids_host, n, layer, out_dtype) -> dict:
    rep = ByteReport()
    _check(ctx, load().scute_predict_bytes(ctx, ptr(ids_host), n, layer, out_dtype, ctypes.byref(rep)))
    return rep.as_dict()


def scute_byte_model_batch(layers, ids_host, n) -> dict:
    """``layers``: sequence of BmLayer (one per call of the batch)."""
    arr = (BmLayer * max(1, len(layers)))(*layers)
    rep = ByteReport()
    code = load().scute_byte_model_batch(arr, len(layers), ptr(ids_host), n, ctypes.byref(rep))
    if code != 0:
        raise ScuteError(code, "scute_byte_model_batch failed")
    return rep.as_dict()


def scute_predict_batch(ctx, layers, ids_host, n, out_dtype) -> dict:
    """Launch list of a batched call over the given layer ids."""
    arr = (Call * max(1, len(layers)))()
    for i, layer in enumerate(layers):
        arr[i].layer = layer
    rep = ByteReport()
    _check(ctx, load().scute_predict_batch(ctx, arr, len(layers), ptr(ids_host), n, out_dtype, ctypes.byref(rep)))
    return rep.as_dict()


def scute_predict_time(report: dict, hbm_gbs: float, tensor_tflops: float, launch_us: float) -> float:
    """Predicted microseconds of a launch list (a report dict as returned above)."""
    rep = ByteReport()
    ks = report["kernels"]
    if len(ks) > BM_MAX_KERNELS:
        raise ValueError("too many launches")
    rep.n_kernels = len(ks)
    for i, (name, b, f) in enumerate(ks):
        rep.name[i].value = name.encode()[:23]
        rep.bytes[i] = int(b)
        rep.flops[i] = int(f)
    us = ctypes.c_double()
    code = load().scute_predict_time(ctypes.byref(rep), float(hbm_gbs), float(tensor_tflops), float(launch_us),
                                     ctypes.byref(us))
    if code != 0:
        raise ScuteError(code, "scute_predict_time failed")
    return us.value


def scute_launch_count(ctx) -> int:
    return load().scute_launch_count(ctx)


def scute_timing_enable(ctx, enable: bool):
    _check(ctx, load().scute_timing_enable(ctx, 1 if enable else 0))


def scute_timing_reset(ctx):
    _check(ctx, load().scute_timing_reset(ctx))


INJECT_STALL = 1


def scute_debug_inject(ctx, what: int) -> None:
    _check(ctx, load().scute_debug_inject(ctx, what))


VARIANT_OFT_PASS, VARIANT_S_PASS = 1, 2


def scute_set_variant(ctx, flags: int) -> None:
    """Place OFT's rotation (1) and / or DoRA's and (IA)^3's s (2) in launches
    of their own around the decode step (byte-model validation)."""
    _check(ctx, load().scute_set_variant(ctx, int(flags)))


PLAN_HEAD, PLAN_CALL_FIELDS = 19, 18


def scute_debug_step_plan(ctx) -> list:
    """The last decode-step launch's plan as a list of ints (layout in scute.h)."""
    n = ctypes.c_int()
    _check(ctx, load().scute_debug_step_plan(ctx, None, 0, ctypes.byref(n)))
    buf = (ctypes.c_int64 * max(n.value, 1))()
    _check(ctx, load().scute_debug_step_plan(ctx, buf, n.value, ctypes.byref(n)))
    return [int(buf[i]) for i in range(n.value)]


def scute_debug_fail_alloc(k: int) -> None:
    """Make the k-th device allocation of the library from now fail as out of
    memory (test hook; k <= 0 switches it off)."""
    load().scute_debug_fail_alloc(int(k))


def scute_timing_read(ctx, max_slots: int = TIMING_SLOTS) -> list:
    buf = (ctypes.c_float * max_slots)()
    n = ctypes.c_int()
    _check(ctx, load().scute_timing_read(ctx, buf, max_slots, ctypes.byref(n)))
    return [float(buf[i]) for i in range(n.value)]


KIND_NAMES = ("step", "index", "rotate", "base_gemm", "lowrank", "vera_shrink", "vera_expand", "oft_pass", "s_pass")


def scute_timing_kinds(ctx, max_slots: int = TIMING_SLOTS) -> list:
    buf = (ctypes.c_int * max_slots)()
    n = ctypes.c_int()
    _check(ctx, load().scute_timing_kinds(ctx, buf, max_slots, ctypes.byref(n)))
    return [KIND_NAMES[buf[i]] for i in range(n.value)]


from .context import Context  # noqa: E402,F401
