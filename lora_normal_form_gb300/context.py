"""A small owner object around a scute context handle (marshalling only)."""
from __future__ import annotations

import numpy as np

from . import (BF16, FP32, METHOD_ID, scute_add_layer, scute_create, scute_debug_index, scute_destroy,
               scute_launch_count, scute_linear, scute_linear_batch, scute_linear_batch_host,
               scute_linear_host, scute_predict_batch, scute_predict_bytes,
               scute_register_adapter, scute_set_shared, scute_set_variant, scute_sync_status,
               scute_timing_enable,
               scute_timing_kinds, scute_timing_read, scute_timing_reset, scute_unregister_adapter)


class Context:
    """Owns one scute context; every method is one C ABI call."""

    def __init__(self, dtype: str = "bf16", max_tokens: int = 1024, max_adapters: int = 64,
                 max_layers: int = 16, device: int = 0):
        self.dtype = dtype
        self.device = device
        self.max_tokens = max_tokens
        self.handle = scute_create(device, BF16 if dtype == "bf16" else FP32, max_tokens, max_adapters,
                                   max_layers)
        self.layer_ids = {}          # layer name -> id
        self.layer_dims = {}         # id -> (d_in, d_out)

    def close(self):
        if self.handle:
            scute_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- setup
    def add_layer(self, layer: int, d_in: int, d_out: int, W):
        scute_add_layer(self.handle, layer, d_in, d_out, W)
        self.layer_dims[layer] = (d_in, d_out)

    def set_shared(self, layer: int, rank: int, A_sh, B_sh):
        scute_set_shared(self.handle, layer, rank, A_sh, B_sh)

    def register(self, method: str, tensors: list) -> int:
        return scute_register_adapter(self.handle, METHOD_ID[method], tensors)

    def unregister(self, adapter_id: int):
        scute_unregister_adapter(self.handle, adapter_id)

    def load_workload(self, w, layer_names=None, drop_host: bool = False):
        """Register the layers, shared pairs and adapters of a synthetic workload
        (``workloads.Workload``) in order, so that adapter ids match."""
        names = [L.name for L in w.layers] if layer_names is None else list(layer_names)
        for L in w.layers:
            if L.name not in names:
                continue
            lid = len(self.layer_ids)
            self.layer_ids[L.name] = lid
            self.add_layer(lid, L.d_in, L.d_out, np.ascontiguousarray(L.get("W")))
            if L.shared_rank:
                self.set_shared(lid, L.shared_rank, np.ascontiguousarray(L.get("A_sh")),
                                np.ascontiguousarray(L.get("B_sh")))
            if drop_host:
                L._cache.pop("W", None)
                L._cache.pop("A_sh", None)
                L._cache.pop("B_sh", None)
        for a in sorted(w.adapters, key=lambda a: a.id):
            tens = []
            for lname in a.layers:
                if lname not in self.layer_ids:
                    continue
                t = {"layer": self.layer_ids[lname], "rank": a.rank, "c": a.c}
                for slot in a.slots(lname):
                    key = {"m": "magnitude"}.get(slot, slot)
                    t[key] = np.ascontiguousarray(a.get(lname, slot))
                tens.append(t)
            # an adapter with no tensors on the chosen layers has identity slots there
            aid = self.register(a.method, tens)
            if aid != a.id:
                raise RuntimeError(f"adapter id mismatch: library gave {aid}, workload has {a.id}")
            if drop_host:
                a.drop()

    # ---------------------------------------------------------------- hot path
    def linear(self, x, ids, layer: int, out, out_dtype: str = "bf16", stream=None, n=None):
        n = int(ids.shape[0]) if n is None else n
        scute_linear(self.handle, x, ids, n, layer, out, BF16 if out_dtype == "bf16" else FP32, stream)

    def linear_host(self, x_host, ids_host, layer: int, out_host, out_dtype: str = "bf16", stream=None):
        scute_linear_host(self.handle, x_host, ids_host, int(ids_host.shape[0]), layer, out_host,
                          BF16 if out_dtype == "bf16" else FP32, stream)

    def linear_batch(self, calls, ids, out_dtype: str = "bf16", stream=None, n=None):
        """``calls``: sequence of (x, layer id, out); every layer sees the same ids."""
        n = int(ids.shape[0]) if n is None else n
        scute_linear_batch(self.handle, list(calls), ids, n, BF16 if out_dtype == "bf16" else FP32, stream)

    def linear_batch_host(self, calls, ids_host, out_dtype: str = "bf16", stream=None):
        scute_linear_batch_host(self.handle, list(calls), ids_host, int(ids_host.shape[0]),
                                BF16 if out_dtype == "bf16" else FP32, stream)

    def sync_status(self) -> int:
        return scute_sync_status(self.handle)

    def debug_index(self, ids, n, perm, aid_sorted, seg_start, seg_aid, counts, stream=None):
        scute_debug_index(self.handle, ids, n, perm, aid_sorted, seg_start, seg_aid, counts, stream)

    def predict_bytes(self, ids_host, layer: int, out_dtype: str = "bf16") -> dict:
        ids_host = np.ascontiguousarray(ids_host, dtype=np.int32)
        return scute_predict_bytes(self.handle, ids_host, int(ids_host.size), layer,
                                   BF16 if out_dtype == "bf16" else FP32)

    def predict_batch(self, layers, ids_host, out_dtype: str = "bf16") -> dict:
        ids_host = np.ascontiguousarray(ids_host, dtype=np.int32)
        return scute_predict_batch(self.handle, list(layers), ids_host, int(ids_host.size),
                                   BF16 if out_dtype == "bf16" else FP32)

    def set_variant(self, flags: int):
        scute_set_variant(self.handle, flags)

    def launch_count(self) -> int:
        return scute_launch_count(self.handle)

    def timing(self, enable: bool):
        scute_timing_enable(self.handle, enable)

    def timing_reset(self):
        scute_timing_reset(self.handle)

    def timing_read(self) -> list:
        return scute_timing_read(self.handle)

    def timing_kinds(self) -> list:
        return scute_timing_kinds(self.handle)
