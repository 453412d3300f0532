"""Seeded synthetic inputs for the adapted linear layer in normal form.

Both the float64 oracle (``oracle/``) and the CUDA path consume these arrays;
this module holds none of the method's arithmetic.  It only draws tensors with
the shapes and distributions of the workloads the Scute article measures
("Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA", paper-daily.com:
Llama-3.1-8B-shaped projections, random adapters drawn away from identity,
section "Does it actually work better?").  No dataset, checkpoint or trained
weight is used: every value is drawn here from a seeded generator.

Storage conventions (what the C ABI receives):
  * matrices (W, A, B, R, shared VeRA A/B, x) in the workload dtype: bf16 is held
    as ``numpy.uint16`` bit patterns (round-to-nearest-even from float32), fp32 as
    ``numpy.float32``;
  * vectors (s, b, d, e, DoRA magnitude m, (IA)^3 l) always as ``numpy.float32``;
  * orientation is row-vector: x [n, d_in], W [d_in, d_out], A [d_in, r],
    B [r, d_out], OFT R as explicit 32x32 blocks [d_in/32, 32, 32].

Every tensor comes from its own stream keyed by (seed, tensor name), so any
tensor can be regenerated alone (the oracle regenerates only what it samples).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Tuple

import numpy as np

METHODS = ("lora", "dora", "ia3", "vera", "oft", "nf")
OFT_BLOCK = 32

# Llama-3-8B projection shapes (d_in, d_out); "ia3" marks the layers that carry
# (IA)^3's l (keys, values and the FFN up projection).
LLAMA_PROJ = {
    "q": (4096, 4096, False),
    "k": (4096, 1024, True),
    "v": (4096, 1024, True),
    "o": (4096, 4096, False),
    "gate": (4096, 14336, False),
    "up": (4096, 14336, True),
    "down": (14336, 4096, False),
}


# --------------------------------------------------------------------------
# storage helpers
# --------------------------------------------------------------------------
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (round-to-nearest-even), as uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 values (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_f64(arr: np.ndarray) -> np.ndarray:
    """Exact float64 view of a stored tensor (bf16 bits or float32)."""
    if arr.dtype == np.uint16:
        return bf16_values(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float64)


def _rng(seed: int, *names) -> np.random.Generator:
    h = hashlib.sha256(repr((int(seed),) + tuple(names)).encode()).digest()
    return np.random.default_rng(np.frombuffer(h[:16], dtype=np.uint32))


def _store(vals: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits(vals)
    return np.ascontiguousarray(vals, dtype=np.float32)


def draw_normal(seed, name, shape, std, dtype, mean=0.0) -> np.ndarray:
    g = _rng(seed, name)
    v = g.standard_normal(size=shape, dtype=np.float32)
    v *= np.float32(std)
    if mean:
        v += np.float32(mean)
    return _store(v, dtype)


def draw_vector(seed, name, n, std=0.1) -> np.ndarray:
    """Adapter vector drawn away from identity: 1 + N(0, std), float32."""
    g = _rng(seed, name)
    return (1.0 + std * g.standard_normal(size=(n,))).astype(np.float32)


def draw_cayley_blocks(seed, name, n_blk, dtype, std=0.05, blk=OFT_BLOCK) -> np.ndarray:
    """Orthogonal blocks R = (I + S)(I - S)^-1 with S skew-symmetric.

    S has its strict upper triangle drawn N(0, std).  The result is rounded to
    the storage dtype, so the stored blocks are orthogonal only to that
    precision; the method consumes whatever blocks it is given.
    """
    g = _rng(seed, name)
    up = np.triu(g.standard_normal(size=(n_blk, blk, blk)) * std, 1)
    S = up - np.transpose(up, (0, 2, 1))
    I = np.eye(blk)[None]
    R = np.linalg.solve(np.transpose(I - S, (0, 2, 1)), np.transpose(I + S, (0, 2, 1)))
    R = np.transpose(R, (0, 2, 1))  # (I+S)(I-S)^-1
    return _store(R, dtype)


# --------------------------------------------------------------------------
# workload description
# --------------------------------------------------------------------------
@dataclass
class Layer:
    name: str
    d_in: int
    d_out: int
    ia3: bool                      # (IA)^3 l is present on this layer
    shared_rank: int               # VeRA shared rank (0: no shared pair)
    _gen: Dict[str, Callable[[], np.ndarray]] = field(default_factory=dict, repr=False)
    _cache: Dict[str, np.ndarray] = field(default_factory=dict, repr=False)

    def get(self, key: str) -> np.ndarray:
        """key in {'W', 'A_sh', 'B_sh', 'x'}."""
        if key not in self._cache:
            self._cache[key] = self._gen[key]()
        return self._cache[key]

    def drop(self):
        self._cache.clear()


@dataclass
class Adapter:
    id: int
    method: str
    c: float
    rank: int
    layers: Tuple[str, ...]                           # layers the adapter has tensors on
    _gen: Dict[Tuple[str, str], Callable[[], np.ndarray]] = field(default_factory=dict, repr=False)
    _cache: Dict[Tuple[str, str], np.ndarray] = field(default_factory=dict, repr=False)

    def slots(self, layer: str) -> List[str]:
        return sorted(k[1] for k in self._gen if k[0] == layer)

    def get(self, layer: str, slot: str) -> np.ndarray:
        k = (layer, slot)
        if k not in self._cache:
            self._cache[k] = self._gen[k]()
        return self._cache[k]

    def drop(self):
        self._cache.clear()


@dataclass
class Workload:
    name: str
    dtype: str                      # "bf16" or "fp32"
    n: int
    ids: np.ndarray                 # int32 [n], -1 = base only
    layers: List[Layer]
    adapters: List[Adapter]
    recipe: str = ""

    def layer(self, name: str) -> Layer:
        for L in self.layers:
            if L.name == name:
                return L
        raise KeyError(name)

    def adapter(self, aid: int) -> Adapter:
        return self._by_id[aid]

    def __post_init__(self):
        self._by_id = {a.id: a for a in self.adapters}

    @property
    def n_adapters(self) -> int:
        return len(self.adapters)


def _make_layer(seed, name, d_in, d_out, ia3, rv, n, dtype, x_std=1.0) -> Layer:
    L = Layer(name=name, d_in=d_in, d_out=d_out, ia3=ia3, shared_rank=rv)
    L._gen["W"] = lambda: draw_normal(seed, f"W/{name}", (d_in, d_out), 0.02, dtype)
    L._gen["x"] = lambda: draw_normal(seed, f"x/{name}", (n, d_in), x_std, dtype)
    if rv:
        L._gen["A_sh"] = lambda: draw_normal(seed, f"Ash/{name}", (d_in, rv), 0.02, dtype)
        L._gen["B_sh"] = lambda: draw_normal(seed, f"Bsh/{name}", (rv, d_out), 0.02, dtype)
    return L


def _make_adapter(seed, aid, method, layers: List[Layer], dtype, rank=16, c=2.0,
                  vec_std=0.1) -> Adapter:
    names = []
    A = Adapter(id=aid, method=method, c=c if method in ("lora", "dora") else 1.0,
                rank=rank if method in ("lora", "dora") else 0, layers=())
    for L in layers:
        pre = f"ad{aid}/{L.name}"
        di, do = L.d_in, L.d_out
        if method in ("lora", "dora"):
            A._gen[(L.name, "A")] = (lambda p=pre, di=di: draw_normal(seed, p + "/A", (di, rank), 0.02, dtype))
            A._gen[(L.name, "B")] = (lambda p=pre, do=do: draw_normal(seed, p + "/B", (rank, do), 0.02, dtype))
            if method == "dora":
                # learned length per output column: about the column norm of W
                # (entries N(0, 0.02) over d_in rows) times 1 + N(0, vec_std).
                scale = 0.02 * np.sqrt(di)
                A._gen[(L.name, "m")] = (lambda p=pre, do=do, sc=scale: (
                    draw_vector(seed, p + "/m", do, vec_std) * np.float32(sc)).astype(np.float32))
            names.append(L.name)
        elif method == "ia3":
            if L.ia3:
                A._gen[(L.name, "l")] = (lambda p=pre, do=do: draw_vector(seed, p + "/l", do, vec_std))
                names.append(L.name)
        elif method == "vera":
            if L.shared_rank:
                rv = L.shared_rank
                A._gen[(L.name, "d")] = (lambda p=pre, rv=rv: draw_vector(seed, p + "/d", rv, vec_std))
                A._gen[(L.name, "e")] = (lambda p=pre, do=do: draw_vector(seed, p + "/e", do, vec_std))
                names.append(L.name)
        elif method == "oft":
            nb = di // OFT_BLOCK
            A._gen[(L.name, "R")] = (lambda p=pre, nb=nb: draw_cayley_blocks(seed, p + "/R", nb, dtype))
            names.append(L.name)
        else:
            raise ValueError(method)
    A.layers = tuple(names)
    return A


def _make_nf_adapter(seed, aid, layers: List[Layer], dtype, with_R=False, rank=0,
                     c=0.5) -> Adapter:
    """A raw normal-form adapter: s and b (scale-and-shift), optionally R and
    one owned low-rank term with live d and e (all folded at registration)."""
    A = Adapter(id=aid, method="nf", c=c, rank=rank, layers=tuple(L.name for L in layers))
    for L in layers:
        pre = f"ad{aid}/{L.name}"
        di, do = L.d_in, L.d_out
        A._gen[(L.name, "s")] = (lambda p=pre, do=do: draw_vector(seed, p + "/s", do, 0.1))
        A._gen[(L.name, "b")] = (lambda p=pre, do=do: (draw_vector(seed, p + "/b", do, 0.3) - 1.0).astype(np.float32))
        if with_R:
            nb = di // OFT_BLOCK
            A._gen[(L.name, "R")] = (lambda p=pre, nb=nb: draw_cayley_blocks(seed, p + "/R", nb, dtype))
        if rank:
            A._gen[(L.name, "A")] = (lambda p=pre, di=di: draw_normal(seed, p + "/A", (di, rank), 0.02, dtype))
            A._gen[(L.name, "B")] = (lambda p=pre, do=do: draw_normal(seed, p + "/B", (rank, do), 0.02, dtype))
            A._gen[(L.name, "d")] = (lambda p=pre: draw_vector(seed, p + "/d", rank, 0.1))
            A._gen[(L.name, "e")] = (lambda p=pre, do=do: draw_vector(seed, p + "/e", do, 0.1))
    return A


MOD5 = ("lora", "dora", "ia3", "vera", "oft")


def uniform_ids(seed, n, n_adapters) -> np.ndarray:
    return _rng(seed, "ids").integers(0, n_adapters, n).astype(np.int32)


def request_ids(seed, n_req, lo, hi, n_adapters, req_adapters=None) -> Tuple[np.ndarray, np.ndarray]:
    """Prefill batch: request lengths U{lo..hi}, one adapter per request (drawn
    uniformly from the pool, or the given ``req_adapters``)."""
    lens = np.random.default_rng(seed).integers(lo, hi + 1, n_req)
    if req_adapters is None:
        ads = _rng(seed, "req_adapters").integers(0, n_adapters, n_req)
    else:
        ads = np.asarray(req_adapters, dtype=np.int64)
        assert ads.shape == (n_req,) and ads.min() >= -1 and ads.max() < n_adapters
    return np.repeat(ads, lens).astype(np.int32), lens


def zipf_ids(seed, n, n_adapters, a=1.0) -> np.ndarray:
    """Finite Zipf(a): P(id = k) proportional to 1/(k+1)^a, k in 0..n_adapters-1."""
    p = 1.0 / np.arange(1, n_adapters + 1, dtype=np.float64) ** a
    p /= p.sum()
    return _rng(seed, "zipf").choice(n_adapters, size=n, p=p).astype(np.int32)


# --------------------------------------------------------------------------
# the workloads
# --------------------------------------------------------------------------
def tiny_fp32(seed: int = 0) -> Workload:
    """Tiny single linear, fp32: d_in = d_out = 256, 16 tokens, 5 adapters one
    per method (LoRA r=8, DoRA r=8, (IA)^3, VeRA shared rank 32, OFT block 32),
    ids uniform over the 5 adapters."""
    n = 16
    L = _make_layer(seed, "lin", 256, 256, True, 32, n, "fp32")
    ads = [_make_adapter(seed, i, m, [L], "fp32", rank=8) for i, m in enumerate(MOD5)]
    ids = uniform_ids(seed, n, 5)
    return Workload("tiny_fp32", "fp32", n, ids, [L], ads,
                    recipe="d=256, n=16, W/A/B ~ N(0,0.02), vectors 1+N(0,0.1), "
                           "R=Cayley(skew N(0,0.05)), x ~ N(0,1), ids uniform over 5")


def decode_mixed(seed: int = 0, n: int = 64, n_adapters: int = 32, rank: int = 16,
                 rv: int = 256, proj=("q", "k", "v", "gate", "up", "down"),
                 shapes: Optional[Dict[str, Tuple[int, int, bool]]] = None,
                 ids: Optional[np.ndarray] = None, dtype: str = "bf16",
                 name: str = "decode_mixed") -> Workload:
    """Llama-3-8B-shaped projections, bf16 decode: n tokens, n_adapters mixed
    evenly across the five methods (method = id mod 5), rank 16, VeRA shared
    rank 256, OFT block 32, ids uniform."""
    shapes = shapes or LLAMA_PROJ
    layers = [_make_layer(seed, p, shapes[p][0], shapes[p][1], shapes[p][2], rv, n, dtype)
              for p in proj]
    ads = [_make_adapter(seed, i, MOD5[i % 5], layers, dtype, rank=rank)
           for i in range(n_adapters)]
    if ids is None:
        ids = uniform_ids(seed, n, n_adapters)
    return Workload(name, dtype, n, ids, layers, ads,
                    recipe=f"n={n}, {n_adapters} adapters, method=id mod 5, r={rank}, "
                           f"r_v={rv}, W/A/B/shared ~ N(0,0.02), vectors 1+N(0,0.1), "
                           "x ~ N(0,1), ids uniform")


def prefill_mixed(seed: int = 0, n_req: int = 16, lo: int = 64, hi: int = 1024,
                  n_adapters: int = 32, rank: int = 16, rv: int = 256,
                  proj=("q", "k", "v", "gate", "up", "down"), shapes=None,
                  dtype: str = "bf16", req_adapters=None) -> Workload:
    """Same shapes, bf16 prefill: n_req requests with lengths U{lo..hi}, each
    request one adapter drawn uniformly from the pool (or the adapters listed
    in ``req_adapters``, one per request: a parity case that puts every method
    in one prefill batch; the seed-0 draw happens to pick no OFT adapter)."""
    ids, lens = request_ids(seed, n_req, lo, hi, n_adapters, req_adapters)
    w = decode_mixed(seed, n=int(ids.size), n_adapters=n_adapters, rank=rank, rv=rv,
                     proj=proj, shapes=shapes, ids=ids, dtype=dtype, name="prefill_mixed")
    w.recipe = (f"{n_req} requests, lengths U{{{lo}..{hi}}} (sum {ids.size}), one adapter "
                f"per request from {n_adapters}; " + w.recipe)
    return w


def scaling_ia3_vera(seed: int = 0, n: int = 256, n_adapters: int = 1024, rv: int = 256,
                     shapes=None) -> Workload:
    """Adapter-count scaling, bf16 decode: 4096->4096 and 4096->14336 layers,
    n=256, 1024 adapters (even ids (IA)^3, odd ids VeRA), ids Zipf(1.0)."""
    shapes = shapes or {"sq": (4096, 4096, True), "up": (4096, 14336, True)}
    layers = [_make_layer(seed, p, *shapes[p], rv, n, "bf16") for p in shapes]
    ads = [_make_adapter(seed, i, "ia3" if i % 2 == 0 else "vera", layers, "bf16")
           for i in range(n_adapters)]
    ids = zipf_ids(seed, n, n_adapters)
    return Workload("scaling_ia3_vera", "bf16", n, ids, layers, ads,
                    recipe=f"n={n}, {n_adapters} adapters half (IA)^3 half VeRA, Zipf(1.0) ids")


def lora_conversion_of(w: Workload, rank: int = 64, seed: int = 1) -> Workload:
    """The same ids with every adapter replaced by a rank-`rank` LoRA of random
    N(0, 0.02) factors (the conversion comparator)."""
    ads = [_make_adapter(seed, a.id, "lora", w.layers, w.dtype, rank=rank)
           for a in w.adapters]
    return Workload(w.name + f"_as_lora{rank}", w.dtype, w.n, w.ids.copy(), w.layers, ads,
                    recipe=f"same ids as {w.name}, rank-{rank} LoRA adapters")


def all_lora_of(w: Workload, rank: int = 16, seed: int = 2) -> Workload:
    """Same n, same ids, every adapter a rank-`rank` LoRA (overhead comparator)."""
    ads = [_make_adapter(seed, a.id, "lora", w.layers, w.dtype, rank=rank)
           for a in w.adapters]
    return Workload(w.name + "_all_lora", w.dtype, w.n, w.ids.copy(), w.layers, ads,
                    recipe=f"same ids as {w.name}, rank-{rank} LoRA adapters")


def stack_32layer(seed: int = 0, n: int = 128, n_adapters: int = 128, n_layers: int = 32,
                  rank: int = 16, rv: int = 256, shapes=None) -> Workload:
    """32-layer stack of all 7 adapted projections per layer, bf16 decode n=128,
    128 adapters mixed evenly across the five methods (OFT on every projection,
    (IA)^3 on k, v, up)."""
    shapes = shapes or LLAMA_PROJ
    layers = []
    for li in range(n_layers):
        for p in ("q", "k", "v", "o", "gate", "up", "down"):
            di, do, ia = shapes[p]
            layers.append(_make_layer(seed, f"L{li}.{p}", di, do, ia, rv, n, "bf16"))
    ads = [_make_adapter(seed, i, MOD5[i % 5], layers, "bf16", rank=rank)
           for i in range(n_adapters)]
    ids = uniform_ids(seed, n, n_adapters)
    return Workload("stack_32layer", "bf16", n, ids, layers, ads,
                    recipe=f"{n_layers} layers x 7 projections, n={n}, {n_adapters} adapters, "
                           "method=id mod 5")


def with_nf_adapters(w: Workload, seed: int = 3, n_extra: int = 2) -> Workload:
    """Append raw normal-form adapters (scale-and-shift s, b; the second also
    carries R and a rank-8 owned term with live d, e, c) and route some tokens
    to them.  Exercises the b slot and fold of live d/e/c."""
    base = len(w.adapters)
    extra = [_make_nf_adapter(seed, base, w.layers, w.dtype)]
    if n_extra > 1:
        extra.append(_make_nf_adapter(seed, base + 1, w.layers, w.dtype, with_R=True, rank=8))
    ids = w.ids.copy()
    g = _rng(seed, "nf_ids")
    pick = g.choice(w.n, size=max(2, w.n // 6), replace=False)
    ids[pick] = base + g.integers(0, len(extra), pick.size)
    # a few base-only tokens too
    pick2 = g.choice(w.n, size=max(1, w.n // 16), replace=False)
    ids[pick2] = -1
    return Workload(w.name + "_nf", w.dtype, w.n, ids.astype(np.int32), w.layers,
                    w.adapters + extra, recipe=w.recipe + "; plus raw normal-form adapters")


# small shapes spanning several tiles with ragged tails (parity cases)
SMALL_PROJ = {
    "q": (544, 1056, False),     # d_in 544 = 8.5 K-blocks of 64; d_out 1056 = 8.25 tiles of 128
    "k": (544, 288, True),
    "up": (544, 1312, True),
    "down": (1312, 544, False),
}


# --------------------------------------------------------------------------
# the same distributions drawn on a CUDA device (bench legs whose host-side
# draws would take minutes: the 32-layer stack, the 1024-adapter scaling
# batch).  Streams are keyed by (seed, name) as above, but the values are
# torch's, not NumPy's: these tensors feed timings, never a parity check.
# --------------------------------------------------------------------------
def _seed_int(seed, *names) -> int:
    h = hashlib.sha256(repr(("device", int(seed)) + tuple(names)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def device_normal(seed, name, shape, std, dtype, device, mean=0.0):
    """N(mean, std^2) drawn on ``device``; bf16 (round-to-nearest-even from
    float32) or float32."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_seed_int(seed, name))
    v = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    v.mul_(std)
    if mean:
        v.add_(mean)
    return v.to(torch.bfloat16) if dtype == "bf16" else v


def device_vector(seed, name, n, device, std=0.1):
    """1 + N(0, std^2), float32, on ``device``."""
    return device_normal(seed, name, (n,), std, "fp32", device, mean=1.0)


def device_cayley_blocks(seed, name, n_blk, dtype, device, std=0.05, blk=OFT_BLOCK):
    """Orthogonal blocks (I + S)(I - S)^-1, S skew with upper entries N(0, std),
    drawn and solved in float64 on ``device``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_seed_int(seed, name))
    up = torch.triu(torch.randn((n_blk, blk, blk), generator=g, device=device, dtype=torch.float64) * std, 1)
    S = up - up.transpose(1, 2)
    I = torch.eye(blk, device=device, dtype=torch.float64).expand(n_blk, blk, blk)
    R = torch.linalg.solve((I - S).transpose(1, 2), (I + S).transpose(1, 2)).transpose(1, 2)
    return R.to(torch.bfloat16 if dtype == "bf16" else torch.float32).contiguous()


def device_layer_tensors(seed, L: Layer, dtype: str, device) -> dict:
    """W [d_in, d_out] and the shared VeRA pair of one layer, on the device."""
    t = {"W": device_normal(seed, f"W/{L.name}", (L.d_in, L.d_out), 0.02, dtype, device)}
    if L.shared_rank:
        t["A_sh"] = device_normal(seed, f"Ash/{L.name}", (L.d_in, L.shared_rank), 0.02, dtype, device)
        t["B_sh"] = device_normal(seed, f"Bsh/{L.name}", (L.shared_rank, L.d_out), 0.02, dtype, device)
    return t


def device_adapter_tensors(seed, a: Adapter, layers: List[Layer], dtype: str, device,
                           vec_std=0.1) -> List[Tuple[str, dict]]:
    """One adapter's raw tensors on every layer it has, drawn on the device
    with the distributions of ``_make_adapter``."""
    out = []
    by_name = {L.name: L for L in layers}
    for lname in a.layers:
        L = by_name[lname]
        pre = f"ad{a.id}/{lname}"
        t = {}
        if a.method in ("lora", "dora"):
            t["A"] = device_normal(seed, pre + "/A", (L.d_in, a.rank), 0.02, dtype, device)
            t["B"] = device_normal(seed, pre + "/B", (a.rank, L.d_out), 0.02, dtype, device)
            if a.method == "dora":
                t["magnitude"] = device_vector(seed, pre + "/m", L.d_out, device, vec_std) * float(
                    0.02 * np.sqrt(L.d_in))
        elif a.method == "ia3":
            t["l"] = device_vector(seed, pre + "/l", L.d_out, device, vec_std)
        elif a.method == "vera":
            t["d"] = device_vector(seed, pre + "/d", L.shared_rank, device, vec_std)
            t["e"] = device_vector(seed, pre + "/e", L.d_out, device, vec_std)
        elif a.method == "oft":
            t["R"] = device_cayley_blocks(seed, pre + "/R", L.d_in // OFT_BLOCK, dtype, device)
        else:
            raise ValueError(a.method)
        out.append((lname, t))
    return out

