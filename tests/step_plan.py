"""Host-side restatement of the decode step's launch plan and of the index
arithmetic its kernel derives from that plan, with a range check of every
index against the buffer it addresses (test infrastructure).

Written from reading ``csrc/api.cu`` (the plan: stream-K ranges, VeRA shrink
units, low-rank items, workspace sizes) and ``csrc/k_step.cu`` (per CTA: the
segments of its range, finisher / sharer roles, partial-tile slots, counter
indices, token-box and weight-box coordinates, epilogue vector accesses).  It
imports nothing from the library: the GPU test compares the plan restated here
with the one the library records for its launch (``scute_debug_step_plan``),
and the CPU test runs the range check over the bench and parity shapes.

The check covers what a bad address in the kernel could come from: an index
or a slot computed from the plan.  It does not cover values read at run time
(ids are restated through the segment counts they produce).
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

# constants of the kernel and its workspace (csrc/internal.h, csrc/k_step.cu)
STEP_MAX_CALLS = 8
STEP_MAX_TOKENS = 128
STEP_MAX_GRID = 190
STEP_MAX_VTILES = 8
STEP_SYNC_INTS = 1 << 16
SY_XS, SY_LR, SY_U, SY_EXIT, SY_ABORT, SY_VTILE, SY_TILE = 0, 8, 16, 24, 25, 32, 96
MAX_RANK = 64
ITEM_FEATURES_PER_BLOCK = 1152
TILE_M = 128
BOX_ROWS = 64
EPI_THREADS = 256
LR_Q = 8
TMEM_COLS = 512
SMEM_OPTIN_GB300 = 232448        # 227 KB opt-in per block


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def fixed_bytes() -> int:
    """sizeof the kernel's shared-memory Fixed block (natural alignment)."""
    off = 8 * (STEP_MAX_GRID + 1)                 # long long start[]
    off += 4 * 2 * STEP_MAX_TOKENS                # key, skey
    off += 4 * 3 * STEP_MAX_TOKENS                # perm, tok_aid, tok_seg
    off += 4 * (STEP_MAX_TOKENS + 1) + 4 * STEP_MAX_TOKENS   # seg_start, seg_aid
    off = ceil_div(off, 8) * 8
    off += 2 * 8 * STEP_MAX_CALLS * STEP_MAX_TOKENS          # segR, segA pointers
    off += 3 * STEP_MAX_CALLS * STEP_MAX_TOKENS              # segRank, oft_list, lr_list
    off += 4 * STEP_MAX_CALLS * (STEP_MAX_TOKENS // 32)      # oft_mask
    off = ceil_div(off, 8) * 8
    off += STEP_MAX_TOKENS * (5 * 8 + 2 * 4)                 # TokMeta: 5 pointers, 2 ints
    return ceil_div(off, 8) * 8


def step_smem_bytes(bn: int, stages: int, rmax: int) -> int:
    xb_floats = 2 * 32 * (TILE_M + 4)
    return 1024 + stages * (TILE_M * 128 + bn * 128) + 512 + fixed_bytes() + 4 * xb_floats


@dataclass
class LayerShape:
    """What the plan reads of a layer: shapes and registered-adapter counts."""
    d_in: int
    d_out: int
    rv: int = 0          # shared VeRA rank (0: no shared pair)
    n_lr: int = 0        # adapters with an owned low-rank term here
    n_vera: int = 0      # adapters with a VeRA term here
    n_rot: int = 0       # adapters with a rotation here
    lr_rmax: int = 0     # largest owned rank here


@dataclass
class Plan:
    head: Dict[str, int]
    calls: List[Dict[str, int]]
    start: List[int]
    flat: List[int] = field(default_factory=list)


HEAD_KEYS = ("n_calls", "n", "bn", "stages", "grid", "n_units", "vs_ch", "n_tiles", "n_items", "rmax",
             "t_main", "hold", "smem_bytes", "smem_optin", "part_floats", "xs_cols", "u_cols", "sync_ints",
             "pre_floats")
CALL_KEYS = ("blk0", "d_in", "kdim", "d_out", "krv", "rv", "kblocks", "vkb", "n_ft", "n_vt", "vs_chunks",
             "vs_unit0", "tile0", "lr_rmax", "lr_items", "lr_item0", "vs_x", "xs_direct")


def layer_shapes(w, names: Sequence[str]) -> List[LayerShape]:
    """Per-layer counts of a ``workloads.Workload`` as the library keeps them
    after registering every adapter (an adapter counts on a layer where it
    has tensors)."""
    out = []
    for name in names:
        L = w.layer(name)
        s = LayerShape(L.d_in, L.d_out, L.shared_rank)
        for a in w.adapters:
            if name not in a.layers:
                continue
            slots = set(a.slots(name))
            if a.method in ("lora", "dora") or (a.method == "nf" and "A" in slots):
                s.n_lr += 1
                s.lr_rmax = max(s.lr_rmax, a.rank)
            if a.method == "vera":
                s.n_vera += 1
            if "R" in slots:
                s.n_rot += 1
        out.append(s)
    return out


def workspace(all_layers: Sequence[LayerShape], max_tokens: int, grid: int) -> Dict[str, int]:
    """Decode workspace sizes a bf16 context reaches after adding these layers."""
    bn_max = 64 if max_tokens <= 64 else 128
    max_ft = max(ceil_div(L.d_out, 128) for L in all_layers)
    max_rank = max(L.lr_rmax for L in all_layers)
    pre = STEP_MAX_CALLS * ceil_div(max_rank, 8) * STEP_MAX_TOKENS * max(L.d_out for L in all_layers)
    return {"part_floats": (2 * grid + STEP_MAX_CALLS * max_ft) * 2 * 128 * bn_max,
            "pre_floats": pre if max_rank else 0,
            "xs_cols": max(L.d_in for L in all_layers),
            "u_cols": max([L.rv for L in all_layers if L.rv] or [0]),
            "bn_max": bn_max}


def plan(layers: Sequence[LayerShape], n: int, grid: int, ws: Dict[str, int],
         smem_optin: int = SMEM_OPTIN_GB300, oft_pass: bool = False, hold: int = 0) -> Plan:
    """The host plan of one decode launch (bf16, 1 <= n <= 128)."""
    assert 1 <= n <= STEP_MAX_TOKENS and 1 <= len(layers) <= STEP_MAX_CALLS
    G = min(grid, STEP_MAX_GRID)
    BN = 64 if n <= 64 else 128
    assert BN <= ws["bn_max"]
    calls = []
    blk = tile = 0
    rmax = 0
    for L in layers:
        vera_on = L.rv > 0 and L.n_vera > 0
        direct = (L.n_rot == 0 or oft_pass) and hold == 0
        k = {"d_in": L.d_in, "kdim": L.d_in, "d_out": L.d_out, "krv": L.rv, "rv": L.rv,
             "kblocks": ceil_div(L.d_in, 64), "vkb": ceil_div(L.rv, 64) if vera_on else 0,
             "n_ft": ceil_div(L.d_out, 128), "n_vt": ceil_div(L.rv, 128) if vera_on else 0,
             "lr_rmax": L.lr_rmax if L.n_lr > 0 else 0,
             "vs_x": 1 if vera_on else 0, "xs_direct": 1 if direct else 0, "n_lr": L.n_lr}
        rmax = max(rmax, k["lr_rmax"])
        k["blk0"] = blk
        blk += k["n_ft"] * (k["kblocks"] + k["vkb"])
        k["tile0"] = tile
        tile += k["n_ft"]
        calls.append(k)
    item = 0
    for k in calls:
        k["lr_items"] = min(k["n_lr"], n) * ceil_div(k["lr_rmax"], 8) if k["lr_rmax"] > 0 else 0
        k["lr_item0"] = item
        item += k["lr_items"]
    if sum(k["n_vt"] for k in calls) > G:
        raise ValueError("more VeRA shrink tiles than CTAs: the library rejects the launch")
    ch = 16
    while True:
        units = sum(k["n_vt"] * ceil_div(k["kblocks"], ch) for k in calls)
        if units <= G:
            break
        ch *= 2
    ublk, u, t_vs = [], 0, 0
    for k in calls:
        k["vs_chunks"] = ceil_div(k["kblocks"], ch)
        k["vs_unit0"] = u
        for _vt in range(k["n_vt"]):
            for cc in range(k["vs_chunks"]):
                b0 = cc * ch
                b1 = min(b0 + ch, k["kblocks"])
                ublk.append(b1 - b0)
                t_vs += b1 - b0
                u += 1
    # low-rank items are dealt with the calls of most work per item first
    # (d_in + d_out, ties in call order), item `it` to CTA G - 1 - it % G; each
    # charges (d_in + d_out) // ITEM_FEATURES_PER_BLOCK stream blocks against
    # its CTA (host bound of items per call)
    order = sorted(range(len(calls)), key=lambda i: (-(calls[i]["d_in"] + calls[i]["d_out"]), i))
    icost = [0] * G
    it = 0
    for i in order:
        k = calls[i]
        pen = (k["d_in"] + k["d_out"]) // ITEM_FEATURES_PER_BLOCK
        for _ in range(k["lr_items"]):
            icost[G - 1 - it % G] += pen
            it += 1
    W = blk + t_vs + sum(icost)
    start, vsb, mono = [], 0, True
    for i in range(G + 1):
        start.append(i * W // G - vsb)
        if i < units:
            vsb += ublk[i]
        if i < G:
            vsb += icost[i]
        if i > 0 and start[i] < start[i - 1]:
            mono = False
    if not mono or start[0] != 0 or start[G] != blk:
        start = [i * blk // G for i in range(G + 1)]
    S = 8
    while S > 2 and step_smem_bytes(BN, S, rmax) > smem_optin:
        S -= 1
    head = {"n_calls": len(calls), "n": n, "bn": BN, "stages": S, "grid": G, "n_units": units, "vs_ch": ch,
            "n_tiles": tile, "n_items": item, "rmax": rmax, "t_main": blk, "hold": hold,
            "smem_bytes": step_smem_bytes(BN, S, rmax), "smem_optin": smem_optin,
            "part_floats": ws["part_floats"], "xs_cols": ws["xs_cols"], "u_cols": ws["u_cols"],
            "sync_ints": STEP_SYNC_INTS, "pre_floats": ws["pre_floats"]}
    flat = [head[key] for key in HEAD_KEYS]
    for k in calls:
        flat += [k[key] for key in CALL_KEYS]
    flat += start
    return Plan(head, calls, start, flat)


def parse(flat: Sequence[int]) -> Plan:
    """A recorded plan (scute_debug_step_plan's layout) as a Plan."""
    head = dict(zip(HEAD_KEYS, flat[:len(HEAD_KEYS)]))
    off = len(HEAD_KEYS)
    calls = []
    for _ in range(head["n_calls"]):
        calls.append(dict(zip(CALL_KEYS, flat[off:off + len(CALL_KEYS)])))
        off += len(CALL_KEYS)
    start = list(flat[off:off + head["grid"] + 1])
    return Plan(head, calls, start, list(flat))


# ------------------------------------------------------------------ the kernel's arithmetic
def mlocate(p: Plan, b: int):
    """(call, tile, kb, nkb, tb0) of stream block b (k_step.cu mlocate)."""
    c = 0
    while c + 1 < len(p.calls) and p.calls[c + 1]["blk0"] <= b:
        c += 1
    k = p.calls[c]
    mpt = k["kblocks"] + k["vkb"]
    l = b - k["blk0"]
    tile = l // mpt
    return c, tile, l - tile * mpt, mpt, k["blk0"] + tile * mpt


def ulocate(p: Plan, u: int):
    """(call, VeRA tile, kb0, kb1) of VeRA shrink unit u (k_step.cu ulocate)."""
    c = 0
    while c + 1 < len(p.calls) and p.calls[c + 1]["vs_unit0"] <= u:
        c += 1
    k = p.calls[c]
    l = u - k["vs_unit0"]
    vt = l // k["vs_chunks"]
    ch = l - vt * k["vs_chunks"]
    kb0 = ch * p.head["vs_ch"]
    return c, vt, kb0, min(k["kblocks"], kb0 + p.head["vs_ch"])


def owner(p: Plan, b: int) -> int:
    """The CTA whose range holds main block b (binary search as in the kernel)."""
    lo, hi = 0, p.head["grid"] - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if p.start[mid] <= b:
            lo = mid
        else:
            hi = mid - 1
    return lo


class AuditError(AssertionError):
    pass


def _need(cond: bool, what: str):
    if not cond:
        raise AuditError(what)


def audit(p: Plan, n_seg_lr: Optional[Sequence[int]] = None) -> Dict[str, int]:
    """Check every plan-derived index of one launch against its buffer.
    n_seg_lr: per call, the number of adapter segments with an owned term
    that the batch's ids form (data-dependent; None skips that check).
    Returns the largest value each index reached (for the report)."""
    h, C = p.head, p.calls
    G, BN, n = h["grid"], h["bn"], h["n"]
    slot_floats = 2 * TILE_M * BN
    part_slots = h["part_floats"] // slot_floats
    mx: Dict[str, int] = {}

    def note(key, v):
        mx[key] = max(mx.get(key, -1), v)

    # launch shape
    _need(1 <= G <= STEP_MAX_GRID, "grid")
    _need(n <= BN <= STEP_MAX_TOKENS, "tokens per tile")
    nb = 4 if BN <= 64 else 2
    _need(2 * nb * BN <= TMEM_COLS, "TMEM columns (buffers x 2 accumulators x BN)")
    _need(h["smem_bytes"] <= h["smem_optin"], "shared memory")
    _need(2 <= h["stages"] <= 8, "stages")
    _need(h["n_units"] <= G, "at most one VeRA unit per CTA")
    _need(len(C) <= STEP_MAX_CALLS, "calls")
    # workspace capacity (the host's own check, restated)
    _need(h["n_units"] + h["n_tiles"] + G <= part_slots, "partial-tile slots")
    _need(SY_TILE + h["n_tiles"] <= h["sync_ints"], "tile counters")
    # stream-K ranges partition the main blocks
    _need(p.start[0] == 0 and p.start[G] == h["t_main"], "range ends")
    _need(all(p.start[i] <= p.start[i + 1] for i in range(G)), "ranges monotone")
    for c, k in enumerate(C):
        _need(k["kdim"] <= h["xs_cols"] or k["xs_direct"], f"call {c}: token-operand slot pitch")
        _need(k["n_vt"] <= STEP_MAX_VTILES, f"call {c}: VeRA tiles")
        _need(k["vkb"] == 0 or k["krv"] <= h["u_cols"], f"call {c}: VeRA intermediate pitch")
        _need(k["lr_rmax"] <= h["rmax"] <= MAX_RANK, f"call {c}: owned rank")
        _need(k["d_out"] % 32 == 0 and k["d_in"] % 32 == 0 and k["krv"] % 32 == 0, f"call {c}: multiples of 32")
        if k["lr_rmax"] > 0:
            # the low-rank rows: planes [ceil(r / 8)][128][d_out] inside the call's slot
            _need(ceil_div(k["lr_rmax"], LR_Q) * STEP_MAX_TOKENS * k["d_out"] <= h["pre_floats"] // STEP_MAX_CALLS,
                  f"call {c}: low-rank row slot")
            note("pre_plane_end", ceil_div(k["lr_rmax"], LR_Q) * STEP_MAX_TOKENS * k["d_out"])
        if n_seg_lr is not None:
            ng = ceil_div(k["lr_rmax"], LR_Q) if k["lr_rmax"] else 0
            _need(n_seg_lr[c] * ng <= k["lr_items"], f"call {c}: low-rank items cover the segments")
    # low-rank items: every item id belongs to exactly one call
    covered = sorted((k["lr_item0"], k["lr_item0"] + k["lr_items"]) for k in C)
    pos = 0
    for a0, a1 in covered:
        _need(a0 == pos, "low-rank item ranges contiguous")
        pos = a1
    _need(pos == h["n_items"], "low-rank items")
    # VeRA shrink units: each (call, tile) has vs_chunks units, all in range
    per_tile: Dict[tuple, int] = {}
    for u in range(h["n_units"]):
        c, vt, kb0, kb1 = ulocate(p, u)
        k = C[c]
        _need(0 <= vt < k["n_vt"] and 0 <= kb0 < kb1 <= k["kblocks"], f"unit {u}")
        _need((kb1 - 1) * 64 < k["kdim"] and (vt + 1) * TILE_M <= max(k["rv"], TILE_M) + TILE_M - 1, f"unit {u} boxes")
        _need(u < part_slots, f"unit {u} slot")
        idx = SY_VTILE + c * STEP_MAX_VTILES + vt
        _need(SY_VTILE <= idx < SY_TILE, f"unit {u} counter")
        per_tile[(c, vt)] = per_tile.get((c, vt), 0) + 1
        note("unit_slot", u)
        u0 = k["vs_unit0"] + vt * k["vs_chunks"]
        _need(u0 + k["vs_chunks"] <= h["n_units"], f"unit {u}: the tile's partial slots")
    for (c, vt), cnt in per_tile.items():
        _need(cnt == C[c]["vs_chunks"], f"VeRA tile ({c},{vt}) arrivals")
    # per CTA: segments, roles, slots, counters, boxes
    publishers: Dict[int, set] = {}
    expected: Dict[int, set] = {}
    for me in range(G):
        ms, mend = p.start[me], p.start[me + 1]
        b = ms
        first = True
        while b < mend:
            c, tl, kb, nkb, tb0 = mlocate(p, b)
            k = C[c]
            se = min(mend, tb0 + nkb)
            _need(0 <= tl < k["n_ft"] and 0 <= kb < nkb, f"CTA {me}: block {b}")
            for bb in range(b, se):
                kk = kb + (bb - b)
                if kk < k["kblocks"]:
                    _need(kk * 64 < k["kdim"], f"CTA {me}: main box")
                else:
                    _need((kk - k["kblocks"]) * 64 < k["krv"], f"CTA {me}: VeRA expand box")
            _need(tl * TILE_M < k["d_out"], f"CTA {me}: weight rows")
            gtile = k["tile0"] + tl
            _need(SY_TILE + gtile < h["sync_ints"], f"CTA {me}: tile counter")
            own = h["n_units"] + gtile + me
            _need(own < part_slots, f"CTA {me}: own slot")
            note("own_slot", own)
            fin = b == tb0
            if not fin:
                _need(first, f"CTA {me}: only a range's first segment can start inside a tile")
                publishers.setdefault(gtile, set()).add(me)
            else:
                lastc = owner(p, tb0 + nkb - 1)
                _need(me <= lastc < G, f"CTA {me}: last sharer")
                others = {j for j in range(me + 1, lastc + 1) if p.start[j + 1] > p.start[j]}
                expected[gtile] = others
                for j in others:
                    _need(h["n_units"] + gtile + j < part_slots, f"CTA {me}: sharer slot")
                    lo, hi = max(tb0, p.start[j]), min(tb0 + nkb, p.start[j + 1])
                    # the planes the finisher reads are the ones the sharer writes
                    sh_base = p.start[j] - tb0 < k["kblocks"]
                    sh_v = k["vkb"] > 0 and min(p.start[j + 1], tb0 + nkb) - tb0 > k["kblocks"]
                    _need((lo - tb0 < k["kblocks"]) == sh_base, f"CTA {me}: base plane of sharer {j}")
                    _need((k["vkb"] > 0 and hi - tb0 > k["kblocks"]) == sh_v, f"CTA {me}: VeRA plane of sharer {j}")
                    note("sharer_slot", h["n_units"] + gtile + j)
            # epilogue vectors: 8 consecutive features, starting at a multiple of 8
            for g in range(16):
                j0 = tl * TILE_M + g * 8
                if j0 < k["d_out"]:
                    _need(j0 + 8 <= k["d_out"], f"CTA {me}: epilogue vector")
            b = se
            first = False
    for gtile, pubs in publishers.items():
        _need(expected.get(gtile) == pubs, f"tile {gtile}: sharers {sorted(pubs)} vs awaited {sorted(expected.get(gtile, []))}")
    for gtile, exp in expected.items():
        _need(publishers.get(gtile, set()) == exp, f"tile {gtile}: awaited sharers that never publish")
    # token rows and the per-token workspace
    _need(n <= STEP_MAX_TOKENS, "token rows of the call slots")
    note("tokens", n)
    return mx


def seg_lr_counts(w, names: Sequence[str], ids) -> List[int]:
    """Per layer, the adapter segments with an owned term the ids form."""
    out = []
    used = {int(i) for i in ids if i >= 0}
    for name in names:
        cnt = 0
        for a in w.adapters:
            if a.id in used and name in a.layers:
                sl = set(a.slots(name))
                if a.method in ("lora", "dora") or (a.method == "nf" and "A" in sl):
                    cnt += 1
        out.append(cnt)
    return out
