"""Token -> segment indexing for a heterogeneous batch.

Test infrastructure only (see ``oracle/__init__``).

The article's batched kernels work per adapter segment ("The big picture":
the shrink and expand run per adapter segment; "Where is the cheapest place to
compute the remaining slots?": each tile belongs to one adapter).  The reading
used here: tokens are ordered by the key (method, adapter id), ties kept in
token order (a stable sort); a segment is a maximal run of one key.  Method
order is LoRA < DoRA < (IA)^3 < VeRA < OFT < raw normal form, and base-only
tokens (id -1, or an id that names no registered adapter) come last.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

METHOD_RANK = {"lora": 0, "dora": 1, "ia3": 2, "vera": 3, "oft": 4, "nf": 5}
BASE_RANK = 6
N_RANKS = 7


@dataclass
class Index:
    perm: np.ndarray          # int32 [n]: sorted position -> token
    aid_sorted: np.ndarray    # int32 [n]: adapter of each sorted row, -1 base
    seg_start: np.ndarray     # int32 [n_seg + 1]
    seg_aid: np.ndarray       # int32 [n_seg]
    count: np.ndarray         # int32 [7]: rows per method rank (base last)
    offset: np.ndarray        # int32 [7]: first sorted row of each method rank
    bad: bool                 # some id named no registered adapter


def sort_keys(ids: np.ndarray, method_of: dict, max_adapters: int):
    """Key of every token: rank(method) * max_adapters + id, base last."""
    ids = np.asarray(ids, dtype=np.int64)
    key = np.empty(ids.shape, dtype=np.int64)
    valid = np.zeros(ids.shape, dtype=bool)
    bad = False
    for t, a in enumerate(ids):
        if 0 <= a < max_adapters and int(a) in method_of:
            key[t] = METHOD_RANK[method_of[int(a)]] * max_adapters + a
            valid[t] = True
        else:
            key[t] = BASE_RANK * max_adapters
            if a != -1:
                bad = True
    return key, valid, bad


def index_tokens(ids: np.ndarray, method_of: dict, max_adapters: int) -> Index:
    key, valid, bad = sort_keys(ids, method_of, max_adapters)
    n = key.size
    perm = np.argsort(key, kind="stable").astype(np.int32)
    ks = key[perm]
    aid_sorted = np.where(valid[perm], np.asarray(ids)[perm], -1).astype(np.int32)
    starts = [i for i in range(n) if i == 0 or ks[i] != ks[i - 1]]
    seg_start = np.array(starts + [n], dtype=np.int32)
    seg_aid = aid_sorted[np.array(starts, dtype=np.int64)] if starts else np.zeros(0, np.int32)
    rank = ks // max_adapters
    count = np.array([int(np.sum(rank == r)) for r in range(N_RANKS)], dtype=np.int32)
    offset = np.concatenate([[0], np.cumsum(count)[:-1]]).astype(np.int32)
    return Index(perm, aid_sorted, seg_start, seg_aid.astype(np.int32), count, offset, bad)
