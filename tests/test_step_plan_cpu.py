"""The decode step's plan-derived index arithmetic, restated on the host
(``step_plan``) and range-checked for the bench and parity shapes, at the
GB300's 152 CTAs and at other grid sizes.  No GPU: the restatement follows
the kernel source; ``test_gpu_parity.py::test_step_plan_matches_restatement``
ties it to the library's own plan."""
import numpy as np
import pytest

import step_plan as SP
import workloads as WL

SMALL = tuple(WL.SMALL_PROJ)


def _shapes_decode(n=64, ids=None):
    w = WL.decode_mixed(n=n, ids=ids)
    names = ("q", "k", "v", "gate", "up", "down")
    return w, names, SP.layer_shapes(w, names)


def _shapes_stack():
    # the stack's per-projection counts: every layer repeats the same shapes
    # and adapters, so one block of seven projections stands for all 32
    w = WL.stack_32layer(n_layers=1)
    names = tuple(L.name for L in w.layers)
    return w, names, SP.layer_shapes(w, names)


@pytest.mark.parametrize("grid", [152, 148, 132, 160, 190, 64, 12])
def test_decode_batch_plan_in_range(grid):
    """The bench step: six Llama-3-8B projections, 64 tokens, one launch."""
    w, names, shapes = _shapes_decode()
    ws = SP.workspace(shapes, 64, grid)
    p = SP.plan(shapes, 64, grid, ws)
    mx = SP.audit(p, SP.seg_lr_counts(w, names, w.ids))
    assert mx["own_slot"] < SP.ceil_div(p.head["part_floats"], 2 * 128 * p.head["bn"])
    if grid == 152:
        # the bench launch: one VeRA unit per CTA for 48 of them, 6 stages
        assert p.head["stages"] == 6 and p.head["n_units"] <= grid and p.head["bn"] == 64


@pytest.mark.parametrize("group", [("L0.q", "L0.k", "L0.v"), ("L0.o",), ("L0.gate", "L0.up"), ("L0.down",),
                                   ("L0.q", "L0.k", "L0.v", "L0.o", "L0.gate", "L0.up", "L0.down")])
@pytest.mark.parametrize("grid", [152, 132])
def test_stack_block_plans_in_range(group, grid):
    """The 32-layer stack's launches: 128 tokens (two token boxes per stage),
    the block groups a transformer block's dependencies allow, and all seven
    projections of a layer in one launch."""
    w, names, shapes = _shapes_stack()
    ws = SP.workspace(shapes, 128, grid)
    sel = [shapes[names.index(g)] for g in group]
    p = SP.plan(sel, 128, grid, ws)
    assert p.head["bn"] == 128
    SP.audit(p, SP.seg_lr_counts(w, list(group), w.ids))


@pytest.mark.parametrize("n", [1, 2, 50, 64, 65, 128])
@pytest.mark.parametrize("grid", [152, 16])
def test_parity_shape_plans_in_range(n, grid):
    """The small parity shapes (ragged K blocks and feature tiles), every
    layer in one launch plus a repeated layer, at several token counts."""
    w = WL.decode_mixed(n=n, shapes=WL.SMALL_PROJ, proj=SMALL)
    if n > 1:
        w = WL.with_nf_adapters(w)
    names = list(SMALL) + ["q"]
    shapes = SP.layer_shapes(w, names)
    ws = SP.workspace(shapes, 128, grid)
    p = SP.plan(shapes, n, grid, ws)
    SP.audit(p, SP.seg_lr_counts(w, names, w.ids))


def test_more_vera_tiles_than_ctas_is_rejected():
    """Six calls with a rank-256 shared pair have 12 VeRA shrink tiles; a grid
    of fewer CTAs cannot give each at most one unit (the kernel's bound), so
    the launch is refused rather than planned."""
    w, names, shapes = _shapes_decode()
    with pytest.raises(ValueError):
        SP.plan(shapes, 64, 11, SP.workspace(shapes, 64, 11))


def test_rank64_and_oft_pass_plans_in_range():
    """Rank-64 owned terms (eight rank groups, eight planes of rows) and the
    separate rotation pass (every call reads its rotated copy directly)."""
    w = WL.decode_mixed(n=64, rank=64)
    names = ("q", "k", "v", "gate", "up", "down")
    shapes = SP.layer_shapes(w, names)
    ws = SP.workspace(shapes, 64, 152)
    for oft_pass in (False, True):
        p = SP.plan(shapes, 64, 152, ws, oft_pass=oft_pass)
        SP.audit(p, SP.seg_lr_counts(w, names, w.ids))
        assert all(k["xs_direct"] == (1 if oft_pass else 0) for k in p.calls)


def test_audit_catches_planted_faults():
    """The audit is not vacuous: a plan with one index pushed out of its
    buffer, or with a sharer that never publishes, fails it."""
    w, names, shapes = _shapes_decode()
    ws = SP.workspace(shapes, 64, 152)
    base = SP.plan(shapes, 64, 152, ws)
    SP.audit(base)

    def mutated(fn):
        p = SP.plan(shapes, 64, 152, ws)
        fn(p)
        return p

    cases = [
        lambda p: p.head.__setitem__("part_floats", (p.head["n_tiles"] + p.head["grid"]) * 2 * 128 * 64),
        lambda p: p.head.__setitem__("pre_floats", 8 * 2 * 128 * 4096),
        lambda p: p.calls[0].__setitem__("vs_chunks", p.calls[0]["vs_chunks"] + 1),
        lambda p: p.start.__setitem__(5, p.start[6] + 10),          # ranges overlap
        lambda p: p.start.__setitem__(p.head["grid"], p.start[-1] - 1),   # the last block has no CTA
        lambda p: p.calls[1].__setitem__("lr_items", 0),
        lambda p: p.head.__setitem__("smem_optin", 100 * 1024),
        lambda p: p.calls[2].__setitem__("n_vt", SP.STEP_MAX_VTILES + 1),
    ]
    for i, fn in enumerate(cases):
        with pytest.raises(AssertionError):
            SP.audit(mutated(fn), SP.seg_lr_counts(w, names, w.ids))


def test_stream_k_ranges_cover_every_block_once():
    """Every main K block of the step belongs to exactly one CTA, and each
    tile has one finisher (the CTA holding its first block)."""
    w, names, shapes = _shapes_decode()
    p = SP.plan(shapes, 64, 152, SP.workspace(shapes, 64, 152))
    owner = np.full(p.head["t_main"], -1)
    for me in range(152):
        assert (owner[p.start[me]:p.start[me + 1]] == -1).all()
        owner[p.start[me]:p.start[me + 1]] = me
    assert (owner >= 0).all()
    for b in range(0, p.head["t_main"], 97):
        assert SP.owner(p, b) == owner[b]


def _lowrank_ks(d_in):
    # the K chunks of the low-rank shrink (csrc/internal.h lowrank_ks)
    ks = min(-(-d_in // 2048), 8)
    kchunk = -(-(-(-d_in // ks)) // 256) * 256
    return -(-d_in // kchunk), kchunk


def test_k_chunks_are_never_empty():
    """Every K chunk of the tensor-core shrinks holds at least one K block, for
    every input width the library accepts (a chunk with none would hand its
    partial an accumulator no MMA wrote): the low-rank shrink's chunks and the
    VeRA shrink's (at most 4)."""
    for d_in in range(32, 16384 + 1, 32):
        kblocks = -(-d_in // 64)
        ks, kchunk = _lowrank_ks(d_in)
        cb = kchunk // 64
        assert ks <= 8 and kchunk % 256 == 0 and (ks - 1) * cb < kblocks, d_in
        vcb = -(-kblocks // 4)
        vks = -(-kblocks // vcb)
        assert vks <= 4 and (vks - 1) * vcb < kblocks <= vks * vcb, d_in
