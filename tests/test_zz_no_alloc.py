"""Context-free token indexing that allocates nothing
(scute_index_tokens_noalloc), graded directly against the oracle's indexing
(a stable sort by (method, adapter id)) bit for bit, and against the context's
own indexing call (scute_debug_index) on the same ids.

Who needs the entry point: callers that cannot allocate device memory, such as
a scheduler that shares the GPU with an engine whose memory pool already holds
most of HBM, or latency-critical code where cudaMalloc may synchronise.  The
tests check the property it is named for too: after a first call, further
calls change neither the device's free memory nor torch's allocations.

The file is named to be collected last, so that it also runs after every other
test has used the device; it needs nothing from them and passes alone too."""
import numpy as np
import pytest

import workloads as WL
from oracle import indexing as IX

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

A = 40   # ids 0..A-3 registered, A-2 and A-1 left free


@pytest.fixture(scope="module")
def setup(gpu_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    scute = gpu_lib
    ctx = scute.Context(dtype="bf16", max_tokens=4096, max_adapters=A, max_layers=1)
    ctx.add_layer(0, 64, 64, WL.draw_normal(0, "Wna", (64, 64), 0.02, "bf16"))
    ctx.set_shared(0, 32, WL.draw_normal(0, "Ana", (64, 32), 0.02, "bf16"),
                   WL.draw_normal(0, "Bna", (32, 64), 0.02, "bf16"))
    order = ["lora", "vera", "ia3", "oft", "nf", "dora"]
    methods = {}
    for i in range(A - 2):
        m = order[(i * 5 + 1) % 6]
        t = {"layer": 0}
        if m in ("lora", "dora"):
            t.update(rank=2, c=1.0, A=WL.draw_normal(i, "na", (64, 2), 0.02, "bf16"),
                     B=WL.draw_normal(i, "nb", (2, 64), 0.02, "bf16"))
            if m == "dora":
                t["magnitude"] = np.ones(64, np.float32)
        elif m == "ia3":
            t["l"] = np.ones(64, np.float32)
        elif m == "vera":
            t["d"] = np.ones(32, np.float32)
        elif m == "oft":
            t["R"] = WL.draw_cayley_blocks(i, "nr", 2, "bf16")
        else:
            t["s"] = np.ones(64, np.float32)
        assert ctx.register(m, [t]) == i
        methods[i] = m
    table = np.full(A, -1, np.int8)
    for i, m in methods.items():
        table[i] = scute.METHOD_ID[m]
    yield scute, ctx, methods, table
    ctx.close()


def _outputs(n):
    i32 = dict(dtype=torch.int32, device="cuda")
    return (torch.full((n,), -7, **i32), torch.full((n,), -7, **i32), torch.full((n + 1,), -7, **i32),
            torch.full((max(n, 1),), -7, **i32), torch.full((22,), -7, **i32))


def _assert_matches_oracle(got, ids, methods):
    """The entry point's arrays against the oracle's stable sort, bit for bit."""
    n = ids.size
    ref = IX.index_tokens(ids, methods, A)
    perm, aid, seg_start, seg_aid, counts = (t.cpu().numpy() for t in got)
    n_seg = int(counts[0])
    assert n_seg == len(ref.seg_aid)
    np.testing.assert_array_equal(perm[:n], ref.perm)
    np.testing.assert_array_equal(aid[:n], ref.aid_sorted)
    np.testing.assert_array_equal(seg_start[:n_seg + 1], ref.seg_start)
    np.testing.assert_array_equal(seg_aid[:n_seg], ref.seg_aid)
    np.testing.assert_array_equal(counts[1:8], ref.count)
    np.testing.assert_array_equal(counts[8:15], ref.offset)
    return ref


@pytest.mark.parametrize("sizes", [(300, 2049), (1, 64)])
def test_noalloc_matches_oracle_and_context_twice(setup, sizes):
    """Two calls in a row: the first with unregistered ids (flag set), the
    second without, so a status word that was not cleared between calls would
    show as a stale flag.  Each is graded against the oracle and against the
    context's indexing call."""
    scute, ctx, methods, table = setup
    for call, n in enumerate(sizes):
        g = np.random.default_rng(1000 + n)
        ids = g.integers(-1, A if call == 0 else A - 2, n).astype(np.int32)
        if call == 0:
            ids[n // 2] = A - 1
        ids_t = torch.from_numpy(ids).cuda()
        got = _outputs(n)
        flags = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        scute.scute_index_tokens_noalloc(table, ids_t, n, *got, flags=flags)
        torch.cuda.synchronize()
        ref = _assert_matches_oracle(got, ids, methods)
        assert (int(flags.item()) != 0) == bool(ref.bad)
        assert bool(ref.bad) == (call == 0)
        # and the context's own indexing call agrees with it
        ctxo = _outputs(n)
        ctx.debug_index(ids_t, n, *ctxo)
        torch.cuda.synchronize()
        n_seg = int(ctxo[4][0].item())
        for a, b, k in zip(got, ctxo, (n, n, n_seg + 1, n_seg, 22)):
            np.testing.assert_array_equal(a.cpu().numpy()[:k], b.cpu().numpy()[:k])
        assert ctx.sync_status() == (5 if ref.bad else 0)


def test_noalloc_allocates_nothing_on_a_side_stream(setup):
    """After a first call, further calls (on a non-default stream, of
    several sizes, n = 0 included) leave the device's free memory and torch's
    allocations unchanged; results are still the oracle's."""
    scute, _, methods, table = setup
    g = np.random.default_rng(7)
    cases = [g.integers(-1, A - 2, n).astype(np.int32) for n in (513, 0, 4096, 1)]
    bufs = [(torch.from_numpy(ids).cuda(), _outputs(ids.size)) for ids in cases]
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    # first call: may load the library's module and look up the scratch array
    with torch.cuda.stream(s):
        scute.scute_index_tokens_noalloc(table, bufs[0][0], cases[0].size, *bufs[0][1], flags=flags,
                                         stream=s)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for rep in range(2):
        for ids, (ids_t, out) in zip(cases, bufs):
            with torch.cuda.stream(s):
                scute.scute_index_tokens_noalloc(table, ids_t, ids.size, *out, flags=flags, stream=s)
            s.synchronize()
            assert int(flags.item()) == 0
            if ids.size == 0:
                c = out[4].cpu().numpy()
                assert int(out[2][0].item()) == 0 and c[0] == 0 and (c[1:] == 0).all()
            else:
                _assert_matches_oracle(out, ids, methods)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"


def test_noalloc_rejects_sizes_beyond_its_limits(setup):
    scute, _, _, table = setup
    n = 8
    ids_t = torch.zeros(n, dtype=torch.int32, device="cuda")
    out = _outputs(n)
    with pytest.raises(scute.ScuteError) as e:
        scute.scute_index_tokens_noalloc(np.zeros(scute.NOALLOC_MAX_ADAPTERS + 1, np.int8), ids_t, n, *out)
    assert e.value.code == 8
    with pytest.raises(scute.ScuteError) as e:
        scute.scute_index_tokens_noalloc(table, ids_t, scute.MAX_TOKENS + 1, *out)
    assert e.value.code == 8
    bad_tab = table.copy()
    bad_tab[0] = 6
    with pytest.raises(scute.ScuteError) as e:
        scute.scute_index_tokens_noalloc(bad_tab, ids_t, n, *out)
    assert e.value.code == 1
    torch.cuda.synchronize()
    assert (out[4].cpu().numpy() == -7).all()   # nothing was launched
