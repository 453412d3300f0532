"""Context-free token indexing that allocates nothing (scute_index_tokens_noalloc),
against the context's own indexing call (scute_debug_index) on the same ids.

Both run the same sorting kernel, so the comparison is bit for bit.  The file
is named to be collected last, so that it also runs after every other test has
used the device; it needs nothing from them and passes alone too."""
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
            torch.full((n,), -7, **i32), torch.full((22,), -7, **i32))


@pytest.mark.parametrize("sizes", [(300, 2049), (1, 64)])
def test_noalloc_matches_context_indexing_twice(setup, sizes):
    scute, ctx, methods, table = setup
    for call, n in enumerate(sizes):
        g = np.random.default_rng(1000 + n)
        # first call: unregistered ids included (flag set); second: none, so a
        # status word that was not cleared would show up as a stale flag
        ids = g.integers(-1, A if call == 0 else A - 2, n).astype(np.int32)
        if call == 0:
            ids[n // 2] = A - 1
        ids_t = torch.from_numpy(ids).cuda()
        ref = _outputs(n)
        ctx.debug_index(ids_t, n, *ref)
        got = _outputs(n)
        flags = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        scute.scute_index_tokens_noalloc(table, ids_t, n, *got, flags=flags)
        torch.cuda.synchronize()
        n_seg = int(ref[4][0].item())
        assert int(got[4][0].item()) == n_seg
        for a, b, k in zip(got, ref, (n, n, n_seg + 1, n_seg, 22)):
            np.testing.assert_array_equal(a.cpu().numpy()[:k], b.cpu().numpy()[:k])
        bad = IX.index_tokens(ids, methods, A).bad
        assert (int(flags.item()) != 0) == bool(bad)
        assert ctx.sync_status() == (5 if bad else 0)
        assert bad == (call == 0)


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
