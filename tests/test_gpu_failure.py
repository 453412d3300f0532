"""Failure path of the decode step, made on purpose and without any GPU fault:
a launch whose token-operand wait can never be met (test hook
scute_debug_inject) must give up within its bounded waits, report
SCUTE_ERR_TIMEOUT through scute_sync_status, and leave the context able to
serve the next call correctly."""
import time

import pytest

import workloads as WL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import gpu_harness as H  # noqa: E402


@pytest.fixture(scope="module")
def scute(gpu_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gpu_lib


def test_stalled_launch_times_out_and_context_recovers(scute):
    w = WL.with_nf_adapters(WL.decode_mixed(n=50, shapes=WL.SMALL_PROJ, proj=("q", "up")))
    ctx = H.make_ctx(scute, w)
    scute.scute_debug_inject(ctx.handle, scute.INJECT_STALL)
    t0 = time.time()
    H.run_layers(ctx, w, ["q"], "fp32")          # synchronises the device
    waited = time.time() - t0
    assert ctx.sync_status() == 7                # SCUTE_ERR_TIMEOUT
    assert 0.5 < waited < 60.0
    # the hook applied to that launch only; counters and status are clean again
    outs = H.run_layers(ctx, w, ["q", "up"], "fp32")
    assert ctx.sync_status() == 0
    for name in ("q", "up"):
        H.grade(w, name, outs[name], "fp32")
    ctx.close()


def test_inject_rejects_unknown_kinds(scute):
    w = WL.decode_mixed(n=8, shapes=WL.SMALL_PROJ, proj=("q",), n_adapters=5)
    ctx = H.make_ctx(scute, w)
    with pytest.raises(scute.ScuteError):
        scute.scute_debug_inject(ctx.handle, 99)
    ctx.close()


def _tiny_layer():
    W = WL.draw_normal(0, "Woom", (64, 96), 0.02, "bf16")
    A = WL.draw_normal(0, "Aoom", (64, 32), 0.02, "bf16")
    B = WL.draw_normal(0, "Boom", (32, 96), 0.02, "bf16")
    return W, A, B


def test_injected_allocation_failures_return_oom(scute):
    """Every device allocation of context creation, layer setup and
    registration is made to fail in turn (host-side hook, no GPU fault): the
    call returns SCUTE_ERR_OOM and the context stays usable; a retry without
    the failure succeeds and the layer then computes the right result."""
    W, A_sh, B_sh = _tiny_layer()
    try:
        # scute_create: its k-th allocation fails until k passes its count
        k = 1
        while True:
            scute.scute_debug_fail_alloc(k)
            try:
                ctx = scute.Context("bf16", max_tokens=64, max_adapters=8, max_layers=2)
            except scute.ScuteError as e:
                assert e.code == 4, e
                k += 1
                assert k < 64
                continue
            break
        n_create = k - 1
        assert n_create >= 10          # creation makes a dozen or more allocations
        scute.scute_debug_fail_alloc(0)
        ctx.close()

        ctx = scute.Context("bf16", max_tokens=64, max_adapters=8, max_layers=2)
        # scute_add_layer: fail each of its allocations, then succeed
        k = 1
        while True:
            scute.scute_debug_fail_alloc(k)
            try:
                ctx.add_layer(0, 64, 96, W)
            except scute.ScuteError as e:
                assert e.code == 4, e
                k += 1
                assert k < 32
                continue
            break
        assert k > 1
        scute.scute_debug_fail_alloc(0)
        # scute_set_shared: the pair and the VeRA intermediates
        k = 1
        while True:
            scute.scute_debug_fail_alloc(k)
            try:
                ctx.set_shared(0, 32, A_sh, B_sh)
            except scute.ScuteError as e:
                assert e.code == 4, e
                k += 1
                assert k < 32
                continue
            break
        assert k > 1
        scute.scute_debug_fail_alloc(0)
        # registration: the adapter's storage; the id is not consumed
        scute.scute_debug_fail_alloc(1)
        l = WL.draw_vector(0, "loom", 96)
        with pytest.raises(scute.ScuteError) as e:
            ctx.register("ia3", [{"layer": 0, "l": l}])
        assert e.value.code == 4
        scute.scute_debug_fail_alloc(0)
        aid = ctx.register("ia3", [{"layer": 0, "l": l}])
        assert aid == 0
        d = WL.draw_vector(0, "doom", 32)
        e_ = WL.draw_vector(0, "eoom", 96)
        assert ctx.register("vera", [{"layer": 0, "d": d, "e": e_, "c": 1.0}]) == 1
    finally:
        scute.scute_debug_fail_alloc(0)
    # the context computes the right result after all the failed calls
    import numpy as np
    from workloads import to_f64
    n = 24
    x = WL.draw_normal(0, "xoom", (n, 64), 1.0, "bf16")
    ids = np.array([0, 1, -1] * 8, np.int32)
    out = torch.empty(n, 96, device="cuda", dtype=torch.float32)
    ctx.linear(H.dev(x), torch.from_numpy(ids).cuda(), 0, out, "fp32")
    torch.cuda.synchronize()
    assert ctx.sync_status() == 0
    from oracle import methods as M
    xf, Wf = to_f64(x), to_f64(W)
    ref = M.base(xf, Wf)
    ref[ids == 0] = M.ia3(xf[ids == 0], Wf, l.astype(np.float64))
    ref[ids == 1] = M.vera(xf[ids == 1], Wf, to_f64(A_sh), to_f64(B_sh), d.astype(np.float64),
                           e_.astype(np.float64))
    g = out.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(g - ref)) <= 1e-3 * np.max(np.abs(ref)) + 1e-4
    ctx.close()
