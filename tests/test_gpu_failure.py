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
