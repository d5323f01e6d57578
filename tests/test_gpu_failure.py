"""The failure path of the bounded device waits, made to run out on purpose.

A self-test kernel waits on a barrier that nothing completes: the short wait
gives up, flags the workspace status and aborts the other waiter.  The host
reads MOE_ERR_TIMEOUT, and the same context and workspace then run a normal
layer call correctly.  Nothing faults or hangs.
"""
import pytest
import torch

import oracle
from _layers import assert_layer_close, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    shape = synth.tiny(M=8)
    d = synth.make_layer(shape, seed=3)
    ws = gbmoe.alloc_workspace(8, shape.H, shape.I, shape.E, shape.topk, gbmoe.MOE_WEIGHT_FP8)
    gave_up = gbmoe.moe_selftest_wait_timeout(ws, limit_cycles=2_000_000)  # about a millisecond
    bad, flags, st = gbmoe.moe_read_status(ws)
    assert st == 5 and flags == 1 and bad == 0       # MOE_ERR_TIMEOUT
    assert int(gave_up.item()) == 2                   # the short wait and the one it aborted
    # the next layer call on the same workspace clears the status and computes normally
    dd = to_device(d)
    out = gbmoe.fused_moe_fp8(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"], dd["w2"],
                              dd["w2_scale"], workspace=ws)
    torch.cuda.synchronize()
    bad, flags, st = gbmoe.moe_read_status(ws)
    assert st == 0 and flags == 0
    assert_layer_close(out.float().cpu().numpy(), oracle.fused_moe_fp8(**d), "layer after the self-test")
