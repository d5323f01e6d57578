"""fused_moe_fp8_static_scratch: the FP8 layer for callers that cannot allocate device memory.

Such callers (a plugin whose host framework owns all device memory, a C caller
with no allocator, a loop that must not pay for cudaMalloc/cudaFree) pass only
inputs and outputs; the library runs the fused_moe_fp8 kernels on its own
static device buffer.  This file is collected last on purpose, so that a run
that stops at the first failure has already run every other test.  It must
pass alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

from _layers import assert_layer_close, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def _args(d):
    return (d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"])


def test_static_scratch_matches_workspace_entry_on_two_calls_in_a_row():
    # two different layers back to back: the second call must not see the first call's leftovers
    a = to_device(synth.make_layer(synth.LayerShape("a", 40, 512, 384, 16, 4, "fp8", "softmax"), seed=21))
    b = to_device(synth.make_layer(synth.LayerShape("b", 7, 512, 384, 16, 4, "fp8", "softmax"), seed=22))
    got_a = gbmoe.fused_moe_fp8_static_scratch(*_args(a))
    got_b = gbmoe.fused_moe_fp8_static_scratch(*_args(b))
    ref_a = gbmoe.fused_moe_fp8(*_args(a))
    ref_b = gbmoe.fused_moe_fp8(*_args(b))
    torch.cuda.synchronize()
    assert_layer_close(got_a.float().cpu().numpy(), ref_a.float().cpu().numpy().astype(np.float64), "call 1")
    assert_layer_close(got_b.float().cpu().numpy(), ref_b.float().cpu().numpy().astype(np.float64), "call 2")


def test_static_scratch_rejects_sizes_beyond_its_buffer():
    shape = synth.LayerShape("big", 128, 4096, 8192, 64, 8, "fp8", "softmax")
    need = gbmoe.moe_workspace_size(shape.M, shape.H, shape.I, shape.E, shape.topk, gbmoe.MOE_WEIGHT_FP8)
    assert need > gbmoe.MOE_STATIC_SCRATCH_BYTES
    dev = torch.device("cuda")
    x = torch.zeros(shape.M, shape.H, dtype=torch.bfloat16, device=dev)
    ids = torch.zeros(shape.M, shape.topk, dtype=torch.int32, device=dev)
    w = torch.zeros(shape.M, shape.topk, dtype=torch.float32, device=dev)
    # no weights are passed: the size check fails on the host before any launch
    lib = gbmoe.load()
    p = lambda t: t.data_ptr()  # noqa: E731
    st = lib.fused_moe_fp8_static_scratch(p(x), p(ids), p(w), p(x), p(w), p(x), p(w), shape.M, shape.H, shape.I,
                                          shape.E, shape.topk, 0, p(x), None)
    assert st == 2  # MOE_ERR_UNSUPPORTED
    assert b"MOE_STATIC_SCRATCH_BYTES" in lib.moe_last_error()
