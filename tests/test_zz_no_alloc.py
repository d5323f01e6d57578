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


def _args(d):
    return (d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"])


def _layer(M, seed, E=16, topk=4):
    return synth.make_layer(synth.LayerShape("s", M, 512, 384, E, topk, "fp8", "softmax"), seed=seed)


# small decode, tcgen05 path, FP8 activations, then a larger decode: the buffer's contents left by each
# call (another layout, another path) must not leak into the next
SEQUENCE = [(7, gbmoe.MOE_PATH_DECODE, "a16"), (40, gbmoe.MOE_PATH_PREFILL, "a16"),
            (24, gbmoe.MOE_ACT_FP8_1X128, "fp8_1x128"), (40, gbmoe.MOE_PATH_DECODE, "a16")]


def test_static_scratch_equals_workspace_entry_and_oracle_over_a_call_sequence():
    for i, (M, flags, act) in enumerate(SEQUENCE):
        host = _layer(M, seed=21 + i)
        d = to_device(host)
        assert gbmoe.moe_workspace_size(M, 512, 384, 16, 4, gbmoe.MOE_WEIGHT_FP8, flags) <= \
            gbmoe.MOE_STATIC_SCRATCH_BYTES
        got = gbmoe.fused_moe_fp8_static_scratch(*_args(d), flags=flags)
        ref = gbmoe.fused_moe_fp8(*_args(d), flags=flags)  # a fresh workspace, the same kernels
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {i + 1} (M={M}, flags={flags:#x}) differs from fused_moe_fp8"
        assert_layer_close(got.float().cpu().numpy(), oracle.fused_moe_fp8(**host, act=act),
                           f"call {i + 1} (M={M}, flags={flags:#x}) against the oracle")
        assert gbmoe.moe_read_static_scratch_status()[2] == 0


def test_static_scratch_status_counts_bad_ids():
    host = _layer(9, seed=31)
    host["topk_ids"][2, 1] = 99  # outside [0, E)
    host["topk_ids"][5, 0] = -3
    got = gbmoe.fused_moe_fp8_static_scratch(*_args(to_device(host)))
    torch.cuda.synchronize()
    bad, flags, st = gbmoe.moe_read_static_scratch_status()
    assert (bad, flags, st) == (2, 0, 6)  # MOE_ERR_BAD_IDS
    assert_layer_close(got.float().cpu().numpy(), oracle.fused_moe_fp8(**host), "dropped ids")
    # the next clean call clears the count
    gbmoe.fused_moe_fp8_static_scratch(*_args(to_device(_layer(9, seed=32))))
    assert gbmoe.moe_read_static_scratch_status() == (0, 0, 0)


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
    # invalid arguments get the layer's own error, however large the sizes
    st = lib.fused_moe_fp8_static_scratch(p(x), p(ids), p(w), p(x), p(w), p(x), p(w), shape.M, shape.H + 64,
                                          shape.I, shape.E, shape.topk, 0, p(x), None)
    assert st == 2 and b"multiples of 128" in lib.moe_last_error()
    st = lib.fused_moe_fp8_static_scratch(p(x), p(ids), p(w), None, p(w), p(x), p(w), shape.M, shape.H, shape.I,
                                          shape.E, shape.topk, 0, p(x), None)
    assert st == 1 and b"NULL" in lib.moe_last_error()  # MOE_ERR_INVALID_ARG
