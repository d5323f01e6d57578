"""Edge cases of the GPU entry points at their limits: most experts, largest top-k, empty batches.

Floating-point outputs must meet the layer tolerance against the oracle; an empty call must
launch nothing and leave its outputs untouched.
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


def _fp8(d, flags=gbmoe.MOE_PATH_AUTO):
    dd = to_device(d)
    out = gbmoe.fused_moe_fp8(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"], dd["w2"],
                              dd["w2_scale"], flags=flags)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("flags", [gbmoe.MOE_PATH_DECODE, gbmoe.MOE_PATH_PREFILL])
def test_most_experts_supported(flags):
    # MOE_MAX_EXPERTS experts, 40 tokens: most experts get no token, a few get one or two
    shape = synth.LayerShape("e", 40, 256, 128, gbmoe.MOE_MAX_EXPERTS, 3, "fp8", "uniform")
    d = synth.make_layer(shape, seed=101)
    assert_layer_close(_fp8(d, flags), oracle.fused_moe_fp8(**d), f"E=1024 flags {flags}")


@pytest.mark.parametrize("flags", [gbmoe.MOE_PATH_DECODE, gbmoe.MOE_PATH_PREFILL])
def test_largest_topk(flags):
    shape = synth.LayerShape("k", 9, 256, 128, 40, 32, "fp8", "softmax")
    d = synth.make_layer(shape, seed=102)
    assert_layer_close(_fp8(d, flags), oracle.fused_moe_fp8(**d), f"topk=32 flags {flags}")


def test_single_expert_every_token():
    shape = synth.LayerShape("one", 50, 256, 256, 1, 1, "fp8", "uniform")
    d = synth.make_layer(shape, seed=103)
    for flags in (gbmoe.MOE_PATH_DECODE, gbmoe.MOE_PATH_PREFILL):
        assert_layer_close(_fp8(d, flags), oracle.fused_moe_fp8(**d), f"E=1 flags {flags}")


def test_empty_batches_are_no_ops():
    dev = "cuda"
    shape = synth.LayerShape("z", 4, 256, 128, 8, 2, "int4", "softmax")
    w13, s13, w2, s2 = [t.to(dev) for t in synth.make_weights(shape, 104)]
    x = torch.empty(0, 256, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(0, 2, dtype=torch.int32, device=dev)
    w = torch.empty(0, 2, dtype=torch.float32, device=dev)
    assert gbmoe.fused_moe_int4(x, ids, w, w13, s13, w2, s2).shape == (0, 256)
    out, gi, gw = gbmoe.fused_moe_gated(gbmoe.MOE_WEIGHT_INT4, x, torch.empty(0, 8, device=dev), gbmoe.gate_config(),
                                        2, w13, s13, w2, s2)
    assert out.shape == (0, 256) and gi.shape == (0, 2)
    # masked layout with every count zero: nothing is written
    xm = synth.make_x(synth.LayerShape("m", 8 * 5, 256, 128, 8, 1, "int4", "uniform"), 105).view(8, 5, 256).to(dev)
    out = torch.full((8, 5, 256), 3.0, dtype=torch.bfloat16, device=dev)
    for flags in (gbmoe.MOE_PATH_DECODE, gbmoe.MOE_PATH_PREFILL):
        gbmoe.fused_moe_masked(gbmoe.MOE_WEIGHT_INT4, xm, torch.zeros(8, dtype=torch.int32, device=dev), w13, s13, w2,
                               s2, out=out, flags=flags)
        torch.cuda.synchronize()
        assert (out.float() == 3.0).all()


def test_all_ids_dropped_gives_zero_output():
    shape = synth.LayerShape("drop", 6, 256, 128, 8, 2, "fp8", "softmax")
    d = synth.make_layer(shape, seed=106)
    d["topk_ids"][:] = -1
    for flags in (gbmoe.MOE_PATH_DECODE, gbmoe.MOE_PATH_PREFILL):
        out = _fp8(d, flags)
        assert np.array_equal(out, np.zeros_like(out)), f"flags {flags}"
