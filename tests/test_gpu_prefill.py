"""GPU parity of the prefill (tcgen05 grouped GEMM) path against the CPU oracle.

Layer outputs must meet rel-L2 <= 5e-3 and max-abs <= 1e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from _layers import assert_layer_close, covering_rows, expert_id_expected, expert_id_layer, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu

PREFILL = gbmoe.MOE_PATH_PREFILL


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def _run(d, kind, flags=PREFILL, ws=None):
    dd = to_device(d)
    fn = gbmoe.fused_moe_fp8 if kind == "fp8" else gbmoe.fused_moe_int8
    out = fn(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"], dd["w2"],
             dd["w2_scale"], flags=flags, workspace=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def test_prefill_fp8_tiny():
    shape = synth.tiny(M=64)
    d = synth.make_layer(shape, seed=31)
    ws = gbmoe.alloc_workspace(64, shape.H, shape.I, shape.E, shape.topk, gbmoe.MOE_WEIGHT_FP8, PREFILL)
    out = _run(d, "fp8", ws=ws)
    bad, flags, st = gbmoe.moe_read_status(ws)
    assert flags == 0, "a bounded device wait gave up"
    assert_layer_close(out, oracle.fused_moe_fp8(**d), "prefill tiny fp8")


def test_prefill_fp8_expert_id_structured_layer():
    d = expert_id_layer(M=48, topk=3, E=8)
    out = _run(d, "fp8")
    want = expert_id_expected(d)
    np.testing.assert_allclose(out, np.repeat(want[:, None], out.shape[1], 1), rtol=1e-2)


@pytest.mark.parametrize("M,H,I,E,k", [
    (300, 512, 384, 6, 3),     # ~150 slots per expert, 3 output tiles, 8 K chunks
    (600, 256, 256, 4, 2),     # ~300 slots per expert: several token tiles per expert
    (129, 1024, 640, 33, 5),   # ragged: many experts with few slots
    (1, 256, 128, 8, 2),       # a single token
])
def test_prefill_fp8_shapes(M, H, I, E, k):
    shape = synth.LayerShape("p", M, H, I, E, k, "fp8", "softmax")
    d = synth.make_layer(shape, seed=M + I)
    out = _run(d, "fp8")
    assert_layer_close(out, oracle.fused_moe_fp8(**d), f"prefill fp8 {M}x{H}x{I} E{E} k{k}")


@pytest.mark.parametrize("M,H,I,E,k", [(200, 512, 256, 8, 4), (520, 256, 384, 4, 2)])
def test_prefill_int8(M, H, I, E, k):
    shape = synth.LayerShape("q", M, H, I, E, k, "int8", "softmax")
    d = synth.make_layer(shape, seed=M * 7)
    out = _run(d, "int8")
    assert_layer_close(out, oracle.fused_moe_int8(**d), f"prefill int8 {M}x{H}x{I}")


def test_prefill_and_decode_agree():
    shape = synth.LayerShape("pd", 96, 512, 256, 16, 4, "fp8", "softmax")
    d = synth.make_layer(shape, seed=41)
    a = _run(d, "fp8", flags=PREFILL)
    b = _run(d, "fp8", flags=gbmoe.MOE_PATH_DECODE)
    ref = oracle.fused_moe_fp8(**d)
    assert_layer_close(a, ref, "prefill")
    assert_layer_close(b, ref, "decode")


def test_prefill_bad_ids():
    shape = synth.tiny(M=40)
    d = synth.make_layer(shape, seed=43)
    ids = d["topk_ids"].clone()
    ids[0, 0] = -5
    ids[7, 1] = 1000
    d["topk_ids"] = ids
    ws = gbmoe.alloc_workspace(40, shape.H, shape.I, shape.E, shape.topk, gbmoe.MOE_WEIGHT_FP8, PREFILL)
    out = _run(d, "fp8", ws=ws)
    assert gbmoe.moe_read_status(ws)[:2] == (2, 0)
    assert_layer_close(out, oracle.fused_moe_fp8(**d), "prefill bad ids")


def test_prefill_deterministic():
    shape = synth.LayerShape("t", 256, 512, 256, 8, 2, "fp8", "softmax")
    d = synth.make_layer(shape, seed=44)
    assert np.array_equal(_run(d, "fp8"), _run(d, "fp8"))


def _full_size_check(shape, seed, kind, flags=gbmoe.MOE_PATH_AUTO):
    """Rows covering every active expert, and the last token of the most loaded experts (the last token
    tile of the heaviest Zipf expert)."""
    ids, w = synth.make_routing(shape, seed)
    rows = covering_rows(ids.numpy(), shape.E_total)
    x = synth.make_x(shape, seed)
    w13, s13, w2, s2 = synth.make_weights(shape, seed, device="cuda")
    fn = gbmoe.fused_moe_fp8 if kind == "fp8" else gbmoe.fused_moe_int8
    out = fn(x.cuda(), ids.cuda(), w.cuda(), w13, s13, w2, s2, flags=flags)
    out = out.float().cpu().numpy()
    ref = oracle.fused_moe_rows(x, ids, w, w13, s13, w2, s2, kind=kind, tokens=rows)
    assert_layer_close(out[rows], ref, shape.name)


def test_deepseek_r1_prefill_2048_zipf_full_size():
    _full_size_check(synth.deepseek_r1(2048, routing="deepseek_zipf"), seed=51, kind="fp8")


def test_deepseek_r1_prefill_16384_zipf_full_size():
    # the compute-bound weight-only point: 16,384 tokens, the alignment split over 36 chunks
    _full_size_check(synth.deepseek_r1(16384, routing="deepseek_zipf"), seed=54, kind="fp8")


def test_qwen3_int8_prefill_256_full_size():
    _full_size_check(synth.qwen3_235b(256), seed=52, kind="int8", flags=PREFILL)


def test_qwen3_int8_prefill_4096_full_size():
    _full_size_check(synth.qwen3_235b(4096), seed=53, kind="int8")
