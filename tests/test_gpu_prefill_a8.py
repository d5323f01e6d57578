"""GPU parity of the FP8-activation (A8, 1 x 128 groups) path against the CPU oracle.

The quantiser is compared bit for bit (its codes are decided in IEEE fp32 on
both sides); layer outputs must meet rel-L2 <= 5e-3 and max-abs <= 1e-2 *
max|ref| against the oracle's act="fp8_1x128" mode.
"""
import numpy as np
import pytest
import torch

import oracle
from _layers import assert_layer_close, covering_rows, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu

A8 = gbmoe.MOE_ACT_FP8_1X128


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def _x_mixed(M, H, seed):
    """bf16 rows with magnitudes from 2^-20 to 2^12, zero groups, and values that land on E4M3 subnormals."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, H, generator=g) * torch.exp2(torch.randint(-20, 13, (M, 1), generator=g).float())
    x[:, 5] *= 1e-4                         # subnormal codes next to a normal amax
    if M > 2:
        x[2, :128] = 0.0                    # an all-zero group
        x[1, 128:256] = -x[1, 128:256].abs()
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("M,H", [(37, 7168), (5, 128), (1, 4096)])
def test_quant_act_fp8_bit_exact(M, H):
    x = _x_mixed(M, H, seed=M + H)
    q, s = gbmoe.moe_quant_act_fp8(x.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_fp8_1x128(x.float().numpy())
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def _run(d, flags=A8, ws=None):
    dd = to_device(d)
    out = gbmoe.fused_moe_fp8(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"], dd["w2"],
                              dd["w2_scale"], flags=flags, workspace=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def test_a8_tiny():
    shape = synth.tiny(M=64)
    d = synth.make_layer(shape, seed=61)
    ws = gbmoe.alloc_workspace(64, shape.H, shape.I, shape.E, shape.topk, gbmoe.MOE_WEIGHT_FP8, A8)
    out = _run(d, ws=ws)
    bad, flags, st = gbmoe.moe_read_status(ws)
    assert flags == 0, "a bounded device wait gave up"
    assert_layer_close(out, oracle.fused_moe_fp8(**d, act="fp8_1x128"), "A8 tiny")


@pytest.mark.parametrize("M,H,I,E,k", [
    (300, 512, 384, 6, 3),     # ~150 slots per expert, 3 gate/up tiles, 4 K blocks
    (600, 256, 256, 4, 2),     # ~300 slots per expert: several token tiles per expert
    (129, 640, 1024, 33, 5),   # ragged: many experts with few slots; GEMM2 ends on a single 128-row block
    (1, 256, 128, 8, 2),       # a single token
    (4, 7168, 256, 16, 3),     # long K (56 K blocks) for GEMM1
])
def test_a8_shapes(M, H, I, E, k):
    shape = synth.LayerShape("a8", M, H, I, E, k, "fp8", "softmax")
    d = synth.make_layer(shape, seed=M + I + 1)
    out = _run(d)
    assert_layer_close(out, oracle.fused_moe_fp8(**d, act="fp8_1x128"), f"A8 {M}x{H}x{I} E{E} k{k}")


def test_a8_differs_from_weight_only_by_quantisation():
    shape = synth.LayerShape("a8", 96, 512, 256, 16, 4, "fp8", "softmax")
    d = synth.make_layer(shape, seed=62)
    a8 = _run(d)
    a16 = _run(d, flags=gbmoe.MOE_PATH_PREFILL)
    rel = np.linalg.norm(a8 - a16) / np.linalg.norm(a16)
    assert 1e-3 < rel < 6e-2
    assert_layer_close(a8, oracle.fused_moe_fp8(**d, act="fp8_1x128"), "A8")
    assert_layer_close(a16, oracle.fused_moe_fp8(**d), "A16")


def test_a8_bad_ids():
    shape = synth.tiny(M=40)
    d = synth.make_layer(shape, seed=63)
    ids = d["topk_ids"].clone()
    ids[0, 0] = -5
    ids[7, 1] = 1000
    d["topk_ids"] = ids
    ws = gbmoe.alloc_workspace(40, shape.H, shape.I, shape.E, shape.topk, gbmoe.MOE_WEIGHT_FP8, A8)
    out = _run(d, ws=ws)
    assert gbmoe.moe_read_status(ws)[:2] == (2, 0)
    assert_layer_close(out, oracle.fused_moe_fp8(**d, act="fp8_1x128"), "A8 bad ids")


def test_a8_deterministic():
    shape = synth.LayerShape("t", 256, 512, 256, 8, 2, "fp8", "softmax")
    d = synth.make_layer(shape, seed=64)
    assert np.array_equal(_run(d), _run(d))


def _full_size_check(shape, seed, rows=None):
    ids, w = synth.make_routing(shape, seed)
    if rows is None:  # rows covering every active expert, and the last token of the most loaded experts
        rows = covering_rows(ids.numpy(), shape.E_total)
    x = synth.make_x(shape, seed)
    w13, s13, w2, s2 = synth.make_weights(shape, seed, device="cuda")
    out = gbmoe.fused_moe_fp8(x.cuda(), ids.cuda(), w.cuda(), w13, s13, w2, s2, flags=A8)
    out = out.float().cpu().numpy()
    ref = oracle.fused_moe_rows(x, ids, w, w13, s13, w2, s2, kind="fp8", tokens=rows, act="fp8_1x128")
    assert_layer_close(out[rows], ref, shape.name + " A8")


def test_deepseek_r1_a8_prefill_2048_zipf_full_size():
    _full_size_check(synth.deepseek_r1(2048, routing="deepseek_zipf"), seed=65)


def test_deepseek_r1_a8_prefill_16384_full_size():
    _full_size_check(synth.deepseek_r1(16384, routing="deepseek_zipf"), seed=66)


def test_deepseek_r1_a8_decode_sized_batch_full_size():
    _full_size_check(synth.deepseek_r1(4), seed=67, rows=[0, 1, 2, 3])
