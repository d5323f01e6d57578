"""GPU parity of the C-ABI library against the CPU oracle (routing, quantisation, decode path).

Integer outputs (routing alignment, INT8 codes) must match bit for bit.
Layer outputs must meet rel-L2 <= 5e-3 and max-abs <= 1e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from _layers import assert_layer_close, covering_rows, expert_id_expected, expert_id_layer, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu

DECODE = gbmoe.MOE_PATH_DECODE


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


# ------------------------------------------------------------------ routing alignment

def _align_both(ids_np, E, B):
    ids = torch.from_numpy(ids_np.astype(np.int32)).cuda()
    s, eid, npp, off = gbmoe.moe_align_block_size(ids, E, B)
    ref = oracle.moe_align_block_size(ids_np, E, B)
    return (s.cpu().numpy(), eid.cpu().numpy(), int(npp.item()), off.cpu().numpy()), ref


@pytest.mark.parametrize("M,topk,E,B", [
    (1, 1, 1, 1), (3, 2, 4, 2), (16, 2, 8, 16), (4, 9, 257, 8), (64, 9, 257, 8),
    (100, 8, 128, 16), (2048, 9, 257, 64), (4096, 8, 128, 128), (777, 3, 1024, 32), (5000, 8, 64, 256),
])
def test_align_bit_exact_random(M, topk, E, B):
    rng = np.random.default_rng(M * 131 + E)
    ids = rng.integers(0, E, size=(M, topk))
    got, ref = _align_both(ids, E, B)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])
    assert got[2] == int(ref[2])
    np.testing.assert_array_equal(got[3], ref[3])


def test_align_bit_exact_skewed_deepseek_routing():
    shape = synth.deepseek_r1(2048, routing="deepseek_zipf")
    ids, _ = synth.make_routing(shape, seed=3)
    for B in (16, 64, 128):
        got, ref = _align_both(ids.numpy(), shape.E_total, B)
        for a, b in zip(got, ref[:4]):
            np.testing.assert_array_equal(np.asarray(a), np.asarray(b))


def test_align_out_of_range_ids_and_duplicates():
    rng = np.random.default_rng(7)
    ids = rng.integers(-3, 12, size=(50, 4))
    ids[5] = [2, 2, 2, 2]  # one token picking one expert several times
    got, ref = _align_both(ids, 9, 4)
    for a, b in zip(got, ref[:4]):
        np.testing.assert_array_equal(np.asarray(a), np.asarray(b))


def test_align_empty_batch():
    got, ref = _align_both(np.zeros((0, 8), np.int64), 16, 8)
    for a, b in zip(got, ref[:4]):
        np.testing.assert_array_equal(np.asarray(a), np.asarray(b))


# ------------------------------------------------------------------ activation quantisation

def test_quant_act_int8_bit_exact():
    g = torch.Generator().manual_seed(4)
    x = (torch.randn(300, 7168, generator=g) * torch.rand(300, 1, generator=g) * 30).to(torch.bfloat16)
    x[7] = 0
    x[8, 100] = 1e30
    x[9, :] = 2.0 ** -130  # bf16 subnormals
    q, s = gbmoe.moe_quant_act_int8(x.cuda())
    rq, rs = oracle.quant_int8_per_row(x.float().numpy())
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


# ------------------------------------------------------------------ fused layer, decode path

def _run(d, kind, flags=DECODE):
    dd = to_device(d)
    fn = gbmoe.fused_moe_fp8 if kind == "fp8" else gbmoe.fused_moe_int8
    out = fn(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"], dd["w2"],
             dd["w2_scale"], flags=flags)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def test_fp8_tiny_config():
    shape = synth.tiny()
    d = synth.make_layer(shape, seed=1)
    out = _run(d, "fp8")
    assert_layer_close(out, oracle.fused_moe_fp8(**d), "tiny fp8")


@pytest.mark.parametrize("M,H,I,E,k", [(40, 512, 384, 16, 4), (1, 256, 128, 8, 2), (128, 384, 256, 6, 3),
                                       (37, 1024, 640, 33, 5)])
def test_fp8_several_tiles_and_ragged_groups(M, H, I, E, k):
    shape = synth.LayerShape("t", M, H, I, E, k, "fp8", "softmax")
    d = synth.make_layer(shape, seed=M + H)
    out = _run(d, "fp8")
    assert_layer_close(out, oracle.fused_moe_fp8(**d), f"fp8 {M}x{H}x{I} E{E} k{k}")


def test_fp8_expert_id_structured_layer():
    d = expert_id_layer(M=20, topk=3, E=8)
    out = _run(d, "fp8")
    want = expert_id_expected(d)
    # bf16 output of a constant row: relative rounding only
    np.testing.assert_allclose(out, np.repeat(want[:, None], out.shape[1], 1), rtol=1e-2)
    assert np.all(out == out[:, :1])


# from under one slot per expert (6 x 2 over 16 experts) to about 51 (128 x 2 over 5: seven 8-slot tiles each)
@pytest.mark.parametrize("M,H,I,E,k", [(16, 256, 128, 8, 2), (50, 512, 384, 12, 4), (128, 256, 256, 5, 2),
                                       (6, 256, 128, 16, 2)])
def test_int8_layer(M, H, I, E, k):
    shape = synth.LayerShape("q", M, H, I, E, k, "int8", "softmax")
    d = synth.make_layer(shape, seed=M * 3 + E)
    out = _run(d, "int8")
    assert_layer_close(out, oracle.fused_moe_int8(**d), f"int8 {M}x{H}x{I}")


def test_bad_ids_are_counted_and_contribute_nothing():
    shape = synth.tiny(M=12)
    d = synth.make_layer(shape, seed=5)
    ids = d["topk_ids"].clone()
    ids[2, 0] = -1
    ids[3, 1] = 99
    d["topk_ids"] = ids
    dd = to_device(d)
    ws = gbmoe.alloc_workspace(12, shape.H, shape.I, shape.E, shape.topk, gbmoe.MOE_WEIGHT_FP8)
    out = gbmoe.fused_moe_fp8(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"],
                              dd["w2"], dd["w2_scale"], workspace=ws)
    bad, flags, st = gbmoe.moe_read_status(ws)
    assert (bad, flags, st) == (2, 0, 6)
    assert_layer_close(out.float().cpu().numpy(), oracle.fused_moe_fp8(**d), "bad ids")


def test_empty_batch_is_noop():
    shape = synth.tiny(M=0)
    d = to_device(synth.make_layer(shape, seed=1))
    out = gbmoe.fused_moe_fp8(d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w13_scale"], d["w2"],
                              d["w2_scale"])
    assert out.shape == (0, shape.H)


def test_deterministic():
    shape = synth.LayerShape("t", 64, 512, 256, 16, 4, "fp8", "softmax")
    d = synth.make_layer(shape, seed=2)
    a = _run(d, "fp8")
    b = _run(d, "fp8")
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ full-size layers
# Every token up to 16 tokens; above, rows that cover every active expert (the oracle dequantises each
# expert once, so that is the bound of its cost) and the last token of the most loaded experts.

def _full_size_check(shape, seed, rows, kind):
    ids, w = synth.make_routing(shape, seed)
    if rows is None:
        rows = list(range(shape.M)) if shape.M <= 16 else covering_rows(ids.numpy(), shape.E_total)
    x = synth.make_x(shape, seed)
    w13, s13, w2, s2 = synth.make_weights(shape, seed, device="cuda")
    fn = gbmoe.fused_moe_fp8 if kind == "fp8" else gbmoe.fused_moe_int8
    out = fn(x.cuda(), ids.cuda(), w.cuda(), w13, s13, w2, s2, flags=DECODE)
    out = out.float().cpu().numpy()
    ref = oracle.fused_moe_rows(x, ids, w, w13, s13, w2, s2, kind=kind, tokens=rows)
    assert_layer_close(out[rows], ref, shape.name)


def test_deepseek_r1_decode_full_size_batch1():
    _full_size_check(synth.deepseek_r1(1), seed=11, rows=[0], kind="fp8")


def test_deepseek_r1_decode_full_size_batch4():
    _full_size_check(synth.deepseek_r1(4), seed=12, rows=None, kind="fp8")


def test_deepseek_r1_decode_sweep_batch64_uniform():
    _full_size_check(synth.deepseek_r1(64, routing="uniform"), seed=13, rows=None, kind="fp8")


def test_qwen3_int8_full_size_batch16():
    _full_size_check(synth.qwen3_235b(16), seed=14, rows=None, kind="int8")


def test_qwen3_int8_full_size_batch1():
    _full_size_check(synth.qwen3_235b(1), seed=15, rows=[0], kind="int8")


def test_qwen3_int8_full_size_batch96():
    # the largest batch MOE_PATH_AUTO gives the weight-streaming kernels: 768 slots over 128 experts, 21 of
    # them with more than one 8-slot tile; rows covering every active expert
    _full_size_check(synth.qwen3_235b(96), seed=16, rows=None, kind="int8")


@pytest.mark.parametrize("M", [2, 8, 16, 32])
def test_deepseek_r1_decode_sweep_uniform(M):
    # the decode batch sweep of DeepSeek-R1 shapes with uniform routing
    _full_size_check(synth.deepseek_r1(M, routing="uniform"), seed=20 + M, rows=None, kind="fp8")
