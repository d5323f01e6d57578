"""GPU parity of the group-wise INT4 layer (fused_moe_int4) against the CPU oracle.

Outputs must meet rel-L2 <= 5e-3 and max-abs <= 1e-2 * max|ref| against
oracle.fused_moe_int4 on the same seeded inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from _layers import assert_layer_close, covering_rows, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def _run(d, flags=gbmoe.MOE_PATH_AUTO, ws=None):
    dd = to_device(d)
    out = gbmoe.fused_moe_int4(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"], dd["w2"],
                               dd["w2_scale"], flags=flags, workspace=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("M,H,I,E,k", [
    (16, 256, 128, 8, 2),      # the tiny layer
    (1, 256, 128, 8, 2),       # a single token
    (37, 512, 384, 6, 3),      # ragged token tiles, three GEMM1 row tiles
    (300, 256, 256, 8, 2),     # more tokens than the decode path takes for the other kinds
    (4, 7168, 256, 16, 3),     # long K for GEMM1 (56 groups)
    (9, 384, 640, 5, 4),       # five K groups in GEMM2, three GEMM2 row tiles
])
def test_int4_shapes(M, H, I, E, k):
    shape = synth.LayerShape("i4", M, H, I, E, k, "int4", "softmax")
    d = synth.make_layer(shape, seed=M + H + I)
    assert_layer_close(_run(d), oracle.fused_moe_int4(**d), f"INT4 {M}x{H}x{I} E{E} k{k}")


@pytest.mark.parametrize("M,H,I,E,k", [
    (300, 256, 256, 8, 2),     # ~75 slots per expert: partial token tiles
    (600, 512, 384, 4, 2),     # several token tiles per expert, three GEMM1 row blocks
    (129, 640, 1024, 33, 5),   # ragged: many experts with few slots
    (4, 7168, 256, 16, 3),     # long K, tiny M on the tcgen05 path
])
def test_int4_tcgen05_path(M, H, I, E, k):
    shape = synth.LayerShape("i4", M, H, I, E, k, "int4", "softmax")
    d = synth.make_layer(shape, seed=M + H + I + 7)
    assert_layer_close(_run(d, flags=gbmoe.MOE_PATH_PREFILL), oracle.fused_moe_int4(**d),
                       f"INT4 tcgen05 {M}x{H}x{I} E{E} k{k}")


def test_int4_qwen3_shape_prefill_4096():
    _full_size(synth.qwen3_235b(4096, weight_kind="int4"), seed=23)


def test_int4_every_code_and_extreme_group_scales():
    # random bytes use all 16 codes (-8 included); scales span 2^-20 .. 2^4 across groups
    shape = synth.LayerShape("i4", 24, 512, 256, 4, 2, "int4", "uniform")
    d = synth.make_layer(shape, seed=77)
    g = torch.Generator().manual_seed(78)
    for wk, sk in (("w13", "w13_scale"), ("w2", "w2_scale")):
        d[wk] = torch.randint(0, 256, tuple(d[wk].shape), generator=g, dtype=torch.uint8)
        d[sk] = (torch.exp2(torch.randint(-20, 5, tuple(d[sk].shape), generator=g).float()) * 0.01).contiguous()
    q = oracle.unpack_int4(d["w13"][0].numpy())
    assert q.min() == -8 and q.max() == 7
    ref = oracle.fused_moe_int4(**d)
    assert_layer_close(_run(d), ref, "INT4 all codes")
    assert_layer_close(_run(d, flags=gbmoe.MOE_PATH_PREFILL), ref, "INT4 all codes, tcgen05 path")


def test_int4_expert_id_closed_form():
    # expert e returns I * silu(1) * (e+1): gate/up rows pick x[:, 0] = 1 with code 1 and scale 1;
    # every W2 code is 1 with group scale e+1
    M, k, E, H, I = 6, 3, 8, 256, 128
    rng = np.random.default_rng(3)
    x = torch.zeros(M, H, dtype=torch.bfloat16)
    x[:, 0] = 1.0
    w13 = torch.zeros(E, 2 * I, H // 2, dtype=torch.uint8)
    w13[:, :, 0] = 0x01                                   # column 0 = 1, column 1 = 0
    s13 = torch.ones(E, 2 * I, H // 128)
    w2 = torch.full((E, H, I // 2), 0x11, dtype=torch.uint8)
    s2 = (torch.arange(E, dtype=torch.float32) + 1)[:, None, None].expand(E, H, I // 128).contiguous()
    ids = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32))
    w = torch.from_numpy(rng.uniform(0.1, 1.0, size=(M, k)).astype(np.float32))
    d = dict(x=x, topk_ids=ids, topk_weights=w, w13=w13, w13_scale=s13, w2=w2, w2_scale=s2)
    silu1 = 1.0 / (1.0 + np.exp(-1.0))
    want = I * silu1 * (w.double().numpy() * (ids.double().numpy() + 1)).sum(axis=1)
    out = _run(d)
    np.testing.assert_allclose(out, np.repeat(want[:, None], H, axis=1), rtol=8e-3)


def test_int4_flags_and_status():
    shape = synth.LayerShape("i4", 8, 256, 128, 8, 2, "int4", "softmax")
    d = synth.make_layer(shape, seed=5)
    ws = gbmoe.alloc_workspace(8, 256, 128, 8, 2, gbmoe.MOE_WEIGHT_INT4)
    with pytest.raises(gbmoe.MoEError) as e:
        _run(d, flags=gbmoe.MOE_ACT_FP8_1X128, ws=ws)
    assert e.value.status == 1
    d["topk_ids"][3, 1] = 99  # dropped id
    out = _run(d, ws=ws)
    bad, flags, st = gbmoe.moe_read_status(ws)
    assert bad == 1 and flags == 0
    assert_layer_close(out, oracle.fused_moe_int4(**d), "INT4 with a dropped id")


def test_int4_deterministic():
    shape = synth.LayerShape("i4", 40, 512, 256, 8, 4, "int4", "softmax")
    d = synth.make_layer(shape, seed=9)
    assert np.array_equal(_run(d), _run(d))


def _full_size(shape, seed, rows=None):
    ids, w = synth.make_routing(shape, seed)
    if rows is None:  # rows covering every active expert, and the last token of the most loaded experts
        rows = covering_rows(ids.numpy(), shape.E_total)
    x = synth.make_x(shape, seed)
    w13, s13, w2, s2 = synth.make_weights(shape, seed, device="cuda")
    out = gbmoe.fused_moe_int4(x.cuda(), ids.cuda(), w.cuda(), w13, s13, w2, s2).float().cpu().numpy()
    ref = oracle.fused_moe_rows(x, ids, w, w13, s13, w2, s2, kind="int4", tokens=rows)
    assert_layer_close(out[rows], ref, shape.name)


def test_int4_deepseek_r1_shape_decode_batch4():
    _full_size(synth.deepseek_r1(4, weight_kind="int4"), seed=21, rows=[0, 1, 2, 3])


def test_int4_qwen3_shape_batch16():
    _full_size(synth.qwen3_235b(16, weight_kind="int4"), seed=22, rows=list(range(16)))


def test_int4_gated_layer():
    shape = synth.LayerShape("g4", 12, 256, 128, 32, 4, "int4", "softmax")
    d = synth.make_layer(shape, seed=31)
    lg = synth.make_router_logits(shape, 31)
    dd = to_device(d)
    out, ids, w = gbmoe.fused_moe_gated(gbmoe.MOE_WEIGHT_INT4, dd["x"], lg.cuda(), gbmoe.gate_config(), 4,
                                        dd["w13"], dd["w13_scale"], dd["w2"], dd["w2_scale"])
    torch.cuda.synchronize()
    ids_o, _ = oracle.gate_softmax_topk(lg.numpy(), 4)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_o)
    d["topk_ids"], d["topk_weights"] = ids.cpu(), w.cpu()
    assert_layer_close(out.float().cpu().numpy(), oracle.fused_moe_int4(**d), "gated INT4 layer")
