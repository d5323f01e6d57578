"""GPU parity of the router gating (moe_gate_topk, fused_moe_gated) against the oracle.

Ids are compared tie-aware (see _gate_check): exactly for the softmax router
and for every sigmoid-router token whose decision margins exceed fp32 error;
weights within 1e-5 relative.  The gated layer must return the routing it
used, identical to moe_gate_topk's, and an output within the layer tolerance
of the oracle layer run on that routing.
"""
import numpy as np
import pytest
import torch

import oracle
from _gate_check import check_grouped, check_softmax
from _layers import assert_layer_close, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu

SIG = gbmoe.MOE_GATE_SIGMOID_GROUPED


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def _logits(M, E, seed, kind="normal"):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(M, E, generator=g)
    if kind == "ties":  # small integers: exact ties
        return torch.randint(-2, 3, (M, E), generator=g).float()
    if kind == "ties_pos":  # 0, 1, 2: exact ties inside and across groups, and every sum of two
        return torch.randint(0, 3, (M, E), generator=g).float()  # scores differs by far more than fp32 error
    raise ValueError(kind)


def _gpu_gate(lg, k, cfg, unaligned=False):
    d = lg.cuda()
    if unaligned:  # rows start 4 bytes past a 16-byte boundary: the scalar-load path
        buf = torch.empty(d.numel() + 1, device="cuda")
        buf[1:] = d.reshape(-1)
        d = buf[1:].view_as(d)
        assert d.data_ptr() % 16 != 0
    ids, w = gbmoe.moe_gate_topk(d, k, cfg)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("M,E,k,shared,kind,unaligned", [
    (4096, 128, 8, False, "normal", False),   # Qwen3-MoE router
    (1, 128, 8, False, "normal", False),
    (300, 8, 2, False, "normal", False),      # 8 experts: one per lane, most lanes empty
    (77, 60, 4, True, "normal", False),       # E not a multiple of 4: scalar loads, a partial lane
    (50, 1000, 8, False, "normal", False),    # 32 experts per lane
    (200, 128, 8, False, "ties", False),
    (33, 256, 32, False, "normal", False),    # topk = 32: every lane holds a result
    (33, 256, 31, True, "normal", False),     # the shared column on the last lane
    (64, 128, 8, False, "normal", True),
])
def test_softmax_gate(M, E, k, shared, kind, unaligned):
    lg = _logits(M, E, seed=M + E + k, kind=kind)
    ids, w = _gpu_gate(lg, k, gbmoe.gate_config(shared_expert=shared), unaligned)
    check_softmax(lg.numpy(), k, ids, w, shared)


@pytest.mark.parametrize("M,E,k,n_group,topk_group,kind", [
    (2048, 256, 8, 8, 4, "normal"),   # DeepSeek-V3/R1 router: 8 groups of 32, keep 4
    (5, 256, 8, 8, 4, "normal"),
    (300, 64, 6, 4, 2, "normal"),     # fast group layout, 8 lanes per group
    (300, 96, 6, 3, 2, "normal"),     # 3 groups: general group path
    (300, 160, 8, 5, 3, "normal"),    # 5 groups of 32 over 8 experts per lane
    (300, 256, 8, 8, 4, "ties_pos"),
    (300, 64, 6, 4, 2, "ties_pos"),
    (300, 256, 8, 8, 8, "normal"),    # every group kept
    (300, 256, 8, 1, 1, "normal"),    # no grouping
    (100, 32, 4, 32, 4, "normal"),    # groups of one expert
    (100, 512, 8, 16, 4, "normal"),   # 16 experts per lane, 2 lanes per group
    (100, 1024, 8, 32, 4, "normal"),  # the largest router: 32 experts per lane, a lane per group
    (100, 1024, 16, 8, 3, "normal"),  # 4 lanes per group of 128
])
def test_grouped_sigmoid_gate(M, E, k, n_group, topk_group, kind):
    lg = _logits(M, E, seed=3 * M + E + n_group, kind=kind)
    bias = None if kind == "ties_pos" else synth.make_router_bias(E, seed=E)
    scale = 2.5
    cfg = gbmoe.gate_config(SIG, n_group, topk_group, scale, bias.cuda() if bias is not None else None, True)
    ids, w = _gpu_gate(lg, k, cfg)
    near = check_grouped(lg.numpy(), k, n_group, topk_group, scale, None if bias is None else bias.numpy(),
                         ids, w, shared=True)
    if kind == "ties_pos":
        assert near == 0  # exact ties are decided by index on both sides


def test_grouped_gate_on_the_zipf_workload_logits():
    shape = synth.deepseek_r1(4096, "deepseek_zipf")
    lg = synth.make_router_logits(shape, seed=3)
    cfg = gbmoe.gate_config(SIG, shape.n_group, shape.topk_group, shape.routed_scaling, None, True)
    ids, w = _gpu_gate(lg, shape.topk, cfg)
    check_grouped(lg.numpy(), shape.topk, shape.n_group, shape.topk_group, shape.routed_scaling, None, ids, w,
                  shared=True)


def test_gate_ids_stay_in_range_for_non_finite_logits():
    lg = _logits(64, 256, seed=5)
    lg[0, :] = float("nan")
    lg[1, 3] = float("inf")
    lg[2, :] = float("-inf")
    lg[3, ::2] = float("nan")
    for cfg in (gbmoe.gate_config(), gbmoe.gate_config(SIG, 8, 4, 1.0, None, False)):
        ids, w = _gpu_gate(lg, 8, cfg)
        assert ((ids >= 0) & (ids < 256)).all()
        # finite rows are unaffected
        if cfg.scoring == SIG:
            check_grouped(lg[4:].numpy(), 8, 8, 4, 1.0, None, ids[4:], w[4:])
        else:
            check_softmax(lg[4:].numpy(), 8, ids[4:], w[4:])


def test_gate_empty_batch():
    ids, w = gbmoe.moe_gate_topk(torch.empty(0, 128, device="cuda"), 8, gbmoe.gate_config())
    assert ids.shape == (0, 8) and w.shape == (0, 8)


# ---------------------------------------------------------------- the gated layer

def _gated_layer(shape, seed, cfg, flags=gbmoe.MOE_PATH_AUTO, full_size=False):
    if full_size:  # weights generated on the device
        x = synth.make_x(shape, seed)
        w13, s13, w2, s2 = synth.make_weights(shape, seed, device="cuda")
        d = dict(x=x, w13=w13, w13_scale=s13, w2=w2, w2_scale=s2)
    else:
        d = synth.make_layer(shape, seed)
    lg = synth.make_router_logits(shape, seed)
    dd = to_device(d)
    kind = gbmoe.MOE_WEIGHT_FP8 if shape.weight_kind == "fp8" else gbmoe.MOE_WEIGHT_INT8
    out, ids, w = gbmoe.fused_moe_gated(kind, dd["x"], lg.cuda(), cfg, shape.topk, dd["w13"], dd["w13_scale"],
                                        dd["w2"], dd["w2_scale"], flags=flags)
    ids_s, w_s = gbmoe.moe_gate_topk(lg.cuda(), shape.topk, cfg)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_s) and torch.equal(w, w_s), "the layer's routing differs from moe_gate_topk's"
    return d, lg.numpy(), out.float().cpu().numpy(), ids.cpu(), w.cpu()


@pytest.mark.parametrize("M,flags", [(4, gbmoe.MOE_PATH_AUTO), (64, gbmoe.MOE_PATH_AUTO),
                                     (65, gbmoe.MOE_PATH_AUTO), (300, gbmoe.MOE_PATH_AUTO),
                                     (40, gbmoe.MOE_ACT_FP8_1X128)])
def test_gated_layer_fp8_sigmoid_router(M, flags):
    # inline ranking (M <= 64) and a separate launch (M > 64), on both paths
    shape = synth.LayerShape("g", M, 256, 128, 64, 6, "fp8", "deepseek", shared_expert=True, n_group=8,
                             topk_group=4, routed_scaling=2.5,
                             act="fp8_1x128" if flags & gbmoe.MOE_ACT_FP8_1X128 else "a16")
    cfg = gbmoe.gate_config(SIG, 8, 4, 2.5, None, True)
    d, lg, out, ids, w = _gated_layer(shape, M, cfg, flags)
    check_grouped(lg, 6, 8, 4, 2.5, None, ids.numpy(), w.numpy(), shared=True)
    d["topk_ids"], d["topk_weights"] = ids, w
    act = "fp8_1x128" if flags & gbmoe.MOE_ACT_FP8_1X128 else "a16"
    assert_layer_close(out, oracle.fused_moe_fp8(**d, act=act), f"gated FP8 layer M{M}")


@pytest.mark.parametrize("M", [3, 200])
def test_gated_layer_int8_softmax_router(M):
    shape = synth.LayerShape("g", M, 512, 256, 32, 4, "int8", "softmax")
    cfg = gbmoe.gate_config()
    d, lg, out, ids, w = _gated_layer(shape, 7 * M, cfg)
    check_softmax(lg, 4, ids.numpy(), w.numpy())
    d["topk_ids"], d["topk_weights"] = ids, w
    assert_layer_close(out, oracle.fused_moe_int8(**d), f"gated INT8 layer M{M}")


def test_gated_layer_deepseek_full_size_decode():
    shape = synth.deepseek_r1(4)
    cfg = gbmoe.gate_config(SIG, shape.n_group, shape.topk_group, shape.routed_scaling, None, True)
    d, lg, out, ids, w = _gated_layer(shape, 11, cfg, full_size=True)
    check_grouped(lg, 8, 8, 4, shape.routed_scaling, None, ids.numpy(), w.numpy(), shared=True)
    ref = oracle.fused_moe_rows(d["x"], ids, w, d["w13"], d["w13_scale"], d["w2"], d["w2_scale"], kind="fp8",
                                tokens=[0, 3])
    assert_layer_close(out[[0, 3]], ref, "gated DeepSeek decode layer")
