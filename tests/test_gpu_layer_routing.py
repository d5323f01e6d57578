"""The routing alignment inside the fused layer, read back with moe_read_routing.

Up to 4096 (token, slot) pairs one CTA aligns them; longer id lists are split
into chunks of consecutive slots, one CTA each, whose cursors start after the
chunks before them.  Either way the result must equal the oracle's stable
argsort bit for bit, ids outside [0, E) must be counted once each, and the
layer's output must still meet the tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from _layers import assert_layer_close, expert_id_expected, expert_id_layer, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def _routing_matches_oracle(ws, ids, M, H, I, E, topk, kind, flags):
    B, s, eid, npp, off = gbmoe.moe_read_routing(ws, M, H, I, E, topk, kind, flags)
    torch.cuda.synchronize()
    ref = oracle.moe_align_block_size(ids, E, B)
    np.testing.assert_array_equal(s.cpu().numpy(), ref[0])
    np.testing.assert_array_equal(eid.cpu().numpy(), ref[1])
    assert int(npp.item()) == int(ref[2])
    np.testing.assert_array_equal(off.cpu().numpy(), ref[3])


@pytest.mark.parametrize("M,topk,E,flags", [
    (4, 9, 257, gbmoe.MOE_PATH_AUTO),                              # one CTA, decode block size
    (300, 8, 64, gbmoe.MOE_PATH_PREFILL),                          # one CTA at 2400 slots
    (2048, 9, 257, gbmoe.MOE_PATH_PREFILL),                        # 5 chunks
    (5000, 8, 1024, gbmoe.MOE_PATH_PREFILL),                       # 10 chunks, most experts
    (16384, 9, 257, gbmoe.MOE_PATH_PREFILL | gbmoe.MOE_ACT_FP8_1X128),  # 36 chunks
    (40000, 8, 16, gbmoe.MOE_PATH_PREFILL),                        # 79 chunks' worth, capped at 64
])
def test_layer_alignment_is_the_stable_argsort(M, topk, E, flags):
    H, I = 256, 128
    if E == 257:  # DeepSeek-R1 routing with Zipf-skewed popularity: 256 routed experts top-8 + the shared one
        shape = synth.LayerShape("r", M, H, I, 256, 8, "fp8", "deepseek_zipf", shared_expert=True, n_group=8,
                                 topk_group=4)
    else:
        shape = synth.LayerShape("r", M, H, I, E, topk, "fp8", "uniform")
    ids, w = synth.make_routing(shape, seed=M + E)
    ids = ids.numpy()
    d = expert_id_layer(M, topk, E, H, I, seed=M)
    d["topk_ids"] = torch.from_numpy(ids.astype(np.int32))
    d["topk_weights"] = w
    dd = to_device(d)
    ws = gbmoe.alloc_workspace(M, H, I, E, topk, gbmoe.MOE_WEIGHT_FP8, flags)
    out = gbmoe.fused_moe_fp8(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"], dd["w2"],
                              dd["w2_scale"], flags=flags, workspace=ws)
    _routing_matches_oracle(ws, ids, M, H, I, E, topk, gbmoe.MOE_WEIGHT_FP8, flags)
    if not flags & gbmoe.MOE_ACT_FP8_1X128:  # the structured layer is exact in the weight-only mode
        exp = expert_id_expected(d)
        got = out.float().cpu().numpy()
        assert_layer_close(got, np.repeat(exp[:, None], H, axis=1), f"expert-id layer M={M}")


def test_split_alignment_counts_every_bad_id_once():
    M, topk, E, H, I = 3000, 8, 32, 256, 128
    rng = np.random.default_rng(5)
    ids = rng.integers(0, E, size=(M, topk))
    bad = rng.random(size=ids.shape) < 0.03
    ids[bad] = rng.choice([-1, E, E + 7, -100], size=int(bad.sum()))
    shape = synth.LayerShape("b", M, H, I, E, topk, "fp8", "uniform")
    d = synth.make_layer(shape, seed=6)
    d["topk_ids"] = torch.from_numpy(ids.astype(np.int32))
    dd = to_device(d)
    flags = gbmoe.MOE_PATH_PREFILL
    ws = gbmoe.alloc_workspace(M, H, I, E, topk, gbmoe.MOE_WEIGHT_FP8, flags)
    for _ in range(2):  # the second call must not carry the first call's count
        out = gbmoe.fused_moe_fp8(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"],
                                  dd["w2"], dd["w2_scale"], flags=flags, workspace=ws)
        n_bad, fl, st = gbmoe.moe_read_status(ws)
        assert (n_bad, fl, st) == (int(bad.sum()), 0, 6)
    _routing_matches_oracle(ws, ids, M, H, I, E, topk, gbmoe.MOE_WEIGHT_FP8, flags)
    assert_layer_close(out.float().cpu().numpy(), oracle.fused_moe_fp8(**d), "split alignment with bad ids")


@pytest.mark.parametrize("kind,M,flags", [
    ("int8", 4096, gbmoe.MOE_PATH_AUTO), ("int4", 700, gbmoe.MOE_PATH_AUTO), ("int8", 16, gbmoe.MOE_PATH_AUTO),
    ("int4", 700, gbmoe.MOE_PATH_DECODE),  # the weight-streaming kernels behind a split alignment
])
def test_layer_alignment_other_weight_kinds(kind, M, flags):
    E, topk, H, I = 128, 8, 256, 128
    shape = synth.LayerShape("k", M, H, I, E, topk, kind, "softmax")
    dh = synth.make_layer(shape, seed=M)
    d = to_device(dh)
    k = {"int8": gbmoe.MOE_WEIGHT_INT8, "int4": gbmoe.MOE_WEIGHT_INT4}[kind]
    fn = {"int8": gbmoe.fused_moe_int8, "int4": gbmoe.fused_moe_int4}[kind]
    ws = gbmoe.alloc_workspace(M, H, I, E, topk, k, flags)
    out = fn(d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
             flags=flags, workspace=ws)
    _routing_matches_oracle(ws, d["topk_ids"].cpu().numpy(), M, H, I, E, topk, k, flags)
    ref = (oracle.fused_moe_int8 if kind == "int8" else oracle.fused_moe_int4)(**dh)
    assert_layer_close(out.float().cpu().numpy(), ref, f"{kind} M={M} flags {flags:#x}")
