"""GPU parity of the masked (fixed-capacity) layout, and CUDA-graph capture of the layer.

The oracle of the masked layout is the plain layer on the flattened rows with
one expert per row (topk 1, weight 1): row (e, i) goes to expert e when
i < masked_m[e] and is dropped otherwise.  Real rows must meet the layer
tolerance; padding rows of the output must be left untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from _layers import assert_layer_close, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def _masked_inputs(E, cap, H, I, kind, seed, counts=None):
    shape = synth.LayerShape("m", E * cap, H, I, E, 1, kind, "uniform")
    w13, s13, w2, s2 = synth.make_weights(shape, seed)
    x = synth.make_x(shape, seed).view(E, cap, H)
    rng = np.random.default_rng(seed)
    m = np.asarray(counts if counts is not None else rng.integers(0, cap + 1, size=E), dtype=np.int32)
    return x, torch.from_numpy(m), (w13, s13, w2, s2)


def _oracle_masked(x, m, weights, kind, rows=None):
    E, cap, H = x.shape
    mc = np.clip(m.numpy(), 0, cap)
    ids = np.full((E * cap, 1), -1, dtype=np.int32)
    for e in range(E):
        ids[e * cap:e * cap + mc[e], 0] = e
    ids_t = torch.from_numpy(ids)
    w = torch.ones(E * cap, 1)
    xf = x.reshape(E * cap, H)
    if rows is not None:
        return oracle.fused_moe_rows(xf, ids_t, w, *weights, kind=kind, tokens=rows), mc
    fn = oracle.fused_moe_fp8 if kind == "fp8" else oracle.fused_moe_int4
    return fn(xf, ids_t, w, *weights), mc


def _run(x, m, weights, kind, out=None, flags=gbmoe.MOE_PATH_AUTO):
    kd = gbmoe.MOE_WEIGHT_FP8 if kind == "fp8" else gbmoe.MOE_WEIGHT_INT4
    w = [t.cuda() for t in weights]
    if out is None:
        out = torch.full(x.shape, SENTINEL, dtype=torch.bfloat16, device="cuda")
    gbmoe.fused_moe_masked(kd, x.cuda(), m.cuda(), *w, out=out, flags=flags)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def _check(out, ref, mc, what):
    E, cap, H = out.shape
    real = np.zeros((E, cap), dtype=bool)
    for e in range(E):
        real[e, :mc[e]] = True
    assert (out[~real] == SENTINEL).all(), f"{what}: padding rows were written"
    if real.any():
        assert_layer_close(out[real], ref.reshape(E, cap, H)[real], what)


@pytest.mark.parametrize("kind", ["fp8", "int4"])
@pytest.mark.parametrize("E,cap,H,I,counts", [
    (8, 16, 256, 128, None),                      # random counts 0..cap
    (4, 21, 512, 256, [21, 0, 8, 13]),            # full, empty, one tile, a ragged tile
    (1, 1, 256, 128, [1]),                        # a single row
    (6, 40, 256, 256, [-3, 99, 40, 17, 0, 1]),    # out-of-range counts are clamped to [0, cap]
    (3, 9, 7168, 256, [9, 4, 2]),                 # long K
])
def test_masked_layout(kind, E, cap, H, I, counts):
    x, m, weights = _masked_inputs(E, cap, H, I, kind, seed=E * cap + H, counts=counts)
    ref, mc = _oracle_masked(x, m, weights, kind)
    _check(_run(x, m, weights, kind), ref, mc, f"masked {kind} E{E} cap{cap}")


@pytest.mark.parametrize("E,cap,H,I,counts", [
    (4, 300, 256, 256, [300, 0, 129, 17]),        # several 128-row tiles, an empty expert, ragged tails
    (8, 16, 256, 128, None),
    (2, 40, 7168, 512, [40, 33]),                 # long K
])
@pytest.mark.parametrize("kind", ["fp8", "int4"])
def test_masked_layout_tcgen05_path(kind, E, cap, H, I, counts):
    x, m, weights = _masked_inputs(E, cap, H, I, kind, seed=E + cap + I, counts=counts)
    ref, mc = _oracle_masked(x, m, weights, kind)
    _check(_run(x, m, weights, kind, flags=gbmoe.MOE_PATH_PREFILL), ref, mc, f"masked {kind} tcgen05 E{E} cap{cap}")


def test_masked_deepseek_local_experts_full_size():
    # 32 local experts of a DeepSeek-R1 layer (256 experts over 8 ranks), up to 64 rows each
    E, cap, H, I = 32, 64, 7168, 2048
    shape = synth.LayerShape("m", E * cap, H, I, E, 1, "fp8", "uniform")
    x = synth.make_x(shape, 5).view(E, cap, H)
    m = torch.from_numpy(np.random.default_rng(5).integers(0, cap + 1, size=E).astype(np.int32))
    w = list(synth.make_weights(shape, 5, device="cuda"))  # the oracle reads them one expert at a time
    mc = np.clip(m.numpy(), 0, cap)
    rows = [e * cap + i for e, i in ((0, 0), (int(np.argmax(mc)), int(mc.max()) - 1)) if mc[e] > i]
    out = torch.full(x.shape, SENTINEL, dtype=torch.bfloat16, device="cuda")
    gbmoe.fused_moe_masked(gbmoe.MOE_WEIGHT_FP8, x.cuda(), m.cuda(), *w, out=out)
    torch.cuda.synchronize()
    ref, _ = _oracle_masked(x, m, w, "fp8", rows=rows)
    got = out.float().cpu().numpy().reshape(E * cap, H)[rows]
    assert_layer_close(got, ref, "masked DeepSeek-R1 local experts")


# both paths: the weight-streaming kernels, and the tcgen05 ones (FP8: the two-term form written by the prologue)
@pytest.mark.parametrize("flags,cap", [(gbmoe.MOE_PATH_AUTO, 24), (gbmoe.MOE_PATH_PREFILL, 150)])
def test_masked_layout_in_a_cuda_graph_replays_with_new_counts(flags, cap):
    E, H, I = 8, 256, 128
    first = [min(c, cap) for c in (cap, 3, 0, 9, 16, 1, 8, cap)]
    x, m, weights = _masked_inputs(E, cap, H, I, "fp8", seed=11, counts=first)
    xd, md = x.cuda(), m.cuda()
    w = [t.cuda() for t in weights]
    out = torch.full(x.shape, SENTINEL, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gbmoe.moe_workspace_size_masked(E, cap, H, I, gbmoe.MOE_WEIGHT_FP8), dtype=torch.uint8,
                     device="cuda")
    gbmoe.fused_moe_masked(gbmoe.MOE_WEIGHT_FP8, xd, md, *w, out=out, workspace=ws, flags=flags)  # eager first
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gbmoe.fused_moe_masked(gbmoe.MOE_WEIGHT_FP8, xd, md, *w, out=out, workspace=ws, flags=flags)
    for counts in (first, [0, cap, 5, 0, 2, cap - 1, 12, 7]):
        md.copy_(torch.tensor(counts, dtype=torch.int32))
        out.fill_(SENTINEL)
        g.replay()
        torch.cuda.synchronize()
        ref, mc = _oracle_masked(x, torch.tensor(counts, dtype=torch.int32), weights, "fp8")
        _check(out.float().cpu().numpy(), ref, mc, f"graph replay {counts}")


# 4 tokens take the weight-streaming kernels, 160 the tcgen05 ones (MOE_PATH_AUTO)
@pytest.mark.parametrize("M", [4, 160])
def test_routed_layer_in_a_cuda_graph_replays_with_new_routing(M):
    shape = synth.LayerShape("g", M, 512, 256, 16, 3, "fp8", "softmax")
    d = to_device(synth.make_layer(shape, seed=12))
    ws = gbmoe.alloc_workspace(M, 512, 256, 16, 3, gbmoe.MOE_WEIGHT_FP8)
    out = torch.empty(M, 512, dtype=torch.bfloat16, device="cuda")
    args = (d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"])
    gbmoe.fused_moe_fp8(*args, out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gbmoe.fused_moe_fp8(*args, out=out, workspace=ws)
    for seed in (13, 14):
        r = synth.make_layer(synth.LayerShape("g", M, 512, 256, 16, 3, "fp8", "softmax"), seed=seed)
        d["topk_ids"].copy_(r["topk_ids"])
        d["topk_weights"].copy_(r["topk_weights"])
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.fused_moe_fp8(d["x"].cpu(), r["topk_ids"], r["topk_weights"], *[t.cpu() for t in args[3:]])
        assert_layer_close(out.float().cpu().numpy(), ref, f"graph replay seed {seed}")
