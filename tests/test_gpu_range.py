"""The weight-only layers over the whole range of their inputs, against the float64 oracle.

The FP8 and INT4 weight-only layers multiply fp16 operands on the tensor cores while
x arrives as bf16 (the exponent range of fp32) and the intermediate h is an fp32
result.  Both are carried in power-of-two frames (one per x row, one per 32-column
block of h, brought to one frame per row before the down projection), and on the
tcgen05 path the FP8 block scales are folded into the weights relative to a frame per
128-row block.  These tests push each of those past fp16's range on both kernel
paths:

* x rows whose magnitudes run from 1e-12 to 1e15 (fp16 holds neither end), each row
  also checked against its own norm;
* an intermediate h far past fp16's largest value (65504);
* rows of h whose 32-column blocks lie up to 18 binades apart, with the down projection
  weighting the small blocks up so that they carry half of every output;
* FP8 block scales drawn log-uniformly from 2^-20 to 2^8.
"""
import numpy as np
import pytest
import torch

import oracle
from _layers import assert_layer_close, errors, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu

PATHS = {"decode": gbmoe.MOE_PATH_DECODE, "prefill": gbmoe.MOE_PATH_PREFILL}


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


def _layer(kind, seed, M=40, H=512, I=256, E=6, topk=2, std=0.02):
    shape = synth.LayerShape("range", M, H, I, E, topk, kind, "softmax")
    d = synth.make_layer(shape, seed)
    if std != 0.02:
        d["w13"], d["w13_scale"], d["w2"], d["w2_scale"] = synth.make_weights(shape, seed, std=std)
    return d


def _row_scaled_x(d, scales, seed):
    """x with row r multiplied by scales[r % len(scales)] (the product rounded to bf16)."""
    M = d["x"].shape[0]
    f = torch.tensor([scales[r % len(scales)] for r in range(M)], dtype=torch.float64)
    d["x"] = (d["x"].double() * f[:, None]).to(torch.bfloat16)
    return f


def _run(kind, d, flags):
    dd = to_device(d)
    fn = gbmoe.fused_moe_fp8 if kind == "fp8" else gbmoe.fused_moe_int4
    out = fn(dd["x"], dd["topk_ids"], dd["topk_weights"], dd["w13"], dd["w13_scale"], dd["w2"], dd["w2_scale"],
             flags=flags)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def _oracle(kind, d):
    fn = oracle.fused_moe_fp8 if kind == "fp8" else oracle.fused_moe_int4
    return fn(d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"])


def _check_rows(out, ref, what):
    """The layer tolerance over the whole output, and the rel-L2 bound on every row by itself."""
    assert np.isfinite(out).all(), f"{what}: non-finite outputs"
    assert_layer_close(out, ref, what)
    for r in range(ref.shape[0]):
        if np.linalg.norm(ref[r]) == 0.0:
            assert np.abs(out[r]).max() == 0.0, f"{what}: row {r} should be zero"
            continue
        rel, mabs = errors(out[r], ref[r])
        assert rel <= 5e-3 and mabs <= 1e-2, f"{what}: row {r}: rel-L2 {rel:.3e}, max-abs {mabs:.3e}"


ROW_SCALES = [1e-12, 1e-5, 1.0, 3e5, 1e9, 1e15]


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("kind", ["fp8", "int4"])
def test_x_rows_beyond_fp16_range(kind, path):
    d = _layer(kind, seed=11)
    _row_scaled_x(d, ROW_SCALES, seed=11)
    ref = _oracle(kind, d)
    assert np.abs(ref).max() > 1e25 and np.abs(ref[0]).max() < 1e-20  # the rows span the range
    _check_rows(_run(kind, d, PATHS[path]), ref, f"{kind} {path}: x rows 1e-12 .. 1e15")


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("kind", ["fp8", "int4"])
def test_h_past_fp16_max(kind, path):
    d = _layer(kind, seed=12, std=0.5)
    d["x"] = (d["x"].float() * 100.0).to(torch.bfloat16)
    # the intermediate of the oracle's first token, first expert, exceeds fp16's range by far
    e = int(d["topk_ids"][0, 0])
    deq = oracle.dequant_fp8_block if kind == "fp8" else oracle.dequant_int4_group
    W13 = deq(d["w13"][e].numpy(), d["w13_scale"][e].numpy())
    I = W13.shape[0] // 2
    C = d["x"][0].double().numpy() @ W13.T
    assert np.abs(oracle.silu(C[:I]) * C[I:]).max() > 1e6
    ref = _oracle(kind, d)
    _check_rows(_run(kind, d, PATHS[path]), ref, f"{kind} {path}: h past 65504")


@pytest.mark.parametrize("path", sorted(PATHS))
def test_h_blocks_in_distant_frames(path):
    """Gate row block rb of every expert scaled by 2^(6 rb): h's 32-column blocks 4 rb .. 4 rb + 3
    then lie 6 binades apart per row block, 18 across the row (several frames, so rows have
    blocks below their frame), and W2's K blocks are scaled by 2^(-6 kb) so each carries as
    much of y."""
    d = _layer("fp8", seed=13, I=512)
    s13 = d["w13_scale"].clone()
    I = d["w13"].shape[1] // 2
    nrb = I // 128
    for rb in range(nrb):
        s13[:, rb, :] *= 2.0 ** (6 * rb)
    d["w13_scale"] = s13
    s2 = d["w2_scale"].clone()
    for kb in range(nrb):
        s2[:, :, kb] *= 2.0 ** (-6 * kb)
    d["w2_scale"] = s2
    ref = _oracle("fp8", d)
    _check_rows(_run("fp8", d, PATHS[path]), ref, f"fp8 {path}: h blocks 6 to 18 binades apart")
    # and without the W2 compensation: the small blocks then matter less, but are still summed
    d["w2_scale"] = _layer("fp8", seed=13, I=512)["w2_scale"]
    ref = _oracle("fp8", d)
    _check_rows(_run("fp8", d, PATHS[path]), ref, f"fp8 {path}: h blocks 6 to 18 binades apart, plain W2")


@pytest.mark.parametrize("path", sorted(PATHS))
def test_fp8_block_scales_2m20_to_2p8(path):
    d = _layer("fp8", seed=14)
    g = torch.Generator().manual_seed(14)
    for k in ("w13_scale", "w2_scale"):
        s = d[k]
        d[k] = torch.exp2(torch.empty(s.shape, dtype=torch.float64).uniform_(-20.0, 8.0, generator=g)).float()
    ref = _oracle("fp8", d)
    _check_rows(_run("fp8", d, PATHS[path]), ref, f"fp8 {path}: block scales 2^-20 .. 2^8")


@pytest.mark.parametrize("path", sorted(PATHS))
def test_fp8_uniform_tiny_and_huge_scales(path):
    """Every block scale of an expert 2^-20 (weights far below fp16's normal range) or 2^8."""
    d = _layer("fp8", seed=15)
    E = d["w13"].shape[0]
    for k in ("w13_scale", "w2_scale"):
        f = torch.tensor([2.0 ** -20 if e % 2 == 0 else 2.0 ** 8 for e in range(E)])
        d[k] = d[k] * f[:, None, None] / d[k].mean()
    ref = _oracle("fp8", d)
    _check_rows(_run("fp8", d, PATHS[path]), ref, f"fp8 {path}: scales 2^-20 and 2^8 per expert")


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("kind", ["fp8", "int4"])
def test_masked_rows_beyond_fp16_range(kind, path):
    E, cap, H, I = 4, 24, 512, 256
    shape = synth.LayerShape("m", E * cap, H, I, E, 1, kind, "uniform")
    w13, s13, w2, s2 = synth.make_weights(shape, 16)
    x = synth.make_x(shape, 16)
    f = torch.tensor([ROW_SCALES[r % len(ROW_SCALES)] for r in range(E * cap)], dtype=torch.float64)
    x = (x.double() * f[:, None]).to(torch.bfloat16).view(E, cap, H)
    m = torch.tensor([cap, 7, 0, 13], dtype=torch.int32)
    ids = np.full((E * cap, 1), -1, dtype=np.int32)
    for e in range(E):
        ids[e * cap:e * cap + int(m[e]), 0] = e
    fn = oracle.fused_moe_fp8 if kind == "fp8" else oracle.fused_moe_int4
    ref = fn(x.reshape(E * cap, H), torch.from_numpy(ids), torch.ones(E * cap, 1), w13, s13, w2, s2)
    kd = gbmoe.MOE_WEIGHT_FP8 if kind == "fp8" else gbmoe.MOE_WEIGHT_INT4
    out = torch.zeros(E, cap, H, dtype=torch.bfloat16, device="cuda")
    gbmoe.fused_moe_masked(kd, x.cuda(), m.cuda(), w13.cuda(), s13.cuda(), w2.cuda(), s2.cuda(), out=out,
                           flags=PATHS[path])
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(E * cap, H).astype(np.float64)
    real = ids[:, 0] >= 0
    _check_rows(got[real], ref[real], f"masked {kind} {path}: x rows 1e-12 .. 1e15")
