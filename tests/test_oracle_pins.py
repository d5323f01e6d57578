"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test ties one oracle function to something independent of it: a library
routine (torch's float8_e4m3fn conversion), a closed form, a hand-worked
fixture, an exact integer identity stated on the pages, brute force, or a
textbook dense FFN.  They run without a GPU.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_moe_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- E4M3 codec

def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF only
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_spec_values():
    d = oracle.e4m3_decode
    assert d(0x38) == 1.0            # 0.0111.000
    assert d(0x7E) == 448.0          # largest finite
    assert d(0x08) == 2.0 ** -6      # smallest normal
    assert d(0x01) == 2.0 ** -9      # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert d(0xB8) == -1.0
    assert d(0x80) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.normal(0, 50, 20000), rng.normal(0, 0.01, 20000),
        rng.uniform(-448, 448, 20000),
    ]).astype(np.float32)
    # exact midpoints between neighbouring grid values: the tie cases
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (grid[:-1] + grid[1:]) / 2)
    v = np.concatenate([v, mids, -mids, grid.astype(np.float32)])
    ours = oracle.e4m3_encode_satfinite(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates():
    v = np.array([448.0, 449.0, 463.9, 464.0, 1e6, np.inf, -1e30, -np.inf], np.float32)
    c = oracle.e4m3_encode_satfinite(v)
    assert list(c) == [0x7E] * 6 + [0xFE] * 2


# --------------------------------------------------------------------------- dequantisation

def test_fp8_block_scale_indexing():
    # all codes 1.0; distinct scales per 128x128 block of a 256 x 384 matrix
    codes = np.full((256, 384), 0x38, np.uint8)
    scale = np.array([[2.0, 3.0, 5.0], [7.0, 11.0, 13.0]], np.float32)
    W = oracle.dequant_fp8_block(codes, scale)
    assert W[0, 0] == 2.0 and W[127, 127] == 2.0
    assert W[128, 0] == 7.0 and W[255, 5] == 7.0
    assert W[5, 128] == 3.0 and W[5, 300] == 5.0
    assert W[200, 383] == 13.0 and W[130, 200] == 11.0


def test_int8_channel_dequant():
    q = np.array([[1, -2], [127, -127]], np.int8)
    s = np.array([0.5, 2.0], np.float32)
    assert np.array_equal(oracle.dequant_int8_channel(q, s), [[0.5, -1.0], [254.0, -254.0]])


# --------------------------------------------------------------------------- dynamic INT8 quant

def test_int8_row_quant_reduces_to_rounding_when_scale_is_one():
    # amax 127 -> s == 1 exactly, so q is plain round-half-even of x
    row = np.array([[127.0, 2.5, 3.5, -2.5, -3.5, 0.49, -0.5, 126.5, -127.0]], np.float32)
    q, s = oracle.quant_int8_per_row(row)
    assert s[0] == 1.0
    assert list(q[0]) == [127, 2, 4, -2, -4, 0, 0, 126, -127]


def test_int8_row_quant_properties():
    rng = np.random.default_rng(1)
    a = (rng.normal(size=(64, 333)) * rng.uniform(0.01, 100, size=(64, 1))).astype(np.float32)
    a[3] = 0.0
    q, s = oracle.quant_int8_per_row(a)
    assert s[3] == 1.0 and not q[3].any()
    nz = np.arange(64) != 3
    assert np.all(np.abs(q[nz]).max(axis=1) == 127)
    err = np.abs(a[nz].astype(np.float64) / s[nz, None] - q[nz])
    assert err.max() <= 0.5 + 1e-5


# --------------------------------------------------------------------------- U8S8 identity (pages)

def test_u8s8_compensation_identity_exact():
    """A x B = (A + 128) x B - 128 x B in exact integers (DA8W8 on VNNI)."""
    rng = np.random.default_rng(2)
    A = rng.integers(-128, 128, size=(37, 300)).astype(np.int64)
    B = rng.integers(-128, 128, size=(300, 53)).astype(np.int64)
    U = A + 128
    assert U.min() >= 0 and U.max() <= 255
    comp = 128 * B.sum(axis=0, keepdims=True)
    assert np.array_equal(U @ B - comp, A @ B)


# --------------------------------------------------------------------------- routing alignment

def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = [int(x) for x in v]
    return out


def test_align_hand_worked_fixture():
    g = _read_golden("align_tiny.txt")
    M, k, E, B = g["M"][0], g["topk"][0], g["E"][0], g["B"][0]
    ids = np.array(g["topk_ids"]).reshape(M, k)
    s, eid, n, off, cnt = oracle.moe_align_block_size(ids, E, B)
    assert list(s) == g["sorted_ids"]
    assert list(eid) == g["expert_ids"]
    assert int(n) == g["num_post_padded"][0]
    assert list(off) == g["expert_offsets"]
    assert list(cnt) == g["counts"]


def _check_align_invariants(ids, E, B, res):
    s, eid, n, off, cnt = res
    M, k = ids.shape
    flat = ids.reshape(-1)
    sentinel = M * k
    assert len(s) == oracle.max_padded(M, k, E, B) and len(eid) == len(s) // B
    seen = []
    for e in range(E):
        assert off[e] % B == 0 and off[e + 1] >= off[e]
        grp = s[off[e]:off[e + 1]]
        real = [int(i) for i in grp if i != sentinel]
        want = [i for i in range(M * k) if flat[i] == e]  # brute force: ascending slots
        assert real == want
        assert list(grp[:len(real)]) == real and all(i == sentinel for i in grp[len(real):])
        assert off[e + 1] - off[e] == -(-len(want) // B) * B
        assert all(eid[b] == e for b in range(off[e] // B, off[e + 1] // B))
        seen += real
    assert int(n) == off[E]
    assert all(x == sentinel for x in s[n:]) and all(x == -1 for x in eid[n // B:])
    assert sorted(seen) == [i for i in range(M * k) if 0 <= flat[i] < E]


def test_align_brute_force_all_tiny_cases():
    for M, k, E in [(1, 1, 1), (1, 2, 3), (2, 2, 3), (3, 1, 4), (3, 2, 2), (2, 2, 4)]:
        for B in (1, 2, 4):
            for combo in itertools.product(range(-1, E + 1), repeat=M * k):
                ids = np.array(combo).reshape(M, k)
                _check_align_invariants(ids, E, B, oracle.moe_align_block_size(ids, E, B))


def test_align_random_larger():
    rng = np.random.default_rng(3)
    for M, k, E, B in [(100, 8, 257, 16), (37, 2, 8, 64), (513, 6, 33, 128)]:
        ids = rng.integers(0, E, size=(M, k))
        _check_align_invariants(ids, E, B, oracle.moe_align_block_size(ids, E, B))


# --------------------------------------------------------------------------- layer

def _torch_dequant_fp8(codes, scale):
    """Library path: torch's float8 conversion, scales broadcast with repeat_interleave."""
    w = torch.as_tensor(codes).view(torch.float8_e4m3fn).double()
    s = torch.as_tensor(scale).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
    return w * s


def _dense_swiglu(x, Wg, Wu, Wd):
    """Textbook gated FFN: down(silu(gate(x)) * up(x)), float64 torch."""
    g = x @ Wg.T
    return (torch.nn.functional.silu(g) * (x @ Wu.T)) @ Wd.T


def test_top1_weight1_equals_dense_swiglu_ffn():
    shape = synth.LayerShape("t", 24, 256, 128, 4, 1, "fp8", "softmax")
    d = synth.make_layer(shape, seed=5)
    rng = np.random.default_rng(5)
    ids = torch.from_numpy(rng.integers(0, 4, size=(24, 1)).astype(np.int32))
    w1 = torch.ones(24, 1)
    out = oracle.fused_moe_fp8(d["x"], ids, w1, d["w13"], d["w13_scale"], d["w2"], d["w2_scale"])
    x = d["x"].double()
    I = shape.I
    for t in range(24):
        e = int(ids[t, 0])
        W13 = _torch_dequant_fp8(d["w13"][e], d["w13_scale"][e])
        W2 = _torch_dequant_fp8(d["w2"][e], d["w2_scale"][e])
        ref = _dense_swiglu(x[t:t + 1], W13[:I], W13[I:], W2)[0].numpy()
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-12)


def _blocked_formulation(d, E, B, kind):
    """The sorted/blocked form: one GEMM-SiLU-GEMM per B-row block, scattered back."""
    x = d["x"].double().numpy()
    ids = d["topk_ids"].numpy()
    tw = d["topk_weights"].double().numpy()
    M, k = ids.shape
    s, eid, n, off, cnt = oracle.moe_align_block_size(ids, E, B)
    I = d["w13"].shape[1] // 2
    Y = np.zeros((M * k, x.shape[1]))
    for b in range(int(n) // B):
        e = int(eid[b])
        rows = [int(i) for i in s[b * B:(b + 1) * B] if i < M * k]
        W13 = _torch_dequant_fp8(d["w13"][e], d["w13_scale"][e]).numpy()
        W2 = _torch_dequant_fp8(d["w2"][e], d["w2_scale"][e]).numpy()
        A = x[[r // k for r in rows]]
        C = A @ W13.T
        Y[rows] = (C[:, :I] / (1 + np.exp(-C[:, :I])) * C[:, I:]) @ W2.T
    return (Y.reshape(M, k, -1) * tw[:, :, None]).sum(axis=1)


def test_naive_masked_loop_equals_blocked_formulation():
    shape = synth.tiny(M=40)
    d = synth.make_layer(shape, seed=7)
    ref = oracle.fused_moe_fp8(d["x"], d["topk_ids"], d["topk_weights"],
                               d["w13"], d["w13_scale"], d["w2"], d["w2_scale"])
    for B in (1, 4, 16):
        blk = _blocked_formulation(d, shape.E, B, "fp8")
        np.testing.assert_allclose(ref, blk, rtol=1e-11, atol=1e-12)


def test_silu_fusion_equals_separate_gemms():
    rng = np.random.default_rng(8)
    A = rng.normal(size=(5, 64))
    B1 = rng.normal(size=(32, 64))
    B2 = rng.normal(size=(32, 64))
    C = A @ np.concatenate([B1, B2]).T          # A x [B1, B2] = [C1, C2]
    fused = oracle.silu(C[:, :32]) * C[:, 32:]
    sep = torch.nn.functional.silu(torch.from_numpy(A @ B1.T)).numpy() * (A @ B2.T)
    np.testing.assert_allclose(fused, sep, rtol=1e-14)


def _expert_id_layer(M, topk, E, H=256, I=128, seed=9):
    """Weights whose expert e returns the constant row I*silu(1)*(e+1).

    x[:, 0] = 1, rest 0; gate and up rows are e_0 (code 1.0, scale 1) so
    g = u = 1 and h = silu(1) on every column; W2 codes are all 1.0 with
    every block scale e+1, so y = I * silu(1) * (e+1) on every output.
    """
    x = torch.zeros(M, H, dtype=torch.bfloat16)
    x[:, 0] = 1.0
    w13 = torch.zeros(E, 2 * I, H, dtype=torch.uint8)
    w13[:, :, 0] = 0x38
    s13 = torch.ones(E, 2 * I // 128, H // 128)
    w2 = torch.full((E, H, I), 0x38, dtype=torch.uint8)
    s2 = (torch.arange(E, dtype=torch.float32) + 1)[:, None, None].expand(E, H // 128, I // 128).contiguous()
    rng = np.random.default_rng(seed)
    ids = torch.from_numpy(np.stack([rng.permutation(E)[:topk] for _ in range(M)]).astype(np.int32))
    w = torch.from_numpy(rng.uniform(0.1, 1.0, size=(M, topk)).astype(np.float32))
    return dict(x=x, topk_ids=ids, topk_weights=w, w13=w13, w13_scale=s13, w2=w2, w2_scale=s2)


def expert_id_expected(d):
    I = d["w13"].shape[1] // 2
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    ids = d["topk_ids"].numpy().astype(np.float64)
    w = d["topk_weights"].numpy().astype(np.float64)
    return I * silu1 * (w * (ids + 1)).sum(axis=1)


def test_expert_id_weights_closed_form():
    d = _expert_id_layer(M=11, topk=3, E=8)
    out = oracle.fused_moe_fp8(**d)
    want = expert_id_expected(d)
    np.testing.assert_allclose(out, np.repeat(want[:, None], out.shape[1], axis=1), rtol=1e-13)


def test_int8_lossless_case_closed_form():
    """DA8W8 where every quantisation step is exact: result is a closed form.

    Row t of x is [127, a_t, 0, ...] so its scale is exactly 1.  Gate rows
    pick column 0 (g = 127, silu(127) == 127 in float64), up rows pick column
    1 (u = a_t); h = 127*a_t on every column, so the requant scale is |a_t|
    and every code is +-127.  Then y[m] = 127 * a_t * s2[m] * sum_j c[m, j].
    """
    M, H, I, E, k = 6, 128, 128, 3, 2
    rng = np.random.default_rng(10)
    a = rng.integers(1, 100, size=M) * rng.choice([-1, 1], size=M)
    x = torch.zeros(M, H, dtype=torch.bfloat16)
    x[:, 0] = 127.0
    x[:, 1] = torch.from_numpy(a.astype(np.float32))
    w13 = torch.zeros(E, 2 * I, H, dtype=torch.int8)
    w13[:, :I, 0] = 1
    w13[:, I:, 1] = 1
    s13 = torch.ones(E, 2 * I)
    c = torch.from_numpy(rng.integers(-127, 128, size=(E, H, I)).astype(np.int8))
    s2 = torch.from_numpy(rng.uniform(0.5, 2.0, size=(E, H)).astype(np.float32))
    ids = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32))
    w = torch.from_numpy(rng.uniform(0.1, 1.0, size=(M, k)).astype(np.float32))
    out = oracle.fused_moe_int8(x, ids, w, w13, s13, c, s2)
    rows = c.double().sum(-1).numpy() * s2.double().numpy()      # [E, H]
    want = np.zeros((M, H))
    for t in range(M):
        for j in range(k):
            want[t] += float(w[t, j]) * 127.0 * a[t] * rows[int(ids[t, j])]
    np.testing.assert_allclose(out, want, rtol=1e-12)


def test_int8_close_to_unquantised_activations():
    """DA8W8 differs from the float-activation layer only by 8-bit rounding of rows."""
    shape = synth.LayerShape("q", 12, 256, 128, 6, 2, "int8", "softmax")
    d = synth.make_layer(shape, seed=11)
    q = oracle.fused_moe_int8(**d)
    # same weights dequantised to float, activations unquantised
    x = d["x"].double()
    ref = np.zeros_like(q)
    I = shape.I
    for t in range(12):
        for j in range(2):
            e = int(d["topk_ids"][t, j])
            W13 = d["w13"][e].double() * d["w13_scale"][e].double()[:, None]
            W2 = d["w2"][e].double() * d["w2_scale"][e].double()[:, None]
            ref[t] += float(d["topk_weights"][t, j]) * _dense_swiglu(x[t:t + 1], W13[:I], W13[I:], W2)[0].numpy()
    rel = np.linalg.norm(q - ref) / np.linalg.norm(ref)
    assert 0 < rel < 2e-2


def test_rows_subset_equals_full_call():
    shape = synth.tiny(M=20)
    d = synth.make_layer(shape, seed=12)
    full = oracle.fused_moe_fp8(**d)
    rows = [0, 7, 19]
    sub = oracle.fused_moe_rows(**d, kind="fp8", tokens=rows)
    np.testing.assert_allclose(sub, full[rows], rtol=1e-11, atol=1e-15)  # BLAS blocking differs by size


def test_ids_out_of_range_contribute_nothing():
    shape = synth.tiny(M=10)
    d = synth.make_layer(shape, seed=13)
    base = oracle.fused_moe_fp8(**d)
    ids = d["topk_ids"].clone()
    ids[3, 1] = -1
    ids[5, 0] = shape.E
    d2 = dict(d, topk_ids=ids)
    out = oracle.fused_moe_fp8(**d2)
    keep = [0, 1, 2, 4, 6, 7, 8, 9]
    np.testing.assert_allclose(out[keep], base[keep], rtol=1e-11, atol=1e-15)
    assert not np.allclose(out[3], base[3]) and not np.allclose(out[5], base[5])


# --------------------------------------------------------------------------- FP8 activations, 1 x 128 groups

def _finite_e4m3_codes():
    c = np.arange(256, dtype=np.uint8)
    return c[(c & 0x7F) != 0x7F]


def test_fp8_1x128_exact_codes_closed_form():
    """Groups built as 2^j * decode(code) with one +-448 element: quantisation returns those codes and s = 2^j."""
    rng = np.random.default_rng(21)
    R, G = 6, 5
    codes = rng.choice(_finite_e4m3_codes(), size=(R, G, 128)).astype(np.uint8)
    codes[:, :, 0] = np.where(rng.random((R, G)) < 0.5, 0x7E, 0xFE)  # amax = 448 * 2^j exactly
    j = rng.integers(-20, 21, size=(R, G))
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * np.exp2(j)[..., None]
    a = vals.astype(np.float32).reshape(R, G * 128)
    assert np.array_equal(a.astype(np.float64), vals.reshape(R, -1))  # exact in float32
    q, s = oracle.quant_fp8_1x128(a)
    assert s.dtype == np.float32 and s.shape == (R, G)
    assert np.array_equal(s.astype(np.float64), np.exp2(j))
    assert np.array_equal(q, codes.reshape(R, -1))
    np.testing.assert_array_equal(oracle.dequant_fp8_1x128(q, s), vals.reshape(R, -1))


def test_fp8_1x128_rounding_error_bound_and_amax():
    rng = np.random.default_rng(22)
    R, G = 16, 4
    a = (rng.standard_normal((R, G * 128)) * np.exp2(rng.integers(-8, 9, size=(R, 1)))).astype(np.float32)
    a[3, 5] = 0.0
    q, s = oracle.quant_fp8_1x128(a)
    g = a.reshape(R, G, 128).astype(np.float64)
    amax = np.abs(g).max(-1)
    assert np.array_equal(s, (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32))
    deq = oracle.dequant_fp8_1x128(q, s).reshape(R, G, 128)
    err = np.abs(deq - g)
    sc = s.astype(np.float64)[..., None]
    normal = np.abs(g) >= 2.0 ** -6 * sc
    # half a unit in the last place: 2^-4 relative (3 mantissa bits), 2^-10 * s among subnormals
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(g)[normal] * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * np.broadcast_to(sc, g.shape)[~normal] * (1 + 1e-6))
    # the largest element of every group lands on +-448
    idx = np.abs(g).argmax(-1)
    top = np.take_along_axis(q.reshape(R, G, 128), idx[..., None], -1)[..., 0]
    assert np.all((top == 0x7E) | (top == 0xFE))


def test_fp8_1x128_zero_group_and_group_boundaries():
    a = np.zeros((2, 384), np.float32)
    a[0, 127] = 3.0      # last column of group 0
    a[0, 128] = -0.5     # first column of group 1
    q, s = oracle.quant_fp8_1x128(a)
    assert s[0].tolist() == [np.float32(3.0) / np.float32(448.0), np.float32(0.5) / np.float32(448.0), 1.0]
    assert s[1].tolist() == [1.0, 1.0, 1.0]
    assert q[0, 127] == 0x7E and q[0, 128] == 0xFE
    assert np.count_nonzero(q) == 2
    with pytest.raises(ValueError):
        oracle.quant_fp8_1x128(np.zeros((1, 100), np.float32))


def test_a8_layer_top1_identity_down_projection_closed_form():
    """Top-1 routing, weight 1, W2 = identity: out = dequant(quant(h)) of h = SiLU(a W1^T) * (a W3^T),
    a = dequant(quant(x)) -- the quantiser is applied per token row, to x and to h."""
    shape = synth.LayerShape("a8", 6, 256, 256, 2, 1, "fp8", "softmax")
    d = synth.make_layer(shape, seed=23)
    rng = np.random.default_rng(23)
    ids = torch.from_numpy(rng.integers(0, 2, size=(6, 1)).astype(np.int32))
    w2 = torch.zeros(2, 256, 256, dtype=torch.uint8)
    w2[:, torch.arange(256), torch.arange(256)] = 0x38  # E4M3 1.0
    s2 = torch.ones(2, 2, 2)
    out = oracle.fused_moe_fp8(d["x"], ids, torch.ones(6, 1), d["w13"], d["w13_scale"], w2, s2, act="fp8_1x128")

    def deq(a):
        q, s = oracle.quant_fp8_1x128(np.asarray(a, np.float32))
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy().reshape(len(q), -1, 128)
        return (v * s.astype(np.float64)[..., None]).reshape(len(q), -1)

    a = torch.from_numpy(deq(d["x"].float().numpy()))
    for t in range(6):
        e = int(ids[t, 0])
        W13 = _torch_dequant_fp8(d["w13"][e], d["w13_scale"][e])
        h = torch.nn.functional.silu(a[t:t + 1] @ W13[:256].T) * (a[t:t + 1] @ W13[256:].T)
        want = deq(h.numpy())[0]
        np.testing.assert_allclose(out[t], want, rtol=1e-12, atol=0)
        # the h quantisation is really applied: the unquantised h differs
        assert np.abs(h.numpy()[0] - want).max() > 0


def test_a8_layer_close_to_a16():
    shape = synth.LayerShape("a8", 24, 512, 256, 8, 3, "fp8", "softmax")
    d = synth.make_layer(shape, seed=24)
    a16 = oracle.fused_moe_fp8(**d)
    a8 = oracle.fused_moe_fp8(**d, act="fp8_1x128")
    rel = np.linalg.norm(a8 - a16) / np.linalg.norm(a16)
    assert 1e-3 < rel < 6e-2
    sub = oracle.fused_moe_rows(**d, kind="fp8", tokens=[2, 17], act="fp8_1x128")
    np.testing.assert_allclose(sub, a8[[2, 17]], rtol=1e-11, atol=1e-15)


# ----------------------------------------------------------------------------
# Power-of-two (UE8M0) scales.  Pins: exhaustive search over exponents, the OCP
# E8M0 code values, equality with the 1 x 128 quantiser wherever its scale is
# already a power of two, torch's E4M3 cast of the exact quotients, and
# hand-worked re-quantisations of stored weights (ties included).
# ----------------------------------------------------------------------------


def test_ue8m0_ceil_is_the_smallest_power_of_two_not_below():
    rng = np.random.default_rng(31)
    s = np.concatenate([np.exp2(rng.uniform(-135.0, 135.0, 400)), np.exp2(np.arange(-127.0, 128.0)),
                        [1.0, np.nextafter(1.0, 2.0), np.nextafter(1.0, 0.0), 448.0 / 448.0, 3.0 / 448.0, 0.75]])
    v, c = oracle.ue8m0_ceil(s)
    assert v.dtype == np.float64 and c.dtype == np.uint8
    for si, vi, ci in zip(s, v, c):
        e = -127
        while e < 127 and math.ldexp(1.0, e) < si:  # search upwards; the format stops at 2^127
            e += 1
        assert vi == math.ldexp(1.0, e) and int(ci) == e + 127, si
    # OCP E8M0 codes: 127 is 1.0, 0 is 2^-127, 254 is 2^127
    assert oracle.ue8m0_ceil([1.0, 2.0 ** -127, 2.0 ** 127])[1].tolist() == [127, 0, 254]
    assert oracle.ue8m0_ceil([1.5])[0][0] == 2.0 and oracle.ue8m0_ceil([0.75])[0][0] == 1.0
    for bad in (0.0, -1.0, np.inf, np.nan):
        with pytest.raises(ValueError):
            oracle.ue8m0_ceil([bad])


def test_fp8_1x128_ue8m0_equals_the_1x128_quantiser_on_power_of_two_scales():
    """Groups whose amax is 448 * 2^j have the scale 2^j already: both quantisers give the same codes and scales."""
    rng = np.random.default_rng(32)
    R, G = 5, 4
    codes = rng.choice(_finite_e4m3_codes(), size=(R, G, 128)).astype(np.uint8)
    codes[:, :, 7] = np.where(rng.random((R, G)) < 0.5, 0x7E, 0xFE)
    j = rng.integers(-30, 31, size=(R, G))
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * np.exp2(j)[..., None]
    a = vals.astype(np.float32).reshape(R, G * 128)
    q8, s8 = oracle.quant_fp8_1x128(a)
    qu, su = oracle.quant_fp8_1x128_ue8m0(a)
    assert su.dtype == np.float32 and np.array_equal(su, s8) and np.array_equal(qu, q8)
    assert np.array_equal(qu, codes.reshape(R, -1))


def test_fp8_1x128_ue8m0_scales_and_torch_codes():
    rng = np.random.default_rng(33)
    R, G = 12, 5
    a = (rng.standard_normal((R, G * 128)) * np.exp2(rng.integers(-12, 13, size=(R, 1)))).astype(np.float32)
    a[4, 128:256] = 0.0                                   # an all-zero group: scale 1, codes 0
    q, s = oracle.quant_fp8_1x128_ue8m0(a)
    g = a.reshape(R, G, 128)
    amax = np.abs(g).max(-1)
    s32 = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    m, _ = np.frexp(s.astype(np.float64))
    assert np.all(m == 0.5)                               # powers of two
    assert np.all(s.astype(np.float64) / 2 < s32) and np.all(s32 <= s)
    assert s[4, 1] == 1.0 and not q.reshape(R, G, 128)[4, 1].any()
    # every code is torch's round-to-nearest-even E4M3 cast of the element over its (power-of-two) scale,
    # a quotient that float32 holds exactly
    quot = g.astype(np.float64) / s.astype(np.float64)[..., None]
    assert np.array_equal(quot.astype(np.float32).astype(np.float64), quot)
    want = torch.from_numpy(quot.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q.reshape(R, G, 128), want)


def test_requant_fp8_block_ue8m0_hand_worked():
    codes = np.full((128, 256), 0x38, np.uint8)        # E4M3 1.0 everywhere
    codes[0, 0] = 0x7E                                  # 448
    codes[0, 1] = 0xB8                                  # -1.0
    codes[2, 3], codes[2, 4], codes[2, 5] = 0x01, 0x02, 0x03   # subnormals 2^-9, 2^-8, 3 * 2^-9
    codes[5, 130] = 0x01
    scale = np.array([[0.75 * 2.0 ** -3, 2.0 ** -5]], np.float32)  # block 0: not a power of two; block 1: one
    q, s = oracle.requant_fp8_block_ue8m0(codes, scale)
    assert s.dtype == np.float32 and s.tolist() == [[2.0 ** -3, 2.0 ** -5]]
    # block 0: every value times 0.75
    assert q[1, 0] == 0x34                              # 1.0 -> 0.75 = 1.5 * 2^-1
    assert q[0, 0] == 0x7A                              # 448 -> 336, halfway between 320 and 352 -> 320 (even)
    assert q[0, 1] == 0xB4                              # -1.0 -> -0.75
    assert q[2, 3] == 0x01                              # 0.75 * 2^-9 -> 2^-9 (nearest)
    assert q[2, 4] == 0x02                              # 1.5 * 2^-9, halfway between 2^-9 and 2^-8 -> 2^-8 (even)
    assert q[2, 5] == 0x02                              # 2.25 * 2^-9 -> 2^-8
    # block 1 already has a power-of-two scale: its codes stay
    assert np.array_equal(q[:, 128:], codes[:, 128:])


def test_requant_fp8_block_ue8m0_rounds_the_exact_product_once():
    """1.5 * r with r the float32 just above 1.0625 / 1.5 lies just above the E4M3 midpoint 1.0625 (between 1.0
    and 1.125), so it rounds to 1.125; its float32 product is 1.0625 exactly, which would tie to 1.0."""
    r = np.nextafter(np.float32(1.0625 / 1.5), np.float32(1.0))
    assert 1.5 * float(r) > 1.0625 and float(np.float32(1.5) * r) == 1.0625
    codes = np.full((128, 128), 0x3C, np.uint8)                 # 1.5
    q, s = oracle.requant_fp8_block_ue8m0(codes, np.array([[r * np.float32(0.125)]], np.float32))
    assert s.tolist() == [[0.125]] and np.all(q == 0x39)        # 1.125


def test_requant_fp8_block_ue8m0_error_bound():
    rng = np.random.default_rng(34)
    codes = rng.choice(_finite_e4m3_codes(), size=(256, 384)).astype(np.uint8)
    scale = (np.exp2(rng.uniform(-20.0, 4.0, size=(2, 3)))).astype(np.float32)
    scale[1, 2] = np.float32(2.0 ** -7)
    q, s = oracle.requant_fp8_block_ue8m0(codes, scale)
    before = oracle.dequant_fp8_block(codes, scale)
    after = oracle.dequant_fp8_block(q, s)
    sc = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)
    err = np.abs(after - before)
    normal = np.abs(before) >= 2.0 ** -6 * sc
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(before)[normal])
    assert np.all(err[~normal] <= 2.0 ** -10 * sc[~normal])
    assert np.array_equal(q[128:, 256:], codes[128:, 256:])   # the power-of-two block


def test_ue8m0_layer_top1_closed_form():
    """Top-1 routing, weight 1: out = dequant(quant(h)) @ W2'^T with power-of-two scales throughout, h from the
    re-quantised W13' and the power-of-two quantisation of x (W13', W2' re-quantised from the stored blocks)."""
    shape = synth.LayerShape("ue", 5, 256, 256, 2, 1, "fp8", "softmax")
    d = synth.make_layer(shape, seed=35)
    rng = np.random.default_rng(35)
    ids = torch.from_numpy(rng.integers(0, 2, size=(5, 1)).astype(np.int32))
    out = oracle.fused_moe_fp8(d["x"], ids, torch.ones(5, 1), d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                               act="fp8_ue8m0")

    def deq(a):
        q, s = oracle.quant_fp8_1x128_ue8m0(np.asarray(a, np.float32))
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy().reshape(len(q), -1, 128)
        return (v * s.astype(np.float64)[..., None]).reshape(len(q), -1)

    a = torch.from_numpy(deq(d["x"].float().numpy()))
    for t in range(5):
        e = int(ids[t, 0])
        q13, s13 = oracle.requant_fp8_block_ue8m0(d["w13"][e].numpy(), d["w13_scale"][e].numpy())
        q2, s2 = oracle.requant_fp8_block_ue8m0(d["w2"][e].numpy(), d["w2_scale"][e].numpy())
        W13 = _torch_dequant_fp8(torch.from_numpy(q13), torch.from_numpy(s13))
        W2 = _torch_dequant_fp8(torch.from_numpy(q2), torch.from_numpy(s2))
        h = torch.nn.functional.silu(a[t:t + 1] @ W13[:256].T) * (a[t:t + 1] @ W13[256:].T)
        want = torch.from_numpy(deq(h.numpy())) @ W2.T
        np.testing.assert_allclose(out[t], want[0].numpy(), rtol=1e-10, atol=1e-12 * np.abs(want.numpy()).max())
    # both weight tensors were really re-quantised (synthetic block scales are not powers of two), and the
    # down projection is not the a8 one
    for w, sc in (("w13", "w13_scale"), ("w2", "w2_scale")):
        assert not np.array_equal(oracle.requant_fp8_block_ue8m0(d[w][0].numpy(), d[sc][0].numpy())[0], d[w][0].numpy())
    a8 = oracle.fused_moe_fp8(d["x"], ids, torch.ones(5, 1), d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                              act="fp8_1x128")
    assert np.abs(out - a8).max() > 0


def test_ue8m0_layer_close_to_a8_and_a16():
    shape = synth.LayerShape("ue", 24, 512, 256, 8, 3, "fp8", "softmax")
    d = synth.make_layer(shape, seed=24)
    a16 = oracle.fused_moe_fp8(**d)
    a8 = oracle.fused_moe_fp8(**d, act="fp8_1x128")
    ue = oracle.fused_moe_fp8(**d, act="fp8_ue8m0")
    rel = lambda u, v: np.linalg.norm(u - v) / np.linalg.norm(v)  # noqa: E731
    assert 1e-3 < rel(ue, a16) < 8e-2 and 1e-3 < rel(ue, a8) < 8e-2
    # power-of-two scales leave up to a factor 2 of each group's range unused: never a smaller error than A8
    # by much, on average a larger one
    assert rel(ue, a16) > 0.8 * rel(a8, a16)
    sub = oracle.fused_moe_rows(**d, kind="fp8", tokens=[0, 23], act="fp8_ue8m0")
    np.testing.assert_allclose(sub, ue[[0, 23]], rtol=1e-11, atol=1e-15)


# ----------------------------------------------------------------------------
# Gating.  Pins: the selection against exhaustive search over expert subsets on
# integer-valued logits (exact sums, planted ties), torch.topk on tie-free
# inputs, closed forms of the weights, and the group rule checked as an
# invariant rather than re-executed.
# ----------------------------------------------------------------------------


def _best_subset_lexmin(score, k):
    """Exhaustive: the k-subset of maximal total score; among equal totals the
    lexicographically smallest index tuple (lower indices win ties)."""
    best = None
    for c in itertools.combinations(range(len(score)), k):
        tot = sum(score[i] for i in c)
        if best is None or tot > best[0]:
            best = (tot, c)
    return best[1]


def test_gate_softmax_selection_brute_force_with_ties():
    rng = np.random.default_rng(31)
    for trial in range(300):
        E = int(rng.integers(2, 8))
        k = int(rng.integers(1, E + 1))
        lg = rng.integers(-3, 4, size=E).astype(np.float64)  # small integers: many exact ties
        ids, w = oracle.gate_softmax_topk(lg[None, :], k)
        want = _best_subset_lexmin(lg, k)
        assert tuple(sorted(ids[0].tolist())) == want
        # output order: descending score, equal scores by ascending index
        order = sorted(want, key=lambda i: (-lg[i], i))
        assert ids[0].tolist() == order


def test_gate_softmax_weights_closed_form():
    rng = np.random.default_rng(32)
    lg = rng.standard_normal((50, 16)).astype(np.float32)
    # k = E: the weights are the softmax itself (computed here with scipy)
    from scipy.special import softmax
    ids, w = oracle.gate_softmax_topk(lg, 16)
    np.testing.assert_allclose(w, np.take_along_axis(softmax(lg.astype(np.float64), axis=-1), ids, -1),
                               rtol=1e-13)
    # k = 1: weight 1; general k: ratios exp(l_i - l_j) and unit sum
    _, w1 = oracle.gate_softmax_topk(lg, 1)
    np.testing.assert_array_equal(w1, 1.0)
    ids, w = oracle.gate_softmax_topk(lg, 4)
    l_sel = np.take_along_axis(lg.astype(np.float64), ids, -1)
    np.testing.assert_allclose(w[:, 1:] / w[:, :1], np.exp(l_sel[:, 1:] - l_sel[:, :1]), rtol=1e-13)
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=1e-14)
    # tie-free input: the same set and order as torch.topk
    tv, ti = torch.topk(torch.from_numpy(lg.astype(np.float64)), 4, dim=-1)
    np.testing.assert_array_equal(ids, ti.numpy())


def test_gate_grouped_single_group_is_plain_sigmoid_topk():
    rng = np.random.default_rng(33)
    lg = rng.standard_normal((40, 64)).astype(np.float32)
    ids, w = oracle.gate_grouped_sigmoid_topk(lg, 6, n_group=1, topk_group=1, routed_scaling=2.5)
    s = torch.sigmoid(torch.from_numpy(lg.astype(np.float64)))
    tv, ti = torch.topk(s, 6, dim=-1)
    np.testing.assert_array_equal(ids, ti.numpy())
    np.testing.assert_allclose(w, (tv / tv.sum(-1, keepdim=True) * 2.5).numpy(), rtol=1e-14)
    # keeping every group changes nothing either
    ids8, w8 = oracle.gate_grouped_sigmoid_topk(lg, 6, n_group=8, topk_group=8, routed_scaling=2.5)
    np.testing.assert_array_equal(ids8, ids)
    np.testing.assert_allclose(w8, w, rtol=0)


def _check_grouped_invariants(lg, bias, ids, w, k, n_group, topk_group, scale):
    """The group rule stated as properties of the answer."""
    M, E = lg.shape
    gs = E // n_group
    s = 1.0 / (1.0 + np.exp(-lg.astype(np.float64)))
    b = s + bias[None, :]
    for t in range(M):
        gscore = np.array([np.sort(b[t, g * gs:(g + 1) * gs])[-2:].sum() for g in range(n_group)])
        chosen = set(ids[t].tolist())
        assert len(chosen) == k
        groups = {i // gs for i in chosen}
        assert len(groups) <= topk_group
        # some kept set of topk_group groups contains them all, and no group outside
        # a kept set scores higher than one inside it: the chosen groups are among
        # the topk_group best (lower index on equal scores)
        rank = sorted(range(n_group), key=lambda g: (-gscore[g], g))
        kept = set(rank[:topk_group])
        assert groups <= kept
        # within the kept groups nothing unchosen beats a chosen expert
        cand = [i for i in range(E) if i // gs in kept]
        worst = min(b[t, i] for i in chosen)
        for i in cand:
            if i not in chosen:
                assert b[t, i] < worst or (b[t, i] == worst and i > max(j for j in chosen if b[t, j] == worst))
        # weights: unbiased scores, renormalised, scaled
        ss = s[t, ids[t]]
        np.testing.assert_allclose(w[t], ss / ss.sum() * scale, rtol=1e-14)


def test_gate_grouped_invariants_random_and_tied():
    rng = np.random.default_rng(34)
    for trial in range(60):
        n_group = int(rng.choice([2, 4, 8]))
        gs = int(rng.choice([2, 4, 8]))
        E = n_group * gs
        topk_group = int(rng.integers(1, n_group + 1))
        k = int(rng.integers(1, min(8, topk_group * gs) + 1))
        if trial % 2:
            lg = rng.integers(-2, 3, size=(5, E)).astype(np.float32)  # ties inside and across groups
            bias = np.zeros(E)
        else:
            lg = rng.standard_normal((5, E)).astype(np.float32)
            bias = rng.standard_normal(E) * 0.1
        scale = float(rng.choice([1.0, 2.5]))
        ids, w = oracle.gate_grouped_sigmoid_topk(lg, k, n_group, topk_group, bias=bias, routed_scaling=scale)
        _check_grouped_invariants(lg, bias, ids, w, k, n_group, topk_group, scale)


def test_gate_grouped_hand_worked_case():
    # 8 experts in 4 groups of 2, keep 2 groups, pick 2.  Sigmoid is monotone, so
    # ranks follow the logits:  group scores (top-2 sums of s) order the groups
    # 3 > 0 > 1 > 2; the best expert overall (5, group 2) is excluded.
    lg = np.array([[1.0, 0.5, 0.2, 0.6, -3.0, 2.0, 0.9, 0.8]])
    ids, w = oracle.gate_grouped_sigmoid_topk(lg, 2, n_group=4, topk_group=2)
    assert ids.tolist() == [[0, 6]]
    s = 1 / (1 + np.exp(-np.array([1.0, 0.9])))
    np.testing.assert_allclose(w[0], s / s.sum(), rtol=1e-14)
    # a bias moves the selection but not the weights
    bias = np.zeros(8)
    bias[4] = 5.0  # group 2 now scores highest and expert 4 is the best biased score
    ids_b, w_b = oracle.gate_grouped_sigmoid_topk(lg, 2, n_group=4, topk_group=2, bias=bias)
    assert ids_b.tolist() == [[4, 5]]
    s4, s5 = 1 / (1 + np.exp(3.0)), 1 / (1 + np.exp(-2.0))
    np.testing.assert_allclose(w_b[0], [s4 / (s4 + s5), s5 / (s4 + s5)], rtol=1e-14)


def test_gate_matches_the_torch_routing_generator():
    # two implementations of the same rules (numpy here, torch in the input
    # generator) agree on the generator's own logits
    for routing, E, k in (("softmax", 128, 8), ("deepseek", 256, 8)):
        shape = synth.LayerShape("g", 200, 256, 128, E, k, "fp8", routing, shared_expert=False,
                                 n_group=8 if routing == "deepseek" else 1,
                                 topk_group=4 if routing == "deepseek" else 1,
                                 routed_scaling=2.5 if routing == "deepseek" else 1.0)
        ids_ref, w_ref = synth.make_routing(shape, 11)
        lg = synth.make_router_logits(shape, 11).numpy()
        if routing == "softmax":
            ids, w = oracle.gate_softmax_topk(lg, k)
        else:
            ids, w = oracle.gate_grouped_sigmoid_topk(lg, k, shape.n_group, shape.topk_group,
                                                      routed_scaling=shape.routed_scaling)
        np.testing.assert_array_equal(ids, ids_ref.numpy())
        np.testing.assert_allclose(w, w_ref.numpy(), rtol=1e-6)


# ----------------------------------------------------------------------------
# INT4 weights (group-wise, one scale per row and 128 columns).  Pins: the
# nibble decoder against sign extension by arithmetic shifts (a different
# route to the same bits) on all 256 bytes and a hand-worked table, the group
# scale indexing in closed form, and the layer against a textbook dense SwiGLU
# on weights unpacked independently.
# ----------------------------------------------------------------------------


def test_int4_unpack_all_bytes_by_arithmetic_shifts():
    b = np.arange(256, dtype=np.uint8)
    lo = (b.astype(np.uint8) << 4).view(np.int8) >> 4        # low nibble, sign-extended
    hi = b.view(np.int8) >> 4                                 # high nibble, sign-extended
    q = oracle.unpack_int4(b[None, :])[0]
    np.testing.assert_array_equal(q[0::2], lo)
    np.testing.assert_array_equal(q[1::2], hi)
    # hand-worked: 0x8F = (-1, -8), 0x70 = (0, 7), 0x19 = (-7, 1)
    np.testing.assert_array_equal(oracle.unpack_int4(np.array([[0x8F, 0x70, 0x19]], dtype=np.uint8)),
                                  [[-1, -8, 0, 7, -7, 1]])


def test_int4_pack_roundtrip_and_group_scale_indexing():
    rng = np.random.default_rng(41)
    q = rng.integers(-8, 8, size=(6, 512))
    packed = synth.pack_int4(torch.from_numpy(q)).numpy()
    assert packed.shape == (6, 256)
    np.testing.assert_array_equal(oracle.unpack_int4(packed), q)
    scale = np.array([[10.0 ** g * (r + 1) for g in range(4)] for r in range(6)], dtype=np.float32)
    W = oracle.dequant_int4_group(packed, scale)
    for r, c in [(0, 0), (0, 127), (0, 128), (3, 300), (5, 511)]:
        assert W[r, c] == q[r, c] * 10.0 ** (c // 128) * (r + 1)


def test_int4_quantiser_bound():
    w = torch.randn(4, 384, generator=torch.Generator().manual_seed(5)) * 0.02
    packed, s = synth.quantize_int4_group(w)
    W = oracle.dequant_int4_group(packed.numpy(), s.numpy())
    err = np.abs(W - w.double().numpy())
    # half a step of each group, and the group maximum lands on +-7 steps exactly
    assert (err <= 0.5 * np.repeat(s.double().numpy(), 128, axis=1) * (1 + 1e-6)).all()
    q = oracle.unpack_int4(packed.numpy()).reshape(4, 3, 128)
    assert (np.abs(q).max(axis=-1) == 7).all()


def test_int4_layer_top1_equals_dense_swiglu():
    shape = synth.LayerShape("i4", 5, 256, 256, 4, 1, "int4", "uniform")
    d = synth.make_layer(shape, seed=43)
    d["topk_weights"] = torch.ones_like(d["topk_weights"])
    out = oracle.fused_moe_int4(**d)

    def unpack(p):  # independent route: arithmetic shifts
        p = p.numpy()
        lo = (p << 4).view(np.int8) >> 4
        hi = p.view(np.int8) >> 4
        q = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.float64)
        q[..., 0::2], q[..., 1::2] = lo, hi
        return q

    x = d["x"].double()
    for t in range(5):
        e = int(d["topk_ids"][t, 0])
        W13 = torch.from_numpy(unpack(d["w13"][e]) * np.repeat(d["w13_scale"][e].double().numpy(), 128, axis=1))
        W2 = torch.from_numpy(unpack(d["w2"][e]) * np.repeat(d["w2_scale"][e].double().numpy(), 128, axis=1))
        np.testing.assert_allclose(out[t], _dense_swiglu(x[t:t + 1], W13[:256], W13[256:], W2)[0].numpy(),
                                   rtol=1e-10, atol=1e-12)


def test_int4_rows_subset_equals_full_call():
    shape = synth.LayerShape("i4", 9, 256, 128, 6, 3, "int4", "softmax")
    d = synth.make_layer(shape, seed=44)
    full = oracle.fused_moe_int4(**d)
    sub = oracle.fused_moe_rows(**d, kind="int4", tokens=[1, 7])
    np.testing.assert_allclose(sub, full[[1, 7]], rtol=1e-12, atol=1e-15)
