"""CPU oracle for the fused MoE (sparse FFN) layer -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the package's smoke check, the CPU-baseline leg of the
benchmark and the report script beside it (numerics_delta.py) may import this
module.  The product path (the CUDA library and its Python binding) never
calls it and shares no code with it.

It is a plain, slow, obviously correct restatement of what the layer
computes, in float64 numpy over dequantised weights:

* routing alignment -- the argsort of topk_ids into per-expert, block-padded
  groups (Xeon 6 / SGLang DeepSeek-R1 blog, section "MoE"; SGLang CPU backend
  write-up, section "(3) FusedMoE", the moe_align_index and thread-offset
  paragraphs);
* the naive masked per-expert loop: for each expert, gather the tokens that
  chose it, run GEMM-SiLU-GEMM, and add the result into each token's output
  with its routing weight (same two sections: the "naive MoE in torch" and
  "experts run serially" paragraphs);
* the gate/up split of W13 as A x [B1, B2] = [C1, C2] with SiLU(C1) * C2
  (same sections, the SiLU-fusion bullet);
* FP8 E4M3 weights with 128x128 block scales, decoded from the OCP FP8
  format definition and scaled per block (DeepSeek-style block quant; the
  post-scaled FP8 GEMV of the OSDI'26 local-MoE paper summary, section "CPU
  decode backend", is the same sum regrouped);
* INT8 per-output-channel weights with dynamic per-token INT8 activations
  (DA8W8; SGLang CPU backend write-up, "(3) FusedMoE", the dynamic-quant
  fusion paragraph);
* INT4 weights with one scale per row and 128 columns, activations at their
  bf16 values (a reading: the pages name INT4 without a layout, see
  unpack_int4);
* the optional FP8 x FP8 ("A8") mode of the FP8 layer, in which the
  activations and the intermediate h are quantised to E4M3 in groups of 1 x 128
  (a reading: the pages keep FP8 activations in BF16, see quant_fp8_1x128);
* the same mode with power-of-two ("UE8M0") scales, the scale format of the
  tensor cores' block-scaled MMA: not on the pages, every scale rounded up to a
  power of two (a reading, see ue8m0_ceil);
* the router's gating functions that produce topk_ids / topk_weights from
  logits (softmax top-k renormalised; sigmoid with a selection bias and
  group-limited top-k).  The pages take the router's output as given; these
  follow the measured layers' model configurations.

Precision: float64 accumulation everywhere, except that every decision that
turns a float into an integer code (activation quantisation) is taken in
float32 with IEEE division and round-half-to-even, the same precision the
GPU kernels use for that decision; re-quantising stored weights to
power-of-two scales rounds each exact product decode(q) * s / s' once.  The
gating functions rank in float64: their results are exact rankings, and the
GPU gate (which ranks in float32) is compared with them only where the
ranking margin exceeds float32 error.
"""
from __future__ import annotations

import numpy as np

FP8_MAX = 448.0
INT8_MAX = 127
QBLOCK = 128

# ----------------------------------------------------------------------------
# FP8 E4M3 codec, from the OCP 8-bit floating point format definition:
# 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
# holds the subnormals 2^-6 * m/8; S.1111.111 is NaN; there is no infinity;
# the largest finite magnitude is 1.1110.110 = 448.
# ----------------------------------------------------------------------------


def e4m3_decode(codes) -> np.ndarray:
    """uint8 E4M3 codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + man / 8.0, (exp - 7).astype(np.int64))
    subnormal = np.ldexp(man / 8.0, -6)
    mag = np.where(exp == 0, subnormal, normal)
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def _e4m3_positive_grid() -> np.ndarray:
    """All 127 finite non-negative E4M3 magnitudes, ascending (codes 0x00..0x7E)."""
    return e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode_satfinite(v) -> np.ndarray:
    """float32 values -> E4M3 codes: round to nearest, ties to even code, clamp to +-448.

    The grid is decoded from the format definition; a value is compared with
    the midpoints between neighbouring grid points.  On a tie the code with an
    even mantissa (even code) wins.  NaN input -> 0x7F.
    """
    return _e4m3_round_satfinite(np.asarray(v, dtype=np.float32).astype(np.float64))


def _e4m3_round_satfinite(v) -> np.ndarray:
    """float64 values -> E4M3 codes, each exact value rounded once (the rule of e4m3_encode_satfinite)."""
    v = np.asarray(v, dtype=np.float64)
    grid = _e4m3_positive_grid()
    a = np.minimum(np.abs(v), FP8_MAX)
    lo = np.clip(np.searchsorted(grid, a, side="right") - 1, 0, 126)
    hi = np.minimum(lo + 1, 126)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(v) & (code != 0), code | 0x80, code)
    code = np.where(np.signbit(v) & (code == 0), np.uint8(0x80), code)
    return np.where(np.isnan(v), np.uint8(0x7F), code).astype(np.uint8)


# ----------------------------------------------------------------------------
# Dequantisation of the stored weights.
# ----------------------------------------------------------------------------


_E4M3_TABLE = None


def _e4m3_table() -> np.ndarray:
    """e4m3_decode of all 256 codes, so large arrays decode by one lookup."""
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = e4m3_decode(np.arange(256, dtype=np.uint8))
    return _E4M3_TABLE


def dequant_fp8_block(codes, scale) -> np.ndarray:
    """codes uint8 [R, C], scale f32 [R/128, C/128] -> float64 W[r, c] = decode(q) * S[r//128, c//128]."""
    codes = np.asarray(codes, dtype=np.uint8)
    scale = np.asarray(scale, dtype=np.float64)
    R, C = codes.shape
    W = _e4m3_table()[codes].reshape(R // QBLOCK, QBLOCK, C // QBLOCK, QBLOCK)
    W *= scale[:, None, :, None]
    return W.reshape(R, C)


def dequant_int8_channel(codes, scale) -> np.ndarray:
    """codes int8 [R, C], scale f32 [R] -> float64 W[r, c] = q * s[r]."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[:, None]


# ----------------------------------------------------------------------------
# INT4 weights with one scale per row and 128 columns (group-wise W4A16).
# The pages name INT4 as the quantised alternative to native FP8 (SGLang CPU
# backend write-up, closing section; OSDI'26 local-MoE summary, evaluation of
# the INT4 decode baseline) without fixing a layout.  Reading: two's-complement
# nibbles in [-8, 7], two per byte (column 2j in the low nibble, 2j+1 in the
# high one), and w = q * s with one fp32 scale per row and 128 columns, the
# same 128-wide K grouping as the FP8 block scales.
# ----------------------------------------------------------------------------


def unpack_int4(packed) -> np.ndarray:
    """uint8 [..., C/2] -> int8 [..., C]: byte j = column 2j (low nibble) and 2j+1 (high nibble)."""
    b = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    nib = np.stack([b & 0x0F, b >> 4], axis=-1).reshape(*b.shape[:-1], 2 * b.shape[-1])
    return np.where(nib >= 8, nib - 16, nib).astype(np.int8)


def dequant_int4_group(packed, scale) -> np.ndarray:
    """packed uint8 [R, C/2], scale f32 [R, C/128] -> float64 W[r, c] = q[r, c] * s[r, c // 128]."""
    q = unpack_int4(packed).astype(np.float64)
    return q * np.repeat(np.asarray(scale, dtype=np.float64), QBLOCK, axis=-1)


# ----------------------------------------------------------------------------
# Dynamic INT8 quantisation (DA8W8), one scale per row.
# ----------------------------------------------------------------------------


def quant_int8_per_row(a):
    """float32 rows [R, C] -> (int8 codes, float32 scales).

    s = amax(|row|) / 127 in float32 (1 when the row is all zero);
    q = round-half-even(row / s) in float32, clamped to [-127, 127].
    """
    a = np.asarray(a, dtype=np.float32)
    amax = np.max(np.abs(a), axis=-1) if a.shape[-1] else np.zeros(a.shape[:-1], np.float32)
    s = np.where(amax > 0, amax / np.float32(INT8_MAX), np.float32(1.0)).astype(np.float32)
    q = np.rint(np.divide(a, s[..., None], dtype=np.float32))
    q = np.clip(q, -INT8_MAX, INT8_MAX).astype(np.int8)
    return q, s


# ----------------------------------------------------------------------------
# FP8 activations in 1 x 128 groups (the optional "A8" mode of the FP8 layer).
#
# The pages run FP8 weights against BF16 activations (Xeon 6 / SGLang blog,
# section "FP8 推理", the weight-only bullet; the author's write-up, section
# "(4) FP8 GEMM").  The DeepGEMM grouped GEMMs that the news rewrite of the LMSYS
# large-scale-EP blog integrates (section "DeepGEMM集成") multiply FP8 by FP8,
# but no page says how the activations are quantised.  Reading: one float32
# scale per row and per 128 consecutive columns, s = amax / 448, and codes by
# the same E4M3 rounding the weights use -- the 128-wide group matches the
# weights' 128 x 128 scale blocks along K.
# ----------------------------------------------------------------------------


def quant_fp8_1x128(a):
    """float32 rows [R, C] (C a multiple of 128) -> (E4M3 codes uint8 [R, C], float32 scales [R, C/128]).

    For every row and every group of 128 consecutive columns:
    s = amax(|group|) / 448 in float32 (1 when the group is all zero);
    q = e4m3_encode_satfinite(group / s), the division in float32 (IEEE).
    """
    a = np.asarray(a, dtype=np.float32)
    R, C = a.shape
    if C % QBLOCK:
        raise ValueError("columns must be a multiple of 128")
    g = a.reshape(R, C // QBLOCK, QBLOCK)
    amax = np.max(np.abs(g), axis=-1) if R else np.zeros((0, C // QBLOCK), np.float32)
    s = np.where(amax > 0, np.divide(amax, np.float32(FP8_MAX), dtype=np.float32), np.float32(1.0))
    s = s.astype(np.float32)
    q = e4m3_encode_satfinite(np.divide(g, s[..., None], dtype=np.float32))
    return q.reshape(R, C), s


def dequant_fp8_1x128(codes, scale) -> np.ndarray:
    """codes uint8 [R, C], scale f32 [R, C/128] -> float64 a[r, c] = decode(q) * s[r, c // 128]."""
    codes = np.asarray(codes, dtype=np.uint8)
    R, C = codes.shape
    a = _e4m3_table()[codes].reshape(R, C // QBLOCK, QBLOCK)
    a = a * np.asarray(scale, dtype=np.float64)[..., None]
    return a.reshape(R, C)


# ----------------------------------------------------------------------------
# Power-of-two (UE8M0) scales.  Not on the pages: the pages' FP8 scales are
# fp32, and the block-scaled MMA of the tensor cores takes its scales as UE8M0
# exponents (the OCP Microscaling format's E8M0: an unsigned 8-bit exponent,
# bias 127, value 2^(code - 127), codes 0..254; 255 is NaN).  The reading taken
# here: every fp32 scale is replaced by the smallest power of two not below it,
# so that no code overflows; activations are quantised against that scale, and
# stored weights are re-quantised from their exact values decode(q) * s.  One
# scale still covers 1 x 128 activations and 128 x 128 weights (a 32-wide MX
# scale block would repeat it four times).
# ----------------------------------------------------------------------------

UE8M0_MIN_EXP = -127
UE8M0_MAX_EXP = 127


def ue8m0_ceil(s):
    """Positive scales -> (float64 2^e, uint8 UE8M0 codes e + 127), e the smallest integer with 2^e >= s,
    clamped to [-127, 127]."""
    s = np.asarray(s, dtype=np.float64)
    if np.any(~(s > 0)) or np.any(~np.isfinite(s)):
        raise ValueError("UE8M0 scales need positive finite inputs")
    m, e = np.frexp(s)                       # s = m * 2^e with m in [0.5, 1)
    e = np.where(m == 0.5, e - 1, e)         # s is 2^(e-1) exactly
    e = np.clip(e, UE8M0_MIN_EXP, UE8M0_MAX_EXP)
    return np.ldexp(1.0, e), (e + 127).astype(np.uint8)


def quant_fp8_1x128_ue8m0(a):
    """float32 rows [R, C] -> (E4M3 codes uint8 [R, C], float32 power-of-two scales [R, C/128]).

    As quant_fp8_1x128, with the group's scale amax / 448 (float32, 1 for an
    all-zero group) replaced by ue8m0_ceil of it; the division by a power of
    two is exact, so each code is the once-rounded value of the element over
    its scale.
    """
    a = np.asarray(a, dtype=np.float32)
    R, C = a.shape
    if C % QBLOCK:
        raise ValueError("columns must be a multiple of 128")
    g = a.reshape(R, C // QBLOCK, QBLOCK)
    amax = np.max(np.abs(g), axis=-1) if R else np.zeros((0, C // QBLOCK), np.float32)
    s = np.where(amax > 0, np.divide(amax, np.float32(FP8_MAX), dtype=np.float32), np.float32(1.0))
    s = ue8m0_ceil(s.astype(np.float32))[0].astype(np.float32)
    q = e4m3_encode_satfinite(np.divide(g, s[..., None], dtype=np.float32))
    return q.reshape(R, C), s


def requant_fp8_block_ue8m0(codes, scale):
    """Stored FP8 block weights (codes uint8 [R, C], fp32 scale [R/128, C/128]) -> the same weights with
    power-of-two block scales: (codes uint8 [R, C], float32 scales [R/128, C/128]).

    Per block: s' = ue8m0_ceil(s); every code becomes the E4M3 rounding
    (ties to even) of the exact value decode(q) * s / s', which lies within
    +-448 because s / s' is in (1/2, 1].
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scale = np.asarray(scale, dtype=np.float32)
    R, C = codes.shape
    s2 = ue8m0_ceil(scale)[0]
    ratio = scale.astype(np.float64) / s2                    # exact: a division by a power of two
    v = _e4m3_table()[codes].reshape(R // QBLOCK, QBLOCK, C // QBLOCK, QBLOCK) * ratio[:, None, :, None]
    return _e4m3_round_satfinite(v).reshape(R, C), s2.astype(np.float32)


# ----------------------------------------------------------------------------
# Gating: router logits -> (topk_ids, topk_weights).  Not on the pages (they
# take the router's choices as given); the two functions follow the layer
# configurations the hot path is measured on: softmax top-k renormalised
# (Qwen3-style) and sigmoid scores with bias-corrected group-limited top-k
# (DeepSeek-style).  Ties always go to the lower index.
# ----------------------------------------------------------------------------


def _stable_desc(v, axis=-1):
    """Indices sorting v in descending order; equal values keep ascending index order."""
    return np.argsort(-v, axis=axis, kind="stable")


def gate_softmax_topk(logits, k: int):
    """logits [M, E] -> (ids int32 [M, k], weights float64 [M, k]).

    p = softmax(logits) in float64; the k largest p (ties to the lower index);
    weights p_sel / sum(p_sel).
    """
    l = np.asarray(logits, dtype=np.float64)
    p = np.exp(l - l.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    ids = _stable_desc(p)[:, :k]
    w = np.take_along_axis(p, ids, axis=-1)
    return ids.astype(np.int32), w / w.sum(axis=-1, keepdims=True)


def gate_grouped_sigmoid_topk(logits, k: int, n_group: int, topk_group: int, bias=None, routed_scaling=1.0):
    """logits [M, E] -> (ids int32 [M, k], weights float64 [M, k]).

    s = sigmoid(logits) in float64 and b = s + bias (selection only).  The E
    experts form n_group consecutive groups; a group's score is the sum of its
    two largest b; the topk_group best groups are kept; the k largest b inside
    them are chosen.  Weights are s_sel / sum(s_sel) times routed_scaling.
    """
    l = np.asarray(logits, dtype=np.float64)
    M, E = l.shape
    s = 1.0 / (1.0 + np.exp(-l))
    b = s + (0.0 if bias is None else np.asarray(bias, dtype=np.float64)[None, :])
    grouped = b.reshape(M, n_group, E // n_group)
    gscore = -np.sort(-grouped, axis=-1)[..., :2].sum(axis=-1)
    keep = _stable_desc(gscore)[:, :topk_group]
    in_kept = np.zeros((M, n_group), dtype=bool)
    np.put_along_axis(in_kept, keep, True, axis=-1)
    masked = np.where(np.repeat(in_kept, E // n_group, axis=-1), b, -np.inf)
    ids = _stable_desc(masked)[:, :k]
    w = np.take_along_axis(s, ids, axis=-1)
    return ids.astype(np.int32), w / w.sum(axis=-1, keepdims=True) * routed_scaling


# ----------------------------------------------------------------------------
# Routing alignment.
# ----------------------------------------------------------------------------


def max_padded(M: int, topk: int, E: int, B: int) -> int:
    """Capacity of sorted_ids: every expert may waste up to B-1 padding slots."""
    n = M * topk + E * (B - 1)
    return (n + B - 1) // B * B


def moe_align_block_size(topk_ids, E: int, B: int):
    """Argsort of the flat topk_ids into per-expert groups padded to multiples of B.

    Flat slot i = t*topk + k.  Slots are grouped by expert in ascending expert
    order; inside one expert they keep ascending slot order (a stable sort).
    Slots whose id lies outside [0, E) are dropped.  Each expert's group is
    padded with the sentinel M*topk up to a multiple of B (an expert with no
    slots gets no block).  expert_ids[b] names the expert that owns block b;
    blocks past the last used one hold -1.  expert_offsets is the exclusive
    prefix sum of the padded group sizes (E+1 entries); num_post_padded its
    last entry.

    Returns (sorted_ids, expert_ids, num_post_padded, expert_offsets, counts)
    with sorted_ids sized max_padded(...) and expert_ids sized that / B.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    M, topk = ids.shape
    flat = ids.reshape(-1)
    sentinel = M * topk
    cap = max_padded(M, topk, E, B)
    sorted_ids = np.full(cap, sentinel, dtype=np.int32)
    expert_ids = np.full(cap // B, -1, dtype=np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    counts = np.zeros(E, dtype=np.int32)
    valid = np.nonzero((flat >= 0) & (flat < E))[0]
    order = valid[np.argsort(flat[valid], kind="stable")]
    pos = 0
    j = 0
    for e in range(E):
        offsets[e] = pos
        n = 0
        while j < len(order) and flat[order[j]] == e:
            sorted_ids[pos + n] = order[j]
            n += 1
            j += 1
        counts[e] = n
        padded = (n + B - 1) // B * B
        expert_ids[pos // B:(pos + padded) // B] = e
        pos += padded
    offsets[E] = pos
    return sorted_ids, expert_ids, np.int32(pos), offsets, counts


# ----------------------------------------------------------------------------
# The layer: naive masked per-expert loop.
# ----------------------------------------------------------------------------


def silu(z):
    return z / (1.0 + np.exp(-z))


def _as_np(t):
    """torch tensors (bf16 included) or arrays -> numpy, exactly."""
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            t = t.float()
        return t.numpy()
    return np.asarray(t)


def fused_moe_fp8(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, experts=None, act="a16"):
    """FP8 block-scaled weights.

    x [M, H] (bf16 values), topk_ids int [M, k], topk_weights f32 [M, k],
    w13 uint8 [E, 2I, H] + scale [E, 2I/128, H/128], w2 uint8 [E, H, I] +
    scale [E, H/128, I/128].  Returns float64 out [M, H].

    act="a16" (the pages' weight-only scheme): activations keep their bf16
    values.  act="fp8_1x128": x is replaced by dequant(quant_fp8_1x128(x)), and
    the intermediate h of every (token, expert) pair, rounded to float32, by
    dequant(quant_fp8_1x128(h)) before the down projection.  act="fp8_ue8m0":
    the same with every scale a power of two -- quant_fp8_1x128_ue8m0 for x and
    h, and both weight tensors re-quantised by requant_fp8_block_ue8m0.

    `experts` restricts the loop to a subset (for sampling large layers);
    contributions of other experts are then left out.
    """
    if act not in ("a16", "fp8_1x128", "fp8_ue8m0"):
        raise ValueError(act)
    return _naive_moe(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, "fp8", experts, act)


def fused_moe_int4(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, experts=None):
    """The layer with group-wise INT4 weights (w13 uint8 [E, 2I, H/2], w13_scale f32 [E, 2I, H/128],
    w2 uint8 [E, H, I/2], w2_scale f32 [E, H, I/128]); activations enter at their bf16 values."""
    return _naive_moe(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, "int4", experts)


def fused_moe_int8(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, experts=None):
    """INT8 per-channel weights with dynamic per-row INT8 activations (DA8W8).

    The token rows are quantised once (quant_int8_per_row of x); the
    intermediate h of each (token, expert) pair is quantised again per row
    before the down projection.  Integer dot products are exact (int64);
    scales are applied afterwards in float64.
    """
    return _naive_moe(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, "int8", experts)


def _naive_moe(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, kind, experts, act="a16"):
    x = _as_np(x).astype(np.float32)
    ids = _as_np(topk_ids).astype(np.int64)
    tw = _as_np(topk_weights).astype(np.float64)
    M, H = x.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    Y = np.zeros(ids.shape + (H,), dtype=np.float64)  # Y[t, k] = expert output of slot (t, k)
    if kind == "int8":
        qx, sx = quant_int8_per_row(x)
    a8 = kind == "fp8" and act in ("fp8_1x128", "fp8_ue8m0")
    quant_act = quant_fp8_1x128_ue8m0 if act == "fp8_ue8m0" else quant_fp8_1x128
    xa = dequant_fp8_1x128(*quant_act(x)) if a8 else x.astype(np.float64)
    for e in (range(E) if experts is None else experts):
        tok, slot = np.nonzero(ids == e)  # the mask of this expert
        if tok.size == 0:
            continue
        # one expert's weights at a time (they may live on a device; copy them here)
        q13, s13, q2, s2 = (_as_np(a[e]) for a in (w13, w13_scale, w2, w2_scale))
        if kind in ("fp8", "int4"):
            deq = dequant_fp8_block if kind == "fp8" else dequant_int4_group
            if kind == "fp8" and act == "fp8_ue8m0":
                q13, s13 = requant_fp8_block_ue8m0(q13, s13)
                q2, s2 = requant_fp8_block_ue8m0(q2, s2)
            W13 = deq(q13, s13)                                    # [2I, H]
            W2 = deq(q2, s2)                                       # [H, I]
            C = xa[tok] @ W13.T                                    # A x [B1, B2] = [C1, C2]
            h = silu(C[:, :I]) * C[:, I:]                          # SiLU(C1) * C2
            if a8:
                h = dequant_fp8_1x128(*quant_act(h.astype(np.float32)))
            y = h @ W2.T
        else:
            acc = qx[tok].astype(np.int64) @ q13.astype(np.int64).T
            C = acc * sx[tok].astype(np.float64)[:, None] * s13.astype(np.float64)[None, :]
            h = silu(C[:, :I]) * C[:, I:]
            qh, sh = quant_int8_per_row(h.astype(np.float32))
            acc2 = qh.astype(np.int64) @ q2.astype(np.int64).T
            y = acc2 * sh.astype(np.float64)[:, None] * s2.astype(np.float64)[None, :]
        Y[tok, slot] = y
    out = np.zeros((M, H), dtype=np.float64)
    for k in range(ids.shape[1]):  # combine in slot order
        valid = (ids[:, k] >= 0) & (ids[:, k] < E)
        out += np.where(valid[:, None], tw[:, k:k + 1] * Y[:, k], 0.0)
    return out


def fused_moe_rows(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, kind, tokens, act="a16"):
    """Oracle output for a subset of token rows only (for layers too large to run whole).

    Computes exactly what the full call gives for those rows: it runs the
    naive loop on the selected tokens alone (every token is independent once
    routed).  Dynamic activation quantisation is per row, so it is unchanged.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    x = _as_np(x)[tokens]
    ids = _as_np(topk_ids)[tokens]
    tw = _as_np(topk_weights)[tokens]
    E = w13.shape[0]
    used = sorted({int(e) for e in np.unique(ids) if 0 <= e < E})
    if kind == "fp8":
        return fused_moe_fp8(x, ids, tw, w13, w13_scale, w2, w2_scale, experts=used, act=act)
    if kind == "int4":
        return fused_moe_int4(x, ids, tw, w13, w13_scale, w2, w2_scale, experts=used)
    if kind != "int8":
        raise ValueError(f"unknown weight kind {kind!r}")
    return fused_moe_int8(x, ids, tw, w13, w13_scale, w2, w2_scale, experts=used)
