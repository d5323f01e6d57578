"""Shared helpers of the test suite: structured layers and the parity check."""
import math

import numpy as np
import torch

# Output tolerance of the floating-point layer (fp32 accumulation on the GPU
# vs the float64 oracle): relative L2 error over the whole output and the
# largest absolute error relative to the largest reference magnitude.
REL_L2_TOL = 5e-3
MAX_ABS_TOL = 1e-2


def expert_id_layer(M, topk, E, H=256, I=128, seed=9):
    """FP8 layer whose expert e returns the constant row I*silu(1)*(e+1).

    x[:, 0] = 1, rest 0; gate and up rows are e_0 (code 1.0, scale 1) so
    g = u = 1 and h = silu(1) everywhere; W2 codes are all 1.0 with every
    block scale e+1, so y = I * silu(1) * (e+1) on every output channel.
    A misrouted or mis-weighted slot shows up as a wrong multiple.
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


def errors(out, ref):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.linalg.norm(out - ref) / max(np.linalg.norm(ref), 1e-300)
    mabs = np.abs(out - ref).max() / max(np.abs(ref).max(), 1e-300)
    return rel, mabs


def assert_layer_close(out, ref, what=""):
    rel, mabs = errors(out, ref)
    assert rel <= REL_L2_TOL and mabs <= MAX_ABS_TOL, f"{what}: rel-L2 {rel:.3e}, max-abs/max|ref| {mabs:.3e}"
    return rel, mabs


def to_device(d, device="cuda"):
    return {k: (v.to(device) if hasattr(v, "to") else v) for k, v in d.items()}


def covering_rows(ids, E_total, limit=None):
    """Token rows whose experts cover every active expert, plus the last token routed to the heaviest
    experts (so the last token tile of the most loaded expert is checked) and the first and last token.

    Each active expert contributes the first token that visits it, unless an earlier pick already does.
    The oracle dequantises each expert once per call, so checking every expert costs about as much as
    checking one token per expert.
    """
    ids = np.asarray(ids)
    M = ids.shape[0]
    valid = (ids >= 0) & (ids < E_total)
    picked, covered = [], set()
    for e in np.unique(ids[valid]):
        if int(e) in covered:
            continue
        t = int(np.nonzero((ids == e).any(axis=1))[0][0])
        picked.append(t)
        covered.update(int(v) for v in ids[t][valid[t]])
    counts = np.bincount(ids[valid].ravel(), minlength=E_total)
    for e in np.argsort(-counts, kind="stable")[:2]:  # the two heaviest experts (the shared one first, if any)
        if counts[e]:
            picked.append(int(np.nonzero((ids == e).any(axis=1))[0][-1]))
    picked += [0, M - 1]
    rows = sorted(set(picked))
    return rows if limit is None else rows[:limit]
