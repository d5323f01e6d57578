"""Seeded synthetic inputs for the fused MoE layer.

This module only draws random inputs: activations, router choices and
quantised expert weights.  It holds none of the layer's own arithmetic
(no expert GEMM, no SiLU, no combine, no routing alignment), so the CUDA
path and the CPU oracle can both consume what it produces.

Shapes follow the workloads the serving pages run the layer on:

* a tiny layer (16 tokens, hidden 256, intermediate 128, 8 experts, top-2);
* a DeepSeek-R1-shaped layer (hidden 7168, intermediate 2048, 256 routed
  experts top-8 with sigmoid scores and 8-group / top-4-group selection,
  plus one shared expert), FP8 E4M3 weights with 128x128 block scales;
* a Qwen3-235B-shaped layer (hidden 4096, intermediate 1536, 128 experts
  top-8 softmax renormalised), INT8 per-output-channel weights.

Weight quantisation here is part of input generation (turning random
N(0, 0.02) weights into the stored formats); it uses torch's own
float8_e4m3fn cast and plain rounding, not code shared with either side.
"""
from __future__ import annotations

import dataclasses
import math

import torch

FP8_MAX = 448.0
INT8_MAX = 127.0
INT4_QMAX = 7.0
QBLOCK = 128


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One MoE layer workload.

    E and topk count routed experts only; a shared expert, when present, is
    appended as expert index E with an extra top-k column of weight 1.0.
    """
    name: str
    M: int
    H: int
    I: int
    E: int
    topk: int
    weight_kind: str  # "fp8" | "int8" | "int4"
    routing: str      # "softmax" | "deepseek" | "deepseek_zipf" | "uniform"
    shared_expert: bool = False
    n_group: int = 1
    topk_group: int = 1
    routed_scaling: float = 1.0
    act: str = "a16"  # FP8 layer: "a16" (bf16 activations) | "fp8_1x128" (E4M3 activations, 1 x 128 groups)

    @property
    def E_total(self) -> int:
        return self.E + (1 if self.shared_expert else 0)

    @property
    def topk_total(self) -> int:
        return self.topk + (1 if self.shared_expert else 0)

    def with_M(self, M: int) -> "LayerShape":
        return dataclasses.replace(self, M=M, name=f"{self.name.rsplit('_M', 1)[0]}_M{M}")


def tiny(M: int = 16) -> LayerShape:
    return LayerShape(f"tiny_M{M}", M, 256, 128, 8, 2, "fp8", "softmax")


def deepseek_r1(M: int, routing: str = "deepseek", E: int = 256, act: str = "a16",
                weight_kind: str = "fp8") -> LayerShape:
    """DeepSeek-R1 layer shapes; a smaller E keeps the per-expert work and shrinks the weight set."""
    return LayerShape(f"dsr1_{routing}_M{M}" + ("" if E == 256 else f"_E{E}") + ("" if act == "a16" else "_a8")
                      + ("" if weight_kind == "fp8" else f"_{weight_kind}"),
                      M, 7168, 2048, E, 8, weight_kind, routing, shared_expert=True, n_group=8, topk_group=4, act=act)


def qwen3_235b(M: int, weight_kind: str = "int8") -> LayerShape:
    return LayerShape(f"qwen3_M{M}" + ("" if weight_kind == "int8" else f"_{weight_kind}"), M, 4096, 1536, 128, 8,
                      weight_kind, "softmax")


def _cpu_gen(seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 1_000_003 + stream * 7_919) % (2 ** 63))
    return g


def _stable_topk_desc(score: torch.Tensor, k: int) -> torch.Tensor:
    """Indices of the k largest entries per row; equal scores keep the lower index."""
    return torch.argsort(-score, dim=-1, stable=True)[:, :k]


def _router_logits(shape: LayerShape, g: torch.Generator) -> torch.Tensor:
    """Router logits [M, E] in float64 for the softmax / deepseek / deepseek_zipf recipes."""
    M, E = shape.M, shape.E
    if shape.routing in ("softmax", "deepseek"):
        return torch.randn(M, E, generator=g, dtype=torch.float32).double()
    if shape.routing == "deepseek_zipf":
        perm = torch.randperm(E, generator=g)
        ranks = torch.arange(1, E + 1, dtype=torch.float64)
        p = ranks.pow(-1.1)
        p = p / p.sum()
        u = torch.rand(M, E, generator=g, dtype=torch.float64).clamp_(1e-300, 1.0 - 1e-16)
        gumbel = -torch.log(-torch.log(u))
        return torch.log(p[perm])[None, :] + gumbel
    raise ValueError(f"routing {shape.routing!r} draws no logits")


def make_router_logits(shape: LayerShape, seed: int) -> torch.Tensor:
    """The router logits make_routing draws for (shape, seed), rounded to fp32 [M, E].

    For the softmax and deepseek recipes the logits are fp32 draws, so this is
    exactly what make_routing ranks; the Zipf recipe's float64 logits are rounded.
    """
    return _router_logits(shape, _cpu_gen(seed, 1)).float().contiguous()


def make_router_bias(E: int, seed: int, std: float = 0.05) -> torch.Tensor:
    """A selection bias per expert (fp32 [E], N(0, std)), standing in for a learnt load-balancing correction."""
    return (torch.randn(E, generator=_cpu_gen(seed, 5), dtype=torch.float32) * std).contiguous()


def make_routing(shape: LayerShape, seed: int):
    """Router choices (topk_ids int32 [M, topk_total], topk_weights fp32) on the CPU.

    The router itself is not part of the layer; it only decides which
    experts each token visits.  The recipes per workload:

    * softmax: logits N(0,1); p = softmax (in float64); top-k of p; weights
      renormalised to sum to 1.
    * deepseek: logits N(0,1); s = sigmoid; per group of E/n_group experts the
      group score is the sum of its two best s; the topk_group best groups
      are kept; top-k experts by s inside them; weights s / sum(s) times the
      routed scaling factor.
    * deepseek_zipf: as deepseek, with logits ln p_pi(e) + Gumbel(0,1), where
      p_r ~ r^-1.1 and pi is a seeded permutation (skewed expert popularity).
    * uniform: each token picks k distinct experts uniformly; weights are
      sigmoid(N(0,1)) renormalised.
    """
    M, E, k = shape.M, shape.E, shape.topk
    g = _cpu_gen(seed, 1)
    if shape.routing == "uniform":
        ids = torch.argsort(torch.rand(M, E, generator=g), dim=-1)[:, :k]
        w = torch.sigmoid(torch.randn(M, k, generator=g, dtype=torch.float64))
        w = w / w.sum(-1, keepdim=True)
    elif shape.routing == "softmax":
        logits = _router_logits(shape, g)
        p = torch.softmax(logits, dim=-1)
        ids = _stable_topk_desc(p, k)
        w = p.gather(1, ids)
        w = w / w.sum(-1, keepdim=True)
    elif shape.routing in ("deepseek", "deepseek_zipf"):
        logits = _router_logits(shape, g)
        s = torch.sigmoid(logits)
        gs = E // shape.n_group
        grouped = s.view(M, shape.n_group, gs)
        top2 = torch.sort(grouped, dim=-1, descending=True).values[..., :2].sum(-1)
        keep = _stable_topk_desc(top2, shape.topk_group)
        mask = torch.zeros(M, shape.n_group, dtype=torch.bool)
        mask.scatter_(1, keep, True)
        masked = torch.where(mask[:, :, None].expand(M, shape.n_group, gs).reshape(M, E), s,
                             torch.full_like(s, -1.0))
        ids = _stable_topk_desc(masked, k)
        w = s.gather(1, ids)
        w = w / w.sum(-1, keepdim=True) * shape.routed_scaling
    else:
        raise ValueError(shape.routing)
    ids = ids.to(torch.int32)
    w = w.to(torch.float32)
    if shape.shared_expert:
        ids = torch.cat([ids, torch.full((M, 1), E, dtype=torch.int32)], dim=1)
        w = torch.cat([w, torch.ones(M, 1, dtype=torch.float32)], dim=1)
    return ids.contiguous(), w.contiguous()


def make_x(shape: LayerShape, seed: int) -> torch.Tensor:
    """Activations x ~ N(0,1), stored bf16 [M, H], on the CPU."""
    g = _cpu_gen(seed, 2)
    return torch.randn(shape.M, shape.H, generator=g).to(torch.bfloat16)


def quantize_fp8_block(w: torch.Tensor):
    """N(0,.02) weights [..., R, C] -> (e4m3 codes as uint8, fp32 scales [..., R/128, C/128]).

    Per 128x128 block: scale = amax / 448 (1 when the block is all zero),
    codes = torch's float8_e4m3fn cast (round to nearest even) of w / scale.
    """
    *lead, R, C = w.shape
    wb = w.reshape(*lead, R // QBLOCK, QBLOCK, C // QBLOCK, QBLOCK)
    amax = wb.abs().amax(dim=(-3, -1))
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax)).float()
    q = (wb / scale[..., :, None, :, None]).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).reshape(*lead, R, C), scale


def quantize_int8_channel(w: torch.Tensor):
    """Weights [..., R, C] -> (int8 codes, fp32 per-row scale amax/127)."""
    amax = w.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / INT8_MAX, torch.ones_like(amax)).float()
    q = torch.round(w / scale[..., None]).clamp(-INT8_MAX, INT8_MAX).to(torch.int8)
    return q, scale


def pack_int4(q: torch.Tensor) -> torch.Tensor:
    """int values in [-8, 7], [..., C] -> uint8 [..., C/2]: column 2j in the low nibble, 2j+1 in the high one."""
    n = (q.to(torch.int16) & 0xF).to(torch.uint8)
    return (n[..., 0::2] | (n[..., 1::2] << 4)).contiguous()


def quantize_int4_group(w: torch.Tensor):
    """Weights [..., R, C] -> (packed int4 codes uint8 [..., R, C/2], fp32 scales [..., R, C/128]).

    Per row and 128 columns: s = amax / 7 (1 when the group is all zero),
    q = round-half-even(w / s), which lies in [-7, 7] (the format also holds -8).
    """
    *lead, R, C = w.shape
    wg = w.reshape(*lead, R, C // QBLOCK, QBLOCK)
    amax = wg.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / INT4_QMAX, torch.ones_like(amax)).float()
    q = torch.round(wg / scale[..., None]).clamp(-8, 7).reshape(*lead, R, C)
    return pack_int4(q), scale


def make_weights(shape: LayerShape, seed: int, device="cpu", std: float = 0.02):
    """Expert weights, one expert at a time (so full-size layers fit), on `device`.

    Returns (w13, w13_scale, w2, w2_scale):
      fp8 : w13 uint8 [E, 2I, H], w13_scale f32 [E, 2I/128, H/128],
            w2  uint8 [E, H, I],  w2_scale  f32 [E, H/128, I/128]
      int8: w13 int8 [E, 2I, H], w13_scale f32 [E, 2I],
            w2  int8 [E, H, I],  w2_scale  f32 [E, H]
      int4: w13 uint8 [E, 2I, H/2] (two codes a byte), w13_scale f32 [E, 2I, H/128],
            w2  uint8 [E, H, I/2],  w2_scale  f32 [E, H, I/128]
    Rows 0..I-1 of w13 are the gate projection, rows I..2I-1 the up projection.
    """
    E, H, I = shape.E_total, shape.H, shape.I
    device = torch.device(device)
    if shape.weight_kind == "fp8":
        w13 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
        s13 = torch.empty(E, 2 * I // QBLOCK, H // QBLOCK, dtype=torch.float32, device=device)
        w2 = torch.empty(E, H, I, dtype=torch.uint8, device=device)
        s2 = torch.empty(E, H // QBLOCK, I // QBLOCK, dtype=torch.float32, device=device)
        quant = quantize_fp8_block
    elif shape.weight_kind == "int8":
        w13 = torch.empty(E, 2 * I, H, dtype=torch.int8, device=device)
        s13 = torch.empty(E, 2 * I, dtype=torch.float32, device=device)
        w2 = torch.empty(E, H, I, dtype=torch.int8, device=device)
        s2 = torch.empty(E, H, dtype=torch.float32, device=device)
        quant = quantize_int8_channel
    elif shape.weight_kind == "int4":
        w13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=device)
        s13 = torch.empty(E, 2 * I, H // QBLOCK, dtype=torch.float32, device=device)
        w2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
        s2 = torch.empty(E, H, I // QBLOCK, dtype=torch.float32, device=device)
        quant = quantize_int4_group
    else:
        raise ValueError(shape.weight_kind)
    g = torch.Generator(device=device)
    for e in range(E):
        g.manual_seed((seed * 1_000_003 + 31 * e + 11) % (2 ** 63))
        a = torch.randn(2 * I, H, generator=g, device=device) * std
        w13[e], s13[e] = quant(a)
        b = torch.randn(H, I, generator=g, device=device) * std
        w2[e], s2[e] = quant(b)
        del a, b
    return w13, s13, w2, s2


def make_layer(shape: LayerShape, seed: int, weight_device="cpu"):
    """All inputs of one layer call. x / ids / weights on the CPU unless asked."""
    ids, w = make_routing(shape, seed)
    x = make_x(shape, seed)
    w13, s13, w2, s2 = make_weights(shape, seed, weight_device)
    return dict(x=x, topk_ids=ids, topk_weights=w, w13=w13, w13_scale=s13, w2=w2, w2_scale=s2)


def distinct_weight_bytes(shape: LayerShape, topk_ids: torch.Tensor) -> int:
    """Bytes of expert weights (codes + scales) a layer call must read at least once."""
    active = torch.unique(topk_ids[(topk_ids >= 0) & (topk_ids < shape.E_total)]).numel()
    H, I = shape.H, shape.I
    if shape.weight_kind == "fp8":
        per = 3 * H * I + 4 * (2 * I // QBLOCK) * (H // QBLOCK) + 4 * (H // QBLOCK) * (I // QBLOCK)
    elif shape.weight_kind == "int4":
        per = 3 * H * I // 2 + 4 * (2 * I * (H // QBLOCK) + H * (I // QBLOCK))
    else:
        per = 3 * H * I + 4 * (2 * I + H)
    return active * per


def algorithmic_flops(shape: LayerShape, topk_ids: torch.Tensor) -> int:
    """2*(M*k_valid)*3*H*I: the three projections over all valid (token, expert) pairs."""
    valid = int(((topk_ids >= 0) & (topk_ids < shape.E_total)).sum())
    return 2 * valid * 3 * shape.H * shape.I


def expert_histogram(shape: LayerShape, topk_ids: torch.Tensor) -> torch.Tensor:
    ids = topk_ids[(topk_ids >= 0) & (topk_ids < shape.E_total)].long()
    return torch.bincount(ids, minlength=shape.E_total)


def balance(hist: torch.Tensor) -> float:
    """mean / max tokens per active expert (1.0 = perfectly even)."""
    act = hist[hist > 0].double()
    return float(act.mean() / act.max()) if act.numel() else 1.0


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("math", "dataclasses", "torch")]
