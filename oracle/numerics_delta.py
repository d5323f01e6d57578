"""Numerics delta of the oracle's power-of-two-scale ("UE8M0") mode -- test infrastructure, a report only.

Runs the oracle's FP8 layer in its three activation modes (bf16 activations;
E4M3 activations with fp32 1 x 128 scales; the same with every scale a power of
two) on one seeded layer of DeepSeek-R1 expert shapes (H 7168, I 2048; 16
tokens, 8 experts, top-2), and prints their differences, and how far
re-quantising one expert's stored gate/up blocks to power-of-two scales moves
the weights.  It calls only the oracle and the seeded input generator, and
takes about a minute of CPU.

    python -m oracle.numerics_delta
"""
import numpy as np

from mixture_experts_ffn_moe_gb300 import synth

from . import moe_oracle as oracle


def rel_l2(u, v):
    return float(np.linalg.norm(u - v) / np.linalg.norm(v))


def max_rel(u, v):
    return float(np.abs(u - v).max() / np.abs(v).max())


def main():
    shape = synth.LayerShape("dsr1_experts_8_top2", 16, 7168, 2048, 8, 2, "fp8", "softmax")
    d = synth.make_layer(shape, seed=41)
    out = {m: oracle.fused_moe_fp8(**d, act=m) for m in ("a16", "fp8_1x128", "fp8_ue8m0")}
    for a, b in (("fp8_1x128", "a16"), ("fp8_ue8m0", "a16"), ("fp8_ue8m0", "fp8_1x128")):
        print(f"{a:10s} vs {b:10s}: rel-L2 {rel_l2(out[a], out[b]):.3e}, "
              f"max-abs / max|ref| {max_rel(out[a], out[b]):.3e}")
    w13, s13 = d["w13"][0].numpy(), d["w13_scale"][0].numpy()
    q, s = oracle.requant_fp8_block_ue8m0(w13, s13)
    before, after = oracle.dequant_fp8_block(w13, s13), oracle.dequant_fp8_block(q, s)
    print(f"expert 0 gate/up weights re-quantised: rel-L2 {rel_l2(after, before):.3e}, "
          f"codes changed {float((q != w13).mean()):.3f}")


if __name__ == "__main__":
    main()
