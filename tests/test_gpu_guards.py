"""Guard bands around every buffer the library writes, and read-only inputs.

The workspace and the output of each layer call are carved out of a larger
device buffer whose bytes before and after them hold a known pattern.  A call
on any path (decode, tcgen05 prefill, FP8 activations, INT8, INT4, gated,
masked) must leave both bands untouched, which checks that
`moe_workspace_size` / `moe_workspace_size_masked` cover everything the
kernels write and that no kernel stores past its output.  Every input must
come back bit-identical, and the result must still meet the layer tolerance
against the oracle, so the guarded layout is also a parity case.
"""
import numpy as np
import pytest
import torch

import oracle
from _layers import assert_layer_close, to_device
from mixture_experts_ffn_moe_gb300 import build, gbmoe, synth

pytestmark = pytest.mark.gpu

BAND = 8192          # guard bytes on each side (a multiple of 512 keeps the caching allocator's alignment)
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return gbmoe.load()


class Guarded:
    """A device byte buffer of n bytes between two guard bands."""

    def __init__(self, n):
        self.n = n
        self.buf = torch.full((BAND + n + BAND,), PATTERN, dtype=torch.uint8, device="cuda")
        self.inner = self.buf[BAND:BAND + n]

    def as_tensor(self, shape, dtype):
        return self.inner.view(dtype).view(*shape)

    def check(self, what):
        host = self.buf.cpu().numpy()
        lo, hi = host[:BAND], host[BAND + self.n:]
        bad_lo = np.flatnonzero(lo != PATTERN)
        bad_hi = np.flatnonzero(hi != PATTERN)
        assert bad_lo.size == 0, f"{what}: {bad_lo.size} bytes written before the buffer (first at -{BAND - bad_lo[0]})"
        assert bad_hi.size == 0, f"{what}: {bad_hi.size} bytes written past the end (first at +{bad_hi[0]})"


def _snapshot(tensors):
    return [t.clone() for t in tensors]


def _assert_unchanged(before, after, what):
    for i, (a, b) in enumerate(zip(before, after)):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                           b.view(torch.uint8) if b.dtype != torch.uint8 else b), f"{what}: input {i} was modified"


_FN = {"fp8": gbmoe.fused_moe_fp8, "int8": gbmoe.fused_moe_int8, "int4": gbmoe.fused_moe_int4}
_KIND = {"fp8": gbmoe.MOE_WEIGHT_FP8, "int8": gbmoe.MOE_WEIGHT_INT8, "int4": gbmoe.MOE_WEIGHT_INT4}
_ORACLE = {"fp8": oracle.fused_moe_fp8, "int8": oracle.fused_moe_int8, "int4": oracle.fused_moe_int4}
A8 = gbmoe.MOE_PATH_PREFILL | gbmoe.MOE_ACT_FP8_1X128


@pytest.mark.parametrize("kind,M,H,I,E,k,flags", [
    ("fp8", 5, 256, 128, 8, 2, gbmoe.MOE_PATH_AUTO),         # weight-streaming decode kernels
    ("fp8", 200, 512, 256, 8, 4, gbmoe.MOE_PATH_PREFILL),    # tcgen05 grouped GEMMs, ragged token tiles
    ("fp8", 200, 512, 256, 8, 4, A8),                        # FP8 x FP8 with per-K-block promotion
    ("int8", 16, 256, 256, 6, 3, gbmoe.MOE_PATH_AUTO),       # requant of h between the GEMMs
    ("int8", 300, 384, 256, 5, 2, gbmoe.MOE_PATH_PREFILL),
    ("int4", 7, 256, 256, 8, 2, gbmoe.MOE_PATH_AUTO),
    ("int4", 150, 512, 256, 6, 3, gbmoe.MOE_PATH_PREFILL),
])
def test_routed_layer_writes_only_its_workspace_and_output(kind, M, H, I, E, k, flags):
    shape = synth.LayerShape("guard", M, H, I, E, k, kind, "softmax")
    d = to_device(synth.make_layer(shape, seed=M * 7 + E))
    inputs = [d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"]]
    before = _snapshot(inputs)
    ws = Guarded(gbmoe.moe_workspace_size(M, H, I, E, k, _KIND[kind], flags))
    out = Guarded(M * H * 2)
    for call in range(2):  # the second call finds the workspace as the first left it
        _FN[kind](*inputs, flags=flags, out=out.as_tensor((M, H), torch.bfloat16), workspace=ws.inner)
        torch.cuda.synchronize()
        ws.check(f"{kind} flags {flags:#x} workspace, call {call}")
        out.check(f"{kind} flags {flags:#x} output, call {call}")
    _assert_unchanged(before, inputs, f"{kind} flags {flags:#x}")
    bad, flags_word, st = gbmoe.moe_read_status(ws.inner)
    assert (bad, flags_word, st) == (0, 0, gbmoe.MOE_OK)
    act = "fp8_1x128" if flags & gbmoe.MOE_ACT_FP8_1X128 else "a16"
    kw = {"act": act} if kind == "fp8" else {}
    ref = _ORACLE[kind](**{n: v.cpu() for n, v in d.items()}, **kw)
    assert_layer_close(out.as_tensor((M, H), torch.bfloat16).float().cpu().numpy(), ref, f"guarded {kind}")


@pytest.mark.parametrize("M", [4, 100])  # ranking inside the prologue / a separate gate launch
def test_gated_layer_writes_only_its_buffers(M):
    E, k, H, I = 32, 4, 256, 128
    shape = synth.LayerShape("gg", M, H, I, E, k, "fp8", "softmax")
    w13, s13, w2, s2 = [t.cuda() for t in synth.make_weights(shape, 31)]
    x = synth.make_x(shape, 31).cuda()
    logits = torch.from_numpy(np.random.default_rng(31).standard_normal((M, E)).astype(np.float32)).cuda()
    before = _snapshot([x, logits, w13, s13, w2, s2])
    gate = gbmoe.gate_config(gbmoe.MOE_GATE_SOFTMAX)
    ws = Guarded(gbmoe.moe_workspace_size(M, H, I, E, k, gbmoe.MOE_WEIGHT_FP8))
    out, ids, wts = Guarded(M * H * 2), Guarded(M * k * 4), Guarded(M * k * 4)
    gbmoe.fused_moe_gated(gbmoe.MOE_WEIGHT_FP8, x, logits, gate, k, w13, s13, w2, s2,
                          out=out.as_tensor((M, H), torch.bfloat16), workspace=ws.inner,
                          topk_ids=ids.as_tensor((M, k), torch.int32), topk_weights=wts.as_tensor((M, k), torch.float32))
    torch.cuda.synchronize()
    for g, what in ((ws, "workspace"), (out, "output"), (ids, "topk_ids"), (wts, "topk_weights")):
        g.check(f"gated M={M} {what}")
    _assert_unchanged(before, [x, logits, w13, s13, w2, s2], f"gated M={M}")
    ref = oracle.fused_moe_fp8(x.cpu(), ids.as_tensor((M, k), torch.int32).cpu(),
                               wts.as_tensor((M, k), torch.float32).cpu(), w13.cpu(), s13.cpu(), w2.cpu(), s2.cpu())
    assert_layer_close(out.as_tensor((M, H), torch.bfloat16).float().cpu().numpy(), ref, f"gated M={M}")


@pytest.mark.parametrize("flags", [gbmoe.MOE_PATH_AUTO, gbmoe.MOE_PATH_PREFILL])
def test_masked_layout_writes_only_its_workspace_and_real_rows(flags):
    E, cap, H, I = 4, 40, 256, 128
    counts = [40, 0, 17, 3]
    shape = synth.LayerShape("mg", E * cap, H, I, E, 1, "fp8", "uniform")
    w13, s13, w2, s2 = [t.cuda() for t in synth.make_weights(shape, 41)]
    x = synth.make_x(shape, 41).view(E, cap, H).cuda()
    m = torch.tensor(counts, dtype=torch.int32, device="cuda")
    before = _snapshot([x, m, w13, s13, w2, s2])
    ws = Guarded(gbmoe.moe_workspace_size_masked(E, cap, H, I, gbmoe.MOE_WEIGHT_FP8))
    out = Guarded(E * cap * H * 2)
    o = out.as_tensor((E, cap, H), torch.bfloat16)
    gbmoe.fused_moe_masked(gbmoe.MOE_WEIGHT_FP8, x, m, w13, s13, w2, s2, flags=flags, out=o, workspace=ws.inner)
    torch.cuda.synchronize()
    ws.check(f"masked flags {flags:#x} workspace")
    out.check(f"masked flags {flags:#x} output")
    _assert_unchanged(before, [x, m, w13, s13, w2, s2], f"masked flags {flags:#x}")
    # rows past each expert's count keep the pattern (0xA5A5 as bf16)
    raw = o.view(torch.int16).cpu().numpy()
    for e, c in enumerate(counts):
        assert (raw[e, c:] == np.int16(-0x5A5B)).all(), f"masked flags {flags:#x}: padding rows of expert {e} written"
