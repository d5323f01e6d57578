"""The C-ABI library builds, loads and exports every entry point of include/gbmoe.h.

These run without a GPU: they only call host-side functions (size queries,
status strings) and argument checks that return before any CUDA call.
"""
import ctypes
import os
import re

import pytest

from mixture_experts_ffn_moe_gb300 import build, gbmoe

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gbmoe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gbmoe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_align_block_size", "fused_moe_fp8", "fused_moe_int8", "moe_workspace_size",
              "moe_read_status", "moe_quant_act_int8"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(gbmoe.EXPORTED) == set(declared_functions())


def test_max_padded_matches_definition(lib):
    assert gbmoe.moe_align_max_padded(3, 2, 4, 2) == 10
    assert gbmoe.moe_align_max_padded(2048, 9, 257, 64) == ((2048 * 9 + 257 * 63 + 63) // 64) * 64
    assert gbmoe.moe_align_max_padded(-1, 2, 4, 2) == 0


def test_workspace_size_queries(lib):
    a = gbmoe.moe_workspace_size(4, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_FP8)
    b = gbmoe.moe_workspace_size(64, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_FP8)
    assert 0 < a < b
    assert gbmoe.moe_workspace_size(4, 4096, 1536, 128, 8, gbmoe.MOE_WEIGHT_INT8) > 0
    assert gbmoe.moe_workspace_size(4, 4096, 1536, 128, 8, 7) == 0
    assert gbmoe.moe_workspace_size(4, 4096, 1536, 2000, 8, gbmoe.MOE_WEIGHT_FP8) == 0


def test_status_strings(lib):
    for st in range(7):
        assert lib.moe_status_string(st)
    assert lib.moe_status_string(99) == b"unknown status"


def _call_fp8(lib, M=4, H=256, I=128, E=8, topk=2, flags=0, null=False):
    p = None if null else ctypes.c_void_p(16)  # never dereferenced: calls fail on the host first
    return lib.fused_moe_fp8(p, p, p, p, p, p, p, M, H, I, E, topk, flags, p, p, 0, None)


def test_host_side_argument_errors(lib):
    assert _call_fp8(lib, M=-1) == 1
    assert _call_fp8(lib, H=200) == 2           # not a multiple of 128
    assert _call_fp8(lib, E=5000) == 2           # more experts than supported
    assert _call_fp8(lib, topk=40) == 2
    assert _call_fp8(lib, flags=0x100) == 1      # unknown flag
    assert _call_fp8(lib, flags=3) == 1          # both paths
    assert _call_fp8(lib, null=True) == 1        # NULL pointers
    assert b"NULL" in lib.moe_last_error()
    assert _call_fp8(lib) == 3                   # workspace NULL / too small
    assert _call_fp8(lib, M=0) == 0              # empty batch is a no-op
    assert lib.moe_align_block_size(None, 4, 2, 8, 0, None, None, None, None, None) == 1
    assert lib.moe_align_block_size(None, 4, 2, 8, 512, None, None, None, None, None) == 2


def test_decode_path_token_limit_and_size_guard(lib):
    dec = gbmoe.MOE_PATH_DECODE
    limit = gbmoe.MOE_MAX_DECODE_TOKENS
    assert _call_fp8(lib, M=limit, flags=dec) == 3              # at the limit: valid, fails on the workspace
    assert _call_fp8(lib, M=limit + 1, flags=dec) == 2          # one past it
    assert b"MOE_MAX_DECODE_TOKENS" in lib.moe_last_error()
    assert _call_fp8(lib, M=limit + 1) == 3                     # MOE_PATH_AUTO takes the tcgen05 path there
    p = ctypes.c_void_p(16)
    assert lib.fused_moe_int8(p, p, p, p, p, p, p, limit + 1, 256, 128, 8, 2, dec, p, p, 0, None) == 2
    # slots M * topk above 2^30 are refused before any size is computed from them
    assert _call_fp8(lib, M=1 << 26, topk=32) == 2
    assert b"too large" in lib.moe_last_error()
    assert _call_fp8(lib, M=1 << 25, topk=32) == 3              # 2^30 slots exactly: still accepted


def test_fp8_activation_flag_host_checks(lib):
    a8 = gbmoe.MOE_ACT_FP8_1X128
    assert _call_fp8(lib, flags=a8 | gbmoe.MOE_PATH_DECODE) == 2   # FP8 x FP8 runs on tcgen05 only
    assert b"prefill" in lib.moe_last_error()
    assert _call_fp8(lib, flags=a8) == 3                            # valid flags: fails on the workspace
    assert _call_fp8(lib, flags=a8 | gbmoe.MOE_PATH_PREFILL) == 3
    p = ctypes.c_void_p(16)
    assert lib.fused_moe_int8(p, p, p, p, p, p, p, 4, 256, 128, 8, 2, a8, p, p, 0, None) == 1  # FP8 layer only
    # workspace: the A8 layout holds codes (1 byte) instead of fp16 rows
    w16 = gbmoe.moe_workspace_size(4096, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_FP8, gbmoe.MOE_PATH_PREFILL)
    w8 = gbmoe.moe_workspace_size(4096, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_FP8, a8)
    assert 0 < w8 < w16
    assert gbmoe.moe_workspace_size(4, 4096, 1536, 128, 8, gbmoe.MOE_WEIGHT_INT8, a8) == 0
    # the standalone quantiser
    assert lib.moe_quant_act_fp8(p, 4, 200, p, p, None) == 2        # H not a multiple of 128
    assert lib.moe_quant_act_fp8(None, 4, 256, p, p, None) == 1
    assert lib.moe_quant_act_fp8(None, 0, 256, None, None, None) == 0


def test_gate_host_checks(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: every call below returns on the host
    G = gbmoe.gate_config

    def gate(M=4, E=8, topk=2, cfg=None):
        cfg = cfg if cfg is not None else G()
        return lib.moe_gate_topk(p, M, E, topk, ctypes.byref(cfg), p, p, None)

    assert lib.moe_gate_topk(p, 4, 8, 2, None, p, p, None) == 1                    # no config
    assert gate(M=0) == 0                                                          # empty batch
    assert gate(topk=9) == 1                                                       # topk > E
    assert gate(E=2000) == 2                                                       # too many experts
    assert gate(E=64, topk=32, cfg=G(shared_expert=True)) == 2                     # 33 columns
    assert gate(cfg=G(n_group=2)) == 1                                             # softmax takes no groups
    assert gate(cfg=G(routed_scaling=2.0)) == 1
    assert gate(cfg=GateCfg_bias()) == 1
    sig = gbmoe.MOE_GATE_SIGMOID_GROUPED
    assert gate(E=12, cfg=G(sig, n_group=8, topk_group=4)) == 1                    # 8 does not divide 12
    assert gate(E=256, cfg=G(sig, n_group=64, topk_group=4)) == 1                  # more than 32 groups
    assert gate(E=256, cfg=G(sig, n_group=8, topk_group=9)) == 1
    assert gate(E=16, topk=5, cfg=G(sig, n_group=8, topk_group=2)) == 1            # 2 groups of 2 hold 4
    assert gate(E=16, topk=4, cfg=G(sig, n_group=8, topk_group=2, routed_scaling=0.0)) == 1
    assert gate(M=0, E=16, topk=4, cfg=G(sig, n_group=8, topk_group=2)) == 0
    assert gate(cfg=G(scoring=7)) == 1
    cfg = G()
    assert lib.moe_gate_topk(None, 4, 8, 2, ctypes.byref(cfg), p, p, None) == 1   # NULL logits
    # the gated layer: weight kind and the layer's own checks
    assert lib.fused_moe_gated(5, p, p, ctypes.byref(cfg), p, p, p, p, 4, 256, 128, 8, 2, 0, p, p, p, p, 0,
                               None) == 1
    assert lib.fused_moe_gated(0, p, p, ctypes.byref(cfg), p, p, p, p, 4, 200, 128, 8, 2, 0, p, p, p, p, 0,
                               None) == 2                                          # H not a multiple of 128
    assert lib.fused_moe_gated(0, p, p, ctypes.byref(cfg), p, p, p, p, 4, 256, 128, 8, 2, 0, p, p, p, p, 0,
                               None) == 3                                          # no workspace


class GateCfg_bias(gbmoe.GateConfig):
    """A softmax config that carries a bias pointer (invalid)."""

    def __init__(self):
        super().__init__(gbmoe.MOE_GATE_SOFTMAX, 1, 1, 1.0, 16, 0)


def test_int4_host_checks(lib):
    p = ctypes.c_void_p(16)

    def call(M=4, H=256, I=128, flags=0):
        return lib.fused_moe_int4(p, p, p, p, p, p, p, M, H, I, 8, 2, flags, p, p, 0, None)

    assert call(flags=gbmoe.MOE_PATH_PREFILL) == 3          # INT4 on the tcgen05 kernels: valid
    assert call(flags=gbmoe.MOE_ACT_FP8_1X128) == 1         # FP8 layer only
    assert call(H=200) == 2
    assert call() == 3                                      # valid: fails on the workspace
    assert call(M=5000) == 3                                # any M (no decode-path token limit for INT4)
    assert gbmoe.moe_workspace_size(4, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_INT4) > 0
    assert gbmoe.moe_workspace_size(4, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_INT4, gbmoe.MOE_ACT_FP8_1X128) == 0
    assert gbmoe.moe_workspace_size(4, 7168, 2048, 257, 9, 3) == 0


def test_masked_host_checks(lib):
    p = ctypes.c_void_p(16)

    def call(kind=0, E=8, cap=16, H=256, I=128, flags=0, null=False):
        q = None if null else p
        return lib.fused_moe_masked(kind, q, q, q, q, q, q, E, cap, H, I, flags, q, q, 0, None)

    assert call(kind=1) == 2                      # INT8 needs per-token scales
    assert call(kind=7) == 1
    assert call(cap=0) == 1
    assert call(E=5000) == 2
    assert call(H=200) == 2
    assert call(flags=gbmoe.MOE_PATH_PREFILL) == 3          # FP8 on the tcgen05 kernels: valid
    assert call(kind=2, flags=gbmoe.MOE_PATH_PREFILL) == 3
    assert call(flags=3) == 1
    assert call(flags=gbmoe.MOE_ACT_FP8_1X128) == 1
    assert call(null=True) == 1
    assert call() == 3                            # valid: fails on the workspace
    assert call(kind=2) == 3
    odd = ctypes.c_void_p(18)  # an output 2-byte aligned only: fine for the weight-streaming kernels
    assert lib.fused_moe_masked(0, p, p, p, p, p, p, 8, 16, 256, 128, 0, odd, p, 0, None) == 3
    assert lib.fused_moe_masked(0, p, p, p, p, p, p, 8, 16, 256, 128, gbmoe.MOE_PATH_PREFILL, odd, p, 0,
                                None) == 1  # the tcgen05 epilogue stores 16-byte row pieces
    a = gbmoe.moe_workspace_size_masked(32, 128, 7168, 2048, gbmoe.MOE_WEIGHT_FP8)
    assert a > 32 * 128 * (7168 + 2048) * 2
    assert gbmoe.moe_workspace_size_masked(32, 128, 7168, 2048, gbmoe.MOE_WEIGHT_INT8) == 0


def test_selftest_host_checks(lib):
    p = ctypes.c_void_p(256)
    assert lib.moe_selftest_wait_timeout(None, 10000, p, None) == 1
    assert lib.moe_selftest_wait_timeout(p, 10, p, None) == 1          # limit below 1000 cycles
    assert lib.moe_selftest_wait_timeout(p, 1 << 40, p, None) == 1     # above 2^31
    assert lib.moe_selftest_wait_timeout(ctypes.c_void_p(16), 10000, p, None) == 3  # misaligned workspace


def test_read_routing_reports_the_block_size_without_a_device(lib):
    bs = ctypes.c_int(0)
    st = lib.moe_read_routing(None, 4, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_FP8, gbmoe.MOE_PATH_AUTO,
                              ctypes.byref(bs), None, None, None, None, None)
    assert st == gbmoe.MOE_OK and bs.value == 8
    st = lib.moe_read_routing(None, 4, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_FP8, gbmoe.MOE_PATH_PREFILL,
                              ctypes.byref(bs), None, None, None, None, None)
    assert st == gbmoe.MOE_OK and bs.value == 16
    assert lib.moe_read_routing(None, 0, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_FP8, 0, ctypes.byref(bs),
                                None, None, None, None, None) == 1
    assert lib.moe_read_routing(None, 4, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_INT8, gbmoe.MOE_ACT_FP8_1X128,
                                ctypes.byref(bs), None, None, None, None, None) == 1
    out = (ctypes.c_int32 * 1)()
    assert lib.moe_read_routing(None, 4, 7168, 2048, 257, 9, gbmoe.MOE_WEIGHT_FP8, 0, None, out, None, None,
                                None, None) == 1  # MOE_ERR_INVALID_ARG: an output but no workspace
