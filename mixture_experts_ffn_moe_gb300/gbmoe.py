"""Thin Python binding of libgbmoe.so (the C ABI declared in include/gbmoe.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  torch supplies device memory and the current CUDA stream.
There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgbmoe.so")

MOE_OK = 0
MOE_PATH_AUTO = 0x0
MOE_PATH_DECODE = 0x1
MOE_PATH_PREFILL = 0x2
MOE_ACT_FP8_1X128 = 0x10
MOE_WEIGHT_FP8 = 0
MOE_WEIGHT_INT8 = 1
MOE_WEIGHT_INT4 = 2
MOE_MAX_EXPERTS = 1024
MOE_MAX_DECODE_TOKENS = 128
MOE_AUTO_PREFILL_TOKENS = 128
MOE_STATIC_SCRATCH_BYTES = 16 << 20
MOE_GATE_SOFTMAX = 0
MOE_GATE_SIGMOID_GROUPED = 1
MOE_GATE_INLINE_TOKENS = 64


class GateConfig(ctypes.Structure):
    """moe_gate_config_t."""
    _fields_ = [("scoring", ctypes.c_int), ("n_group", ctypes.c_int), ("topk_group", ctypes.c_int),
                ("routed_scaling", ctypes.c_float), ("bias", ctypes.c_void_p), ("shared_expert", ctypes.c_int)]

_STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_BAD_IDS"}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)} ({detail})")


_lib = None

_vp, _i, _u, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
_SIGS = {
    "moe_align_max_padded": (_sz, [_i, _i, _i, _i]),
    "moe_align_block_size": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "moe_gate_topk": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "fused_moe_gated": (_i, [_i] + [_vp] * 7 + [_i] * 5 + [_u, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_quant_act_int8": (_i, [_vp, _i, _i, _vp, _vp, _vp]),
    "moe_quant_act_fp8": (_i, [_vp, _i, _i, _vp, _vp, _vp]),
    "moe_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _u]),
    "fused_moe_fp8": (_i, [_vp] * 7 + [_i] * 5 + [_u, _vp, _vp, _sz, _vp]),
    "fused_moe_int8": (_i, [_vp] * 7 + [_i] * 5 + [_u, _vp, _vp, _sz, _vp]),
    "fused_moe_int4": (_i, [_vp] * 7 + [_i] * 5 + [_u, _vp, _vp, _sz, _vp]),
    "moe_workspace_size_masked": (_sz, [_i, _i, _i, _i, _i]),
    "fused_moe_masked": (_i, [_i] + [_vp] * 6 + [_i] * 4 + [_u, _vp, _vp, _sz, _vp]),
    "fused_moe_fp8_static_scratch": (_i, [_vp] * 7 + [_i] * 5 + [_u, _vp, _vp]),
    "moe_read_status": (_i, [_vp, _vp, _vp]),
    "moe_read_static_scratch_status": (_i, [_vp, _vp]),
    "moe_read_routing": (_i, [_vp] + [_i] * 6 + [_u] + [_vp] * 6),
    "moe_selftest_wait_timeout": (_i, [_vp, ctypes.c_longlong, _vp, _vp]),
    "moe_profile_enable": (_i, [_i]),
    "moe_profile_read": (_i, [_vp, _vp, _i, _vp, _vp]),
    "moe_status_string": (ctypes.c_char_p, [_i]),
    "moe_last_error": (ctypes.c_char_p, []),
}
EXPORTED = tuple(_SIGS)


def load(path: str = LIB_PATH):
    """Loads libgbmoe.so (built in-tree by build.py) and declares its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m mixture_experts_ffn_moe_gb300.build` "
                           "(the CUDA library is required; there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(st: int, where: str):
    if st != MOE_OK:
        detail = load().moe_last_error().decode() or load().moe_status_string(st).decode()
        raise MoEError(st, where, detail)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t: torch.Tensor, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def moe_align_max_padded(M: int, topk: int, num_experts: int, block_size: int) -> int:
    return int(load().moe_align_max_padded(M, topk, num_experts, block_size))


def moe_align_block_size(topk_ids: torch.Tensor, num_experts: int, block_size: int, with_offsets: bool = True):
    """Returns (sorted_ids, expert_ids, num_tokens_post_padded, expert_offsets) as device tensors."""
    _need(topk_ids, torch.int32, "topk_ids")
    M, topk = topk_ids.shape
    cap = moe_align_max_padded(M, topk, num_experts, block_size)
    dev = topk_ids.device
    sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(cap // block_size, dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    offs = torch.empty(num_experts + 1, dtype=torch.int32, device=dev) if with_offsets else None
    st = load().moe_align_block_size(_ptr(topk_ids), M, topk, num_experts, block_size, _ptr(sorted_ids),
                                     _ptr(expert_ids), _ptr(npp), _ptr(offs), _stream(topk_ids))
    _check(st, "moe_align_block_size")
    return sorted_ids, expert_ids, npp, offs


def gate_config(scoring=MOE_GATE_SOFTMAX, n_group=1, topk_group=1, routed_scaling=1.0, bias=None,
                shared_expert=False):
    """A moe_gate_config_t.  `bias` (fp32 [E] CUDA tensor or None) is kept alive by the config."""
    if bias is not None:
        _need(bias, torch.float32, "bias")
    cfg = GateConfig(scoring, n_group, topk_group, routed_scaling,
                     bias.data_ptr() if bias is not None else None, 1 if shared_expert else 0)
    cfg.bias_tensor = bias  # the struct holds a raw pointer into this tensor
    return cfg


def moe_gate_topk(logits: torch.Tensor, topk: int, gate: GateConfig):
    """fp32 router logits [M, E] -> (topk_ids int32, topk_weights fp32), both [M, topk + shared_expert]."""
    _need(logits, torch.float32, "logits")
    M, E = logits.shape
    ld = topk + gate.shared_expert
    ids = torch.empty(M, ld, dtype=torch.int32, device=logits.device)
    w = torch.empty(M, ld, dtype=torch.float32, device=logits.device)
    st = load().moe_gate_topk(_ptr(logits), M, E, topk, ctypes.byref(gate), _ptr(ids), _ptr(w), _stream(logits))
    _check(st, "moe_gate_topk")
    return ids, w


def fused_moe_gated(weight_kind, x, router_logits, gate: GateConfig, topk, w13, w13_scale, w2, w2_scale,
                    flags=MOE_PATH_AUTO, out=None, workspace=None, topk_ids=None, topk_weights=None):
    """The layer from router logits: gating, then the fused layer (see include/gbmoe.h).

    Returns (out, topk_ids, topk_weights); the weights hold E + gate.shared_expert experts.
    """
    wdt = torch.int8 if weight_kind == MOE_WEIGHT_INT8 else torch.uint8
    _need(x, torch.bfloat16, "x")
    _need(router_logits, torch.float32, "router_logits")
    if w13.dtype == torch.float8_e4m3fn:
        w13 = w13.view(torch.uint8)
    if w2.dtype == torch.float8_e4m3fn:
        w2 = w2.view(torch.uint8)
    _need(w13, wdt, "w13")
    _need(w2, wdt, "w2")
    _need(w13_scale, torch.float32, "w13_scale")
    _need(w2_scale, torch.float32, "w2_scale")
    M, H = x.shape
    E = router_logits.shape[1]
    sh = gate.shared_expert
    Et, I = _weight_dims(weight_kind, x, w13, w2)
    if router_logits.shape[0] != M or Et != E + sh:
        raise ValueError("inconsistent shapes")
    ids = topk_ids if topk_ids is not None else torch.empty(M, topk + sh, dtype=torch.int32, device=x.device)
    w = topk_weights if topk_weights is not None else torch.empty(M, topk + sh, dtype=torch.float32,
                                                                  device=x.device)
    _need(ids, torch.int32, "topk_ids")
    _need(w, torch.float32, "topk_weights")
    if tuple(ids.shape) != (M, topk + sh) or tuple(w.shape) != (M, topk + sh):
        raise ValueError("topk_ids / topk_weights must be [M, topk + shared_expert]")
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        workspace = alloc_workspace(M, H, I, Et, topk + sh, weight_kind, flags, x.device)
    st = load().fused_moe_gated(weight_kind, _ptr(x), _ptr(router_logits), ctypes.byref(gate), _ptr(w13),
                                _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), M, H, I, E, topk, flags, _ptr(ids),
                                _ptr(w), _ptr(out), _ptr(workspace), workspace.numel(), _stream(x))
    _check(st, "fused_moe_gated")
    return out, ids, w


def moe_quant_act_int8(x: torch.Tensor):
    """bf16 [M, H] -> (int8 codes [M, H], fp32 scales [M])."""
    _need(x, torch.bfloat16, "x")
    M, H = x.shape
    q = torch.empty(M, H, dtype=torch.int8, device=x.device)
    s = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(load().moe_quant_act_int8(_ptr(x), M, H, _ptr(q), _ptr(s), _stream(x)), "moe_quant_act_int8")
    return q, s


def moe_quant_act_fp8(x: torch.Tensor):
    """bf16 [M, H] -> (E4M3 codes uint8 [M, H], fp32 scales [M, H/128]), one scale per 1 x 128 group."""
    _need(x, torch.bfloat16, "x")
    M, H = x.shape
    q = torch.empty(M, H, dtype=torch.uint8, device=x.device)
    s = torch.empty(M, max(H // 128, 1), dtype=torch.float32, device=x.device)
    _check(load().moe_quant_act_fp8(_ptr(x), M, H, _ptr(q), _ptr(s), _stream(x)), "moe_quant_act_fp8")
    return q, s


def moe_workspace_size(M, H, I, E, topk, weight_kind, flags=MOE_PATH_AUTO) -> int:
    return int(load().moe_workspace_size(M, H, I, E, topk, weight_kind, flags))


def alloc_workspace(M, H, I, E, topk, weight_kind, flags=MOE_PATH_AUTO, device="cuda") -> torch.Tensor:
    n = moe_workspace_size(M, H, I, E, topk, weight_kind, flags)
    if n == 0:
        raise MoEError(2, "moe_workspace_size", "unsupported sizes")
    return torch.empty(n, dtype=torch.uint8, device=device)  # caching allocator blocks are 512-byte aligned


def _weight_dims(kind, x, w13, w2):
    """(E, I) of the stored weights; checks their shapes against x [M, H]."""
    H = x.shape[1]
    E, I2, Hs = w13.shape
    pack = 2 if kind == MOE_WEIGHT_INT4 else 1  # INT4 stores two codes per byte along K
    if Hs * pack != H or tuple(w2.shape) != (E, H, I2 // 2 // pack):
        raise ValueError("inconsistent shapes")
    return E, I2 // 2


def _fused(fn_name, kind, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, flags, out, workspace):
    wdt = torch.int8 if kind == MOE_WEIGHT_INT8 else torch.uint8
    _need(x, torch.bfloat16, "x")
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    if w13.dtype == torch.float8_e4m3fn:
        w13 = w13.view(torch.uint8)
    if w2.dtype == torch.float8_e4m3fn:
        w2 = w2.view(torch.uint8)
    _need(w13, wdt, "w13")
    _need(w2, wdt, "w2")
    _need(w13_scale, torch.float32, "w13_scale")
    _need(w2_scale, torch.float32, "w2_scale")
    M, H = x.shape
    E, I = _weight_dims(kind, x, w13, w2)
    if topk_ids.shape[0] != M:
        raise ValueError("inconsistent shapes")
    if tuple(topk_weights.shape) != tuple(topk_ids.shape):
        raise ValueError("topk_weights and topk_ids must have the same shape")
    topk = topk_ids.shape[1]
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        workspace = alloc_workspace(M, H, I, E, topk, kind, flags, x.device)
    fn = getattr(load(), fn_name)
    st = fn(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale),
            M, H, I, E, topk, flags, _ptr(out), _ptr(workspace), workspace.numel(), _stream(x))
    _check(st, fn_name)
    return out


def fused_moe_fp8(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, flags=MOE_PATH_AUTO, out=None,
                  workspace=None):
    """The MoE layer with FP8 E4M3 128x128-block-scaled weights (see include/gbmoe.h)."""
    return _fused("fused_moe_fp8", MOE_WEIGHT_FP8, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale,
                  flags, out, workspace)


def fused_moe_int8(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, flags=MOE_PATH_AUTO, out=None,
                   workspace=None):
    """The MoE layer with INT8 per-channel weights and dynamic INT8 activations (see include/gbmoe.h)."""
    return _fused("fused_moe_int8", MOE_WEIGHT_INT8, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale,
                  flags, out, workspace)


def fused_moe_int4(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, flags=MOE_PATH_AUTO, out=None,
                   workspace=None):
    """The MoE layer with group-wise INT4 weights: w13 uint8 [E, 2I, H/2] + scales [E, 2I, H/128],
    w2 uint8 [E, H, I/2] + scales [E, H, I/128] (see include/gbmoe.h)."""
    return _fused("fused_moe_int4", MOE_WEIGHT_INT4, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale,
                  flags, out, workspace)


def moe_workspace_size_masked(E, cap, H, I, weight_kind) -> int:
    return int(load().moe_workspace_size_masked(E, cap, H, I, weight_kind))


def fused_moe_masked(weight_kind, x, masked_m, w13, w13_scale, w2, w2_scale, flags=MOE_PATH_AUTO, out=None,
                     workspace=None):
    """Expert FFNs on the masked layout: x bf16 [E, cap, H], masked_m int32 [E] (device) -> out bf16 [E, cap, H].

    Rows i >= masked_m[e] of `out` are left untouched (see include/gbmoe.h).
    """
    _need(x, torch.bfloat16, "x")
    _need(masked_m, torch.int32, "masked_m")
    if w13.dtype == torch.float8_e4m3fn:
        w13 = w13.view(torch.uint8)
    if w2.dtype == torch.float8_e4m3fn:
        w2 = w2.view(torch.uint8)
    _need(w13, torch.uint8, "w13")
    _need(w2, torch.uint8, "w2")
    _need(w13_scale, torch.float32, "w13_scale")
    _need(w2_scale, torch.float32, "w2_scale")
    E, cap, H = x.shape
    Ew, I = _weight_dims(weight_kind, x.view(E * cap, H), w13, w2)
    if Ew != E or tuple(masked_m.shape) != (E,):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.zeros(E, cap, H, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        n = moe_workspace_size_masked(E, cap, H, I, weight_kind)
        if n == 0:
            raise MoEError(2, "moe_workspace_size_masked", "unsupported sizes or weight kind")
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    st = load().fused_moe_masked(weight_kind, _ptr(x), _ptr(masked_m), _ptr(w13), _ptr(w13_scale), _ptr(w2),
                                 _ptr(w2_scale), E, cap, H, I, flags, _ptr(out), _ptr(workspace), workspace.numel(),
                                 _stream(x))
    _check(st, "fused_moe_masked")
    return out


def fused_moe_fp8_static_scratch(x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, flags=MOE_PATH_AUTO,
                                 out=None):
    """fused_moe_fp8 without a workspace, for callers that cannot allocate device memory.

    The library runs the same kernels on a fixed static device buffer of
    MOE_STATIC_SCRATCH_BYTES; sizes that need more are rejected.  Calls that
    overlap on the GPU share that buffer and must be serialised.
    """
    _need(x, torch.bfloat16, "x")
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    if w13.dtype == torch.float8_e4m3fn:
        w13 = w13.view(torch.uint8)
    if w2.dtype == torch.float8_e4m3fn:
        w2 = w2.view(torch.uint8)
    for t, n in ((w13, "w13"), (w2, "w2")):
        _need(t, torch.uint8, n)
    _need(w13_scale, torch.float32, "w13_scale")
    _need(w2_scale, torch.float32, "w2_scale")
    M, H = x.shape
    E, I2, _ = w13.shape
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    st = load().fused_moe_fp8_static_scratch(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13),
                                             _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), M, H, I2 // 2, E,
                                             topk_ids.shape[1], flags, _ptr(out), _stream(x))
    _check(st, "fused_moe_fp8_static_scratch")
    return out


def moe_read_static_scratch_status(device=None):
    """(bad_id_count, flags, status) of the last fused_moe_fp8_static_scratch call on the current device."""
    buf = (ctypes.c_int32 * 2)()
    stream = torch.cuda.current_stream(device).cuda_stream
    st = load().moe_read_static_scratch_status(ctypes.cast(buf, ctypes.c_void_p), ctypes.c_void_p(stream))
    return int(buf[0]), int(buf[1]), int(st)


def moe_read_status(workspace: torch.Tensor):
    """(bad_id_count, flags, status) of the last fused call that used `workspace`."""
    buf = (ctypes.c_int32 * 2)()
    st = load().moe_read_status(_ptr(workspace), ctypes.cast(buf, ctypes.c_void_p), _stream(workspace))
    return int(buf[0]), int(buf[1]), int(st)


def moe_read_routing(workspace: torch.Tensor, M, H, I, E, topk, weight_kind, flags=MOE_PATH_AUTO):
    """The alignment a routed fused call on `workspace` used, with the same sizes and flags.

    Returns (block_size, sorted_ids, expert_ids, num_tokens_post_padded, expert_offsets) as
    moe_align_block_size would give them for that block size (see include/gbmoe.h).
    """
    L = load()
    bs = ctypes.c_int(0)
    _check(L.moe_read_routing(None, M, H, I, E, topk, weight_kind, flags, ctypes.byref(bs), None, None, None, None,
                              None), "moe_read_routing")
    B = bs.value
    cap = moe_align_max_padded(M, topk, E, B)
    dev = workspace.device
    sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(cap // B, dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    _check(L.moe_read_routing(_ptr(workspace), M, H, I, E, topk, weight_kind, flags, None, _ptr(sorted_ids),
                              _ptr(expert_ids), _ptr(npp), _ptr(offs), _stream(workspace)), "moe_read_routing")
    return B, sorted_ids, expert_ids, npp, offs


def moe_selftest_wait_timeout(workspace: torch.Tensor, limit_cycles: int = 2_000_000) -> torch.Tensor:
    """Runs the bounded-wait failure self-test on `workspace`; returns the device count of waits that gave up."""
    gave_up = torch.zeros(1, dtype=torch.int32, device=workspace.device)
    st = load().moe_selftest_wait_timeout(_ptr(workspace), limit_cycles, _ptr(gave_up), _stream(workspace))
    _check(st, "moe_selftest_wait_timeout")
    return gave_up


def moe_profile_enable(max_calls: int) -> None:
    """Record per-kernel CUDA events for the next `max_calls` fused calls of this thread (0 = stop)."""
    _check(load().moe_profile_enable(max_calls), "moe_profile_enable")


def moe_profile_read(max_stages: int = 8):
    """Waits for the recorded events; returns (calls, [(kernel name, summed ms), ...]) and forgets them."""
    ms = (ctypes.c_float * max_stages)()
    names = (ctypes.c_char_p * max_stages)()
    n_st = ctypes.c_int(0)
    n_calls = ctypes.c_int(0)
    st = load().moe_profile_read(ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(names, ctypes.c_void_p),
                                 max_stages, ctypes.byref(n_st), ctypes.byref(n_calls))
    _check(st, "moe_profile_read")
    return n_calls.value, [(names[i].decode(), float(ms[i])) for i in range(n_st.value)]
