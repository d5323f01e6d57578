"""bench.py's work accounting on the CPU: the algorithmic bytes and flops behind the roofline, and the rule
that keeps a DRAM traffic record only while the sources it was taken on are unchanged."""
import numpy as np

import bench
from mixture_experts_ffn_moe_gb300 import synth


def _default_layer():
    shape = bench.all_workloads()["dsr1_decode_M4"]
    ids, _ = synth.make_routing(shape, 1234)  # the bench's own seed
    return shape, ids


def test_default_layer_routing_is_33_experts_over_36_slots():
    shape, ids = _default_layer()
    flat = ids.numpy().ravel()
    assert flat.size == 4 * 9 and len(np.unique(flat)) == 33


def test_decode_gemm1_algorithmic_bytes_at_four_tokens():
    # 33 active experts x (gate and up codes, 2 x 2048 x 7168 bytes, + 7,168 bytes of 128 x 128 block scales)
    # + x in fp16 (4 x 7168 x 2) + h in fp16 (36 slots x 2048 x 2): 969,325,568 bytes
    shape, ids = _default_layer()
    gemm1_bytes, gemm1_flops = bench.stage_work(shape, ids)["decode_gemm1"]
    assert gemm1_bytes == 33 * (2 * 2048 * 7168 + 7168) + 4 * 7168 * 2 + 36 * 2048 * 2 == 969_325_568
    assert gemm1_flops == 2 * 36 * (2 * 2048) * 7168


def test_decode_gemm2_algorithmic_bytes_at_four_tokens():
    # 33 experts x (7168 x 2048 codes + 3,584 bytes of scales) + h in (fp16) + y out (fp32 by slot)
    shape, ids = _default_layer()
    gemm2_bytes, gemm2_flops = bench.stage_work(shape, ids)["decode_gemm2"]
    assert gemm2_bytes == 33 * (7168 * 2048 + 4 * 56 * 16) + 36 * 2048 * 2 + 36 * 7168 * 4
    assert gemm2_flops == 2 * 36 * 7168 * 2048


def test_roofline_of_the_default_layer_is_hbm_bound():
    shape, ids = _default_layer()
    peaks = {"hbm_gbs": 6775.6, "bf16_tflops": 1886.9, "bf16_tflops_sustained": 1700.0, "source": "measured"}
    n = 20
    stages = [("prologue_align_prep", 0.010 * n), ("decode_gemm1", 0.165 * n), ("decode_gemm2", 0.083 * n),
              ("combine", 0.008 * n)]
    r = bench.roofline_of(shape, ids, stages, n, "dsr1_decode_M4", peaks)
    assert r["bound"] == "hbm" and r["kernel"] == "decode_gemm1" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 969_325_568 / 0.165e-3 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 6775.6) < 1e-12


def test_prefill_at_16384_tokens_is_tensor_bound_against_the_fp8_rate():
    shape = bench.all_workloads()["dsr1_prefill_M16384_a8"]
    ids, _ = synth.make_routing(shape, 1234)
    peaks = {"hbm_gbs": 6775.6, "bf16_tflops": 1886.9, "bf16_tflops_sustained": 1700.0, "source": "measured"}
    stages = [("prefill_gemm1", 4.5), ("prefill_gemm2", 2.7)]
    r = bench.roofline_of(shape, ids, stages, 1, "dsr1_prefill_M16384_a8", peaks)
    flops = 2 * 16384 * 9 * (2 * 2048) * 7168
    assert r["bound"] == "tensor" and r["kernel"] == "prefill_gemm1" and r["peak"] == 2 * 1886.9
    assert abs(r["achieved"] - flops / 4.5e-3 / 1e12) < 1e-6


def test_traffic_record_is_dropped_once_its_sources_change(monkeypatch):
    rec = bench.ncu_traffic("dsr1_decode_M4", "decode_gemm1")
    if rec is not None:  # a record taken on the current sources is returned as is
        assert rec > 969_325_568
    monkeypatch.setattr(bench, "source_hash", lambda kernel, a8=False: "0000000000000000")
    assert bench.ncu_traffic("dsr1_decode_M4", "decode_gemm1") is None
