"""Benchmark of the GB300 fused MoE layer (one JSON line on stdout).

A step is one call of the whole layer (routing alignment, activation
preparation, gate/up GEMM with SiLU*mul, down projection and weighted
combine) on one batch of synthetic, seeded input.  After the default line's
own measurements, the line's "also" object times every other configuration
of the layer the same way (DeepSeek-R1 decode at 1 token and the 1..64-token
sweep, the 2048- and 16,384-token prefill with bf16 and FP8 activations,
Qwen3 INT8 at 1/16/256/4096 tokens), each with its clocks, routing histogram
and a parity check of one token against the oracle (--no-also skips it).  The default workload is a
DeepSeek-R1-shaped MoE decode layer: 4 tokens, hidden 7168, expert
intermediate 2048, 256 routed experts top-8 (sigmoid scores, 8 groups / top-4
groups) plus 1 shared expert, FP8 E4M3 weights with 128x128 block scales,
bf16 activations N(0,1).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

--impl reference times the CPU oracle (a deliberately plain float64 restatement
of the layer) on the host cores, one bounded sample of the workload per step.
Under torchrun (N > 1) every rank runs an independent replica of the layer on
its own GPU (the layer is not sharded across GPUs); rank 0 prints.
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_ffn_moe_gb300 import gbmoe, synth  # noqa: E402

METRIC = "fused-MoE tokens/s per layer; decode HBM GB/s, prefill TFLOPS vs GB300 peak"
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


def workloads():
    return {
        "dsr1_decode_M1": synth.deepseek_r1(1),
        "dsr1_decode_M4": synth.deepseek_r1(4),
        "dsr1_prefill_M2048": synth.deepseek_r1(2048, routing="deepseek_zipf"),
        "dsr1_prefill_M16384": synth.deepseek_r1(16384, routing="deepseek_zipf"),
        # FP8 activations in 1 x 128 groups (FP8 x FP8 tensor-core products)
        "dsr1_prefill_M2048_a8": synth.deepseek_r1(2048, routing="deepseek_zipf", act="fp8_1x128"),
        "dsr1_prefill_M16384_a8": synth.deepseek_r1(16384, routing="deepseek_zipf", act="fp8_1x128"),
        **{f"dsr1_sweep_M{m}": synth.deepseek_r1(m, routing="uniform") for m in (1, 2, 4, 8, 16, 32, 64)},
        **{f"qwen3_M{m}": synth.qwen3_235b(m) for m in (1, 16, 256, 4096)},
        **{f"qwen3_M{m}": synth.qwen3_235b(m) for m in (64, 96, 128)},
        **{f"dsr1_decode_M{m}": synth.deepseek_r1(m) for m in (64, 96, 128)},
        "tiny_M16": synth.tiny(),
        # same per-expert work with 32+1 experts: small enough for full ncu captures
        "dsr1_decode_M4_E32": synth.deepseek_r1(4, E=32),
        "dsr1_prefill_M2048_E32": synth.deepseek_r1(2048, routing="deepseek_zipf", E=32),
        "dsr1_prefill_M2048_E32_a8": synth.deepseek_r1(2048, routing="deepseek_zipf", E=32, act="fp8_1x128"),
        "qwen3_M1024": synth.qwen3_235b(1024),
        # group-wise INT4 weights (one scale per row and 128 columns), bf16 activations
        "dsr1_decode_M1_int4": synth.deepseek_r1(1, weight_kind="int4"),
        "dsr1_decode_M4_int4": synth.deepseek_r1(4, weight_kind="int4"),
        "dsr1_sweep_M64_int4": synth.deepseek_r1(64, routing="uniform", weight_kind="int4"),
        "qwen3_M1_int4": synth.qwen3_235b(1, weight_kind="int4"),
        "qwen3_M16_int4": synth.qwen3_235b(16, weight_kind="int4"),
        "dsr1_decode_M4_E32_int4": synth.deepseek_r1(4, E=32, weight_kind="int4"),
        "qwen3_M4096_int4": synth.qwen3_235b(4096, weight_kind="int4"),
        "dsr1_prefill_M2048_int4": synth.deepseek_r1(2048, routing="deepseek_zipf", weight_kind="int4"),
    }


DEFAULT_WORKLOAD = "dsr1_decode_M4"

# Workloads whose step starts from router logits: GPU gating, then the layer (fused_moe_gated).
GATED = {f"{n}_gated": n for n in ("dsr1_decode_M1", "dsr1_decode_M4", "dsr1_prefill_M2048", "dsr1_prefill_M16384",
                                   "qwen3_M16", "qwen3_M4096")}


# Masked fixed-capacity layout of expert-parallel low-latency decode: the 32 local experts of
# one of 8 ranks of a DeepSeek-R1 layer, 128 rows each; the counts are the rows the
# DeepSeek router sends to experts 0..31 from a global batch of M tokens.
# (local experts, rows per expert, global tokens, path flag: the caller picks the path, since the counts
# live on the device)
MASKED = {"dsr1_masked_ep8_M64": (32, 128, 64, 0), "dsr1_masked_ep8_M512": (32, 128, 512, 0),
          "dsr1_masked_ep8_M512_tc": (32, 128, 512, 2), "dsr1_masked_ep8_M4096_tc": (32, 1024, 4096, 2)}


def masked_problem(name, seed=1234):
    """(local layer shape [M = E*cap rows, topk 1], x [E*cap, H], flat ids [E*cap, 1] with -1 on
    padding rows, unit weights, counts [E])."""
    E, cap, M, _ = MASKED[name]
    full = synth.deepseek_r1(M)
    ids, _ = synth.make_routing(full, seed)
    counts = torch.bincount(ids[:, :full.topk].reshape(-1).long(), minlength=full.E)[:E].clamp(max=cap)
    shape = synth.LayerShape(name, E * cap, full.H, full.I, E, 1, "fp8", "uniform")
    x = synth.make_x(shape, seed)
    flat = torch.full((E * cap, 1), -1, dtype=torch.int32)
    for e in range(E):
        flat[e * cap:e * cap + int(counts[e]), 0] = e
    return shape, x, flat, torch.ones(E * cap, 1), counts.to(torch.int32)


def all_workloads():
    w = workloads()
    masked = {n: synth.LayerShape(n, E * cap, 7168, 2048, E, 1, "fp8", "uniform") for n, (E, cap, _, _) in MASKED.items()}
    return {**w, **{g: w[base] for g, base in GATED.items()}, **masked}


def gate_config_of(shape):
    """The router of the workload's model configuration."""
    if shape.routing.startswith("deepseek"):
        return gbmoe.gate_config(gbmoe.MOE_GATE_SIGMOID_GROUPED, shape.n_group, shape.topk_group,
                                 shape.routed_scaling, None, shape.shared_expert)
    return gbmoe.gate_config(shared_expert=shape.shared_expert)


KERNEL_SOURCES = {  # kernel -> the source files that define it
    "decode_gemm1": "moe_decode.cu", "decode_gemm2": "moe_decode.cu",
    "prefill_gemm1": "moe_prefill.cu", "prefill_gemm2": "moe_prefill.cu",
}


def source_hash(kernel: str, a8: bool = False) -> str:
    """Hash of the kernel's own source file and the headers it includes (a8: the FP8-operand prefill kernels,
    which run every FP8-weight layer on the tcgen05 path)."""
    csrc = os.path.join(ROOT, "mixture_experts_ffn_moe_gb300", "csrc")
    h = hashlib.sha256()
    src = "moe_prefill_a8.cu" if a8 and kernel.startswith("prefill") else KERNEL_SOURCES.get(kernel, "")
    for name in (src, "common.cuh", "sm100_ptx.cuh", "internal.h"):
        path = os.path.join(csrc, name)
        if name and os.path.exists(path):
            h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def ncu_traffic(workload: str, kernel: str, a8: bool = False):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    rec = d.get(workload, {}).get(kernel)
    if not rec or rec.get("source_hash") != source_hash(kernel, a8):
        return None
    return rec.get("dram_bytes_per_launch")


def roofline_of(shape, ids, stages, n_calls, workload, peaks):
    """Roofline of the dominant kernel of a call: its algorithmic bytes (or flops, above the ridge) over its
    average per-kernel event time, against the measured peak."""
    work = stage_work(shape, ids)
    stage_avg = {name: ms / max(n_calls, 1) for name, ms in stages}
    dominant = max((n for n in stage_avg if n in work), key=lambda n: stage_avg[n])
    dbytes, dflops = work[dominant]
    secs = stage_avg[dominant] * 1e-3
    # Tensor peak of the kernel's operand type, burst figure: fp16 MMA runs at the measured dense
    # bf16 rate; E4M3 x E4M3 at twice it (the nominal FP8:BF16 ratio, 4.5 : 2.25 PFLOP/s).
    if shape.act == "fp8_1x128":
        tpeak, tsrc = 2.0 * peaks["bf16_tflops"], peaks["source"] + " bf16 dense x 2 (nominal FP8:BF16 ratio)"
    elif shape.weight_kind == "fp8" and shape.M >= gbmoe.MOE_AUTO_PREFILL_TOKENS and dominant.startswith("prefill"):
        # two E4M3 products per product at the FP8 rate (twice bf16): the same bound as one bf16 product
        tpeak, tsrc = peaks["bf16_tflops"], peaks["source"] + (" bf16 dense (two-term E4M3 activations: two FP8 "
                                                                "products per product at twice the bf16 rate)")
    else:
        tpeak, tsrc = peaks["bf16_tflops"], peaks["source"] + " bf16 dense (fp16 same rate)"
    ridge = tpeak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    a8 = shape.weight_kind == "fp8" and dominant.startswith("prefill")  # FP8 weights: the FP8-operand kernels
    if dflops / dbytes > ridge:
        achieved = dflops / secs / 1e12
        return {"bound": "tensor", "kernel": dominant, "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                "frac": achieved / tpeak, "traffic": ncu_traffic(workload, dominant, a8),
                "algorithmic_flops": dflops, "algorithmic_bytes": dbytes, "peak_source": tsrc}
    achieved = dbytes / secs / 1e9
    return {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(workload, dominant, a8),
            "algorithmic_bytes": dbytes, "algorithmic_flops": dflops, "peak_source": peaks["source"]}


def routing_summary(shape, ids):
    """The realised expert histogram of a call: active experts, tokens per active expert and the balance
    (mean / max, 1.0 = even), over all experts and over the routed ones alone (a shared expert takes
    every token)."""
    hist = synth.expert_histogram(shape, ids)

    def stats(h):
        act = h[h > 0].double()
        if not act.numel():
            return None
        q = torch.quantile(act, torch.tensor([0.0, 0.5, 0.9, 1.0], dtype=torch.float64)).tolist()
        return {"active_experts": int(act.numel()), "min": q[0], "median": q[1], "p90": q[2], "max": q[3],
                "mean": float(act.mean()), "balance_mean_over_max": float(act.mean() / act.max())}

    return {"experts": shape.E_total, "all": stats(hist),
            "routed": stats(hist[:shape.E]) if shape.shared_expert else None}


def parity_rows(shape, x, ids, w, weights, out, tokens):
    """rel-L2 and max-abs / max|ref| of the layer's output rows `tokens` against the oracle."""
    import oracle
    ref = oracle.fused_moe_rows(x, ids, w, *weights, kind=shape.weight_kind, tokens=tokens, act=shape.act)
    got = out[torch.as_tensor(tokens, dtype=torch.long, device=out.device)].float().cpu().numpy().astype(np.float64)
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    mabs = float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))
    experts = int(np.unique(ids[tokens].numpy()).size)
    return {"rel_l2": rel, "max_abs_over_max_ref": mabs, "tokens": len(tokens), "experts_covered": experts,
            "within_tolerance": rel <= 5e-3 and mabs <= 1e-2, "tolerance": "rel-L2 <= 5e-3, max-abs <= 1e-2 max|ref|"}


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


ONE_CORE_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                "BLIS_NUM_THREADS": "1", "NUMEXPR_NUM_THREADS": "1"}


def oracle_one_core(shape, x, ids, w, weights, tokens):
    """Seconds the oracle takes for `tokens` in a child process limited to one thread (its BLAS and
    OpenMP pools set to 1 before numpy loads).  Only the involved experts' weights are handed over."""
    import tempfile
    used = sorted({int(e) for e in ids[tokens].reshape(-1).tolist() if 0 <= e < shape.E_total})
    remap = {e: i for i, e in enumerate(used)}
    sub_ids = ids[tokens].clone().apply_(lambda e: remap.get(int(e), -1))
    payload = {"x": x[tokens], "ids": sub_ids, "w": w[tokens], "kind": shape.weight_kind, "act": shape.act,
               "weights": [t[used].cpu() for t in weights]}
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "sample.pt")
        torch.save(payload, path)
        code = ("import sys, time, torch; sys.path.insert(0, %r); import oracle; p = torch.load(%r); "
                "t0 = time.perf_counter(); oracle.fused_moe_rows(p['x'], p['ids'], p['w'], *p['weights'], "
                "kind=p['kind'], tokens=list(range(p['x'].shape[0])), act=p['act']); "
                "print(time.perf_counter() - t0)") % (ROOT, path)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                           env={**os.environ, **ONE_CORE_ENV})
    if r.returncode != 0:
        return None
    return float(r.stdout.strip().splitlines()[-1])


def stage_work(shape, ids: torch.Tensor):
    """Algorithmic (bytes, flops) per kernel of one call.

    Bytes: distinct activated weights (codes + scales) read once, plus the
    activation rows each kernel must read or write once.  Flops: 2 per
    multiply-add of the unpadded (token, expert) pairs.
    """
    hist = synth.expert_histogram(shape, ids)
    active = int((hist > 0).sum())
    valid = int(hist.sum())
    H, I, M = shape.H, shape.I, shape.M
    ab = 1 if shape.act == "fp8_1x128" else 2  # bytes per gathered activation element (E4M3 or fp16)
    wb = 0.5 if shape.weight_kind == "int4" else 1  # bytes per weight code
    if shape.weight_kind == "fp8":
        s13 = 4 * (2 * I // 128) * (H // 128)
        s2 = 4 * (H // 128) * (I // 128)
    elif shape.weight_kind == "int4":
        s13, s2 = 4 * 2 * I * (H // 128), 4 * H * (I // 128)
    else:
        s13, s2 = 4 * 2 * I, 4 * H
    f1 = 2 * valid * 2 * I * H
    f2 = 2 * valid * H * I
    return {
        "decode_gemm1": (int(active * (2 * I * H * wb + s13)) + M * H * 2 + valid * I * 2, f1),
        "decode_gemm2": (int(active * (H * I * wb + s2)) + valid * I * 2 + valid * H * 4, f2),
        "prefill_gemm1": (active * (2 * I * H + s13) + valid * H * ab + valid * I * ab, f1),
        "prefill_gemm2": (active * (H * I + s2) + valid * I * ab + valid * H * 2, f2),  # y in bf16
    }


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    _count = 0

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        ClockSampler._count += 1  # one file per sampler: several may run in one process
        self.path = os.path.join("/tmp", f"gbmoe_clocks_{os.getpid()}_{ClockSampler._count}.csv")
        self.samples = None

    def _lines(self):
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        # the sampler's start-up takes a moment: time nothing before its first sample is written
        t0 = time.time()
        while self.proc is not None and self._lines() < 1 and time.time() - t0 < 5.0:
            time.sleep(0.05)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            n, t0 = self._lines(), time.time()
            while self._lines() < n + 2 and time.time() - t0 < 2.0:  # samples that follow the timed work
                time.sleep(0.05)
            self.proc.terminate()
            self.proc.wait()

    def _read(self):
        """[(unix time, sm MHz, max sm MHz, set of active reasons)], read once after the sampler stops."""
        if self.samples is not None:
            return self.samples
        self.samples = []
        if self.proc is None or not os.path.exists(self.path):
            return self.samples
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax = float(f[2]), float(f[3])
            except ValueError:
                continue
            self.samples.append((ts, sm, smax, {n for n, v in zip(names, f[6:10]) if v.lower() == "active"}))
        os.unlink(self.path)
        return self.samples

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and throttle reasons of the samples taken in [t0, t1] widened by one
        sampling period (unix time; all samples when not given)."""
        sel = [x for x in self._read() if (t0 is None or x[0] >= t0 - 0.2) and (t1 is None or x[0] <= t1 + 0.2)]
        if not sel:
            return None
        reasons = set().union(*(x[3] for x in sel))
        return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_max_mhz": max(x[2] for x in sel),
                "reasons": sorted(reasons), "samples": len(sel)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def make_inputs(shape, seed=1234):
    ids, w = synth.make_routing(shape, seed)
    x = synth.make_x(shape, seed)
    w13, s13, w2, s2 = synth.make_weights(shape, seed, device="cuda")
    return x, ids, w, (w13, s13, w2, s2)


def cpu_cores() -> int:
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        blas = [i["num_threads"] for i in info if i.get("user_api") == "blas"]
        if blas:
            return int(blas[0])
    except ImportError:
        pass
    return os.cpu_count() or 1


def oracle_sample(shape, x, ids, w, weights, token=0):
    """Times the oracle on one token of the batch (all of its experts); returns (tokens/s, seconds, text)."""
    import oracle
    w13, s13, w2, s2 = weights
    t0 = time.perf_counter()
    oracle.fused_moe_rows(x, ids, w, w13, s13, w2, s2, kind=shape.weight_kind, tokens=[token], act=shape.act)
    dt = time.perf_counter() - t0
    return 1.0 / dt, dt, (f"1 token of the {shape.M}-token batch ({int((ids[token] >= 0).sum())} experts), "
                          "float64 numpy")


def run_reference(args, shape):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    wdev = "cuda" if torch.cuda.is_available() else "cpu"
    if args.workload in MASKED:
        shape, x, ids, w, _ = masked_problem(args.workload)
    else:
        ids, w = synth.make_routing(shape, 1234)
        x = synth.make_x(shape, 1234)
    weights = synth.make_weights(shape, 1234, device=wdev)
    tok = int((ids[:, 0] >= 0).nonzero()[0])
    for _ in range(args.warmup):
        oracle_sample(shape, x, ids, w, weights, tok)
    times = [oracle_sample(shape, x, ids, w, weights, tok)[1] for _ in range(args.steps)]
    total = sum(times)
    value = args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(shape, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": oracle_sample(shape, x, ids, w, weights, tok)[2] + " per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(shape, args):
    if args.workload in MASKED:
        E, cap, M, path = MASKED[args.workload]
        return {"workload": args.workload, "layout": f"masked: {E} local experts x {cap} rows (rank 0 of 8)",
                "path": "tcgen05 (MOE_PATH_PREFILL)" if path == 2 else "weight-streaming",
                "global_tokens": M, "H": shape.H, "I": shape.I, "weights": "fp8_e4m3_block128",
                "activations": "bf16", "unit": "a token is one dispatched (token, local expert) row",
                "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas{args.gpus}"}
    return {"workload": args.workload, "M": shape.M, "H": shape.H, "I": shape.I, "E": shape.E_total,
            "topk": shape.topk_total, "weights": {"fp8": "fp8_e4m3_block128", "int8": "int8_per_channel",
                                                  "int4": "int4_group128"}[shape.weight_kind],
            "activations": "fp8_e4m3_1x128" if shape.act == "fp8_1x128" else
            ("int8_per_row" if shape.weight_kind == "int8" else "bf16"),
            "routing": shape.routing + (" (gated on the GPU from router logits)" if args.workload in GATED else ""),
            "l2": "flushed between steps (256 MiB write)",
            "parallelism": f"replicas{args.gpus}"}


def run_ours(args, shape):
    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    torch.cuda.set_device(local)
    from mixture_experts_ffn_moe_gb300 import build
    build.build()
    gbmoe.load()
    dev = torch.device("cuda", local)
    masked = args.workload in MASKED
    if masked:
        shape, x, ids, w, counts = masked_problem(args.workload)
        w13, s13, w2, s2 = synth.make_weights(shape, 1234, device="cuda")
        units = int(counts.sum())  # dispatched rows processed per step
    else:
        x, ids, w, (w13, s13, w2, s2) = make_inputs(shape)
        units = shape.M
    xd, idsd, wd = x.to(dev), ids.to(dev), w.to(dev)
    kind = {"fp8": gbmoe.MOE_WEIGHT_FP8, "int8": gbmoe.MOE_WEIGHT_INT8, "int4": gbmoe.MOE_WEIGHT_INT4}[shape.weight_kind]
    fn = {gbmoe.MOE_WEIGHT_FP8: gbmoe.fused_moe_fp8, gbmoe.MOE_WEIGHT_INT8: gbmoe.fused_moe_int8,
          gbmoe.MOE_WEIGHT_INT4: gbmoe.fused_moe_int4}[kind]
    flags = gbmoe.MOE_ACT_FP8_1X128 if shape.act == "fp8_1x128" else gbmoe.MOE_PATH_AUTO
    if masked:
        E_loc, cap = shape.E, shape.M // shape.E
        ws = torch.empty(gbmoe.moe_workspace_size_masked(E_loc, cap, shape.H, shape.I, kind), dtype=torch.uint8,
                         device=dev)
        md = counts.to(dev)
    else:
        ws = gbmoe.alloc_workspace(shape.M, shape.H, shape.I, shape.E_total, shape.topk_total, kind, flags, dev)
    out = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    gated = args.workload in GATED
    if gated:
        lg = synth.make_router_logits(shape, 1234)
        lgd = lg.to(dev)
        gcfg = gate_config_of(shape)

        def step():
            gbmoe.fused_moe_gated(kind, xd, lgd, gcfg, shape.topk, w13, s13, w2, s2, flags=flags, out=out,
                                  workspace=ws, topk_ids=idsd, topk_weights=wd)
    elif masked:
        def step():
            gbmoe.fused_moe_masked(kind, xd.view(E_loc, cap, shape.H), md, w13, s13, w2, s2,
                                   out=out.view(E_loc, cap, shape.H), workspace=ws, flags=MASKED[args.workload][3])
    else:
        def step():
            fn(xd, idsd, wd, w13, s13, w2, s2, flags=flags, out=out, workspace=ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    bad, dev_flags, st = gbmoe.moe_read_status(ws)
    if st != 0:
        raise SystemExit(f"device status after warm-up: bad ids {bad}, flags {dev_flags}")

    # ---- timed region: K steps, device time per step with CUDA events on the launch stream.
    # The layer's kernels overlap their launches (programmatic dependent launch), so no
    # event is recorded between them here; per-kernel times come from the pass below.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index if world == 1 else local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - wall0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # ---- per-kernel pass: the same K steps with CUDA events recorded between the kernels
    gbmoe.moe_profile_enable(args.steps)
    prof_start = torch.cuda.Event(enable_timing=True)
    prof_end = torch.cuda.Event(enable_timing=True)
    prof_ms = 0.0
    for i in range(args.steps):
        flush.zero_()
        prof_start.record(stream)
        step()
        prof_end.record(stream)
        prof_end.synchronize()
        prof_ms += prof_start.elapsed_time(prof_end)
    n_calls, stages = gbmoe.moe_profile_read()
    gbmoe.moe_profile_enable(0)
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = world * units * args.steps / (total_ms / 1e3)

    # ---- roofline of the dominant kernel
    peaks = measured_peaks()
    # (masked: the activation terms count the real rows only)
    roofline = roofline_of(dataclasses.replace(shape, M=units) if masked else shape, ids, stages, n_calls,
                           args.workload, peaks)
    layer_bytes = synth.distinct_weight_bytes(shape, ids)
    flops = synth.algorithmic_flops(shape, ids)

    # ---- end to end through the public API with host buffers (pinned), copies inside the timing
    # (gated workloads copy the router logits instead of the routing)
    xh, idsh, wh = x.pin_memory(), ids.pin_memory(), w.pin_memory()
    lgh = lg.pin_memory() if gated else None
    mh = counts.pin_memory() if masked else None
    outh = torch.empty(shape.M, shape.H, dtype=torch.bfloat16).pin_memory()
    h2d = xh.numel() * 2 + (lgh.numel() * 4 if gated else mh.numel() * 4 if masked else
                            idsh.numel() * 4 + wh.numel() * 4)
    d2h = outh.numel() * 2
    e_start = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_end = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        e_start[i].record(stream)
        xd.copy_(xh, non_blocking=True)
        if gated:
            lgd.copy_(lgh, non_blocking=True)
        elif masked:
            md.copy_(mh, non_blocking=True)
        else:
            idsd.copy_(idsh, non_blocking=True)
            wd.copy_(wh, non_blocking=True)
        step()
        outh.copy_(out, non_blocking=True)
        e_end[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(e_start, e_end)), world)
    e2e_value = world * units * args.steps / (e2e_ms / 1e3)

    if rank != 0:
        return
    stage_avg = {name: ms / max(n_calls, 1) for name, ms in stages}
    # ---- parity of the timed output against the oracle (rank 0): every token up to 16 tokens, else a
    # bounded sample; the routing the call realised
    real = [int(t) for t in ((ids >= 0) & (ids < shape.E_total)).any(dim=1).nonzero().flatten()]
    ptoks = real if len(real) <= 16 else real[:: max(1, len(real) // 8)][:8]
    parity = parity_rows(shape, x, ids, w, (w13, s13, w2, s2), out, ptoks) if ptoks and not masked else None
    routing = routing_summary(shape, ids)
    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only), on every host core and on
    # one, with the host's CPU model
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        tok = int((ids[:, 0] >= 0).nonzero()[0])
        v, dt, text = oracle_sample(shape, x, ids, w, (w13, s13, w2, s2), token=tok)
        one = oracle_one_core(shape, x, ids, w, (w13, s13, w2, s2), [tok])
        cpu = {"value": v, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle", "sample": text,
               "seconds": dt, "cpu_model": cpu_model(),
               "one_core": {"value": 1.0 / one, "unit": "tokens/s", "cores": 1, "seconds": one} if one else None,
               "tiny_layer": tiny_cpu_baseline()}
    main_clocks = clocks.summary()
    # ---- the other configurations of the layer, each timed the same way (N = 1 only)
    also = None
    if world == 1 and not args.no_also and args.workload == DEFAULT_WORKLOAD:
        also = run_also(dev, flush, peaks, (w13, s13, w2, s2), shape)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype_of(shape, kind),
        "data": "synthetic", "config": config_of(shape, args),
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": sum(1 for _ in stages) * n_calls,
        "clocks": main_clocks,
        "parity": parity,
        "routing": routing,
        "layer": {"weight_gbs": layer_bytes / (ms_per_step * 1e-3) / 1e9,
                  "weight_bytes": layer_bytes, "hbm_frac": layer_bytes / (ms_per_step * 1e-3) / 1e9 / peaks["hbm_gbs"],
                  "tflops": flops / (ms_per_step * 1e-3) / 1e12,
                  # context: the layer's rate against the dense bf16 peak and the FP8 peak (2x bf16, nominal ratio)
                  "tflops_frac_bf16": flops / (ms_per_step * 1e-3) / 1e12 / peaks["bf16_tflops"],
                  "tflops_frac_fp8": flops / (ms_per_step * 1e-3) / 1e12 / (2.0 * peaks["bf16_tflops"]),
                  "active_experts":
                  int((synth.expert_histogram(shape, ids) > 0).sum()),
                  "stages_ms": {n: round(v, 5) for n, v in stage_avg.items()},
                  "ms_per_step_with_kernel_events": prof_ms / args.steps},
        "also": also,
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def dtype_of(shape, kind):
    """The arithmetic the call's path computes in (MOE_PATH_AUTO: the weight-streaming kernels up to
    MOE_AUTO_PREFILL_TOKENS tokens, the tcgen05 kernels from there; FP8 activations always on tcgen05)."""
    if kind == gbmoe.MOE_WEIGHT_FP8:
        if shape.act == "fp8_1x128":
            return "fp8 x fp8 mma, f32 acc"
        if shape.M >= gbmoe.MOE_AUTO_PREFILL_TOKENS:
            return "fp8 x fp8 mma (bf16 x and fp32 h as two e4m3 terms), f32 acc"
        return "fp8->f16 mma, f32 acc"
    return "int8->f16 mma, f32 acc" if kind == gbmoe.MOE_WEIGHT_INT8 else "int4->f16 mma, f32 acc"


def tiny_cpu_baseline():
    """The oracle on the whole tiny layer (16 tokens), on every host core and on one."""
    import oracle
    shape = synth.tiny()
    d = synth.make_layer(shape, 1234)
    args = [d[k] for k in ("x", "topk_ids", "topk_weights", "w13", "w13_scale", "w2", "w2_scale")]
    t0 = time.perf_counter()
    reps = 5
    for _ in range(reps):
        oracle.fused_moe_fp8(*args)
    dt = (time.perf_counter() - t0) / reps
    one = oracle_one_core(shape, d["x"], d["topk_ids"], d["topk_weights"], args[3:], list(range(shape.M)))
    return {"workload": "tiny_M16", "tokens_per_s": shape.M / dt, "cores": cpu_cores(),
            "tokens_per_s_one_core": shape.M / one if one else None}


# The other workloads of the layer's configurations, timed after the default line: DeepSeek-R1 single-token
# decode, the uniform-routing decode sweep, the 2048-token Zipf prefill and the 16,384-token prefill
# (weight-only and FP8 activations), and the Qwen3 INT8 layer at 1, 16, 256 and 4096 tokens.
ALSO_WORKLOADS = (["dsr1_decode_M1"] + [f"dsr1_sweep_M{m}" for m in (1, 2, 4, 8, 16, 32, 64)] +
                  ["dsr1_prefill_M2048", "dsr1_prefill_M2048_a8", "dsr1_prefill_M16384", "dsr1_prefill_M16384_a8",
                   "qwen3_M1", "qwen3_M16", "qwen3_M256", "qwen3_M4096"])
ALSO_MIN_SECONDS = 0.3   # timed work per entry (so the clock sampler sees it)


def run_also(dev, flush, peaks, main_weights, main_shape):
    """Times every ALSO_WORKLOADS entry as the default line is timed (L2 flushed between steps, CUDA events
    on the launch stream, a per-kernel pass for the roofline) and checks one token against the oracle."""
    stream = torch.cuda.current_stream(dev)
    cache = {(main_shape.E_total, main_shape.H, main_shape.I, main_shape.weight_kind): main_weights}
    results, windows = {}, {}
    with ClockSampler(dev.index) as clocks:
        for name in ALSO_WORKLOADS:
            shape = workloads()[name]
            key = (shape.E_total, shape.H, shape.I, shape.weight_kind)
            if key not in cache:
                cache = {key: synth.make_weights(shape, 1234, device="cuda")}
                torch.cuda.empty_cache()
            weights = cache[key]
            ids, tw = synth.make_routing(shape, 1234)
            x = synth.make_x(shape, 1234)
            xd, idsd, twd = x.to(dev), ids.to(dev), tw.to(dev)
            kind = {"fp8": gbmoe.MOE_WEIGHT_FP8, "int8": gbmoe.MOE_WEIGHT_INT8,
                    "int4": gbmoe.MOE_WEIGHT_INT4}[shape.weight_kind]
            fn = {gbmoe.MOE_WEIGHT_FP8: gbmoe.fused_moe_fp8, gbmoe.MOE_WEIGHT_INT8: gbmoe.fused_moe_int8,
                  gbmoe.MOE_WEIGHT_INT4: gbmoe.fused_moe_int4}[kind]
            flags = gbmoe.MOE_ACT_FP8_1X128 if shape.act == "fp8_1x128" else gbmoe.MOE_PATH_AUTO
            ws = gbmoe.alloc_workspace(shape.M, shape.H, shape.I, shape.E_total, shape.topk_total, kind, flags, dev)
            o = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device=dev)

            def step():
                fn(xd, idsd, twd, *weights, flags=flags, out=o, workspace=ws)

            for _ in range(3):
                flush.zero_()
                step()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(3):
                flush.zero_()
                step()
            e1.record(stream)
            e1.synchronize()
            steps = int(min(4000, max(5, ALSO_MIN_SECONDS * 1e3 / (e0.elapsed_time(e1) / 3))))
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            torch.cuda.synchronize()
            t0 = time.time()
            for i in range(steps):
                flush.zero_()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize()
            windows[name] = (t0, time.time())
            ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
            bad, dev_flags, st = gbmoe.moe_read_status(ws)
            if st != 0:
                raise SystemExit(f"{name}: device status bad ids {bad}, flags {dev_flags}")
            npass = min(steps, 10)
            gbmoe.moe_profile_enable(npass)
            for _ in range(npass):
                flush.zero_()
                step()
            n_calls, stages = gbmoe.moe_profile_read()
            gbmoe.moe_profile_enable(0)
            roof = roofline_of(shape, ids, stages, n_calls, name, peaks)
            layer_bytes = synth.distinct_weight_bytes(shape, ids)
            flops = synth.algorithmic_flops(shape, ids)
            tok = int((ids[:, 0] >= 0).nonzero()[0])
            results[name] = {
                "M": shape.M, "ms": ms, "tokens_per_s": shape.M / (ms * 1e-3), "steps": steps,
                "dtype": dtype_of(shape, kind),
                "roofline": {k: roof[k] for k in ("kernel", "bound", "achieved", "unit", "peak", "frac")},
                "layer": {"weight_gbs": layer_bytes / (ms * 1e-3) / 1e9,
                          "hbm_frac": layer_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                          "tflops": flops / (ms * 1e-3) / 1e12,
                          "tflops_frac_bf16": flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                          "tflops_frac_fp8": flops / (ms * 1e-3) / 1e12 / (2.0 * peaks["bf16_tflops"])},
                "stages_ms": {n: round(v / max(n_calls, 1), 5) for n, v in stages},
                "routing": routing_summary(shape, ids),
                "parity": parity_rows(shape, x, ids, tw, weights, o, [tok]),
            }
            del ws, o, xd, idsd, twd
    for name, (t0, t1) in windows.items():
        results[name]["clocks"] = clocks.summary(t0, t1)
    return results


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(all_workloads()))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-also", action="store_true", help="time the default workload only")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    shape = all_workloads()[args.workload]
    if args.impl == "reference":
        run_reference(args, shape)
    else:
        run_ours(args, shape)


if __name__ == "__main__":
    main()
