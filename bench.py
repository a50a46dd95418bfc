"""Benchmark of the DeepSeekMoE FP8 layer forward + bias update on B300.

One step = the whole path over one batch: route (logits, sigmoid, biased
top-K, gates, counts) -> dispatch -> 1x128 quantisation of the gathered
activations -> grouped FP8 GEMM gate/up + SiLU + re-quantisation -> grouped
FP8 GEMM down -> combine with shared expert and residual -> bias update.
Every step runs in libmoefp8's kernels, called through its C ABI.

Default workload: the V3-shape prefill batch (T=4096 tokens, d=7168, 256
routed experts top-8 + 1 shared, intermediate 2048), synthetic seeded data
and weights.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain C implementation used as
the correctness reference) on the host cores, on a bounded sample of the
same workload.  With N > 1 (torchrun) every rank runs an independent replica
of the layer on its own GPU (the path has no cross-GPU exchange step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from fine_grained_fp8_bias_b300 import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/s at d=7168,256e top-8; FP8 GEMM % peak; decode HBM GB/s"
FP8_OVER_BF16 = 2.0   # nominal dense FP8 : BF16 tensor rate (4.5 : 2.25 PFLOP/s)
STAGES = ["route", "permute", "quant", "gemm_gate_up", "gemm_down", "combine", "bias_update"]
KERNELS_PER_STAGE = {"route": 2, "permute": 3, "quant": 1, "gemm_gate_up": 1, "gemm_down": 1,
                     "combine": 1, "bias_update": 1}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest replica's time for the timed region (all-reduce MAX; the
    process group is NCCL on GPUs, gloo in the CPU tests)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, T: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every replica processed T tokens per step, and the
    job took as long as its slowest replica."""
    return world * T * steps / (ms / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# --------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())}


# ----------------------------------------------------------- GPU path
class Step:
    """Buffers and the component calls of one step (the same sequence moe_forward runs)."""

    def __init__(self, layer, u, gamma):
        from fine_grained_fp8_bias_b300 import lib
        self.lib = lib
        self.L = layer
        self.u = u
        self.gamma = gamma
        T, d, E, K, S, I = u.shape[0], layer.d, layer.E, layer.K, layer.S, layer.I
        self.T, self.M = T, T * (K + S)
        dev = u.device
        M = self.M
        self.route_ws = torch.empty(lib.route_workspace_bytes(T, E, d), dtype=torch.uint8,
                                    device=dev)
        nchunks = (T + 63) // 64
        self.perm_ws = torch.empty(2 * ((4 * nchunks * E + 255) // 256 * 256) + 256,
                                   dtype=torch.uint8, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.rout = {"idx": torch.empty((T, K), dtype=torch.int32, device=dev),
                     "gate": torch.empty((T, K), dtype=torch.float32, device=dev),
                     "tie": torch.empty((T,), dtype=torch.uint8, device=dev),
                     "counts": torch.empty((E,), dtype=torch.int32, device=dev)}
        self.pout = {"offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev),
                     "group_offsets": torch.empty((E + S + 1,), dtype=torch.int32, device=dev),
                     "perm_token": torch.empty((M,), dtype=torch.int32, device=dev),
                     "inv_row": torch.empty((T, K), dtype=torch.int32, device=dev)}
        self.A = torch.empty((M, d), dtype=torch.uint8, device=dev)
        self.sa = torch.empty((d // 128, M), dtype=torch.float32, device=dev)
        self.H = torch.empty((M, I), dtype=torch.uint8, device=dev)
        self.sh = torch.empty((I // 128, M), dtype=torch.float32, device=dev)
        self.Y = torch.empty((T * K, d), dtype=torch.bfloat16, device=dev)
        self.Ysh = torch.empty((T * S, d), dtype=torch.float32, device=dev)
        self.h = torch.empty((T, d), dtype=torch.float32, device=dev)

    def stage(self, name):
        lib, L = self.lib, self.L
        if name == "route":
            if L.n_groups:
                lib.moe_route_grouped(self.u, L.centroids, L.bias, L.K, L.n_groups, L.topk_groups,
                                      L.group_topk, ws=self.route_ws, out=self.rout)
            elif self.T < 256:
                # below 256 tokens moe_forward sums all logits on CUDA cores: the
                # kernels of moe_route_noalloc
                lib.moe_route_noalloc(self.u, L.centroids, L.bias, L.K, out=self.rout)
            else:
                lib.moe_route(self.u, L.centroids, L.bias, L.K, ws=self.route_ws, out=self.rout)
        elif name == "permute":
            lib.moe_permute(self.rout["idx"], L.E, L.S, ws=self.perm_ws, status=self.status,
                            out=self.pout)
        elif name == "quant":
            lib.moe_quant_1x128_dispatch(self.u, self.pout["inv_row"], L.K, L.S, q=self.A,
                                         scales=self.sa, status=self.status)
        elif name == "gemm_gate_up":
            gemm = lib.moe_grouped_gemm_fp8_small if self.T <= 64 else lib.moe_grouped_gemm_fp8
            gemm(lib.MOE_GEMM_GATE_UP_SILU_QUANT, self.A, self.sa,
                                     self.pout["group_offsets"], L.w_gate, L.w_up, L.s_gate,
                                     L.s_up, out=self.H, out_scales=self.sh, status=self.status)
        elif name == "gemm_down":
            # routed rows bf16, shared rows float32; the small-group tiles for the
            # gate/up GEMM up to 64 tokens and for the down GEMM up to 4 (as moe_forward)
            lib.moe_grouped_gemm_fp8_down(self.H, self.sh, self.pout["group_offsets"], L.w_down,
                                          L.s_down, L.E, self.T * L.K, self.Y, self.Ysh,
                                          small_tiles=self.T <= 4, status=self.status)
        elif name == "combine":
            lib.moe_combine(self.u, self.Y, self.rout["gate"], self.pout["inv_row"],
                            self.Ysh if L.S else None, L.S, h=self.h)
        elif name == "bias_update":
            lib.moe_update_bias(self.rout["counts"], L.bias, self.T, L.K, self.gamma)

    def run(self, events=None):
        for i, name in enumerate(STAGES):
            self.stage(name)
            if events is not None:
                events[i].record()


def algorithmic_bytes(cfg, T, touched: int) -> dict:
    """Minimal HBM bytes of each stage (each input read once, each output written once)."""
    d, E, K, S, I = cfg.d, cfg.E, cfg.K, cfg.S, cfg.I
    M = T * (K + S)
    wsc = lambda n, k: (n // 128) * (k // 128) * 4
    return {
        "route": T * d * 2 + E * d * 4 + E * 4 + T * K * 8 + T + E * 4,
        "permute": T * K * 4 + M * 4 + T * K * 4 + (E + S + 1) * 4 * 2,
        "quant": T * d * 2 + M * 4 + M * d + M * (d // 128) * 4,
        "gemm_gate_up": touched * 2 * (I * d + wsc(I, d)) + M * d + M * (d // 128) * 4
        + M * I + M * (I // 128) * 4,
        # expert outputs y: routed rows bf16, shared rows float32
        "gemm_down": touched * (d * I + wsc(d, I)) + M * I + M * (I // 128) * 4
        + T * K * d * 2 + T * S * d * 4,
        "combine": T * d * 2 + T * K * d * 2 + T * S * d * 4 + T * K * 8 + T * d * 4,
        "bias_update": E * 4 * 3,
    }


def gemm_flops(cfg, T) -> dict:
    M = T * (cfg.K + cfg.S)
    return {"gemm_gate_up": 2.0 * M * 2 * cfg.I * cfg.d, "gemm_down": 2.0 * M * cfg.d * cfg.I}


def kernel_traffic(stage: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source and the same workload (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    src = os.path.join(ROOT, "fine_grained_fp8_bias_b300", "csrc", d.get("source_file", ""))
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    e = d.get("kernels", {}).get(stage)
    if e is None or d.get("source_sha256_16") != h or d.get("workload_name") != workload:
        return None
    return e.get("dram_bytes_per_launch")


def time_steps(step, steps):
    """Times `steps` whole steps on the current stream with CUDA events: total
    ms and the per-stage ms summed over the steps (an event after each stage)."""
    stream = torch.cuda.current_stream()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in STAGES] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(steps):
        step.run(evs[k])
    stop.record(stream)
    torch.cuda.synchronize()
    per_stage = {s: 0.0 for s in STAGES}
    for k in range(steps):
        for i, s in enumerate(STAGES):
            a = start if (k == 0 and i == 0) else (evs[k][i - 1] if i > 0 else evs[k - 1][-1])
            per_stage[s] += a.elapsed_time(evs[k][i])
    return start.elapsed_time(stop), per_stage


def kernel_table(cfg, T, touched, per_stage, steps):
    abytes = algorithmic_bytes(cfg, T, touched)
    flops = gemm_flops(cfg, T)
    kernels = {}
    for s in STAGES:
        ms = per_stage[s] / steps
        kernels[s] = {"ms": round(ms, 4), "share": round(per_stage[s] / sum(per_stage.values()), 4),
                      "GBps": round(abytes[s] / (ms * 1e-3) / 1e9, 1)}
        if s in flops:
            kernels[s]["TFLOPs"] = round(flops[s] / (ms * 1e-3) / 1e12, 1)
    return kernels, abytes, flops


def run_ours(args, world, rank, local):
    from fine_grained_fp8_bias_b300 import lib
    from fine_grained_fp8_bias_b300.layer import MoELayer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = wl.CONFIGS[args.workload]
    if args.tokens:
        cfg = cfg.with_(T=args.tokens)
    pk = peaks()
    layer = MoELayer.from_config(cfg, dev)
    u = wl.tokens(cfg, dev)
    step = Step(layer, u, cfg.gamma)

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if lib.moe_check_device_status(step.status) != 0:
        raise RuntimeError("device status flagged during warm-up")

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    launches0 = lib.kernel_launches()
    total_ms, per_stage = time_steps(step, args.steps)
    launches = lib.kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if lib.moe_check_device_status(step.status) != 0:
        raise RuntimeError("device status flagged during the timed region")

    counts = step.rout["counts"].cpu()
    touched = int((counts > 0).sum()) + cfg.S
    T = cfg.T
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_step = total_ms / args.steps
    value = job_tokens_per_s(world, T, args.steps, total_ms)

    # per-kernel roofline
    kernels, abytes, flops = kernel_table(cfg, T, touched, per_stage, args.steps)
    dom = max(STAGES, key=lambda s: per_stage[s])
    dom_ms = per_stage[dom] / args.steps
    # FP8 dense peak: measured on this GPU (cuBLASLt e4m3 GEMM), burst for a kernel
    # timed alone, sustained for a kernel timed inside a long loop of steps (the
    # GEMMs here); without the probe, the bf16 figures x the nominal FP8:BF16 ratio.
    fp8 = fp8_peak_probe(dev) if not args.no_fp8_probe else None
    if fp8 and fp8.get("sustained_TFLOPs"):
        fp8_sus, fp8_src = fp8["sustained_TFLOPs"], "measured e4m3 GEMM, sustained"
    else:
        fp8_sus = (pk.get("bf16_tflops_sustained") or pk["bf16_tflops"]) * FP8_OVER_BF16
        fp8_src = f"{pk['source']} cuBLAS bf16 sustained x nominal FP8:BF16 ratio 2"
    intensity = flops.get(dom, 0.0) / abytes[dom]
    ridge = fp8_sus * 1e12 / (pk["hbm_gbs"] * 1e9)
    if intensity > ridge:
        achieved = flops[dom] / (dom_ms * 1e-3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": round(fp8_sus, 1), "unit": "TFLOP/s",
                    "frac": round(achieved / fp8_sus, 4),
                    "traffic": kernel_traffic(dom, cfg.name), "algorithmic_flops": flops[dom],
                    "algorithmic_bytes": abytes[dom], "flop_per_byte": round(intensity, 1),
                    "peak_source": fp8_src}
    else:
        achieved = abytes[dom] / (dom_ms * 1e-3) / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1),
                    "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                    "traffic": kernel_traffic(dom, cfg.name), "algorithmic_bytes": abytes[dom],
                    "flop_per_byte": round(intensity, 1),
                    "peak_source": f"{pk['source']} HBM copy bandwidth"}
    fp8_gemm = {s: {"TFLOPs": kernels[s]["TFLOPs"],
                    "frac_of_fp8_peak": round(kernels[s]["TFLOPs"] / fp8_sus, 4)} for s in flops}
    fp8_gemm["peak_TFLOPs"] = round(fp8_sus, 1)
    fp8_gemm["peak_source"] = fp8_src

    e2e = run_e2e(layer, cfg, dev, max(3, min(args.steps, 50)), world)
    legs = args.workload == "v3_prefill" and not args.no_legs and not args.tokens
    decode = run_decode(layer, cfg, dev, pk) if legs else None
    backward = run_backward(layer, cfg, dev, pk) if legs else None
    wgrad = run_wgrad(layer, cfg, dev, pk) if legs else None
    skew = run_skew(layer, dev, pk, fp8_sus) if legs else None
    pipelined = run_pipelined(layer, cfg, dev) if legs else None
    balance = run_balance(layer, cfg, dev) if args.workload == "v3_long" else None

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded counter-based generator; random-init weights quantised 128x128)",
        "config": {**wl.describe(cfg), "inputs": "resident in HBM; weights 11.3 GB > L2, no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline, "fp8_gemm": fp8_gemm, "kernels": kernels,
        "gpu_launches": launches, "clocks": clk, "e2e": e2e,
    }
    if fp8:
        line["fp8_peak_measured"] = fp8
    if decode:
        line["decode"] = decode
    if balance:
        line["balance"] = balance
    if backward:
        line["backward_dgrad"] = backward
    if wgrad is not None:
        line["backward_wgrad"] = wgrad
    if skew:
        line["skew"] = skew
    if pipelined:
        line["pipelined"] = pipelined
    if legs:
        # the tensor-bound configuration: its own layer (weights of its seed), after
        # the prefill layer's memory is released
        del step, layer
        torch.cuda.empty_cache()
        line["long"] = run_long(dev, pk, fp8_sus, fp8_src)
    return line


def fp8_peak_probe(dev, n=8192, burst_reps=10, sustain_s=3.0):
    """Dense FP8 (e4m3) tensor rate of this GPU: an n^3 GEMM through cuBLASLt
    (torch._scaled_mm, bf16 output), best single call (burst) and back-to-back
    calls for a few seconds (sustained, under the power cap), with the SM
    clocks sampled meanwhile.  A measurement probe only: the layer never calls it."""
    try:
        g = torch.Generator(device=dev).manual_seed(7)
        a = (torch.randn((n, n), device=dev, generator=g) * 0.5).to(torch.float8_e4m3fn)
        b = (torch.randn((n, n), device=dev, generator=g) * 0.5).to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=dev)
        f = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        flop = 2.0 * n ** 3
        best = float("inf")
        for _ in range(burst_reps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            f()
            e.record()
            torch.cuda.synchronize()
            best = min(best, s.elapsed_time(e))
        clocks = ClockSampler(dev.index or 0)
        clocks.start()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(10, int(sustain_s / (best * 1e-3)))
        s.record()
        for _ in range(reps):
            f()
        e.record()
        torch.cuda.synchronize()
        clk = clocks.stop()
        ms = s.elapsed_time(e) / reps
        del a, b
        return {"burst_TFLOPs": round(flop / (best * 1e-3) / 1e12, 1),
                "sustained_TFLOPs": round(flop / (ms * 1e-3) / 1e12, 1),
                "shape": f"{n}x{n}x{n} e4m3 -> bf16", "sustained_calls": reps,
                "clocks_sustained": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
                "how": "torch._scaled_mm (cuBLASLt), unit scales; best of "
                       f"{burst_reps} (burst) and {reps} back-to-back calls (sustained)"}
    except Exception as exc:                    # the probe is context; never fail the bench on it
        return {"error": f"{type(exc).__name__}: {exc}"[:200]}


def run_skew(layer, dev, pk, fp8_sus, steps=50, warmup=5):
    """The V3 prefill batch with skewed expert popularity (16 hot experts with
    ~40% of the selections; the prefill weights, the skewed centroids): tokens/s
    and the per-kernel breakdown."""
    cfg = wl.V3_SKEW
    saved_c, saved_b = layer.centroids.clone(), layer.bias.clone()
    layer.centroids.copy_(wl.centroids(cfg, dev))
    layer.bias.copy_(wl.bias(cfg, dev))
    try:
        step = Step(layer, wl.tokens(cfg, dev), cfg.gamma)
        for _ in range(warmup):
            step.run()
        torch.cuda.synchronize()
        total_ms, per_stage = time_steps(step, steps)
        counts = step.rout["counts"].cpu()
        from fine_grained_fp8_bias_b300 import lib
        if lib.moe_check_device_status(step.status) != 0:
            raise RuntimeError("device status flagged in the skew leg")
    finally:
        layer.centroids.copy_(saved_c)
        layer.bias.copy_(saved_b)
    touched = int((counts > 0).sum()) + cfg.S
    kernels, abytes, _ = kernel_table(cfg, cfg.T, touched, per_stage, steps)
    hot = float(counts[:cfg.hot_experts].sum()) / (cfg.T * cfg.K)
    gu = kernels["gemm_gate_up"]
    return {"workload": cfg.name, "steps": steps, "ms_per_step": round(total_ms / steps, 4),
            "tokens_per_s": round(cfg.T * steps / (total_ms / 1e3), 1),
            "hot_fraction": round(hot, 3), "max_expert_rows": int(counts.max()),
            "gemm_gate_up_frac_of_hbm": round(gu["GBps"] / pk["hbm_gbs"], 4),
            "kernels": kernels}


def run_pipelined(layer, cfg, dev, n_batches=12, reserves=(0, 8, 16, 24, 32)):
    """Two micro-batches in flight (moe_forward_pipelined) against the same
    batches run one after another (moe_forward + moe_update_bias each): ms per
    batch for each number of SMs the GEMMs leave to the routing / dispatch /
    combine of the other batch.  CUDA events on the current stream, which waits
    for both of the pipeline's streams."""
    us = [wl.tokens(cfg, dev, step=k % 4) for k in range(n_batches)]
    outs = [dict(layer.outputs(cfg.T), u=u) for u in us]
    saved = layer.bias.clone()

    def timed(fn):
        fn()                                    # warm-up (workspaces, streams)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / n_batches

    def seq():
        for o in outs:
            layer.forward(o["u"], o)
            layer.update_bias(o["counts"], cfg.T, cfg.gamma)

    res = {"batches": n_batches, "sequential_ms_per_batch": round(timed(seq), 4)}
    for r in reserves:
        res[f"pipelined_reserve_{r}_ms_per_batch"] = round(
            timed(lambda: layer.forward_pipelined(us, cfg.gamma, r, outs)), 4)
    if layer.pipelined_status() != 0:
        raise RuntimeError("device status flagged in the pipelined leg")
    layer.bias.copy_(saved)
    best = min((v, k) for k, v in res.items() if k.startswith("pipelined"))
    res["best"] = best[1]
    res["speedup_vs_sequential"] = round(res["sequential_ms_per_batch"] / best[0], 4)
    return res


def run_long(dev, pk, fp8_sus, fp8_src, steps=10, warmup=3):
    """The tensor-bound configuration (T = 32768, V3 shapes, 4-component mixture
    tokens, its own weights): tokens/s of the whole step, each GEMM's TFLOP/s as
    a fraction of the measured FP8 peak, and the 100-step load-balancing run."""
    from fine_grained_fp8_bias_b300 import lib
    from fine_grained_fp8_bias_b300.layer import MoELayer
    cfg = wl.V3_LONG
    layer = MoELayer.from_config(cfg, dev)
    step = Step(layer, wl.tokens(cfg, dev), cfg.gamma)
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    total_ms, per_stage = time_steps(step, steps)
    clk = clocks.stop()
    if lib.moe_check_device_status(step.status) != 0:
        raise RuntimeError("device status flagged in the long leg")
    counts = step.rout["counts"].cpu()
    touched = int((counts > 0).sum()) + cfg.S
    kernels, _, flops = kernel_table(cfg, cfg.T, touched, per_stage, steps)
    out = {"workload": cfg.name, "T": cfg.T, "steps": steps,
           "ms_per_step": round(total_ms / steps, 4),
           "tokens_per_s": round(cfg.T * steps / (total_ms / 1e3), 1),
           "fp8_peak_TFLOPs": round(fp8_sus, 1), "fp8_peak_source": fp8_src,
           "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
           "kernels": kernels}
    for s in flops:
        out[s] = {"TFLOPs": kernels[s]["TFLOPs"],
                  "frac_of_fp8_peak": round(kernels[s]["TFLOPs"] / fp8_sus, 4)}
    del step
    out["balance"] = run_balance(layer, cfg, dev)
    del layer
    torch.cuda.empty_cache()
    return out


def run_e2e(layer, cfg, dev, steps, world):
    """Whole-job throughput through moe_forward_host with host buffers: every
    step uploads its batch from pinned memory, runs the layer and the bias
    update, and downloads h'; the uploads and downloads of neighbouring steps
    overlap the compute (three streams).  Wall clock from an idle device to
    the last download, max over ranks."""
    u_host = [wl.pinned_like(wl.tokens(cfg, "cpu", step=s)) for s in range(2)]
    h_host = [torch.empty((cfg.T, cfg.d), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    layer.forward_host(u_host, h_host, cfg.gamma)           # warm-up (streams, buffers)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    layer.forward_host([u_host[k % 2] for k in range(steps)], [h_host[k % 2] for k in range(steps)],
                       cfg.gamma)
    torch.cuda.synchronize()
    ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
    if layer.status() != 0:
        raise RuntimeError("device status flagged in the end-to-end loop")
    return {"value": round(job_tokens_per_s(world, cfg.T, steps, ms), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 4,
            "steps": steps, "ms_per_step": round(ms / steps, 4),
            "api": "moe_forward_host (pinned host batches; upload, compute and download "
                   "overlapped across steps)"}


def run_decode(layer, cfg, dev, pk, Ts=(1, 16, 64, 256), steps=50):
    """Decode-sized batches on the V3 weights with the skewed decode routing
    (centroids and bias of the decode workload: 16 hot experts take 40% of the
    selections at T = 256), each step a replay of a CUDA graph of moe_forward:
    forward time and the HBM rate of the weights each forward touches
    (distinct experts + shared)."""
    dcfg = wl.V3_DECODE
    saved_c, saved_b = layer.centroids.clone(), layer.bias.clone()
    layer.centroids.copy_(wl.centroids(dcfg, dev))
    layer.bias.copy_(wl.bias(dcfg, dev))
    res = []
    try:
        for T in Ts:
            u = wl.tokens(dcfg.with_(T=T), dev)
            # one decode step = one replay of the captured moe_forward
            graph, out = layer.capture_forward(u)
            for _ in range(5):
                graph.replay()
            torch.cuda.synchronize()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(steps):
                graph.replay()
            e.record()
            torch.cuda.synchronize()
            if layer.status() != 0:
                raise RuntimeError("device status flagged in the decode leg")
            us = s.elapsed_time(e) / steps * 1e3
            counts = out["counts"].cpu()
            touched = int((counts > 0).sum()) + cfg.S
            wbytes = touched * 3 * cfg.d * cfg.I * (1 + 4 / 128 ** 2)
            hot = float(counts[:dcfg.hot_experts].sum()) / (T * cfg.K)
            res.append({"T": T, "us_per_forward": round(us, 1), "experts_touched": touched,
                        "hot_fraction": round(hot, 3),
                        "weight_GBps": round(wbytes / (us * 1e-6) / 1e9, 1),
                        "frac_of_hbm": round(wbytes / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4)})
    finally:
        layer.centroids.copy_(saved_c)
        layer.bias.copy_(saved_b)
    return res


def run_backward(layer, cfg, dev, pk, steps=20):
    """Input gradient of the layer (moe_backward_dgrad) after a forward of the
    same batch: time of the backward alone (CUDA events), its GEMM FLOP rate
    (10 M d I: dH, the recomputed gate/up, dA) and the rate of the weight bytes
    it reads (W_down^T, W_gate, W_up, [W_gate^T | W_up^T] of the touched groups)."""
    u = wl.tokens(cfg, dev)
    dh = wl.normal(wl.stream_key(cfg.seed, 99), (cfg.T, cfg.d), 1.0, dev).to(torch.bfloat16)
    out = layer.forward(u)
    layer.prepare_backward()
    for _ in range(3):
        layer.backward_dgrad(u, dh, out)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        layer.backward_dgrad(u, dh, out)
    e.record()
    torch.cuda.synchronize()
    if layer.backward_status() != 0:
        raise RuntimeError("device status flagged in the backward leg")
    ms = s.elapsed_time(e) / steps
    M = cfg.T * (cfg.K + cfg.S)
    flops = 10.0 * M * cfg.d * cfg.I
    touched = int((out["counts"].cpu() > 0).sum()) + cfg.S
    wbytes = touched * 5 * cfg.d * cfg.I
    return {"ms": round(ms, 4), "TFLOPs": round(flops / (ms * 1e-3) / 1e12, 1),
            "weight_GBps": round(wbytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(wbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "what": "du from dh' (bf16) for the V3 batch: quantise dy, dH GEMM, gate/up recompute "
                    "+ SiLU backward + re-quantise, dA GEMM, gather, gate term"}


def run_wgrad(layer, cfg, dev, pk, steps=10):
    """Weight gradients of every expert (moe_backward_wgrad) for the batch of
    the backward leg: time of the call alone (CUDA events; four 128x1
    re-quantisations and two token-contracted GEMMs), the float32 gradient
    bytes it writes (3 d I per group) as a rate, and its GEMM FLOP rate
    (6 M d I over the dispatch rows)."""
    T = cfg.T
    dW = layer.backward_wgrad(T)
    for _ in range(2):
        layer.backward_wgrad(T, dW)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        layer.backward_wgrad(T, dW)
    e.record()
    torch.cuda.synchronize()
    if layer.backward_status() != 0:
        raise RuntimeError("device status flagged in the weight-gradient leg")
    ms = s.elapsed_time(e) / steps
    G = cfg.E + cfg.S
    out_bytes = G * 3 * cfg.d * cfg.I * 4
    M = T * (cfg.K + cfg.S)
    flops = 6.0 * M * cfg.d * cfg.I
    del dW
    torch.cuda.empty_cache()
    return {"ms": round(ms, 4), "out_GB": round(out_bytes / 1e9, 2),
            "out_GBps": round(out_bytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(out_bytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "TFLOPs": round(flops / (ms * 1e-3) / 1e12, 1),
            "what": "dW_gate, dW_up, dW_down (float32) of all 257 experts for the V3 batch: "
                    "A, h, dy, [dG | dU] re-quantised 128x1, then dy^T h and [dG | dU]^T A"}


def run_balance(layer, cfg, dev, steps=100):
    """Long-prefill leg: every step routes a fresh batch (generated on the device
    from the same stream of seeds), runs the layer and the bias update.  Reports
    the max over experts of c_e / (T K / E) per step and the layer's tokens/s
    over these steps (CUDA events around forward + bias update only)."""
    out = layer.outputs(cfg.T)
    ratios, ms = [], 0.0
    mean_load = cfg.T * cfg.K / cfg.E
    for step in range(steps):
        u = wl.tokens(cfg, dev, step)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        layer.forward(u, out)
        layer.update_bias(out["counts"], cfg.T, cfg.gamma)
        e.record()
        torch.cuda.synchronize()
        ms += s.elapsed_time(e)
        ratios.append(float(out["counts"].max().item()) / mean_load)
    if layer.status() != 0:
        raise RuntimeError("device status flagged in the balance leg")
    return {"steps": steps, "tokens_per_s": round(cfg.T * steps / (ms / 1e3), 1),
            "max_load_over_mean": {"first": round(ratios[0], 3), "last": round(ratios[-1], 3),
                                   "min": round(min(ratios), 3), "max": round(max(ratios), 3),
                                   "mean_last_10": round(statistics.mean(ratios[-10:]), 3)},
            "inputs": "fresh batch per step (4-component mixture), bias updated every step"}


# ------------------------------------------------------ CPU oracle arm
def oracle_setup(cfg, n_tok):
    from oracle import oracle as orc
    orc.build()
    u = wl.tokens(cfg, "cpu")[:n_tok]
    ub = u.view(torch.int16).numpy().view("uint16")
    cent = wl.centroids(cfg).numpy()
    b = wl.bias(cfg).numpy()
    r = orc.route(ub, cent, b, cfg.K)
    groups = set(range(cfg.E, cfg.E + cfg.S)) | {int(e) for e in r["idx"].ravel()}
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    W = orc.quantised_weights(cfg, sorted(groups),
                              lambda which, g: wl.master_weight(cfg, which, g, gen_dev).cpu().numpy())
    return orc, ub, cent, b, W


def oracle_step(orc, cfg, ub, cent, b, W, toks):
    r = orc.route(ub[toks], cent, b, cfg.K)
    orc.layer_forward(ub[toks], r["idx"], r["gate"], W, cfg.d, cfg.E, cfg.K, cfg.S, cfg.I,
                      list(range(len(toks))))
    orc.update_bias(r["counts"], b, len(toks), cfg.K, cfg.gamma)


def cpu_baseline(cfg, n_tok=2, reps=2):
    """The oracle as it stands, on the host cores: one thread, then one thread
    per core, each thread running the same sample (ctypes releases the GIL
    inside the C oracle, so the threads run in parallel)."""
    from concurrent.futures import ThreadPoolExecutor
    orc, ub, cent, b, W = oracle_setup(cfg, n_tok)
    toks = list(range(n_tok))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(orc, cfg, ub, cent, b.copy(), W, toks)
    one = reps * n_tok / (time.perf_counter() - t0)
    threads = max(1, min(os.cpu_count() or 1, 64))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        list(ex.map(lambda _: oracle_step(orc, cfg, ub, cent, b.copy(), W, toks), range(threads)))
        dt = time.perf_counter() - t0
    return {"value": round(threads * n_tok / dt, 3), "unit": "tokens/s", "cores": threads,
            "kind": "oracle", "single_core": round(one, 3),
            "sample": f"{n_tok} tokens of the {cfg.name} batch per thread ({threads} threads, one "
                      f"pass each; single core: {reps} passes): routing over all {cfg.E} experts, "
                      f"1x128 quantisation, {cfg.K} routed + {cfg.S} shared expert FFNs per token, "
                      f"combine, bias update"}


def run_reference(args):
    cfg = wl.CONFIGS[args.workload]
    n_tok = 2
    orc, ub, cent, b, W = oracle_setup(cfg, n_tok)
    for k in range(args.warmup):
        oracle_step(orc, cfg, ub, cent, b, W, [k % n_tok])
    t0 = time.perf_counter()
    for k in range(args.steps):
        oracle_step(orc, cfg, ub, cent, b, W, [k % n_tok])
    dt = time.perf_counter() - t0
    value = args.steps / dt
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 (E4M3 emulated)",
            "data": "synthetic", "config": wl.describe(cfg),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1,
                             "kind": "oracle",
                             "sample": f"each step one token of the {cfg.name} batch (cycling over "
                                       f"its first {n_tok}): routing, quantisation, {cfg.K}+{cfg.S} "
                                       f"expert FFNs, combine, bias update"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="v3_prefill", choices=sorted(wl.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-legs", action="store_true",
                    help="only the main workload (no decode, backward, skew, long legs)")
    ap.add_argument("--no-fp8-probe", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (profiling-size decode steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_ours(args, world, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl.CONFIGS[args.workload])
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
