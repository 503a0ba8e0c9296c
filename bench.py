"""Benchmark of the fused MoE layer on GB300 (one JSON line on stdout).

Headline workload: Mixtral-8x7B MoE decode (T=32 tokens, H=4096, I=14336,
E=8 experts, top-2, bf16 weights/activations, fp32 accumulation).  A step is
one whole forward of the layer (route, sort, gather, stage-1 and stage-2
group GEMMs, combine) through the C ABI on device-resident inputs.  The
default run also times, one after another, the tiny layer, Mixtral prefill
(T=8192 with uneven expert loads), the block-scaled FP8 layer (T=4096) and
the fine-grained skewed layer (T=4096, E=256, top-8), each with its own
clocks and rooflines under "per_config".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--no-per-config]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Under torchrun (N > 1) each rank runs an independent replica on its own GPU
(the layer is independent per token: weak scaling, no collective on the data
path); rank 0 prints the line with the max time over ranks.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-MoE TFLOP/s & HBM GB/s per shape on 1 GB300; % of roofline; tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ["route", "sort", "gather", "stage1", "stage2", "combine"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash(files):
    """Digest of the source files a profiled kernel is built from (names under the package's csrc/)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_grouped_moe_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's sources are unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d.get(workload, {}).get(kernel)
        if not ent or ent.get("source_hash") != kernel_source_hash(ent["sources"]):
            return None
        return ent["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        return None


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings over the process group (the slowest replica sets the time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_throughput(world, tokens_per_rank, ms_max):
    """Tokens per second over all replicas: every rank processes its own batch (weak scaling)."""
    return world * tokens_per_rank / (ms_max * 1e-3)


def algorithmic_counts(cfg, counts, dtype_bytes):
    """FLOPs and bytes of the layer from the actual routing (counts per expert), as the roofline
    definition states them: routed FLOPs 2*S*3*H*I + 2*T*H*E; bytes = weights (+ scales) of the
    experts that received a slot, x and out once (bf16), the router weights."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    S = T * k
    flops = 2.0 * S * 3 * H * I + 2.0 * T * H * E
    active = int(sum(1 for c in counts if c > 0))
    s1_scale = s2_scale = 0
    if cfg.dtype == "fp8":
        s1_scale = active * (2 * I // 128) * (H // 128) * 4
        s2_scale = active * (H // 128) * (I // 128) * 4
    elif cfg.dtype == "fp8_token":
        s1_scale, s2_scale = active * 2 * I * 4, active * H * 4
    elif cfg.dtype == "mxfp4":
        s1_scale, s2_scale = active * 2 * I * H // 32, active * H * I // 32
    s1_bytes = int(active * 2 * I * H * dtype_bytes) + s1_scale
    s2_bytes = int(active * H * I * dtype_bytes) + s2_scale
    bytes_ = s1_bytes + s2_bytes + T * H * 2 + T * H * 2 + E * H * 2
    return flops, bytes_, active, s1_bytes, s2_bytes


def make_weights(moe, cfg, inp, dev):
    """The layer's weights in the workload's format (quantised on the GPU by the library)."""
    import torch
    w = {"W_router": inp["W_router"], "bias": inp["bias"]}
    E, I, H = cfg.E, cfg.I, cfg.H
    if cfg.dtype == "fp8":
        q1 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
        s1 = torch.empty(E * 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
        q2 = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
        s2 = torch.empty(E * H // 128, I // 128, dtype=torch.float32, device=dev)
        moe.moe_quantize_fp8_weights(inp["W_gate_up"], E * 2 * I, H, q1, s1)
        moe.moe_quantize_fp8_weights(inp["W_down"], E * H, I, q2, s2)
        w.update(W_gate_up=q1, w1_scale=s1, W_down=q2, w2_scale=s2)
    elif cfg.dtype == "fp8_token":
        q1 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
        s1 = torch.empty(E * 2 * I, dtype=torch.float32, device=dev)
        q2 = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
        s2 = torch.empty(E * H, dtype=torch.float32, device=dev)
        moe.moe_quantize_fp8_rows(inp["W_gate_up"], E * 2 * I, H, q1, s1)
        moe.moe_quantize_fp8_rows(inp["W_down"], E * H, I, q2, s2)
        w.update(W_gate_up=q1, w1_scale=s1, W_down=q2, w2_scale=s2)
    elif cfg.dtype == "mxfp4":
        q1 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=dev)
        s1 = torch.empty(E * 2 * I * H // 32, dtype=torch.uint8, device=dev)
        q2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=dev)
        s2 = torch.empty(E * H * I // 32, dtype=torch.uint8, device=dev)
        moe.moe_quantize_mxfp4(inp["W_gate_up"], E * 2 * I, H, q1, s1, tiled=True)
        moe.moe_quantize_mxfp4(inp["W_down"], E * H, I, q2, s2, tiled=True)
        w.update(W_gate_up=q1, w1_scale=s1, W_down=q2, w2_scale=s2)
    else:
        w.update(W_gate_up=inp["W_gate_up"], W_down=inp["W_down"])
    return w


L2_BYTES = 129 * 2 ** 20


def layer_bytes_exceed_l2(cfg):
    eb = {"fp8": 1, "fp8_token": 1, "mxfp4": 0.5}.get(cfg.dtype, 2)
    return cfg.E * 3 * cfg.H * cfg.I * eb > 2 * L2_BYTES


def measure(args, cfg, rank, world, local_rank, e2e=False):
    """Time K whole-layer steps of one workload on this rank's GPU (after W warm-ups): the
    device-resident step, the per-stage split (a second pass with events between launches), and
    optionally the end-to-end step through the host-buffer entry."""
    import numpy as np
    import torch

    from mixture_experts_grouped_moe_gb300 import moe, synth

    dev = torch.device("cuda", local_rank)
    dtype = {"fp8": moe.MOE_FP8_BLOCK128, "fp8_token": moe.MOE_FP8_TOKEN, "mxfp4": moe.MOE_MXFP4}.get(
        cfg.dtype, moe.MOE_BF16)
    inp = synth.make_inputs(cfg, seed=0, device=dev)
    w = make_weights(moe, cfg, inp, dev)
    if cfg.dtype != "bf16":
        del inp["W_gate_up"], inp["W_down"]  # only the quantised stacks are used
    one_stage = cfg.dtype == "bf16" and cfg.T <= 128 and not args.two_launch
    opts = moe.Options(one_stage=1 if one_stage else 0)
    layer = moe.FusedMoE(dtype, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, host_staging=e2e, options=opts)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup
    # inputs smaller than L2 (the tiny workload): a buffer larger than L2 is written between steps
    flush = None if layer_bytes_exceed_l2(cfg) else torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(W):
        layer(inp["x"], w, out)
    torch.cuda.synchronize()
    if layer.status() != moe.MOE_OK:
        raise RuntimeError(f"{cfg.name}: device wait timed out during warm-up")
    # Small layers finish on the GPU before the host has prepared the next call: there the step
    # is one CUDA graph of the call (all of its kernels), replayed; large layers are called
    # directly (consecutive calls then overlap at the launch boundary).
    graph = layer.capture(inp["x"], w, out) if flush is not None else None

    def step():
        if graph is not None:
            graph.replay()
        else:
            layer(inp["x"], w, out)
    counts = layer.view("expert_counts", torch.int32, (cfg.E,)).cpu().numpy().tolist()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(K)]
    for row in ev:  # torch creates the CUDA event on first record; the handles must exist before use
        for e in row:
            e.record(stream)
    steps_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.15)
    if flush is None:
        # timed region: K whole-layer steps back to back, nothing between the library's launches
        start.record(stream)
        for _ in range(K):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        ms_total = start.elapsed_time(stop)
    else:
        for i in range(K):
            flush.fill_(float(i))
            steps_ev[i][0].record(stream)
            step()
            steps_ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms_total = sum(a.elapsed_time(b) for a, b in steps_ev)
    clocks = sampler.stop() if sampler else None
    # per-kernel timing: the same steps again with the library recording an event between its
    # launches (events between kernels stop the launch overlap, so this pass does not set `value`)
    for i in range(K):
        if flush is not None:
            flush.fill_(float(i))
        layer(inp["x"], w, out, options=moe.Options(one_stage=opts.one_stage, stage_events=ev[i]))
    torch.cuda.synchronize()
    stage_ms = {st: 0.0 for st in STAGES}
    for i in range(K):
        for j, st in enumerate(STAGES):
            stage_ms[st] += ev[i][j].elapsed_time(ev[i][j + 1])
    stage_ms = {st: v / K for st, v in stage_ms.items()}

    e2e_ms = None
    if e2e:
        # end to end: host (pinned) x in, host out back, through the C-ABI host entry
        x_host = inp["x"].cpu().pin_memory()
        out_host = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory()
        for _ in range(max(3, W // 4)):
            layer.forward_host(x_host, w, out_host)
        torch.cuda.synchronize()
        K2 = max(1, K // 2)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K2):
            layer.forward_host(x_host, w, out_host)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / K2
        assert np.isfinite(out_host.float().numpy()).all()
    assert torch.isfinite(out.float()).all()

    ms = ms_total / K
    if world > 1:
        ms, e2e_max = max_over_ranks([ms, e2e_ms or 0.0], dev)
        e2e_ms = e2e_max if e2e else None
    plan = layer.plan
    r = dict(ms=ms, e2e_ms=e2e_ms, stage_ms=stage_ms, counts=counts, clocks=clocks, plan=plan, K=K, W=W,
             one_stage=one_stage, l2="L2 flushed between steps (256 MiB written)" if flush is not None
             else "inputs larger than L2 (expert weights streamed every step)",
             launch="one CUDA graph of the layer call per step" if graph is not None
             else "direct library calls", timed_ms=ms_total)
    del layer, w, inp, out, flush, graph
    torch.cuda.empty_cache()
    return r


def summarize(cfg, r, peaks, peak_kind, world):
    """Throughput, the layer roofline and the dominant kernel's roofline of one measured workload."""
    eb = {"fp8": 1, "fp8_token": 1, "mxfp4": 0.5}.get(cfg.dtype, 2)
    flops, bytes_, active, s1_bytes, s2_bytes = algorithmic_counts(cfg, r["counts"], eb)
    ms = r["ms"]
    # a timed region of a second or more runs under the power cap: the sustained GEMM peak applies
    sustained = r.get("timed_ms", 0.0) >= 1000.0
    peak_t = (peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]) if sustained
              else peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tensor_kind = f"{peak_kind}, {'sustained' if sustained else 'burst'}"
    if eb == 1:
        peak_t = peaks.get("fp8_tflops", 2.0 * peak_t)  # nominal dense FP8 / bf16 ratio
    elif eb == 0.5:
        peak_t = peaks.get("fp4_tflops", 6.0 * peak_t)  # nominal dense FP4 / bf16 ratio on GB300 (13.5 / 2.25)
    hbm = peaks["hbm_gbs"]
    t_roof = max(flops / (peak_t * 1e12), bytes_ / (hbm * 1e9))
    T, H, I, S = cfg.T, cfg.H, cfg.I, cfg.S
    plan = r["plan"]
    npp_rows = sum(-(-c // plan.block_m) * plan.block_m for c in r["counts"])
    h_bytes = {"fp8": 1, "mxfp4": 0.5}.get(cfg.dtype, 2)
    x_bytes = T * H * 2
    if r["one_stage"]:
        # one launch runs both stages and reads x itself
        kname, kms = "one-kernel stage 1 + stage 2 (swap-AB)", r["stage_ms"]["stage1"]
        k_flops = 2.0 * S * 3 * H * I
        k_bytes = s1_bytes + s2_bytes + x_bytes
        impl = int(k_bytes + 2 * npp_rows * I * 2 + plan.split_k2 * npp_rows * H * 4)  # h out and back, partials
    else:
        kname, kms = "stage 1 gate/up group GEMM" + (" (swap-AB)" if plan.mode == 1 else ""), r["stage_ms"]["stage1"]
        k_flops = 2.0 * S * 2 * I * H
        k_bytes = s1_bytes + x_bytes
        impl = int(s1_bytes + npp_rows * H * eb + npp_rows * I * h_bytes)  # gathered x rows in, h out
    mem_bound = k_bytes / (hbm * 1e9) >= k_flops / (peak_t * 1e12)
    if mem_bound:
        achieved = k_bytes / (kms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "alg_bytes_per_launch": int(k_bytes)}
    else:
        achieved = k_flops / (kms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak_t, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak_t, 4), "alg_flops_per_launch": k_flops}
    roof.update(kernel=kname, impl_bytes_per_launch=impl, peak_source=peak_kind if mem_bound else tensor_kind,
                kernel_ms=round(kms, 5),
                traffic=profiled_traffic(cfg.name, "one_kernel" if r["one_stage"] else "stage1"))
    return {
        "value": round(whole_job_throughput(world, T, ms), 2), "unit": "tokens/s", "ms_per_step": round(ms, 5),
        "steps": r["K"], "warmup": r["W"],
        "tflops": round(flops / (ms * 1e-3) / 1e12, 2), "hbm_gbs": round(bytes_ / (ms * 1e-3) / 1e9, 1),
        "layer_roofline": {"t_roof_ms": round(t_roof * 1e3, 4), "frac": round(t_roof / (ms * 1e-3), 4),
                           "bound": "hbm" if bytes_ / (hbm * 1e9) >= flops / (peak_t * 1e12) else "tensor",
                           "alg_bytes": bytes_, "alg_flops": flops, "active_experts": active},
        "stage_ms": {k2: round(v, 5) for k2, v in r["stage_ms"].items()},
        "roofline": roof,
        "gpu_launches": launches_per_step(cfg, r["one_stage"]) * r["K"],
        "clocks": r["clocks"],
        "plan": {"mode": "swap" if plan.mode == 1 else "grouped", "block_m": plan.block_m,
                 "split_k2": plan.split_k2},
        "l2": r["l2"],
        "launch": r.get("launch", "direct library calls"),
    }


def cpu_baseline(cfg, host, budget_s=20.0):
    """The oracle as it stands on this host's cores, on a bounded token sample."""
    import numpy as np

    import oracle
    from mixture_experts_grouped_moe_gb300 import synth

    n = max(1, min(cfg.T, oracle.default_threads()))
    toks = synth.token_sample(cfg.T, n).numpy()
    t0 = time.perf_counter()
    run_oracle(cfg, host, toks)
    first = time.perf_counter() - t0
    reps = 1 + max(0, min(9, int(budget_s / max(first, 1e-6)) - 1))
    for _ in range(reps - 1):
        run_oracle(cfg, host, toks)
    dt = (time.perf_counter() - t0) / reps
    return {"value": n / dt, "unit": "tokens/s", "cores": oracle.default_threads(), "kind": "oracle",
            "sample": f"{n} of the {cfg.T} tokens, full layer per token (fp64 CPU oracle), {reps} run(s)"}


def run_oracle(cfg, host, toks):
    import oracle
    if cfg.dtype == "fp8":
        return oracle.moe_forward_fp8(host["x"], host["W_router"], host["bias"], host["q1"], host["s1"],
                                      host["q2"], host["s2"], cfg.k, toks)
    if cfg.dtype == "mxfp4":
        return oracle.moe_forward_mxfp4(host["x"], host["W_router"], host["bias"], host["q1"], host["s1"],
                                        host["q2"], host["s2"], cfg.k, toks)
    if cfg.dtype == "fp8_token":
        return oracle.moe_forward_fp8_token(host["x"], host["W_router"], host["bias"], host["q1"], host["s1"],
                                            host["q2"], host["s2"], cfg.k, toks)
    return oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"],
                                   cfg.k, toks)


def host_inputs(cfg, device):
    import torch

    import oracle
    from mixture_experts_grouped_moe_gb300 import synth
    inp = synth.make_inputs(cfg, seed=0, device=device)
    host = {k: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
            for k, v in inp.items()}
    if cfg.dtype == "fp8":
        host["q1"], host["s1"] = oracle.quant_128x128(host["W_gate_up"])
        host["q2"], host["s2"] = oracle.quant_128x128(host["W_down"])
    elif cfg.dtype == "fp8_token":
        host["q1"], host["s1"] = oracle.quant_rows(host["W_gate_up"])
        host["q2"], host["s2"] = oracle.quant_rows(host["W_down"])
    elif cfg.dtype == "mxfp4":
        host["q1"], host["s1"] = oracle.quant_mx4(host["W_gate_up"])
        host["q2"], host["s2"] = oracle.quant_mx4(host["W_down"])
    return host


def launches_per_step(cfg, one_stage=False):
    """Kernels the library launches per forward: router (+ top-k pass for large T*E), sort
    (one launch up to 1024 slots, else three), gather, stage 1 (+ the per-token re-quantisation
    of h), stage 2, combine; the one-kernel decode path replaces gather, stage 1 and stage 2 by
    one launch that fetches the token rows itself."""
    router = 2 if cfg.T * cfg.E > 4096 else 1
    sort = 1 if cfg.T * cfg.k <= 1024 else 3
    if one_stage:
        return router + sort + 2
    return router + sort + 4 + (1 if cfg.dtype == "fp8_token" else 0)


def workload_desc(cfg):
    d = {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} top-{cfg.k} SwiGLU"
                     + {"fp8": " block-scaled FP8 e4m3", "fp8_token": " per-token FP8 e4m3",
                        "mxfp4": " MXFP4 (E2M1, E8M0 per 1x32)"}.get(cfg.dtype, " bf16")
                     + ("" if cfg.bias is None else f" router bias {cfg.bias}({cfg.bias_param})"),
         "tokens_per_step": cfg.T, "seq_len": 1 if cfg.T <= 128 else cfg.T}
    return d


# The workloads timed beside the headline in the default run (one after another on the same GPU,
# each allocated, timed and freed in turn): the small case, Mixtral prefill with uneven loads, the
# block-scaled FP8 layer and the fine-grained skewed layer.
PER_CONFIG = ["tiny", "mixtral_prefill", "mixtral_fp8", "finegrained_zipf"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--workload", default=None,
                    help="time only this workload (default: Mixtral decode as the headline, plus the other "
                         "workloads under per_config)")
    ap.add_argument("--no-per-config", action="store_true", help="the headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--train", action="store_true",
                    help="bf16 training step: training forward + backward (dx and all weight gradients)")
    ap.add_argument("--two-launch", action="store_true",
                    help="bf16 decode: stage 1 and stage 2 as two launches instead of the one-kernel path")
    ap.add_argument("--experts", type=int, default=0, help="profiling aid: override E (not a bench line)")
    ap.add_argument("--tokens", type=int, default=0, help="profiling aid: override T (not a bench line)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from mixture_experts_grouped_moe_gb300 import synth
    explicit = args.workload is not None
    cfg = synth.CONFIGS[args.workload or "mixtral_decode"]
    if args.experts:
        cfg = cfg.with_(name=cfg.name + f"_E{args.experts}", E=args.experts)
    if args.tokens:
        cfg = cfg.with_(name=cfg.name + f"_T{args.tokens}", T=args.tokens)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, cfg)

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    from mixture_experts_grouped_moe_gb300 import build as moe_build
    from mixture_experts_grouped_moe_gb300 import moe
    moe_build.build()
    moe.load()
    torch.cuda.set_device(local_rank)
    if args.train:
        return run_train(args, cfg, rank, world, local_rank)
    peaks, peak_kind = load_peaks()
    r = measure(args, cfg, rank, world, local_rank, e2e=True)
    others = []
    if not explicit and not args.no_per_config:
        for name in PER_CONFIG:
            c = synth.CONFIGS[name]
            others.append((c, measure(args, c, rank, world, local_rank)))
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    head = summarize(cfg, r, peaks, peak_kind, world)
    eb = {"fp8": 1, "fp8_token": 1, "mxfp4": 0.5}.get(cfg.dtype, 2)
    T, H = cfg.T, cfg.H
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": r["K"], "warmup": r["W"], "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {1: "fp8-e4m3/fp32-acc", 0.5: "mxfp4-e2m1/fp32-acc"}.get(eb, "bf16"),
        "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights; random init, no checkpoint)",
        "config": dict(workload_desc(cfg), parallelism=f"replicas x{world}",
                       **({"one_stage": True} if r["one_stage"] else {}), l2=head["l2"]),
        "tflops": head["tflops"], "hbm_gbs": head["hbm_gbs"],
        "layer_roofline": head["layer_roofline"],
        "stage_ms": head["stage_ms"],
        "roofline": head["roofline"],
        "gpu_launches": head["gpu_launches"],
        "stage_ms_note": "per-kernel CUDA-event times from a second pass of the same steps with an event "
                         "between launches; value is timed without them",
        "clocks": head["clocks"],
        "e2e": {"value": round(whole_job_throughput(world, T, r["e2e_ms"]), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
                "ms_per_step": round(r["e2e_ms"], 5)},
        "plan": head["plan"],
    }
    if others:
        line["per_config"] = {}
        for c, rc in others:
            ent = summarize(c, rc, peaks, peak_kind, world)
            ent["workload"] = workload_desc(c)["workload"]
            line["per_config"][c.name] = ent
    if not args.no_cpu_baseline:
        host = host_inputs(cfg, torch.device("cuda", local_rank))
        line["cpu_baseline"] = cpu_baseline(cfg, host)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_train(args, cfg, rank, world, local_rank):
    """One training step = moe_fused_forward_train + moe_fused_backward on device-resident inputs."""
    import torch

    from mixture_experts_grouped_moe_gb300 import build as moe_build
    from mixture_experts_grouped_moe_gb300 import moe, synth

    if cfg.dtype != "bf16":
        raise SystemExit("--train runs the bf16 layer")
    moe_build.build()
    moe.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_kind = load_peaks()
    inp = synth.make_inputs(cfg, seed=0, device=dev)
    w = {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": inp["W_gate_up"], "W_down": inp["W_down"]}
    dout = torch.randn(cfg.T, cfg.H, generator=torch.Generator(device=dev).manual_seed(1), device=dev).to(
        torch.bfloat16)
    tr = moe.MoETrain(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, device=dev)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    K, W = args.steps, args.warmup
    for _ in range(W):
        tr.forward(inp["x"], w, out)
        g = tr.backward(inp["x"], w, dout)
    torch.cuda.synchronize()
    if tr.status() != moe.MOE_OK:
        raise RuntimeError("device wait timed out during warm-up")
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    fw = bw = 0.0
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.15)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(K):
        tr.forward(inp["x"], w, out)
        g = tr.backward(inp["x"], w, dout)
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = start.elapsed_time(stop) / K
    for _ in range(K):  # split of the step (events between the two calls)
        ev[0].record(stream)
        tr.forward(inp["x"], w, out)
        ev[1].record(stream)
        g = tr.backward(inp["x"], w, dout)
        ev[2].record(stream)
        torch.cuda.synchronize()
        fw += ev[0].elapsed_time(ev[1])
        bw += ev[1].elapsed_time(ev[2])
    fw, bw = fw / K, bw / K
    assert all(torch.isfinite(v.float()).all() for v in g.values())
    if world > 1:
        ms, = max_over_ranks([ms], dev)
    if rank != 0:
        return 0
    S, H, I = cfg.S, cfg.H, cfg.I
    fwd_flops = 2.0 * S * 3 * H * I
    flops = 3 * fwd_flops  # forward, input gradient, weight gradients
    peak_t = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    bwd_tflops = 2 * fwd_flops / (bw * 1e-3) / 1e12
    line = {
        "metric": METRIC + " (training step)", "value": round(whole_job_throughput(world, cfg.T, ms), 2),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations and output gradient, N(0,1/fan_in) weights)",
        "config": dict(workload_desc(cfg), parallelism=f"replicas x{world}", step="forward + backward"),
        "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "stage_ms": {"forward_train": round(fw, 5), "backward": round(bw, 5)},
        "roofline": {"bound": "tensor", "achieved": round(bwd_tflops, 1), "peak": peak_t, "unit": "TFLOP/s",
                     "frac": round(bwd_tflops / peak_t, 4), "kernel": "backward (its GEMMs, transposes and aux)",
                     "alg_flops_per_launch": 2 * fwd_flops, "peak_source": peak_kind, "traffic": None},
        "clocks": clocks,
        "e2e": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, cfg):
    """The CPU oracle as the reference arm: each step runs the layer on a bounded token sample."""
    import torch

    import oracle
    from mixture_experts_grouped_moe_gb300 import synth
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    host = host_inputs(cfg, dev)
    nthr = oracle.default_threads()
    n = max(1, min(cfg.T, nthr))
    toks = synth.token_sample(cfg.T, n).numpy()
    t0 = time.perf_counter()
    run_oracle(cfg, host, toks)
    t_step = time.perf_counter() - t0
    budget = 150.0
    if (args.steps + args.warmup) * t_step > budget:
        n = 1  # smallest sample: one token per step
        toks = toks[:1]
    for _ in range(args.warmup):
        run_oracle(cfg, host, toks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle(cfg, host, toks)
    dt = (time.perf_counter() - t0) / args.steps
    value = n / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
            "data": "synthetic", "config": dict(workload_desc(cfg), parallelism="host cores"),
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": nthr, "kind": "oracle",
                             "sample": f"{n} token(s) of the {cfg.T}-token batch per step"},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
