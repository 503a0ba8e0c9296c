"""bench.py's output contract and host-side accounting (CPU only).

The reference arm (the CPU oracle timed on the host cores) prints the same
JSON line as the CUDA arm; its keys and types are checked here.  The helper
that counts the library's launches per forward and the rule that reports ncu
traffic only for unchanged kernel sources are checked on their own.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mixture_experts_grouped_moe_gb300 import synth  # noqa: E402


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC
    for key, typ in (("value", float), ("ms_per_step", float), ("n_gpus", int), ("steps", int), ("warmup", int)):
        assert isinstance(d[key], typ), key
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 1 and d["warmup"] >= 3
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("mixtral_decode")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_launches_per_step():
    # decode, one-kernel path: router, sort, both GEMM stages with the token-row fetch, combine
    assert bench.launches_per_step(synth.CONFIGS["mixtral_decode"], one_stage=True) == 4
    # two launches for the stages: + gather, stage 1, stage 2
    assert bench.launches_per_step(synth.CONFIGS["mixtral_decode"], one_stage=False) == 6
    # large T*E: logit pass + top-k pass; more than 1024 slots: three-launch sort
    assert bench.launches_per_step(synth.CONFIGS["finegrained_zipf"]) == 2 + 3 + 4
    # per-token FP8: + the row re-quantisation of h
    cfg = synth.CONFIGS["mixtral_fp8_token"]
    assert bench.launches_per_step(cfg) == 2 + 3 + 5


def test_traffic_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "mixture_experts_grouped_moe_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    (csrc / "h.cuh").write_text("header v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.kernel_source_hash(["k.cu", "h.cuh"])
    assert digest == bench.kernel_source_hash(["h.cuh", "k.cu"])  # order of the list does not matter
    (tmp_path / "profiles").mkdir()
    entry = {"w": {"stage1": {"dram_bytes_per_launch": 1234, "sources": ["k.cu", "h.cuh"], "source_hash": digest}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entry))
    assert bench.profiled_traffic("w", "stage1") == 1234
    assert bench.profiled_traffic("w", "one_kernel") is None
    assert bench.profiled_traffic("other", "stage1") is None
    (csrc / "h.cuh").write_text("header v2")  # any source change voids the recorded traffic
    assert bench.profiled_traffic("w", "stage1") is None


class _Plan:
    mode, block_m, split_k2 = 1, 16, 7


def test_summarize_reports_algorithmic_counts():
    """The dominant kernel's roofline uses the layer definition's algorithmic bytes (weights of the
    active experts and x once); implementation bytes (h round trip, split partials) are separate."""
    cfg = synth.CONFIGS["mixtral_decode"]
    stage_ms = {s: 0.01 for s in bench.STAGES}
    stage_ms["stage1"] = 0.42
    r = dict(ms=0.44, stage_ms=stage_ms, counts=[8] * 8, clocks=None, plan=_Plan, K=20, W=5, one_stage=True,
             l2="inputs larger than L2")
    peaks = {"hbm_gbs": 6700.0, "bf16_tflops": 1900.0}
    d = bench.summarize(cfg, r, peaks, "measured", 1)
    H, I, T = cfg.H, cfg.I, cfg.T
    alg = 8 * 3 * H * I * 2 + T * H * 2
    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["alg_bytes_per_launch"] == alg
    assert abs(roof["achieved"] - alg / 0.42e-3 / 1e9) < 0.1
    assert abs(roof["frac"] - roof["achieved"] / 6700.0) < 1e-4
    assert roof["impl_bytes_per_launch"] > alg
    assert d["layer_roofline"]["alg_bytes"] == alg + T * H * 2 + cfg.E * H * 2
    assert d["gpu_launches"] == 4 * 20 and d["value"] == round(T / 0.44e-3, 2)
    # a compute-bound workload reports tensor FLOPs of stage 1
    cfg2 = synth.CONFIGS["mixtral_prefill"]
    r2 = dict(r, one_stage=False, plan=type("P", (), {"mode": 0, "block_m": 128, "split_k2": 1}),
              counts=[2048] * 8, ms=3.5)
    d2 = bench.summarize(cfg2, r2, peaks, "measured", 1)
    assert d2["roofline"]["bound"] == "tensor"
    assert d2["roofline"]["alg_flops_per_launch"] == 2.0 * cfg2.S * 2 * cfg2.I * cfg2.H
    assert d2["roofline"]["peak"] == 1900.0 and d2["roofline"]["peak_source"] == "measured, burst"
    # a timed region of a second or more is measured against the sustained GEMM peak
    d3 = bench.summarize(cfg2, dict(r2, timed_ms=1750.0), dict(peaks, bf16_tflops_sustained=1700.0), "measured", 1)
    assert d3["roofline"]["peak"] == 1700.0 and d3["roofline"]["peak_source"] == "measured, sustained"
    assert abs(d3["roofline"]["frac"] - d2["roofline"]["frac"] * 1900.0 / 1700.0) < 1e-3
