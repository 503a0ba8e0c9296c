"""A layer call captured in a CUDA graph (FusedMoE.capture): the library allocates nothing and
never synchronises, so the whole call -- router, sort, gather, both GEMM stages, combine --
replays from one graph launch.  The replay must give exactly the direct call's bytes, and it
must read its inputs at replay time (new x in the same buffer, new result)."""
import pytest
import torch

from mixture_experts_grouped_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_moe_gb300 import build
    build.build()
    from mixture_experts_grouped_moe_gb300 import moe as m
    m.load()
    return m


def _weights(moe, cfg, inp):
    if cfg.dtype != "fp8":
        return {k: inp[k] for k in ("W_router", "bias", "W_gate_up", "W_down")}
    E, I, H = cfg.E, cfg.I, cfg.H
    q1 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device="cuda")
    s1 = torch.empty(E * 2 * I // 128, H // 128, dtype=torch.float32, device="cuda")
    q2 = torch.empty(E, H, I, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(E * H // 128, I // 128, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_weights(inp["W_gate_up"], E * 2 * I, H, q1, s1)
    moe.moe_quantize_fp8_weights(inp["W_down"], E * H, I, q2, s2)
    return {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": q1, "w1_scale": s1, "W_down": q2,
            "w2_scale": s2}


CASES = [
    synth.CONFIGS["tiny"],                                                               # one-launch decode
    synth.MoEConfig("grouped", T=700, H=256, I=512, E=16, k=2, bias="normal", bias_param=0.5),  # CTA pairs
    synth.MoEConfig("fp8_grouped", T=600, H=256, I=384, E=8, k=2, dtype="fp8"),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_graph_replay_matches_direct_call(moe, cfg):
    dtype = moe.MOE_FP8_BLOCK128 if cfg.dtype == "fp8" else moe.MOE_BF16
    inp = synth.make_inputs(cfg, seed=5, device="cuda")
    w = _weights(moe, cfg, inp)
    layer = moe.FusedMoE(dtype, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    x = inp["x"].clone()
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    graph = layer.capture(x, w, out)
    ref = torch.empty_like(out)
    for seed in (5, 6):
        x.copy_(synth.make_inputs(cfg, seed=seed, device="cuda")["x"])
        layer(x, w, ref)
        out.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        assert layer.status() == moe.MOE_OK
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), seed
