"""One-kernel ("1-stage") bf16 decode path vs the oracle and vs the two-launch path.

Both stages run in one persistent launch (tiles of both stages claimed from
one counter, the intermediate kept in L2); the per-call option one_stage = 0
selects the two launches.  The tiles, MMAs and epilogues are
the same as in the two-launch kernels, so the outputs must be bit-identical
to them, and within 5e-3 of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_grouped_moe_gb300 import synth
from moe_checks import check_rows, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_moe_gb300 import build
    build.build()
    from mixture_experts_grouped_moe_gb300 import moe as m
    m.load()
    return m


def _run(moe, cfg, inp, one_stage, block_m=0, split_k=0):
    layer = moe.FusedMoE(moe.MOE_BF16, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, block_m, split_k,
                         options=moe.Options(one_stage=1 if one_stage else 0))
    assert layer.plan.mode == moe.MOE_MODE_SWAP
    w = {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": inp["W_gate_up"], "W_down": inp["W_down"]}
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    layer(inp["x"], w, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    return out


CASES = [
    # (name, T, H, I, E, k, bias, block_m, split_k)
    ("t1", 1, 128, 256, 4, 2, None, 0, 0),
    ("t3_e2", 3, 128, 256, 2, 2, None, 0, 0),
    ("t17_e5", 17, 256, 384, 5, 2, "normal", 0, 0),
    ("e1k1", 9, 128, 128, 1, 1, None, 0, 0),
    ("k_eq_e", 11, 128, 256, 3, 3, None, 0, 0),
    ("t128", 128, 256, 256, 4, 2, None, 0, 0),
    ("b32_sk2", 40, 256, 512, 4, 2, None, 32, 2),
    ("b128_sk1", 20, 256, 512, 4, 2, None, 128, 1),
    ("sk8", 8, 512, 1024, 8, 2, None, 0, 8),
    ("h_odd", 50, 640, 256, 8, 2, "normal", 0, 0),
    ("t128_e1k1", 128, 256, 256, 1, 1, None, 0, 0),   # one 128-row tile of real token rows
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_one_stage_edge_cases(moe, case):
    name, T, H, I, E, k, bias, bm, sk = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5)
    inp = synth.make_inputs(cfg, seed=3, device="cuda")
    one = _run(moe, cfg, inp, True, bm, sk)
    two = _run(moe, cfg, inp, False, bm, sk)
    assert torch.equal(one.view(torch.int16), two.view(torch.int16))
    host = {kk: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
            for kk, v in inp.items()}
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"], k)
    assert rel_l2(one.float().cpu().numpy(), ref) <= 5e-3


def test_one_stage_mixtral_decode(moe):
    cfg = synth.CONFIGS["mixtral_decode"]
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    one = _run(moe, cfg, inp, True)
    two = _run(moe, cfg, inp, False)
    assert torch.equal(one.view(torch.int16), two.view(torch.int16))
    again = _run(moe, cfg, inp, True)
    assert torch.equal(one.view(torch.int16), again.view(torch.int16))
    host = {kk: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
            for kk, v in inp.items()}
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"],
                                  cfg.k, expert_major=True)
    check_rows(one.float().cpu().numpy(), ref, 5e-3, label="mixtral decode, one kernel")


def test_one_stage_option_rejects_bad_value(moe):
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg, seed=3, device="cuda")
    layer = moe.FusedMoE(moe.MOE_BF16, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, options=moe.Options(one_stage=2))
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer(inp["x"], inp, out)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG


def test_two_layers_choose_independently(moe):
    """Two layer objects in one process keep their own launch choice (no process-wide switch)."""
    cfg = synth.CONFIGS["tiny"].with_(T=24)
    inp = synth.make_inputs(cfg, seed=4, device="cuda")
    a = _run(moe, cfg, inp, True)
    b = _run(moe, cfg, inp, False)
    c = _run(moe, cfg, inp, True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))
