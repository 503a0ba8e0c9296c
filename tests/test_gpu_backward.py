"""Backward of the bf16 layer (grouped dgrad / wgrad, router) through the C ABI vs the CPU oracle.

Tolerance, derived: the GPU path rounds three intermediates to bf16 (the
weighted output gradient dY, the saved pre-activations g | u, and dg | du),
each a relative 2^-9 step, and accumulates in fp32; a relative L2 error of
1e-2 per gradient leaves margin above that.  Gradients are also bitwise
reproducible run to run, and experts without tokens get exact zeros.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_grouped_moe_gb300 import synth
from moe_checks import rel_l2

pytestmark = pytest.mark.gpu

TOL_GRAD = 1e-2


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_moe_gb300 import build
    build.build()
    from mixture_experts_grouped_moe_gb300 import moe as m
    m.load()
    return m


def _run(moe, cfg, inp, dout, options=None):
    tr = moe.MoETrain(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, options=options)
    w = {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": inp["W_gate_up"], "W_down": inp["W_down"]}
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    tr.forward(inp["x"], w, out)
    g = tr.backward(inp["x"], w, dout)
    torch.cuda.synchronize()
    assert tr.status() == moe.MOE_OK
    return out, g


CASES = [
    # (name, T, H, I, E, k, bias)
    ("t40_e4", 40, 256, 256, 4, 2, None),
    ("t300_ragged", 300, 384, 512, 6, 3, "normal"),
    ("e1k1", 150, 256, 256, 1, 1, None),
    ("empty_experts", 20, 256, 256, 16, 2, None),
    ("h_odd", 200, 640, 256, 8, 2, "normal"),
    ("medium", 1024, 1024, 1024, 8, 2, "normal"),   # long K loops; about 128 tokens per expert segment
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_backward_parity(moe, case, options=None):
    name, T, H, I, E, k, bias = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5)
    inp = synth.make_inputs(cfg, seed=17, device="cuda")
    dout = torch.randn(T, H, generator=torch.Generator(device="cuda").manual_seed(18), device="cuda").to(
        torch.bfloat16)
    out, g = _run(moe, cfg, inp, dout, options)
    host = {kk: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
            for kk, v in inp.items()}
    ref_out = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"], k)
    assert rel_l2(out.float().cpu().numpy(), ref_out) <= 5e-3
    ref = oracle.moe_backward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"],
                                   synth.bf16_bits(dout), k)
    for key in ("dx", "dW_gate_up", "dW_down", "dW_router", "dbias"):
        got = g[key].float().cpu().numpy()
        r = ref[key]
        if not np.abs(r).max() > 0:
            assert not got.any(), key
            continue
        err = rel_l2(got, r)
        print(f"{name} {key}: relL2 {err:.3e}")
        assert err <= TOL_GRAD, (key, err)
    ids, _, _ = oracle.route(host["x"], host["W_router"], host["bias"], k)
    for e in set(range(E)) - set(ids.ravel().tolist()):
        assert not g["dW_gate_up"][e].any() and not g["dW_down"][e].any()


def test_backward_reproducible(moe):
    cfg = synth.MoEConfig("rep", T=130, H=256, I=256, E=4, k=2)
    inp = synth.make_inputs(cfg, seed=19, device="cuda")
    dout = torch.randn(cfg.T, cfg.H, generator=torch.Generator(device="cuda").manual_seed(20), device="cuda").to(
        torch.bfloat16)
    _, a = _run(moe, cfg, inp, dout)
    _, b = _run(moe, cfg, inp, dout)
    for key in a:
        assert torch.equal(a[key].view(torch.int16) if a[key].dtype == torch.bfloat16 else a[key],
                           b[key].view(torch.int16) if b[key].dtype == torch.bfloat16 else b[key]), key


def test_train_workspace_rejects_unsupported(moe):
    assert moe.moe_train_workspace_size(16, 256, 384, 4, 2) == 0   # I not a multiple of 256
    assert moe.moe_train_workspace_size(16, 256, 256, 4, 2) > 0


@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[4]], ids=lambda c: c[0] + "_pairs")
def test_backward_parity_cta_pairs(moe, case):
    """The same gradients with the CTA-pair GEMMs forced (training forward, both backward GEMMs, and
    the weight gradients whose row count is a multiple of 256)."""
    test_backward_parity(moe, case, options=moe.Options(gemm_pair=1))
