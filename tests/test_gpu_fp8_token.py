"""Per-token FP8 ("per_Token" quantisation on the AITER page) through the C ABI vs the CPU oracle.

Codes and scales of the per-row quantiser are compared bit for bit, both
standalone and inside the fused call (the gathered activations, and the
intermediate re-quantised from the call's own bf16 SwiGLU output).  The
layer output must meet relative L2 error <= 3e-2 against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_grouped_moe_gb300 import synth
from moe_checks import E4M3_LEADERS, check_rows, every_bf16_below, parity_tokens, rel_l2

pytestmark = pytest.mark.gpu

TOL_FP8 = 3e-2


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_moe_gb300 import build
    build.build()
    from mixture_experts_grouped_moe_gb300 import moe as m
    m.load()
    return m


def _host(inp):
    return {k: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
            for k, v in inp.items()}


def quantize_rows_gpu(moe, inp, cfg):
    E, I, H = cfg.E, cfg.I, cfg.H
    q1 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device="cuda")
    s1 = torch.empty(E * 2 * I, dtype=torch.float32, device="cuda")
    q2 = torch.empty(E, H, I, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(E * H, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(inp["W_gate_up"], E * 2 * I, H, q1, s1)
    moe.moe_quantize_fp8_rows(inp["W_down"], E * H, I, q2, s2)
    return {"W_gate_up": q1, "w1_scale": s1, "W_down": q2, "w2_scale": s2}


def run_fused(moe, cfg, inp, w8, block_m=0, split_k=0):
    layer = moe.FusedMoE(moe.MOE_FP8_TOKEN, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, block_m, split_k)
    w = dict(w8, W_router=inp["W_router"], bias=inp["bias"])
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    layer(inp["x"], w, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    return out, layer


@pytest.mark.parametrize("R,C", [(300, 1024), (37, 20480), (5, 16)], ids=["regs", "two_pass", "narrow"])
def test_quant_rows_bit_exact(moe, R, C):
    g = torch.Generator(device="cuda").manual_seed(12)
    X = (torch.randn(R, C, generator=g, device="cuda") *
         torch.exp(torch.randn(R, 1, generator=g, device="cuda") * 3)).to(torch.bfloat16)
    X[1] = 0
    q = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    s = torch.empty(R, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(X, R, C, q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_rows(synth.bf16_bits(X))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quant_rows_every_bf16_value(moe):
    # every bf16 value within 21 binades below a row's largest, for eight row scales (one whose
    # reciprocal is not a normal float): each code must be e4m3 of the IEEE quotient v / scale
    X = every_bf16_below(E4M3_LEADERS, 5504, 5504).cuda()
    R, C = X.shape
    q = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    s = torch.empty(R, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(X, R, C, q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_rows(synth.bf16_bits(X))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quant_rows_rejects_bad_shapes(moe):
    X = torch.zeros(4, 24, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(4, 24, dtype=torch.uint8, device="cuda")
    s = torch.empty(4, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError):
        moe.moe_quantize_fp8_rows(X, 4, 24, q, s)  # C not a multiple of 16


def _check_codes_in_workspace(moe, layer, cfg, host):
    """The gathered x codes / scales and the re-quantised intermediate are bit-exact
    re-quantisations of their own inputs (the bf16 x rows, the call's bf16 h)."""
    T, k, E = cfg.T, cfg.k, cfg.E
    r_ids, _, _ = oracle.route(host["x"], host["W_router"], host["bias"], k)
    assert np.array_equal(layer.view("topk_ids", torch.int32, (T, k)).cpu().numpy(), r_ids)
    P = layer.plan.max_padded
    npp = int(layer.view("num_tokens_post_padded", torch.int32, (1,)).item())
    s_ids = layer.view("sorted_ids", torch.int32, (P,)).cpu().numpy()[:npp]
    o_ids, _, o_npp, _ = oracle.align_sort(r_ids, E, layer.plan.block_m)
    assert npp == o_npp and np.array_equal(s_ids, o_ids[:npp])
    S = T * k
    xrows = np.where((s_ids < S)[:, None], host["x"][np.minimum(s_ids, S - 1) // k], np.uint16(0))
    rq, rs = oracle.quant_rows(xrows)
    xq = layer.view("x_sorted", torch.uint8, (P, cfg.H)).cpu().numpy()[:npp]
    xs = layer.view("x_scales", torch.float32, (P,)).cpu().numpy()[:npp]
    assert np.array_equal(xq, rq) and np.array_equal(xs.view(np.uint32), rs.view(np.uint32))
    h = layer.view("inter_h", torch.int16, (P, cfg.I)).cpu().numpy()[:npp].view(np.uint16)
    hq, hs = oracle.quant_rows(h)
    gq = layer.view("inter", torch.uint8, (P, cfg.I)).cpu().numpy()[:npp]
    gs = layer.view("inter_scales", torch.float32, (P,)).cpu().numpy()[:npp]
    assert np.array_equal(gq, hq) and np.array_equal(gs.view(np.uint32), hs.view(np.uint32))
    return r_ids


@pytest.mark.parametrize("name", ["mixtral_fp8_token_decode", "mixtral_fp8_token"])
def test_fused_fp8_token_parity(moe, name):
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    host = _host(inp)
    w8 = quantize_rows_gpu(moe, inp, cfg)
    out, layer = run_fused(moe, cfg, inp, w8)
    assert layer.plan.mode == (moe.MOE_MODE_SWAP if cfg.T <= 128 else moe.MOE_MODE_GROUPED)
    r_ids = _check_codes_in_workspace(moe, layer, cfg, host)
    q1, s1 = oracle.quant_rows(host["W_gate_up"])
    q2, s2 = oracle.quant_rows(host["W_down"])
    assert np.array_equal(w8["w1_scale"].cpu().numpy().view(np.uint32), s1.view(np.uint32))
    assert np.array_equal(w8["W_down"].cpu().numpy(), q2) and np.array_equal(w8["W_gate_up"].cpu().numpy(), q1)
    toks = np.arange(cfg.T) if cfg.T <= 128 else parity_tokens(r_ids, cfg.E, layer.plan.block_m)
    ref = oracle.moe_forward_fp8_token(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, cfg.k, toks,
                                       expert_major=True)
    check_rows(out.float().cpu().numpy()[toks], ref, TOL_FP8, label=name)


EDGE = [
    # (name, T, H, I, E, k, bias, block_m, split_k)
    ("t1", 1, 128, 256, 4, 2, None, 0, 0),
    ("e1k1", 9, 128, 128, 1, 1, None, 0, 0),
    ("swap_b32_sk2", 40, 256, 512, 4, 2, None, 32, 2),
    ("swap_sk4", 8, 512, 512, 8, 2, None, 0, 4),
    ("swap_t128", 128, 256, 256, 4, 2, "normal", 0, 0),
    ("grouped_t129", 129, 256, 256, 4, 2, None, 0, 0),
    ("grouped_ragged", 257, 384, 256, 6, 3, "normal", 0, 0),
    ("grouped_h_odd", 200, 640, 384, 8, 2, "normal", 0, 0),
    ("grouped_many_experts", 1024, 256, 256, 128, 4, "zipf", 0, 0),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: c[0])
def test_fused_fp8_token_edge_cases(moe, case):
    name, T, H, I, E, k, bias, bm, sk = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5, dtype="fp8_token")
    inp = synth.make_inputs(cfg, seed=4, device="cuda")
    host = _host(inp)
    w8 = quantize_rows_gpu(moe, inp, cfg)
    out, layer = run_fused(moe, cfg, inp, w8, block_m=bm, split_k=sk)
    _check_codes_in_workspace(moe, layer, cfg, host)
    q1, s1 = oracle.quant_rows(host["W_gate_up"])
    q2, s2 = oracle.quant_rows(host["W_down"])
    ref = oracle.moe_forward_fp8_token(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, k, np.arange(T))
    err = rel_l2(out.float().cpu().numpy(), ref)
    assert err <= TOL_FP8, err


def test_fused_fp8_token_deterministic(moe):
    cfg = synth.MoEConfig("det", T=48, H=256, I=384, E=6, k=2, dtype="fp8_token")
    inp = synth.make_inputs(cfg, seed=6, device="cuda")
    w8 = quantize_rows_gpu(moe, inp, cfg)
    a, _ = run_fused(moe, cfg, inp, w8)
    b, _ = run_fused(moe, cfg, inp, w8)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
