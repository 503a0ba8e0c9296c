"""Grouped-mode GEMMs on CTA pairs (two-SM tensor core) vs the one-SM kernels.

Each case runs the fused layer with the kernel choice forced both ways
(per-call option gemm_pair 1 and 0): both must meet the tolerance against the
oracle, and the routing / sort outputs stay bit-exact.  The cases cover odd
block counts per expert (half-used pairs), experts without tokens, a ragged
last N tile of stage 2 and the Mixtral prefill shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_grouped_moe_gb300 import synth
from moe_checks import check_rows, parity_tokens, rel_l2

pytestmark = pytest.mark.gpu


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


def _run(moe, cfg, inp, w, dtype, pair_mode):
    layer = moe.FusedMoE(dtype, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, options=moe.Options(gemm_pair=pair_mode))
    assert layer.plan.mode == moe.MOE_MODE_GROUPED
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    layer(inp["x"], w, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    return out.float().cpu().numpy(), layer


CASES = [
    # (name, T, H, I, E, k, bias)
    ("t129_e4", 129, 256, 256, 4, 2, None),
    ("t300_ragged", 300, 384, 640, 6, 3, "normal"),
    ("h_odd", 200, 640, 384, 8, 2, "normal"),
    ("many_experts", 700, 256, 256, 40, 4, "normal"),   # some experts empty, many with one block
    ("e1k1", 520, 256, 384, 1, 1, None),                # one expert, odd block count
]


@pytest.mark.parametrize("mode", [1, 0], ids=["pair", "one_sm"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_bf16_grouped_both_kernels(moe, case, mode):
    name, T, H, I, E, k, bias = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5)
    inp = synth.make_inputs(cfg, seed=11, device="cuda")
    host = _host(inp)
    w = {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": inp["W_gate_up"], "W_down": inp["W_down"]}
    got, layer = _run(moe, cfg, inp, w, moe.MOE_BF16, mode)
    r_ids, _, _ = oracle.route(host["x"], host["W_router"], host["bias"], k)
    assert np.array_equal(layer.view("topk_ids", torch.int32, (T, k)).cpu().numpy(), r_ids)
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"], k)
    assert rel_l2(got, ref) <= 5e-3


@pytest.mark.parametrize("mode", [1, 0], ids=["pair", "one_sm"])
@pytest.mark.parametrize("case", CASES[:4], ids=lambda c: c[0])
def test_fp8_token_grouped_both_kernels(moe, case, mode):
    name, T, H, I, E, k, bias = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5, dtype="fp8_token")
    inp = synth.make_inputs(cfg, seed=12, device="cuda")
    host = _host(inp)
    q1 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device="cuda")
    s1 = torch.empty(E * 2 * I, dtype=torch.float32, device="cuda")
    q2 = torch.empty(E, H, I, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(E * H, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(inp["W_gate_up"], E * 2 * I, H, q1, s1)
    moe.moe_quantize_fp8_rows(inp["W_down"], E * H, I, q2, s2)
    w = {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": q1, "w1_scale": s1, "W_down": q2,
         "w2_scale": s2}
    got, _ = _run(moe, cfg, inp, w, moe.MOE_FP8_TOKEN, mode)
    o1, os1 = oracle.quant_rows(host["W_gate_up"])
    o2, os2 = oracle.quant_rows(host["W_down"])
    ref = oracle.moe_forward_fp8_token(host["x"], host["W_router"], host["bias"], o1, os1, o2, os2, k)
    assert rel_l2(got, ref) <= 3e-2


def _fp8_block_weights(moe, inp, cfg):
    E, I, H = cfg.E, cfg.I, cfg.H
    q1 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device="cuda")
    s1 = torch.empty(E * 2 * I // 128, H // 128, dtype=torch.float32, device="cuda")
    q2 = torch.empty(E, H, I, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(E * H // 128, I // 128, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_weights(inp["W_gate_up"], E * 2 * I, H, q1, s1)
    moe.moe_quantize_fp8_weights(inp["W_down"], E * H, I, q2, s2)
    return {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": q1, "w1_scale": s1, "W_down": q2,
            "w2_scale": s2}


def _fp8_block_both(moe, cfg, inp, w):
    """The block-FP8 layer with the pair kernels and with the one-SM kernels: outputs, the stage-1
    h codes and their 1x128 scales of the real sorted rows."""
    res = []
    for mode in (1, 0):
        out, layer = _run(moe, cfg, inp, w, moe.MOE_FP8_BLOCK128, mode)
        P = layer.plan.max_padded
        npp = int(layer.view("num_tokens_post_padded", torch.int32, (1,)).item())
        ids = layer.view("sorted_ids", torch.int32, (P,))[:npp]
        real = (ids < cfg.T * cfg.k).cpu()
        h = layer.view("inter", torch.uint8, (P, cfg.I))[:npp].cpu()[real]
        hs = layer.view("inter_scales", torch.float32, (cfg.I // 128, P))[:, :npp].cpu()[:, real]
        res.append((out, h, hs))
    return res


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_fp8_block_pair_bit_identical(moe, case):
    """Block-FP8 on CTA pairs: each CTA promotes the same per-128 products in the same order as the
    one-SM kernel, so the h codes, their scales and the output are bit-identical to it (half-used
    pairs, empty experts, a ragged last stage-2 tile included), and within the FP8 tolerance of the
    oracle."""
    name, T, H, I, E, k, bias = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5, dtype="fp8")
    inp = synth.make_inputs(cfg, seed=13, device="cuda")
    w = _fp8_block_weights(moe, inp, cfg)
    (o_p, h_p, s_p), (o_1, h_1, s_1) = _fp8_block_both(moe, cfg, inp, w)
    assert torch.equal(h_p, h_1)
    assert torch.equal(s_p.view(torch.int32), s_1.view(torch.int32))
    assert np.array_equal(o_p.view(np.uint32), o_1.view(np.uint32))
    host = _host(inp)
    q1, s1 = oracle.quant_128x128(host["W_gate_up"])
    q2, s2 = oracle.quant_128x128(host["W_down"])
    ref = oracle.moe_forward_fp8(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, k)
    assert rel_l2(o_p, ref) <= 3e-2


def test_fp8_block_pair_full_size_bit_identical(moe):
    """Mixtral shapes at T=4096 (block FP8): the pair kernels reproduce the one-SM kernels' h codes,
    scales and outputs bit for bit on every token."""
    cfg = synth.CONFIGS["mixtral_fp8"]
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    w = _fp8_block_weights(moe, inp, cfg)
    (o_p, h_p, s_p), (o_1, h_1, s_1) = _fp8_block_both(moe, cfg, inp, w)
    assert torch.equal(h_p, h_1)
    assert torch.equal(s_p.view(torch.int32), s_1.view(torch.int32))
    assert np.array_equal(o_p.view(np.uint32), o_1.view(np.uint32))


def test_prefill_pair_matches_one_sm(moe):
    """Mixtral prefill shapes: both kernels against the oracle on the full-size parity sample (every
    M-block, the least-loaded experts, each expert's last row), and against each other on every token."""
    cfg = synth.CONFIGS["mixtral_prefill"]
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    w = {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": inp["W_gate_up"], "W_down": inp["W_down"]}
    outs = [_run(moe, cfg, inp, w, moe.MOE_BF16, mode)[0] for mode in (1, 0)]
    host = _host(inp)
    r_ids, _, _ = oracle.route(host["x"], host["W_router"], host["bias"], cfg.k)
    toks = parity_tokens(r_ids, cfg.E, 128)
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"],
                                  cfg.k, toks, expert_major=True)
    check_rows(outs[0][toks], ref, 5e-3, label="prefill pairs")
    check_rows(outs[1][toks], ref, 5e-3, label="prefill one-SM")
    assert rel_l2(outs[0], outs[1]) <= 5e-3


def test_gemm_pair_option_rejects_bad_value(moe):
    cfg = synth.MoEConfig("bad", T=200, H=256, I=256, E=4, k=2)
    inp = synth.make_inputs(cfg, seed=1, device="cuda")
    layer = moe.FusedMoE(moe.MOE_BF16, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, options=moe.Options(gemm_pair=2))
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer(inp["x"], inp, out)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG


# Light experts (all rows in one 128-row block) on swap-AB pair tiles: routings with empty,
# single-token, one-block and multi-block experts; I a multiple of 256 (the light stage-1 tile
# covers 256 intermediate columns); a ragged last tile of H in stage 2.
LIGHT_CASES = [
    # (name, T, H, I, E, k, bias)
    ("all_light", 200, 256, 256, 64, 2, None),
    ("zipf_mix", 1000, 512, 512, 64, 4, "zipf"),
    ("ragged_h", 300, 640, 256, 32, 3, "normal"),
    ("few_experts", 260, 256, 768, 4, 1, "normal"),
]


@pytest.mark.parametrize("light", [1, 0], ids=["light", "pairs_only"])
@pytest.mark.parametrize("case", LIGHT_CASES, ids=lambda c: c[0])
def test_light_expert_tiles(moe, case, light):
    name, T, H, I, E, k, bias = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=1.2 if bias == "zipf" else 0.5)
    inp = synth.make_inputs(cfg, seed=13, device="cuda")
    host = _host(inp)
    w = {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": inp["W_gate_up"], "W_down": inp["W_down"]}
    layer = moe.FusedMoE(moe.MOE_BF16, T, H, I, E, k, options=moe.Options(gemm_pair=1, light_tiles=light))
    assert layer.plan.mode == moe.MOE_MODE_GROUPED
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    layer(inp["x"], w, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    counts = layer.view("expert_counts", torch.int32, (E,)).cpu().numpy()
    print(name, "counts", sorted(counts.tolist()))
    assert ((counts > 0) & (counts <= 128)).any()   # some light experts in every case
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"], k)
    check_rows(out.float().cpu().numpy(), ref, 5e-3, label=f"{name} light={light}")
    # bitwise reproducible
    out2 = torch.empty_like(out)
    layer(inp["x"], w, out2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_light_tiles_need_i_multiple_of_256(moe):
    cfg = synth.MoEConfig("bad_light", T=200, H=256, I=384, E=8, k=2)
    inp = synth.make_inputs(cfg, seed=1, device="cuda")
    layer = moe.FusedMoE(moe.MOE_BF16, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k,
                         options=moe.Options(gemm_pair=1, light_tiles=1))
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer(inp["x"], inp, out)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED


def test_finegrained_light_tiles_on_and_off(moe):
    """The fine-grained workload (most experts hold a few tokens): both tile choices against the oracle
    on the full-size parity sample."""
    cfg = synth.CONFIGS["finegrained_zipf"]
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    host = _host(inp)
    w = {"W_router": inp["W_router"], "bias": inp["bias"], "W_gate_up": inp["W_gate_up"], "W_down": inp["W_down"]}
    outs = []
    for light in (1, 0):
        layer = moe.FusedMoE(moe.MOE_BF16, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k,
                             options=moe.Options(gemm_pair=1, light_tiles=light))
        out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
        layer(inp["x"], w, out)
        torch.cuda.synchronize()
        assert layer.status() == moe.MOE_OK
        outs.append(out.float().cpu().numpy())
        del layer
    r_ids, _, _ = oracle.route(host["x"], host["W_router"], host["bias"], cfg.k)
    toks = parity_tokens(r_ids, cfg.E, 128)
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"],
                                  cfg.k, toks, expert_major=True)
    check_rows(outs[0][toks], ref, 5e-3, label="fine-grained light tiles")
    check_rows(outs[1][toks], ref, 5e-3, label="fine-grained pair tiles only")


@pytest.mark.parametrize("case", [("e512_light_limit", 2048, 256, 256, 512, 8, "zipf", 1),
                                  ("e1024_pair_limit", 2048, 256, 256, 1024, 8, "zipf", -1)],
                         ids=lambda c: c[0])
def test_many_experts_at_the_table_limits(moe, case):
    """The largest expert counts of the per-expert tables: 512 with light-expert tiles (their limit),
    1024 on plain pair tiles (the pair kernel's and the router's limit; light tiles are not
    supported there, so the automatic choice leaves them off).  The tensor-core router, the
    chunked sort and the pair kernels' tile tables at full size, against the oracle."""
    name, T, H, I, E, k, bias, light = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=1.2)
    inp = synth.make_inputs(cfg, seed=31, device="cuda")
    host = _host(inp)
    layer = moe.FusedMoE(moe.MOE_BF16, T, H, I, E, k, options=moe.Options(gemm_pair=1, light_tiles=light))
    assert layer.plan.mode == moe.MOE_MODE_GROUPED
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    layer(inp["x"], inp, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    r_ids, _, _ = oracle.route(host["x"], host["W_router"], host["bias"], k)
    assert np.array_equal(layer.view("topk_ids", torch.int32, (T, k)).cpu().numpy(), r_ids)
    counts = layer.view("expert_counts", torch.int32, (E,)).cpu().numpy()
    assert (counts == 0).any() and (counts > 128).any()   # empty, light and multi-block experts
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"], k,
                                  expert_major=True)
    check_rows(out.float().cpu().numpy(), ref, 5e-3, label=name)
