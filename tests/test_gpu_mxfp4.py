"""MXFP4 ("per_1x32": E2M1 elements, one E8M0 scale per 32) through the C ABI vs the CPU oracle.

The quantiser's codes and scales are compared bit for bit in both scale
orders (row-major and the tiled weight order), standalone and inside the
fused call (the gathered activations).  The layer output must be within
relative L2 1e-2 of the oracle: both sides round the same quantities to the
same E2M1 grid, so the difference is the bf16 rounding of the output
(about 2^-9) plus the rare intermediate code that lands on the other side of
a rounding boundary because the two accumulate in different precisions.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_grouped_moe_gb300 import synth
from moe_checks import check_rows, parity_tokens, rel_l2

pytestmark = pytest.mark.gpu

TOL_MX4 = 1e-2


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


def unpack(qp):
    """Two codes per byte (element 2j in the low nibble) -> one code per byte."""
    q = np.asarray(qp, dtype=np.uint8)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = q & 15
    out[..., 1::2] = q >> 4
    return out


def untile(st, R, C):
    """Tiled E8M0 scales [R/128][C/128][512] -> row-major [R][C/32]."""
    t = np.asarray(st, dtype=np.uint8).reshape(R // 128, C // 128, 32, 4, 4)   # [rb][cb][r%32][r%128/32][g%4]
    return t.transpose(0, 3, 2, 1, 4).reshape(R, C // 32)


def quantize_weights_gpu(moe, inp, cfg):
    E, I, H = cfg.E, cfg.I, cfg.H
    q1 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device="cuda")
    s1 = torch.empty(E * 2 * I * H // 32, dtype=torch.uint8, device="cuda")
    q2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(E * H * I // 32, dtype=torch.uint8, device="cuda")
    moe.moe_quantize_mxfp4(inp["W_gate_up"], E * 2 * I, H, q1, s1, tiled=True)
    moe.moe_quantize_mxfp4(inp["W_down"], E * H, I, q2, s2, tiled=True)
    return {"W_gate_up": q1, "w1_scale": s1, "W_down": q2, "w2_scale": s2}


@pytest.mark.parametrize("tiled", [False, True], ids=["row_major", "tiled"])
def test_quant_mxfp4_bit_exact(moe, tiled):
    R, C = 256, 384
    g = torch.Generator(device="cuda").manual_seed(21)
    X = (torch.randn(R, C, generator=g, device="cuda") *
         torch.exp(torch.randn(R, C // 32, generator=g, device="cuda").repeat_interleave(32, 1) * 4))
    X = X.to(torch.bfloat16)
    X[7, 32:64] = 0
    X[9, :32] = torch.tensor([4.0, 2.5, 1.25, 0.75, 0.25, 5.0, 3.5, 1.75] * 4, device="cuda")  # exact ties
    X[11, :32] = 1e-39  # subnormal block
    q = torch.empty(R, C // 2, dtype=torch.uint8, device="cuda")
    s = torch.empty(R * C // 32, dtype=torch.uint8, device="cuda")
    moe.moe_quantize_mxfp4(X, R, C, q, s, tiled=tiled)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_mx4(synth.bf16_bits(X))
    gs = s.cpu().numpy()
    gs = untile(gs, R, C) if tiled else gs.reshape(R, C // 32)
    assert np.array_equal(gs, rs)
    assert np.array_equal(unpack(q.cpu().numpy()), rq)


def _every_rounding_boundary(R, C):
    """Groups of 32 bf16 values: a leader 7.875 * 2^j that fixes the group's scale at 2^j (2^-127,
    the clamp, for the subnormal j), then every finite bf16 value v with 2^(j-3) <= |v| <= leader,
    both signs, 31 to a group -- each scaled value from 1/8 up into the saturation range meets the
    rounding rule.  Padded with zero groups to R x C."""
    vals = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    groups = []
    for j in (-130, -127, -3, 0, 9, 125):
        lead = 7.875 * 2.0 ** j
        v = vals[torch.isfinite(vals) & (vals.abs() <= lead) & (vals.abs() >= 2.0 ** (j - 3))]
        v = torch.cat([v, torch.zeros((-len(v)) % 31)]).view(-1, 31)
        groups.append(torch.cat([torch.full((v.shape[0], 1), lead), v], 1))
    g = torch.cat(groups).reshape(-1)
    X = torch.zeros(R * C)
    X[: g.numel()] = g
    return X.view(R, C).to(torch.bfloat16)


@pytest.mark.parametrize("tiled", [False, True], ids=["row_major", "tiled"])
def test_quant_mxfp4_every_rounding_boundary(moe, tiled):
    R, C = 128, 384
    X = _every_rounding_boundary(R, C).cuda()
    q = torch.empty(R, C // 2, dtype=torch.uint8, device="cuda")
    s = torch.empty(R * C // 32, dtype=torch.uint8, device="cuda")
    moe.moe_quantize_mxfp4(X, R, C, q, s, tiled=tiled)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_mx4(synth.bf16_bits(X))
    gs = s.cpu().numpy()
    gs = untile(gs, R, C) if tiled else gs.reshape(R, C // 32)
    assert np.array_equal(gs, rs)
    assert np.array_equal(unpack(q.cpu().numpy()), rq)


def test_quant_mxfp4_rejects_bad_shapes(moe):
    X = torch.zeros(4, 48, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(4, 24, dtype=torch.uint8, device="cuda")
    s = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoEError):
        moe.moe_quantize_mxfp4(X, 4, 48, q, s)            # C not a multiple of 32
    X = torch.zeros(100, 128, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(100, 64, dtype=torch.uint8, device="cuda")
    s = torch.empty(400, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoEError):
        moe.moe_quantize_mxfp4(X, 100, 128, q, s, tiled=True)  # tiled needs R % 128 == 0


def run_fused(moe, cfg, inp, w4, block_m=0, split_k=0):
    layer = moe.FusedMoE(moe.MOE_MXFP4, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, block_m, split_k)
    w = dict(w4, W_router=inp["W_router"], bias=inp["bias"])
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    layer(inp["x"], w, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    return out, layer


def untile_scales(tiled, R, C):
    """Row-major [R][C/32] E8M0 bytes from the 128 x 4 blocked order of 128-row x 128-column tiles
    ([R/128][C/128][512]; row r, group g at byte (r % 32) * 16 + (r % 128 // 32) * 4 + g % 4)."""
    r = np.arange(R)[:, None]
    g = np.arange(C // 32)[None, :]
    off = ((r // 128) * (C // 128) + g // 4) * 512 + (r % 32) * 16 + (r % 128 // 32) * 4 + g % 4
    return np.asarray(tiled)[off]


def _check_workspace(moe, layer, cfg, host):
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
    rq, rs = oracle.quant_mx4(xrows)
    xq = layer.view("x_sorted", torch.uint8, (P, cfg.H // 2)).cpu().numpy()[:npp]
    xs = layer.view("x_scales", torch.uint8, (P * cfg.H // 32,)).cpu().numpy()
    if layer.plan.mode == moe.MOE_MODE_GROUPED:
        # grouped mode keeps them in the tensor core's blocked order (npp: whole 128-row blocks)
        assert npp % 128 == 0
        xs = untile_scales(xs, npp, cfg.H)
    else:
        xs = xs.reshape(P, cfg.H // 32)[:npp]
    assert np.array_equal(unpack(xq), rq) and np.array_equal(xs, rs)


def test_fused_mxfp4_decode_parity(moe):
    cfg = synth.CONFIGS["mixtral_mxfp4_decode"]
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    host = _host(inp)
    w4 = quantize_weights_gpu(moe, inp, cfg)
    out, layer = run_fused(moe, cfg, inp, w4)
    assert layer.plan.mode == moe.MOE_MODE_SWAP and layer.plan.split_k2 > 1
    _check_workspace(moe, layer, cfg, host)
    q1, s1 = oracle.quant_mx4(host["W_gate_up"])
    q2, s2 = oracle.quant_mx4(host["W_down"])
    assert np.array_equal(unpack(w4["W_gate_up"][cfg.E - 1, -8:].cpu().numpy()), q1[cfg.E - 1, -8:])
    toks = np.arange(cfg.T)
    ref = oracle.moe_forward_mxfp4(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, cfg.k, toks)
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    err = rel_l2(got, ref)
    print(f"mxfp4 decode: relL2 {err:.3e}")
    assert err <= TOL_MX4


EDGE = [
    # (name, T, H, I, E, k, bias, block_m, split_k)
    ("t1", 1, 256, 256, 4, 2, None, 0, 0),
    ("t17_e5", 17, 256, 512, 5, 2, "normal", 0, 0),
    ("e1k1", 9, 256, 256, 1, 1, None, 0, 0),
    ("k_eq_e", 11, 256, 256, 3, 3, None, 0, 0),
    ("t64_max", 64, 512, 512, 4, 2, None, 0, 0),
    ("b32_sk2", 40, 256, 512, 4, 2, None, 32, 2),
    ("b64_sk1", 20, 512, 256, 4, 2, None, 64, 1),
    ("h_odd", 24, 768, 256, 6, 2, "normal", 0, 0),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: c[0])
def test_fused_mxfp4_edge_cases(moe, case):
    name, T, H, I, E, k, bias, bm, sk = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5, dtype="mxfp4")
    inp = synth.make_inputs(cfg, seed=5, device="cuda")
    host = _host(inp)
    w4 = quantize_weights_gpu(moe, inp, cfg)
    out, layer = run_fused(moe, cfg, inp, w4, block_m=bm, split_k=sk)
    _check_workspace(moe, layer, cfg, host)
    q1, s1 = oracle.quant_mx4(host["W_gate_up"])
    q2, s2 = oracle.quant_mx4(host["W_down"])
    ref = oracle.moe_forward_mxfp4(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, k, np.arange(T))
    err = rel_l2(out.float().cpu().numpy(), ref)
    assert err <= TOL_MX4, err


GROUPED = [
    # (name, T, H, I, E, k, bias): grouped mode (T > 64), 128-row blocks
    ("t65", 65, 256, 256, 4, 2, None),
    ("t300_ragged", 300, 512, 256, 6, 3, "normal"),
    ("e1k1_t200", 200, 256, 512, 1, 1, None),
    ("h_odd", 150, 768, 256, 5, 2, "normal"),
    ("many_experts", 500, 256, 256, 40, 4, "normal"),
    ("e128_zipf", 1024, 256, 256, 128, 4, "zipf"),
]


@pytest.mark.parametrize("case", GROUPED, ids=lambda c: c[0])
def test_fused_mxfp4_grouped_edge_cases(moe, case):
    name, T, H, I, E, k, bias = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5, dtype="mxfp4")
    inp = synth.make_inputs(cfg, seed=6, device="cuda")
    host = _host(inp)
    w4 = quantize_weights_gpu(moe, inp, cfg)
    out, layer = run_fused(moe, cfg, inp, w4)
    assert layer.plan.mode == moe.MOE_MODE_GROUPED
    _check_workspace(moe, layer, cfg, host)
    q1, s1 = oracle.quant_mx4(host["W_gate_up"])
    q2, s2 = oracle.quant_mx4(host["W_down"])
    ref = oracle.moe_forward_mxfp4(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, k, np.arange(T))
    err = rel_l2(out.float().cpu().numpy(), ref)
    assert err <= TOL_MX4, err


def test_fused_mxfp4_prefill_parity(moe):
    cfg = synth.CONFIGS["mixtral_mxfp4"]
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    host = _host(inp)
    w4 = quantize_weights_gpu(moe, inp, cfg)
    out, layer = run_fused(moe, cfg, inp, w4)
    assert layer.plan.mode == moe.MOE_MODE_GROUPED
    _check_workspace(moe, layer, cfg, host)
    q1, s1 = oracle.quant_mx4(host["W_gate_up"])
    q2, s2 = oracle.quant_mx4(host["W_down"])
    r_ids, _, _ = oracle.route(host["x"], host["W_router"], host["bias"], cfg.k)
    toks = parity_tokens(r_ids, cfg.E, layer.plan.block_m)
    ref = oracle.moe_forward_mxfp4(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, cfg.k, toks,
                                   expert_major=True)
    check_rows(out.float().cpu().numpy()[toks], ref, TOL_MX4, label="mxfp4 T=4096")
