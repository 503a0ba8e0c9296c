"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Integer outputs (expert ids, sort order, padding, FP8 codes) must match
bit for bit; floating-point outputs must meet relative L2 error <= 5e-3
(bf16) and <= 3e-2 (block-scaled FP8) against the oracle fed the same
inputs, and every compared token row within 4x that; top-k weights within
1e-5 relative.  Large workloads compare every routing/sort output in full
and the layer output on the full-size parity sample of moe_checks
(512 seeded tokens, a row of every sorted M-block, the last row of every
expert, the tokens of the least-loaded experts).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_grouped_moe_gb300 import synth
from moe_checks import E4M3_LEADERS, check_rows, check_sort_invariants, every_bf16_below, parity_tokens, rel_l2

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3
TOL_FP8 = 3e-2


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_moe_gb300 import build
    build.build()
    from mixture_experts_grouped_moe_gb300 import moe as m
    m.load()
    return m


_cache = {}


def gpu_inputs(cfg, seed=0):
    key = (cfg, seed)
    if key not in _cache:
        if len(_cache) > 1:
            _cache.clear()
            torch.cuda.empty_cache()
        inp = synth.make_inputs(cfg, seed=seed, device="cuda")
        host = {k: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
                for k, v in inp.items()}
        _cache[key] = (inp, host)
    return _cache[key]


def bias_np(host):
    return host["bias"]


def run_fused(moe, cfg, inp, dtype=0, block_m=0, split_k=0, fp8w=None):
    layer = moe.FusedMoE(dtype, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, block_m, split_k)
    w = {"W_router": inp["W_router"], "bias": inp["bias"]}
    if dtype == moe.MOE_BF16:
        w.update(W_gate_up=inp["W_gate_up"], W_down=inp["W_down"])
    else:
        w.update(fp8w)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    layer(inp["x"], w, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    return out, layer


def quantize_weights_gpu(moe, inp, cfg):
    E, I, H = cfg.E, cfg.I, cfg.H
    q1 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device="cuda")
    s1 = torch.empty(E * 2 * I // 128, H // 128, dtype=torch.float32, device="cuda")
    q2 = torch.empty(E, H, I, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(E * H // 128, I // 128, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_weights(inp["W_gate_up"], E * 2 * I, H, q1, s1)
    moe.moe_quantize_fp8_weights(inp["W_down"], E * H, I, q2, s2)
    return {"W_gate_up": q1, "w1_scale": s1, "W_down": q2, "w2_scale": s2}


# ---------------------------------------------------------------- router

ROUTER_CASES = [
    synth.CONFIGS["tiny"],
    synth.CONFIGS["mixtral_decode"],
    synth.CONFIGS["mixtral_prefill"],
    synth.CONFIGS["finegrained_zipf"],
    synth.CONFIGS["tiny"].with_(name="t1", T=1),
    synth.CONFIGS["tiny"].with_(name="t3_e1", T=3, E=1, k=1),
    synth.CONFIGS["tiny"].with_(name="t17_k_eq_e", T=17, E=5, k=5),
    synth.CONFIGS["tiny"].with_(name="e1000_k32", T=40, H=384, E=1000, k=32, bias="normal", bias_param=0.5),
    synth.CONFIGS["tiny"].with_(name="h_ragged", T=70, H=384, E=40, k=6),
]


@pytest.mark.parametrize("cfg", ROUTER_CASES, ids=lambda c: c.name)
def test_router_parity(moe, cfg):
    inp = synth.make_inputs(cfg, seed=0, device="cuda", weights=False)
    T, E, k = cfg.T, cfg.E, cfg.k
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    moe.moe_route_topk(inp["x"], inp["W_router"], inp["bias"], T, cfg.H, E, k, ids, w, logits)
    torch.cuda.synchronize()
    xb, wb = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"])
    b = None if inp["bias"] is None else inp["bias"].cpu().numpy()
    r_ids, r_w, r_logits = oracle.route(xb, wb, b, k)
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), r_logits.view(np.uint32))
    assert np.array_equal(ids.cpu().numpy(), r_ids)
    np.testing.assert_allclose(w.cpu().numpy(), r_w, rtol=1e-5, atol=1e-7)
    assert np.allclose(w.sum(1).cpu().numpy(), 1.0, atol=1e-5)
    if cfg.name == "finegrained_zipf":
        counts = np.bincount(r_ids.ravel(), minlength=E)
        assert (counts == 0).sum() >= 1
        assert (counts > 0.05 * cfg.S).sum() >= 2
    # the softmax over all E at the selected experts (renormalize = 0): same ids
    ids3 = torch.empty_like(ids)
    w3 = torch.empty_like(w)
    moe.moe_route_topk(inp["x"], inp["W_router"], inp["bias"], T, cfg.H, E, k, ids3, w3, logits, renormalize=False)
    torch.cuda.synchronize()
    _, r_w3, _ = oracle.route(xb, wb, b, k, renormalize=False)
    assert torch.equal(ids3, ids)
    np.testing.assert_allclose(w3.cpu().numpy(), r_w3, rtol=1e-5, atol=1e-7)
    if T * E > 4096 and T <= 2048:
        # without a logits buffer the fused one-launch router runs instead: same bits
        ids2 = torch.empty_like(ids)
        w2 = torch.empty_like(w)
        moe.moe_route_topk(inp["x"], inp["W_router"], inp["bias"], T, cfg.H, E, k, ids2, w2, None)
        torch.cuda.synchronize()
        assert torch.equal(ids2, ids) and torch.equal(w2, w)


# ------------------------------------------------------------ align-sort

# single-CTA sorts: S <= 1024 with E <= 32 (one-warp scan) and with E > 32 (block scan), each at
# its limits; then the three-launch sort
SORT_CASES = [(16, 2, 4, 16), (32, 2, 8, 16), (8192, 2, 8, 128), (4096, 8, 256, 128), (1, 1, 1, 1),
              (3, 2, 3, 4), (700, 3, 1000, 32), (5000, 1, 7, 64), (2049, 4, 16, 128),
              (512, 2, 32, 16), (100, 4, 64, 16), (128, 8, 256, 32)]


@pytest.mark.parametrize("T,k,E,B", SORT_CASES)
def test_align_sort_parity(moe, T, k, E, B):
    rng = np.random.default_rng(T * 7 + E)
    # skewed expert popularity so that some experts get nothing
    p = rng.dirichlet(np.full(E, 0.3))
    ids = np.stack([rng.choice(E, k, replace=False, p=p) if E > k else rng.permutation(E)[:k]
                    for _ in range(T)]).astype(np.int32)
    wts = rng.random((T, k)).astype(np.float32)
    P, NB = oracle.align_sort_sizes(T, k, E, B)
    d_ids = torch.from_numpy(ids).cuda()
    d_w = torch.from_numpy(wts).cuda()
    s_ids = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    s_w = torch.full((P,), -7.0, dtype=torch.float32, device="cuda")
    s_e = torch.full((NB,), -7, dtype=torch.int32, device="cuda")
    npp = torch.zeros(1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(E, dtype=torch.int32, device="cuda")
    wsb = moe.moe_align_sort_workspace_size(T, k, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    moe.moe_align_sort(d_ids, d_w, T, k, E, B, s_ids, s_w, s_e, npp, cnt, ws, wsb)
    torch.cuda.synchronize()
    r_ids, r_e, r_npp, r_cnt = oracle.align_sort(ids, E, B)
    g_ids = s_ids.cpu().numpy()
    assert np.array_equal(g_ids, r_ids)
    assert np.array_equal(s_e.cpu().numpy(), r_e)
    assert int(npp.item()) == r_npp
    assert np.array_equal(cnt.cpu().numpy(), r_cnt)
    S = T * k
    ref_w = np.where(r_ids < S, wts.ravel()[np.minimum(r_ids, S - 1)], 0.0).astype(np.float32)
    assert np.array_equal(s_w.cpu().numpy(), ref_w)
    check_sort_invariants(ids, E, B, g_ids, s_e.cpu().numpy(), int(npp.item()), cnt.cpu().numpy())


@pytest.mark.parametrize("T,k,E,B", [(16, 2, 4, 16), (100, 4, 64, 16), (2049, 4, 16, 128)],
                         ids=["one_warp", "one_cta", "chunked"])
def test_align_sort_reports_bad_ids(moe, T, k, E, B):
    """An id outside [0, E) from the caller is never used as an index: its slot is left out and
    num_tokens_post_padded reports -1 (all three sort kernels).  The GPU must stay usable."""
    rng = np.random.default_rng(5)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids[T // 2, 0] = E + 3
    ids[T - 1, k - 1] = -2
    wts = rng.random((T, k)).astype(np.float32)
    P, NB = oracle.align_sort_sizes(T, k, E, B)
    d_ids = torch.from_numpy(ids).cuda()
    d_w = torch.from_numpy(wts).cuda()
    s_ids = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    s_w = torch.zeros(P, dtype=torch.float32, device="cuda")
    s_e = torch.zeros(NB, dtype=torch.int32, device="cuda")
    npp = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = moe.moe_align_sort_workspace_size(T, k, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    moe.moe_align_sort(d_ids, d_w, T, k, E, B, s_ids, s_w, s_e, npp, None, ws, wsb)
    torch.cuda.synchronize()
    assert int(npp.item()) == moe.MOE_ERR_INVALID_ARG
    got = s_ids.cpu().numpy()
    assert not np.isin([(T // 2) * k, T * k - 1], got).any()   # the two bad slots are placed nowhere
    # the same call with valid ids still sorts correctly afterwards
    ids[T // 2, 0] = 0
    ids[T - 1, k - 1] = E - 1
    d_ids.copy_(torch.from_numpy(ids))
    moe.moe_align_sort(d_ids, d_w, T, k, E, B, s_ids, s_w, s_e, npp, None, ws, wsb)
    torch.cuda.synchronize()
    r_ids, r_e, r_npp, _ = oracle.align_sort(ids, E, B)
    assert int(npp.item()) == r_npp
    assert np.array_equal(s_ids.cpu().numpy(), r_ids)


# ------------------------------------------------------------ FP8 codes

def test_quant_act_bit_exact(moe):
    g = torch.Generator(device="cuda").manual_seed(11)
    X = (torch.randn(300, 1024, generator=g, device="cuda") *
         torch.exp(torch.randn(300, 1, generator=g, device="cuda") * 3)).to(torch.bfloat16)
    X[5, 256:384] = 0
    q = torch.empty(300, 1024, dtype=torch.uint8, device="cuda")
    s = torch.empty(300, 8, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_act(X, 300, 1024, q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_1x128(synth.bf16_bits(X))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quant_act_every_bf16_value(moe):
    # every bf16 value within 21 binades below a group's largest, for eight group scales
    X = every_bf16_below(E4M3_LEADERS, 5504, 128).cuda()
    R, C = X.shape
    q = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    s = torch.empty(R, C // 128, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_act(X, R, C, q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_1x128(synth.bf16_bits(X))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quant_weights_bit_exact(moe):
    cfg = synth.CONFIGS["tiny"].with_(E=3, H=256, I=384)
    inp = synth.make_inputs(cfg, seed=3, device="cuda")
    inp["W_down"][1, :128, :128] *= 1000.0  # a block with a very different scale
    w = quantize_weights_gpu(moe, inp, cfg)
    torch.cuda.synchronize()
    for name, sname in (("W_gate_up", "w1_scale"), ("W_down", "w2_scale")):
        rq, rs = oracle.quant_128x128(synth.bf16_bits(inp[name]))
        assert np.array_equal(w[sname].cpu().numpy().view(np.uint32), rs.view(np.uint32))
        assert np.array_equal(w[name].cpu().numpy(), rq)


# --------------------------------------------------------- fused layer

def _oracle_bf16(host, cfg, tokens):
    return oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"],
                                   cfg.k, tokens)


def _check_intermediates(moe, layer, cfg, host):
    """Routing and sort outputs inside the fused call's workspace are bit-exact."""
    T, k, E = cfg.T, cfg.k, cfg.E
    r_ids, r_w, _ = oracle.route(host["x"], host["W_router"], host["bias"], k)
    ids = layer.view("topk_ids", torch.int32, (T, k)).cpu().numpy()
    assert np.array_equal(ids, r_ids)
    B = layer.plan.block_m
    P, NB = layer.plan.max_padded, layer.plan.max_blocks
    s_ids = layer.view("sorted_ids", torch.int32, (P,)).cpu().numpy()
    s_e = layer.view("sorted_expert_ids", torch.int32, (NB,)).cpu().numpy()
    o_ids, o_e, o_npp, o_cnt = oracle.align_sort(r_ids, E, B)
    assert np.array_equal(s_ids, o_ids)
    assert np.array_equal(s_e, o_e)
    assert int(layer.view("num_tokens_post_padded", torch.int32, (1,)).item()) == o_npp
    return r_ids


FUSED_CASES = ["tiny", "mixtral_decode", "mixtral_prefill", "finegrained_zipf"]


@pytest.mark.parametrize("name", FUSED_CASES)
def test_fused_bf16_parity(moe, name):
    cfg = synth.CONFIGS[name]
    inp, host = gpu_inputs(cfg)
    out, layer = run_fused(moe, cfg, inp)
    r_ids = _check_intermediates(moe, layer, cfg, host)
    toks = np.arange(cfg.T) if cfg.T <= 128 else parity_tokens(r_ids, cfg.E, layer.plan.block_m)
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"],
                                  cfg.k, toks, expert_major=True)
    check_rows(out.float().cpu().numpy()[toks], ref, TOL_BF16, label=name)


def _check_fp8_block_gathered_codes(layer, cfg, host):
    """The block-FP8 call's own gather + quantise: the e4m3 codes of x in sorted order and their
    1x128 scales (stored transposed, [H/128][max_padded]) equal the oracle's quantiser applied to
    the gathered rows, bit for bit; padding rows are zero rows (codes 0, scale 1)."""
    T, H, k = cfg.T, cfg.H, cfg.k
    P = layer.plan.max_padded
    npp = int(layer.view("num_tokens_post_padded", torch.int32, (1,)).item())
    s_ids = layer.view("sorted_ids", torch.int32, (P,)).cpu().numpy()[:npp]
    rows = np.zeros((npp, H), np.uint16)
    real = s_ids < T * k
    rows[real] = host["x"][s_ids[real] // k]
    rq, rs = oracle.quant_1x128(rows)
    gq = layer.view("x_sorted", torch.uint8, (P, H)).cpu().numpy()[:npp]
    gs = layer.view("x_scales", torch.float32, (H // 128, P)).cpu().numpy()[:, :npp].T
    assert np.array_equal(gq, rq)
    assert np.array_equal(np.ascontiguousarray(gs).view(np.uint32), rs.view(np.uint32))


def test_fused_fp8_parity(moe):
    cfg = synth.CONFIGS["mixtral_fp8"]
    inp, host = gpu_inputs(cfg)
    fp8w = quantize_weights_gpu(moe, inp, cfg)
    out, layer = run_fused(moe, cfg, inp, dtype=moe.MOE_FP8_BLOCK128, fp8w=fp8w)
    r_ids = _check_intermediates(moe, layer, cfg, host)
    # the oracle quantises the weights itself; its codes and scales equal the GPU's, in full
    q1, s1 = oracle.quant_128x128(host["W_gate_up"])
    q2, s2 = oracle.quant_128x128(host["W_down"])
    for name, ref_q, sname, ref_s in (("W_gate_up", q1, "w1_scale", s1), ("W_down", q2, "w2_scale", s2)):
        assert np.array_equal(fp8w[name].cpu().numpy(), ref_q), name
        assert np.array_equal(fp8w[sname].cpu().numpy().view(np.uint32), ref_s.view(np.uint32)), sname
    _check_fp8_block_gathered_codes(layer, cfg, host)
    toks = parity_tokens(r_ids, cfg.E, layer.plan.block_m)
    ref = oracle.moe_forward_fp8(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, cfg.k, toks,
                                 expert_major=True)
    check_rows(out.float().cpu().numpy()[toks], ref, TOL_FP8, label="fp8 block")


EDGE_CASES = [
    # (name, T, H, I, E, k, bias, block_m, split_k)
    ("t1", 1, 128, 256, 4, 2, None, 0, 0),
    ("t3_e2", 3, 128, 256, 2, 2, None, 0, 0),
    ("t17_e5", 17, 256, 384, 5, 2, "normal", 0, 0),
    ("e1k1", 9, 128, 128, 1, 1, None, 0, 0),
    ("k_eq_e", 11, 128, 256, 3, 3, None, 0, 0),
    ("swap_t128", 128, 256, 256, 4, 2, None, 0, 0),
    ("grouped_t129", 129, 256, 256, 4, 2, None, 0, 0),
    ("grouped_ragged", 300, 384, 640, 6, 3, "normal", 0, 0),
    ("swap_b32_sk2", 40, 256, 512, 4, 2, None, 32, 2),
    ("swap_b128_sk1", 20, 256, 512, 4, 2, None, 128, 1),
    ("swap_sk8", 8, 512, 1024, 8, 2, None, 0, 8),
    ("grouped_h_odd", 200, 640, 256, 8, 2, "normal", 0, 0),
    ("grouped_k32", 200, 128, 256, 64, 32, "normal", 0, 0),   # the token-major gather at its k limit
]


@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: c[0])
def test_fused_bf16_edge_cases(moe, case):
    name, T, H, I, E, k, bias, bm, sk = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5)
    inp = synth.make_inputs(cfg, seed=1, device="cuda")
    host = {kk: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
            for kk, v in inp.items()}
    out, layer = run_fused(moe, cfg, inp, block_m=bm, split_k=sk)
    _check_intermediates(moe, layer, cfg, host)
    ref = _oracle_bf16(host, cfg, np.arange(T))
    err = rel_l2(out.float().cpu().numpy(), ref)
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("case", [("fp8_small", 40, 256, 384, 4, 2, None), ("fp8_ragged", 257, 384, 256, 6, 3, "normal"),
                                  ("fp8_t1", 1, 128, 256, 4, 2, None),
                                  ("fp8_many_experts", 1024, 256, 256, 128, 4, "zipf")], ids=lambda c: c[0])
def test_fused_fp8_edge_cases(moe, case):
    name, T, H, I, E, k, bias = case
    cfg = synth.MoEConfig(name, T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5, dtype="fp8")
    inp = synth.make_inputs(cfg, seed=2, device="cuda")
    host = {kk: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
            for kk, v in inp.items()}
    fp8w = quantize_weights_gpu(moe, inp, cfg)
    out, layer = run_fused(moe, cfg, inp, dtype=moe.MOE_FP8_BLOCK128, fp8w=fp8w)
    _check_intermediates(moe, layer, cfg, host)
    _check_fp8_block_gathered_codes(layer, cfg, host)
    q1, s1 = oracle.quant_128x128(host["W_gate_up"])
    q2, s2 = oracle.quant_128x128(host["W_down"])
    ref = oracle.moe_forward_fp8(host["x"], host["W_router"], host["bias"], q1, s1, q2, s2, k, np.arange(T))
    err = rel_l2(out.float().cpu().numpy(), ref)
    assert err <= TOL_FP8, err


def test_fused_deterministic_and_unused_experts_not_read(moe):
    cfg = synth.MoEConfig("nan_test", T=24, H=256, I=256, E=16, k=2)
    inp = synth.make_inputs(cfg, seed=5, device="cuda")
    out1, layer = run_fused(moe, cfg, inp)
    out2, _ = run_fused(moe, cfg, inp)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    ids = layer.view("topk_ids", torch.int32, (cfg.T, cfg.k)).cpu().numpy()
    unused = sorted(set(range(cfg.E)) - set(ids.ravel().tolist()))
    assert unused
    for e in unused:
        inp["W_gate_up"][e] = float("nan")
        inp["W_down"][e] = float("nan")
    out3, _ = run_fused(moe, cfg, inp)
    assert torch.equal(out1.view(torch.int16), out3.view(torch.int16))
    # the grouped kernel too
    cfg2 = cfg.with_(T=300)
    inp2 = synth.make_inputs(cfg2, seed=6, device="cuda")
    o1, lay2 = run_fused(moe, cfg2, inp2)
    ids2 = lay2.view("topk_ids", torch.int32, (cfg2.T, cfg2.k)).cpu().numpy()
    unused2 = sorted(set(range(cfg2.E)) - set(ids2.ravel().tolist()))
    for e in unused2:
        inp2["W_gate_up"][e] = float("nan")
        inp2["W_down"][e] = float("nan")
    o2, _ = run_fused(moe, cfg2, inp2)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_fused_host_entry_matches_device_entry(moe):
    cfg = synth.CONFIGS["tiny"].with_(T=50)
    inp = synth.make_inputs(cfg, seed=8, device="cuda")
    out_dev, _ = run_fused(moe, cfg, inp)
    layer = moe.FusedMoE(0, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, host_staging=True)
    x_host = inp["x"].cpu().pin_memory()
    out_host = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory()
    layer.forward_host(x_host, {"W_router": inp["W_router"], "bias": None, "W_gate_up": inp["W_gate_up"],
                                "W_down": inp["W_down"]}, out_host)
    torch.cuda.synchronize()
    assert torch.equal(out_host.view(torch.int16), out_dev.cpu().view(torch.int16))


# ------------------------------------------------ tensor-core router

def _route_in_layer(moe, cfg, inp, tc):
    """Run the layer with the tensor-core router on or off; return its workspace's ids, weights, layer."""
    layer = moe.FusedMoE(moe.MOE_BF16, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, options=moe.Options(tc_router=tc))
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    layer(inp["x"], inp, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    ids = layer.view("topk_ids", torch.int32, (cfg.T, cfg.k)).cpu().numpy()
    w = layer.view("topk_weights", torch.float32, (cfg.T, cfg.k)).cpu().numpy()
    return ids, w, layer


TC_ROUTER_CASES = [
    synth.CONFIGS["finegrained_zipf"],
    synth.MoEConfig("e64_k2", T=300, H=512, I=256, E=64, k=2),
    synth.MoEConfig("e128_k8_bias", T=1000, H=1024, I=256, E=128, k=8, bias="normal", bias_param=0.5),
    synth.MoEConfig("e1024_k28", T=70, H=256, I=256, E=1024, k=28, bias="zipf", bias_param=1.2),
]


@pytest.mark.parametrize("cfg", TC_ROUTER_CASES, ids=lambda c: c.name)
def test_tc_router_bit_identical_to_fixed_order(moe, cfg):
    """Ids and weights of the tensor-core router equal the fixed-order router's and the oracle's ids
    bit for bit; few tokens need the all-exact fall-back."""
    if cfg.name == "finegrained_zipf":
        inp, host = gpu_inputs(cfg)
    else:
        inp = synth.make_inputs(cfg, seed=4, device="cuda")
        host = {kk: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
                for kk, v in inp.items()}
    ids1, w1, layer = _route_in_layer(moe, cfg, inp, 1)
    ids0, w0, _ = _route_in_layer(moe, cfg, inp, 0)
    assert np.array_equal(ids1, ids0)
    assert np.array_equal(w1.view(np.uint32), w0.view(np.uint32))
    r_ids, _, r_logits = oracle.route(host["x"], host["W_router"], host["bias"], cfg.k)
    assert np.array_equal(ids1, r_ids)
    st = layer.ws[layer.layout.status:layer.layout.status + 32].view(torch.int32).cpu().numpy()
    fallbacks = int(st[4])
    print(f"{cfg.name}: {fallbacks} of {cfg.T} tokens fell back to all fixed-order logits")
    assert fallbacks <= max(2, cfg.T // 10)
    # the tensor-core logits against the fixed-order ones: far inside the bound the check assumes
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    rows = (cfg.T + 127) // 128 * 128
    s, nkb, tiles1 = 1, cfg.H // 64, (rows // 128) * ((cfg.E + 255) // 256)
    while s < 8 and tiles1 * s < nsm // 2 and nkb % (2 * s) == 0:
        s *= 2
    part = layer.view("router_logits", torch.float32, (s, rows, cfg.E)).double().sum(0)[:cfg.T].cpu().numpy()
    if host["bias"] is not None:
        part = part + host["bias"][None, :].astype(np.float64)
    xf = host["x"].astype(np.uint32) << 16
    wf = host["W_router"].astype(np.uint32) << 16
    xn = np.linalg.norm(xf.view(np.float32).astype(np.float64), axis=1)
    wn = np.linalg.norm(wf.view(np.float32).astype(np.float64), axis=1)
    rel = np.abs(part - r_logits.astype(np.float64)) / (xn[:, None] * wn[None, :])
    print(f"{cfg.name}: max |tensor-core - fixed-order| / (||x|| ||w||) = {rel.max():.3e}")
    assert rel.max() < 2.0 ** -16


def test_tc_router_exact_ties_fall_back(moe):
    """Experts with identical router rows tie exactly: the check must fall back to the fixed order
    and give the tie to the lower expert, as the fixed-order router does."""
    cfg = synth.MoEConfig("ties", T=256, H=512, I=256, E=64, k=4)
    inp = synth.make_inputs(cfg, seed=6, device="cuda")
    for e in range(64):  # four groups of 16 identical rows: the leading group ties well past k + 4
        inp["W_router"][e] = inp["W_router"][e - e % 16]
    ids1, w1, layer = _route_in_layer(moe, cfg, inp, 1)
    ids0, w0, _ = _route_in_layer(moe, cfg, inp, 0)
    assert np.array_equal(ids1, ids0)
    assert np.array_equal(w1.view(np.uint32), w0.view(np.uint32))
    r_ids, _, _ = oracle.route(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"]), None, cfg.k)
    assert np.array_equal(ids1, r_ids)
    st = layer.ws[layer.layout.status:layer.layout.status + 32].view(torch.int32).cpu().numpy()
    assert st[4] == cfg.T   # every token's leading group ties beyond its candidates: all fell back


def test_tc_router_near_ties_settled_by_candidates(moe):
    """Experts in pairs whose router rows differ in one element by one bf16 step: their fixed-order
    logits differ, by far less than the tensor core's error bound.  The two of a pair rank next to
    each other, so with an odd k the k-th and (k+1)-th candidates are a pair for every token and
    only their fixed-order logits can order them.  The result must still be the fixed-order
    router's and the oracle's, bit for bit, and the pairs inside the candidate set must not force
    the all-expert fall-back."""
    cfg = synth.MoEConfig("twins", T=512, H=512, I=256, E=64, k=3)
    inp = synth.make_inputs(cfg, seed=8, device="cuda")
    bits = inp["W_router"].view(torch.int16)
    for e in range(1, 64, 2):
        bits[e] = bits[e - 1]
        bits[e, 5 + e] += 1   # one bf16 step in one element (nonzero rows: no sign or zero crossing)
    ids1, w1, layer = _route_in_layer(moe, cfg, inp, 1)
    ids0, w0, _ = _route_in_layer(moe, cfg, inp, 0)
    assert np.array_equal(ids1, ids0)
    assert np.array_equal(w1.view(np.uint32), w0.view(np.uint32))
    r_ids, _, _ = oracle.route(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"]), None, cfg.k)
    assert np.array_equal(ids1, r_ids)
    st = layer.ws[layer.layout.status:layer.layout.status + 32].view(torch.int32).cpu().numpy()
    print(f"twins: {st[4]} of {cfg.T} tokens fell back to all fixed-order logits")
    assert st[4] < cfg.T // 4
