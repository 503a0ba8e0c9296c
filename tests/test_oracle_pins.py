"""Pins for the CPU oracle: each test ties the oracle to something other than
itself -- values worked by hand from the pages' formulas, brute-force
enumeration, an independent formulation (masked dense MoE), closed cases
(E=1/k=1 is a plain SwiGLU MLP; k=E is a softmax mixture) evaluated with
library routines, and PyTorch's own E4M3 encoder.  CPU only.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import heuristics
from mixture_experts_grouped_moe_gb300 import synth
from moe_checks import check_sort_invariants

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _bf16_bits_of(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    """bf16 bits -> float64 values."""
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------ e4m3

def test_e4m3_decode_known_values():
    # OCP FP8 E4M3: bias 7, max finite 448, min normal 2^-6, min subnormal 2^-9, S.1111.111 = NaN
    d = oracle.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x40, 0x7E, 0xFE, 0x80], np.uint8))
    assert list(d) == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 2.0, 448.0, -448.0, 0.0]
    assert math.isnan(oracle.e4m3_decode(np.array([0x7F], np.uint8))[0])
    assert math.isnan(oracle.e4m3_decode(np.array([0xFF], np.uint8))[0])


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_table()
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), ~finite)
    assert np.array_equal(ours[finite], ref[finite])


def test_e4m3_encode_roundtrip_and_midpoints():
    tab = oracle.e4m3_table()
    finite = [c for c in range(256) if not math.isnan(tab[c])]
    enc = oracle.e4m3_encode(np.array([tab[c] for c in finite], np.float32))
    assert list(enc) == finite  # includes -0 -> 0x80
    # exact midpoints between neighbouring positive codes go to the even code
    pos = [c for c in range(0x00, 0x7F)]
    for a, b in zip(pos[:-1], pos[1:]):
        mid = np.float32((tab[a] + tab[b]) / 2)
        assert float(mid) == (tab[a] + tab[b]) / 2
        got = int(oracle.e4m3_encode(np.array([mid], np.float32))[0])
        assert got == (a if a % 2 == 0 else b), (a, b, got)
    # saturation instead of NaN above 448
    assert list(oracle.e4m3_encode(np.array([448, 460, 1e4, -1e30, np.inf], np.float32))) == \
        [0x7E, 0x7E, 0x7E, 0xFE, 0x7E]


def test_e4m3_encode_matches_torch_random():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000))).astype(np.float32)
    v = v[np.abs(v) < 448]
    ours = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_quant_1x128_against_torch_encoder():
    g = torch.Generator().manual_seed(3)
    X = (torch.randn(7, 512, generator=g) * torch.exp(torch.randn(7, 1, generator=g) * 3)).to(torch.bfloat16)
    X[2, 128:256] = 0  # an all-zero group takes scale 1
    bits = X.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.quant_1x128(bits)
    xf = X.float().reshape(7, 4, 128)
    amax = xf.abs().amax(-1)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    assert np.array_equal(s, sc.numpy())
    ref = (xf / sc[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(7, 512).numpy()
    assert np.array_equal(q, ref)
    tab = oracle.e4m3_table()
    for r in range(7):
        for gi in range(4):
            vals = np.abs(tab[q[r, gi * 128:(gi + 1) * 128]])
            assert vals.max() == (0.0 if (r, gi) == (2, 1) else 448.0)


def test_quant_128x128_block_scales():
    g = torch.Generator().manual_seed(4)
    W = (torch.randn(256, 384, generator=g) / 16).to(torch.bfloat16)
    W[128:, 256:] *= 64
    bits = W.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.quant_128x128(bits)
    assert s.shape == (2, 3)
    Wf = W.float().reshape(2, 128, 3, 128).permute(0, 2, 1, 3)
    amax = Wf.abs().amax((-1, -2))
    assert np.array_equal(s, (amax / 448.0).numpy())
    ref = (Wf / (amax / 448.0)[..., None, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    ref = ref.permute(0, 2, 1, 3).reshape(256, 384).numpy()
    assert np.array_equal(q, ref)


def test_quant_rows_against_torch_encoder():
    """Per-row ("per_Token") scales: amax of the whole row / 448, codes from torch's e4m3 cast."""
    g = torch.Generator().manual_seed(5)
    X = (torch.randn(9, 640, generator=g) * torch.exp(torch.randn(9, 1, generator=g) * 3)).to(torch.bfloat16)
    X[4] = 0  # an all-zero row takes scale 1
    X[6, 17] = -300.0  # one large entry sets the row's scale
    bits = X.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.quant_rows(bits)
    xf = X.float()
    amax = xf.abs().amax(-1)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    assert np.array_equal(s, sc.numpy())
    ref = (xf / sc[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    tab = oracle.e4m3_table()
    for r in range(9):
        assert np.abs(tab[q[r]]).max() == (0.0 if r == 4 else 448.0)
    assert tab[q[6, 17]] == -448.0


def test_quant_rows_is_1x128_on_single_group_rows():
    """With 128 columns a row is one 1x128 group: both quantisers must agree."""
    g = torch.Generator().manual_seed(6)
    X = (torch.randn(33, 128, generator=g) * 7).to(torch.bfloat16)
    bits = X.view(torch.int16).numpy().view(np.uint16)
    q1, s1 = oracle.quant_rows(bits)
    q2, s2 = oracle.quant_1x128(bits)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2[:, 0])


# ----------------------------------------------------------------- MXFP4

def test_e2m1_codes_golden():
    tab = oracle.e2m1_decode(np.arange(16))
    assert list(tab[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(tab[8:]) == [-v for v in tab[:8]]
    for v, code in _golden_rows("e2m1_codes.txt"):
        assert int(oracle.e2m1_encode([v])[0]) == int(code), (v, code)
    # every representable value encodes to itself
    assert np.array_equal(oracle.e2m1_encode(tab.astype(np.float32)), np.arange(16, dtype=np.uint8))


def test_mx_exponent_golden():
    for amax, e in _golden_rows("mx_exponent.txt"):
        assert oracle.mx_exponent(amax) == int(e), (amax, e)


def _mx4_numpy(xf):
    """Independent restatement of the MX FP4 rule on a float array [R, C]."""
    R, C = xf.shape
    g = xf.astype(np.float64).reshape(R, C // 32, 32)
    amax = np.abs(g).max(-1)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, 0).astype(np.int64)
    y = g / np.exp2(e)[..., None]
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    a = np.minimum(np.abs(y), 6.0)
    d = np.abs(a[..., None] - grid)
    best = d.argmin(-1)
    # ties: argmin keeps the lower index; move to the upper one when it is the even index
    upper = np.minimum(best + 1, 7)
    tie = (np.abs(a - grid[upper]) == d.min(-1)) & (upper != best) & (upper % 2 == 0)
    idx = np.where(tie, upper, best)
    code = (idx + np.where(np.signbit(y), 8, 0)).astype(np.uint8)
    return code.reshape(R, C), (e + 127).astype(np.uint8)


def test_quant_mx4_against_numpy_restatement():
    g = torch.Generator().manual_seed(13)
    X = (torch.randn(11, 256, generator=g) * torch.exp(torch.randn(11, 8, generator=g).repeat_interleave(32, 1) * 3))
    X = X.to(torch.bfloat16)
    X[3, 64:96] = 0  # an all-zero block
    X[5, 0:32] = torch.tensor([4.0, 2.5, 1.25, 0.75, 0.25, 5.0, 3.5, 1.75] * 4)  # block scale 1: exact ties
    bits = X.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.quant_mx4(bits)
    rq, rs = _mx4_numpy(X.float().numpy())
    assert np.array_equal(s, rs)
    assert np.array_equal(q, rq)
    assert s[3, 2] == 127 and not q[3, 64:96].any()
    # every non-zero block reaches 4 or 6 in magnitude (amax / X lies in [4, 8))
    tab = oracle.e2m1_decode(np.arange(16))
    for r in range(11):
        for b in range(8):
            if (r, b) != (3, 2):
                assert np.abs(tab[q[r, b * 32:(b + 1) * 32]]).max() in (4.0, 6.0)


def test_forward_mxfp4_against_dense_dequantised_reference():
    cfg = synth.CONFIGS["tiny"].with_(T=6, H=256, I=384, E=3, k=2)
    inp = synth.make_inputs(cfg, seed=14)
    xb, wrb = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"])
    q1, s1 = oracle.quant_mx4(synth.bf16_bits(inp["W_gate_up"]))
    q2, s2 = oracle.quant_mx4(synth.bf16_bits(inp["W_down"]))
    assert s1.shape == (cfg.E * 2 * cfg.I, cfg.H // 32) and s2.shape == (cfg.E * cfg.H, cfg.I // 32)
    got = oracle.moe_forward_mxfp4(xb, wrb, None, q1, s1, q2, s2, cfg.k)

    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
    deq = lambda q, s: grid[q] * np.repeat(np.exp2(s.astype(np.float64) - 127), 32, -1).reshape(q.shape)
    Wgu = deq(q1, s1.reshape(cfg.E, 2 * cfg.I, -1))
    Wd = deq(q2, s2.reshape(cfg.E, cfg.H, -1))
    xq, xs = _mx4_numpy(inp["x"].float().numpy())
    x = deq(xq, xs)
    ids, w, _ = oracle.route(xb, wrb, None, cfg.k)
    ref = np.zeros((cfg.T, cfg.H))
    I = cfg.I
    for t in range(cfg.T):
        for j in range(cfg.k):
            e = ids[t, j]
            g, u = Wgu[e, :I] @ x[t], Wgu[e, I:] @ x[t]
            a = (g / (1 + np.exp(-g)) * u).astype(np.float32)[None]
            aq, as_ = _mx4_numpy(a)
            ref[t] += w[t, j] * (Wd[e] @ deq(aq, as_)[0])
    assert _rel(got, ref) < 1e-12
    sub = np.array([5, 1], np.int64)
    assert np.array_equal(oracle.moe_forward_mxfp4(xb, wrb, None, q1, s1, q2, s2, cfg.k, tokens=sub), got[sub])


# ---------------------------------------------------------------- router

def test_router_order_hand_worked_cases():
    for case, H, bias, expected, triples in _golden_rows("router_order.txt"):
        H = int(H)
        x = np.zeros(H, np.float32)
        w = np.zeros(H, np.float32)
        for t in triples.split(","):
            h, xv, wv = t.split(":")
            x[int(h)] = float(xv)
            w[int(h)] = float(wv)
        b = None if bias == "none" else np.array([float(bias)], np.float32)
        got = oracle.router_logit(_bf16_bits_of(x), _bf16_bits_of(w), b, 0)
        assert got == np.float32(float(expected)), (case, got, expected)


def test_router_logit_within_fp32_bound_of_exact():
    g = torch.Generator().manual_seed(5)
    for H in (8, 128, 1000, 4096, 7168):
        x = torch.randn(H, generator=g).to(torch.bfloat16)
        w = (torch.randn(H, generator=g) / math.sqrt(H)).to(torch.bfloat16)
        xb, wb = x.view(torch.int16).numpy().view(np.uint16), w.view(torch.int16).numpy().view(np.uint16)
        got = float(oracle.router_logit(xb, wb))
        prod = _f(xb) * _f(wb)
        exact = prod.sum()
        # each partial adds at most ceil(H/256)*8 terms, then 5 butterfly levels
        depth = 8 * -(-H // 256) + 5
        bound = depth * 2.0 ** -24 * np.abs(prod).sum() * 1.01
        assert abs(got - exact) <= bound


def test_route_topk_against_fp64_softmax_topk_renorm():
    cfg = synth.CONFIGS["tiny"].with_(T=64, E=6, k=3)
    inp = synth.make_inputs(cfg, seed=1, weights=False)
    xb, wb = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"])
    ids, w, logits = oracle.route(xb, wb, None, cfg.k)
    # independent formulation: exact logits, softmax over all E, top-k, renormalise
    L = _f(xb) @ _f(wb).T
    P = np.exp(L - L.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    for t in range(cfg.T):
        order = sorted(range(cfg.E), key=lambda e: (-L[t, e], e))
        gaps = np.abs(np.diff(np.sort(L[t])[::-1][:cfg.k + 1]))
        if gaps.min() < 1e-5:
            continue  # near-tie: fp32 vs exact may legitimately differ
        assert list(ids[t]) == order[:cfg.k]
        ref = P[t, ids[t]] / P[t, ids[t]].sum()
        np.testing.assert_allclose(w[t], ref, rtol=1e-6)
        assert abs(w[t].sum() - 1.0) < 1e-12
        assert np.all(np.diff(w[t]) <= 0)
    # returned logits are the fixed-order fp32 values
    for t in (0, 7):
        for e in range(cfg.E):
            assert logits[t, e] == oracle.router_logit(xb[t], wb[e])
    # without renormalisation: the same ids, weights = the softmax over all E at those ids
    ids2, w2, _ = oracle.route(xb, wb, None, cfg.k, renormalize=False)
    assert np.array_equal(ids2, ids)
    for t in range(cfg.T):
        gaps = np.abs(np.diff(np.sort(L[t])[::-1][:cfg.k + 1]))
        if gaps.min() < 1e-5:
            continue
        np.testing.assert_allclose(w2[t], P[t, ids[t]], rtol=1e-6)
        assert w2[t].sum() < 1.0


def test_route_ties_go_to_lower_expert():
    H = 64
    x = np.ones((2, H), np.float32)
    W = np.zeros((4, H), np.float32)
    W[1] = W[2] = 0.5   # experts 1 and 2 tie for the top logit
    W[3] = 0.25
    ids, w, _ = oracle.route(_bf16_bits_of(x), _bf16_bits_of(W), None, 3)
    assert list(ids[0]) == [1, 2, 3]
    assert w[0, 0] == w[0, 1]
    # a bias breaks the tie and changes the weights too
    ids, w, _ = oracle.route(_bf16_bits_of(x), _bf16_bits_of(W), np.array([0, 0, 1, 0], np.float32), 2)
    assert list(ids[0]) == [2, 1]
    np.testing.assert_allclose(w[0], [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))], rtol=1e-12)


# ------------------------------------------------------------ align-sort

def test_align_sort_sizes_golden():
    for T, k, E, B, P, NB in _golden_rows("align_sort_sizes.txt"):
        assert oracle.align_sort_sizes(int(T), int(k), int(E), int(B)) == (int(P), int(NB))


def _sort_by_definition(ids, E, B):
    """Stable grouping of slots by expert with per-expert padding, from Python's sorted()."""
    T, k = ids.shape
    S = T * k
    slots = sorted(range(S), key=lambda s: (ids.flat[s], s))
    P, NB = oracle.align_sort_sizes(T, k, E, B)
    out, eids = [], []
    for e in range(E):
        seg = [s for s in slots if ids.flat[s] == e]
        pad = -(-len(seg) // B) * B
        out += seg + [S] * (pad - len(seg))
        eids += [e] * (pad // B)
    n = len(out)
    return np.array(out + [S] * (P - n), np.int32), np.array(eids + [-1] * (NB - len(eids)), np.int32), n


def test_align_sort_brute_force_all_small_routings():
    n_cases = 0
    for E in (1, 2, 3):
        for k in range(1, E + 1):
            choices = list(itertools.permutations(range(E), k))
            for T in (1, 2, 3):
                for routing in itertools.product(choices, repeat=T):
                    ids = np.array(routing, np.int32).reshape(T, k)
                    for B in (1, 2, 3, 4):
                        si, se, npp, cnt = oracle.align_sort(ids, E, B)
                        ri, re_, rn = _sort_by_definition(ids, E, B)
                        assert np.array_equal(si, ri) and np.array_equal(se, re_) and npp == rn
                        assert list(cnt) == [int((ids == e).sum()) for e in range(E)]
                        n_cases += 1
    assert n_cases > 1000


def test_align_sort_invariants_random():
    rng = np.random.default_rng(7)
    for T, k, E, B in [(100, 2, 8, 16), (33, 8, 256, 128), (4096, 8, 64, 64), (5, 1, 1, 128)]:
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        si, se, npp, cnt = oracle.align_sort(ids, E, B)
        check_sort_invariants(ids, E, B, si, se, npp, cnt)


# --------------------------------------------------------------- forward

def _dense_masked_reference(inp, k):
    """Masked dense MoE (every expert evaluated, weighted by the routing mask): the
    formulation the group-GEMM talk says grouped GEMMs replace.  fp64 numpy."""
    x = _f(synth.bf16_bits(inp["x"]))
    Wr = _f(synth.bf16_bits(inp["W_router"]))
    Wgu = _f(synth.bf16_bits(inp["W_gate_up"]))
    Wd = _f(synth.bf16_bits(inp["W_down"]))
    E, twoI, H = Wgu.shape
    I = twoI // 2
    ids, w, _ = oracle.route(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"]),
                             None if inp["bias"] is None else inp["bias"].numpy(), k)
    mask = np.zeros((x.shape[0], E))
    for t in range(x.shape[0]):
        mask[t, ids[t]] = w[t]
    out = np.zeros_like(x)
    for e in range(E):
        g = x @ Wgu[e, :I].T
        u = x @ Wgu[e, I:].T
        a = g / (1 + np.exp(-g)) * u
        out += mask[:, e:e + 1] * (a @ Wd[e].T)
    return out


def _oracle_bf16(inp, k, tokens=None):
    b = None if inp["bias"] is None else inp["bias"].numpy()
    return oracle.moe_forward_bf16(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"]), b,
                                   synth.bf16_bits(inp["W_gate_up"]), synth.bf16_bits(inp["W_down"]), k, tokens)


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("T,E,k,bias", [(16, 4, 2, None), (1, 1, 1, None), (3, 2, 2, "normal"),
                                        (17, 5, 2, "normal"), (9, 5, 5, None)])
def test_forward_equals_masked_dense(T, E, k, bias):
    cfg = synth.CONFIGS["tiny"].with_(T=T, E=E, k=k, bias=bias, bias_param=0.5)
    inp = synth.make_inputs(cfg, seed=2)
    assert _rel(_oracle_bf16(inp, k), _dense_masked_reference(inp, k)) < 1e-12


def test_forward_e1_k1_is_plain_swiglu_mlp():
    cfg = synth.CONFIGS["tiny"].with_(T=12, E=1, k=1)
    inp = synth.make_inputs(cfg, seed=3)
    x = inp["x"].double()
    Wg, Wu = inp["W_gate_up"][0, :cfg.I].double(), inp["W_gate_up"][0, cfg.I:].double()
    Wd = inp["W_down"][0].double()
    ref = torch.nn.functional.linear(torch.nn.functional.silu(x @ Wg.T) * (x @ Wu.T), Wd)
    assert _rel(_oracle_bf16(inp, 1), ref.numpy()) < 1e-12


def test_forward_k_equals_e_is_softmax_mixture():
    cfg = synth.CONFIGS["tiny"].with_(T=10, E=3, k=3)
    inp = synth.make_inputs(cfg, seed=4)
    x = inp["x"].double()
    logits = x @ inp["W_router"].double().T
    p = torch.softmax(logits, -1)
    ref = torch.zeros_like(x)
    for e in range(3):
        Wg, Wu = inp["W_gate_up"][e, :cfg.I].double(), inp["W_gate_up"][e, cfg.I:].double()
        ref += p[:, e:e + 1] * (torch.nn.functional.silu(x @ Wg.T) * (x @ Wu.T)) @ inp["W_down"][e].double().T
    assert _rel(_oracle_bf16(inp, 3), ref.numpy()) < 1e-6  # logits fp32 vs fp64 only


def test_forward_unused_expert_weights_never_read():
    cfg = synth.CONFIGS["tiny"].with_(T=8, E=6, k=2)
    inp = synth.make_inputs(cfg, seed=5)
    ids, _, _ = oracle.route(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"]), None, 2)
    unused = sorted(set(range(6)) - set(ids.ravel().tolist()))
    assert unused, "seed should leave an expert without tokens"
    ref = _oracle_bf16(inp, 2)
    for e in unused:
        inp["W_gate_up"][e] = float("nan")
        inp["W_down"][e] = float("nan")
    got = _oracle_bf16(inp, 2)
    assert np.array_equal(got, ref)


def test_forward_token_permutation_and_subset():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg, seed=6)
    full = _oracle_bf16(inp, 2)
    perm = torch.randperm(cfg.T, generator=torch.Generator().manual_seed(0))
    inp2 = dict(inp, x=inp["x"][perm].contiguous())
    assert np.array_equal(_oracle_bf16(inp2, 2), full[perm.numpy()])
    sub = np.array([0, 5, 15], np.int64)
    assert np.array_equal(_oracle_bf16(inp, 2, sub), full[sub])


@pytest.mark.parametrize("T,H,I,E,k,bias", [(37, 256, 384, 6, 3, "normal"), (20, 128, 256, 4, 2, None),
                                            (50, 256, 256, 16, 4, "zipf"), (5, 128, 128, 1, 1, None),
                                            (40, 128, 256, 3, 3, None)])
def test_forward_expert_major_bit_identical_to_per_token(T, H, I, E, k, bias):
    """The expert-by-expert evaluation computes the same fp64 sums in the same order as the
    per-token loop, in all four number formats: equal bit for bit (token lists with repeats,
    any order, experts with one slot and with more than one 16-slot group)."""
    cfg = synth.MoEConfig("em", T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5 if bias == "normal" else 1.2)
    inp = synth.make_inputs(cfg, seed=7)
    h = {n: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.numpy()))
         for n, v in inp.items()}
    toks = np.array([T - 1, 0, 3 % T, 3 % T] + list(range(T)), np.int64)
    args = (h["x"], h["W_router"], h["bias"])
    runs = [(oracle.moe_forward_bf16, (h["W_gate_up"], h["W_down"]))]
    q1, s1 = oracle.quant_128x128(h["W_gate_up"])
    q2, s2 = oracle.quant_128x128(h["W_down"])
    runs.append((oracle.moe_forward_fp8, (q1, s1, q2, s2)))
    q1, s1 = oracle.quant_rows(h["W_gate_up"])
    q2, s2 = oracle.quant_rows(h["W_down"])
    runs.append((oracle.moe_forward_fp8_token, (q1, s1, q2, s2)))
    q1, s1 = oracle.quant_mx4(h["W_gate_up"])
    q2, s2 = oracle.quant_mx4(h["W_down"])
    runs.append((oracle.moe_forward_mxfp4, (q1, s1, q2, s2)))
    for fn, w in runs:
        a = fn(*args, *w, k, toks)
        b = fn(*args, *w, k, toks, expert_major=True)
        assert np.array_equal(a.view(np.uint64), b.view(np.uint64)), fn.__name__


def test_forward_fp8_against_dense_dequantised_reference():
    """FP8 path vs an independent dense formulation: torch's e4m3 encoder for
    the 1x128 re-quantisation of the SwiGLU output, numpy matmuls."""
    cfg = synth.CONFIGS["tiny"].with_(T=6, H=256, I=256, E=3, k=2)
    inp = synth.make_inputs(cfg, seed=7)
    xb, wrb = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"])
    qgu, s1 = oracle.quant_128x128(synth.bf16_bits(inp["W_gate_up"]))
    qd, s2 = oracle.quant_128x128(synth.bf16_bits(inp["W_down"]))
    got = oracle.moe_forward_fp8(xb, wrb, None, qgu, s1, qd, s2, cfg.k)

    tab = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    Wgu = tab[qgu] * np.repeat(np.repeat(s1, 128, 0), 128, 1).reshape(qgu.shape)
    Wd = tab[qd] * np.repeat(np.repeat(s2, 128, 0), 128, 1).reshape(qd.shape)
    xq, xs = oracle.quant_1x128(xb)
    x = tab[xq] * np.repeat(xs, 128, 1)
    ids, w, _ = oracle.route(xb, wrb, None, cfg.k)
    ref = np.zeros((cfg.T, cfg.H))
    I = cfg.I
    for t in range(cfg.T):
        for j in range(cfg.k):
            e = ids[t, j]
            g, u = Wgu[e, :I] @ x[t], Wgu[e, I:] @ x[t]
            a = torch.from_numpy(g / (1 + np.exp(-g)) * u).float().reshape(-1, 128)
            amax = a.abs().amax(-1, keepdim=True)
            sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
            aq = (a / sc).clamp(-448, 448).to(torch.float8_e4m3fn).double() * sc.double()
            ref[t] += w[t, j] * (Wd[e] @ aq.reshape(-1).numpy())
    assert _rel(got, ref) < 1e-12


def test_forward_fp8_token_against_dense_dequantised_reference():
    """Per-token FP8 path vs an independent dense formulation: scales broadcast
    by row with numpy, torch's e4m3 encoder for the per-token re-quantisation
    of the SwiGLU output, numpy matmuls."""
    cfg = synth.CONFIGS["tiny"].with_(T=7, H=256, I=384, E=3, k=2)
    inp = synth.make_inputs(cfg, seed=8)
    xb, wrb = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"])
    qgu, s1 = oracle.quant_rows(synth.bf16_bits(inp["W_gate_up"]))
    qd, s2 = oracle.quant_rows(synth.bf16_bits(inp["W_down"]))
    assert s1.shape == (cfg.E * 2 * cfg.I,) and s2.shape == (cfg.E * cfg.H,)
    got = oracle.moe_forward_fp8_token(xb, wrb, None, qgu, s1, qd, s2, cfg.k)

    tab = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    Wgu = tab[qgu] * s1.astype(np.float64).reshape(cfg.E, 2 * cfg.I, 1)
    Wd = tab[qd] * s2.astype(np.float64).reshape(cfg.E, cfg.H, 1)
    xf = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).float()
    xs = xf.abs().amax(-1, keepdim=True) / 448.0
    x = (xf / xs).to(torch.float8_e4m3fn).double().numpy() * xs.double().numpy()
    ids, w, _ = oracle.route(xb, wrb, None, cfg.k)
    ref = np.zeros((cfg.T, cfg.H))
    I = cfg.I
    for t in range(cfg.T):
        for j in range(cfg.k):
            e = ids[t, j]
            g, u = Wgu[e, :I] @ x[t], Wgu[e, I:] @ x[t]
            a = torch.from_numpy(g / (1 + np.exp(-g)) * u).float()
            sc = a.abs().amax() / 448.0
            aq = (a / sc).to(torch.float8_e4m3fn).double() * sc.double()
            ref[t] += w[t, j] * (Wd[e] @ aq.numpy())
    assert _rel(got, ref) < 1e-12
    sub = np.array([6, 0, 3], np.int64)
    assert np.array_equal(oracle.moe_forward_fp8_token(xb, wrb, None, qgu, s1, qd, s2, cfg.k, tokens=sub), got[sub])


def test_forward_fp8_token_close_to_bf16_layer():
    """Quantisation only perturbs the layer: the per-token FP8 output stays
    within the e4m3 error budget of the bf16 layer (and is not identical)."""
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg, seed=9)
    xb, wrb = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"])
    gub, db = synth.bf16_bits(inp["W_gate_up"]), synth.bf16_bits(inp["W_down"])
    qgu, s1 = oracle.quant_rows(gub)
    qd, s2 = oracle.quant_rows(db)
    got = oracle.moe_forward_fp8_token(xb, wrb, None, qgu, s1, qd, s2, cfg.k)
    ref = oracle.moe_forward_bf16(xb, wrb, None, gub, db, cfg.k)
    r = _rel(got, ref)
    assert 1e-3 < r < 0.15, r  # three e4m3 roundings (x, W, h), each about 3 % relative RMS


def _autograd_reference(inp, ids, dout, k):
    """Plain fp64 torch model of the layer with the routing choice fixed to `ids`."""
    X = inp["x"].double().clone().requires_grad_()
    Wr = inp["W_router"].double().clone().requires_grad_()
    b = (inp["bias"].double() if inp["bias"] is not None else torch.zeros(Wr.shape[0], dtype=torch.float64))
    b = b.clone().requires_grad_()
    Wgu = inp["W_gate_up"].double().clone().requires_grad_()
    Wd = inp["W_down"].double().clone().requires_grad_()
    I = Wgu.shape[1] // 2
    L = X @ Wr.T + b
    ids_t = torch.from_numpy(ids.astype(np.int64))
    w = torch.softmax(L.gather(1, ids_t), dim=1)
    out = []
    for t in range(X.shape[0]):
        acc = torch.zeros(X.shape[1], dtype=torch.float64)
        for j in range(k):
            e = int(ids[t, j])
            h = torch.nn.functional.silu(Wgu[e, :I] @ X[t]) * (Wgu[e, I:] @ X[t])
            acc = acc + w[t, j] * (Wd[e] @ h)
        out.append(acc)
    out = torch.stack(out)
    (out * dout.double()).sum().backward()
    return {"dx": X.grad, "dW_gate_up": Wgu.grad, "dW_down": Wd.grad, "dW_router": Wr.grad, "dbias": b.grad}


@pytest.mark.parametrize("shape", [(9, 96, 80, 4, 2, "normal"), (5, 64, 48, 7, 3, None), (6, 32, 32, 1, 1, None)],
                         ids=["t9_e4_k2_bias", "t5_e7_k3", "e1_k1"])
def test_backward_against_torch_autograd(shape):
    T, H, I, E, k, bias = shape
    cfg = synth.CONFIGS["tiny"].with_(T=T, H=H, I=I, E=E, k=k, bias=bias, bias_param=0.5)
    inp = synth.make_inputs(cfg, seed=15)
    dout = (torch.randn(T, H, generator=torch.Generator().manual_seed(16))).to(torch.bfloat16)
    xb, wrb = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["W_router"])
    b = None if inp["bias"] is None else inp["bias"].numpy()
    got = oracle.moe_backward_bf16(xb, wrb, b, synth.bf16_bits(inp["W_gate_up"]), synth.bf16_bits(inp["W_down"]),
                                   synth.bf16_bits(dout), k)
    ids, _, _ = oracle.route(xb, wrb, b, k)
    ref = _autograd_reference(inp, ids, dout, k)
    for name in ("dx", "dW_gate_up", "dW_down", "dW_router", "dbias"):
        r = ref[name].numpy()
        if not np.abs(r).max() > 1e-30:  # k = 1: the softmax over one logit passes no gradient
            assert np.abs(got[name]).max() < 1e-30, name
            continue
        # the oracle's softmax weights come from the fp32 logits that decide the routing: ~1e-7 relative
        assert _rel(got[name], r) < 1e-5, (name, _rel(got[name], r))
    # experts without tokens get exactly zero weight gradients
    used = set(ids.ravel().tolist())
    for e in range(E):
        if e not in used:
            assert not got["dW_gate_up"][e].any() and not got["dW_down"][e].any()


# ------------------------------------------------------------ heuristics

def test_heuristics_golden():
    for kind, token, topk, expert, inter, model, units, bm, expected in _golden_rows("heuristics.txt"):
        token, topk, expert, inter, model, units, bm, expected = map(
            int, (token, topk, expert, inter, model, units, bm, expected))
        if kind == "bsm":
            assert heuristics.block_size_m(token, topk, expert, inter, units) == expected
        else:
            assert heuristics.ksplit(token, topk, expert, inter, model, units, bm) == expected
