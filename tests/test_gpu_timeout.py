"""The bounded device waits give up with a status, and the GPU stays usable.

The one-launch decode kernel's stage-2 tiles wait, on a global counter, for
every stage-1 epilogue to have stored its part of the intermediate.  With
the test option unsatisfiable_h_wait that wait's target is one more than the
number of epilogues, so nothing ever satisfies it: after h_wait_limit_us the
waiting thread records MOE_ERR_TIMEOUT in the workspace status word and
raises its CTA's abort flag; the CTA retires the copies it announced but will
not issue, waits for the copies and MMAs already in flight, frees its tensor
memory and returns.  The host reads the status; the next ordinary call on the
same GPU and workspace must give the oracle's result.  No fault, trap or
endless loop is involved: the wait is bounded and simply runs out.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_grouped_moe_gb300 import synth
from moe_checks import check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_moe_gb300 import build
    build.build()
    from mixture_experts_grouped_moe_gb300 import moe as m
    m.load()
    return m


@pytest.mark.parametrize("T,H,I,E,k,split_k", [(24, 128, 256, 4, 2, 0), (32, 512, 1024, 8, 2, 2)],
                         ids=["tiny", "split2"])
def test_wait_runs_out_then_next_call_is_clean(moe, T, H, I, E, k, split_k):
    cfg = synth.MoEConfig("timeout", T=T, H=H, I=I, E=E, k=k)
    inp = synth.make_inputs(cfg, seed=21, device="cuda")
    layer = moe.FusedMoE(moe.MOE_BF16, T, H, I, E, k, 0, split_k)
    assert layer.plan.mode == moe.MOE_MODE_SWAP   # the one-launch decode path (the default there)
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    limit_us = 20000
    stuck = moe.Options(unsatisfiable_h_wait=1, h_wait_limit_us=limit_us)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    layer(inp["x"], inp, out, options=stuck)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert layer.status() == moe.MOE_ERR_TIMEOUT
    assert limit_us * 1e-6 <= elapsed < 1.5, elapsed   # it waited its limit, not the 2 s default

    # the next ordinary call on the same workspace: status cleared, the definition's result
    layer(inp["x"], inp, out)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    host = {n: (None if v is None else (synth.bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()))
            for n, v in inp.items()}
    ref = oracle.moe_forward_bf16(host["x"], host["W_router"], host["bias"], host["W_gate_up"], host["W_down"], k)
    check_rows(out.float().cpu().numpy(), ref, 5e-3, label="after timeout")
    # and it is the same result as from a fresh workspace
    fresh = moe.FusedMoE(moe.MOE_BF16, T, H, I, E, k, 0, split_k)
    out2 = torch.empty_like(out)
    fresh(inp["x"], inp, out2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert np.isfinite(out.float().cpu().numpy()).all()
