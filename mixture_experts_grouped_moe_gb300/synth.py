"""Seeded synthetic inputs for the fused MoE layer.

This module only draws random tensors.  It holds none of the layer's
arithmetic (no routing, sorting, GEMM, activation or quantisation), so both
the CUDA path and the CPU oracle can take their inputs from it without
sharing any of the method.

Workloads (sizes from the fused-MoE pages' Mixtral-8x7B and fine-grained
DeepSeek-style shapes; tensors are random, there are no trained weights):

  tiny              T=16   H=128  I=256   E=4   k=2
  mixtral_decode    T=32   H=4096 I=14336 E=8   k=2
  mixtral_prefill   T=8192 H=4096 I=14336 E=8   k=2  router bias ~ N(0, var 0.5)
  mixtral_fp8       T=4096 H=4096 I=14336 E=8   k=2  (block-scaled FP8, quantised by the path)
  mixtral_fp8_token T=4096 H=4096 I=14336 E=8   k=2  (per-token FP8)
  mixtral_fp8_token_decode  T=32, same shapes (per-token FP8)
  mixtral_mxfp4_decode      T=32, same shapes (MXFP4, per 1x32)
  mixtral_mxfp4             T=4096, same shapes (MXFP4)
  finegrained_zipf  T=4096 H=7168 I=2048  E=256 k=8  Zipf(s=1.2) router bias

Distributions: x ~ N(0, 1); W_router, W_gate, W_up ~ N(0, 1/H);
W_down ~ N(0, 1/I); each drawn in fp32 and rounded to bf16 (RNE).  Draw
order is fixed: x, W_router, bias, then W_gate[e] and W_up[e] for e = 0..E-1,
then W_down[e] for e = 0..E-1.  W_gate_up[e] is [W_gate[e]; W_up[e]] (gate rows first).

The Zipf bias gives each expert a rank r (1..E) from a seeded permutation and
sets bias_e = -s * beta * ln(r_e): the log of a Zipf(s) mass up to a
constant, so that a few experts take a large share of the slots and the
tail experts receive none.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    bias: str | None = None  # None | "normal" | "zipf"
    bias_param: float = 0.0  # variance for "normal", exponent s for "zipf"
    zipf_beta: float = 1.0
    dtype: str = "bf16"      # "bf16" | "fp8" (block-scaled e4m3) | "fp8_token" (per-token e4m3) | "mxfp4"

    @property
    def S(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": MoEConfig("tiny", T=16, H=128, I=256, E=4, k=2),
    "mixtral_decode": MoEConfig("mixtral_decode", T=32, H=4096, I=14336, E=8, k=2),
    "mixtral_prefill": MoEConfig("mixtral_prefill", T=8192, H=4096, I=14336, E=8, k=2,
                                 bias="normal", bias_param=0.5),
    "mixtral_fp8": MoEConfig("mixtral_fp8", T=4096, H=4096, I=14336, E=8, k=2, dtype="fp8"),
    "mixtral_fp8_token": MoEConfig("mixtral_fp8_token", T=4096, H=4096, I=14336, E=8, k=2, dtype="fp8_token"),
    "mixtral_fp8_token_decode": MoEConfig("mixtral_fp8_token_decode", T=32, H=4096, I=14336, E=8, k=2,
                                          dtype="fp8_token"),
    "mixtral_mxfp4_decode": MoEConfig("mixtral_mxfp4_decode", T=32, H=4096, I=14336, E=8, k=2, dtype="mxfp4"),
    "mixtral_mxfp4": MoEConfig("mixtral_mxfp4", T=4096, H=4096, I=14336, E=8, k=2, dtype="mxfp4"),
    "finegrained_zipf": MoEConfig("finegrained_zipf", T=4096, H=7168, I=2048, E=256, k=8,
                                  bias="zipf", bias_param=1.2),
}


def _randn_bf16(shape, std, gen, device):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def make_inputs(cfg: MoEConfig, seed: int = 0, device="cpu", weights: bool = True) -> dict:
    """Draw the layer's inputs.  Returns a dict of torch tensors on `device`:

    x [T,H] bf16, W_router [E,H] bf16, bias [E] fp32 or None,
    W_gate_up [E,2I,H] bf16, W_down [E,H,I] bf16 (weights only if `weights`).
    The same seed on the same device type gives the same bytes.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    T, H, I, E = cfg.T, cfg.H, cfg.I, cfg.E
    out = {}
    out["x"] = _randn_bf16((T, H), 1.0, gen, device)
    out["W_router"] = _randn_bf16((E, H), 1.0 / math.sqrt(H), gen, device)
    if cfg.bias == "normal":
        out["bias"] = torch.randn((E,), generator=gen, device=device) * math.sqrt(cfg.bias_param)
    elif cfg.bias == "zipf":
        perm = torch.randperm(E, generator=gen, device=device)
        rank = perm.to(torch.float64) + 1.0
        out["bias"] = (-cfg.bias_param * cfg.zipf_beta * torch.log(rank)).to(torch.float32)
    else:
        out["bias"] = None
    if not weights:
        return out
    wgu = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=device)
    wd = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
    sg = 1.0 / math.sqrt(H)
    sd = 1.0 / math.sqrt(I)
    for e in range(E):
        wgu[e, :I] = _randn_bf16((I, H), sg, gen, device)
        wgu[e, I:] = _randn_bf16((I, H), sg, gen, device)
    for e in range(E):
        wd[e] = _randn_bf16((H, I), sd, gen, device)
    out["W_gate_up"] = wgu
    out["W_down"] = wd
    return out


def token_sample(T: int, n: int, seed: int = 1234) -> torch.Tensor:
    """A seeded, sorted subset of n token indices out of T (all if n >= T)."""
    if n >= T:
        return torch.arange(T, dtype=torch.int64)
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(T, generator=g)[:n].sort().values


def bf16_bits(t: torch.Tensor):
    """A host numpy uint16 view of a bf16 tensor's bits (copies to host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
