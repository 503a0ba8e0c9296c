"""Host heuristics of the fused-MoE pages, restated -- TEST INFRASTRUCTURE ONLY.

AITER page, section 3.3 (get_block_size_M): for each candidate block size
BM, count the tile groups ceil(inter_dim / 128) * ceil(max_padded / BM)
with max_padded = token*topk + expert*BM - topk, then the rounds
ceil(tiles / units) each compute unit runs and the units left idle in the
last round, units - tiles % units; pick the candidate with the fewest
rounds, then the fewest idle units (then the smaller BM).

AITER page, section 3.4 (get_ksplit): no split when token*topk > expert or
when the tile groups already cover every unit; otherwise the largest
i <= ceil(units / tiles), i >= 2, that divides model_dim with
(model_dim / i) % 256 == 0, else no split.  The page leaves tgN and tgM
undefined in that function; read here as tgN = ceil(inter_dim / 128) (the
same tileN as section 3.3) and tgM = ceil(token*topk / BM).

`units` is the GPU's compute-unit count (the streaming-multiprocessor count
on this hardware).
"""
from __future__ import annotations


def block_size_m(token: int, topk: int, expert: int, inter_dim: int, units: int,
                 candidates=(32, 64, 128)) -> int:
    tgN = -(-inter_dim // 128)
    scored = []
    for bm in candidates:
        max_padded = token * topk + expert * bm - topk
        tiles = tgN * (-(-max_padded // bm))
        rounds = -(-tiles // units)
        idle = units - tiles % units
        scored.append((rounds, idle, bm))
    scored.sort()
    return scored[0][2]


def ksplit(token: int, topk: int, expert: int, inter_dim: int, model_dim: int, units: int,
           block_m: int) -> int:
    if token * topk > expert:
        return 0
    tgN = -(-inter_dim // 128)
    tgM = -(-(token * topk) // block_m)
    tiles = tgN * tgM
    if tiles >= units:
        return 0
    split_max = -(-units // tiles)
    for i in range(split_max, 1, -1):
        if model_dim % i == 0 and (model_dim // i) % 256 == 0:
            return i
    return 0
