"""Host heuristics of the fused-MoE pages, restated -- TEST INFRASTRUCTURE ONLY.

AITER page, section 3.3 (get_block_size_M): for each candidate block size
BM, the tile-group count is the page's expression
tgN * (max_padded + BM - 1) // BM, evaluated as Python evaluates it (* and
// bind equally and group left to right: (tgN * (max_padded + BM - 1)) // BM,
not tgN * ceil(max_padded / BM), which the page's comment "total tile groups"
might suggest), with tgN = ceil(inter_dim / 128) and max_padded =
token*topk + expert*BM - topk; then the rounds ceil(tiles / units) each
compute unit runs and the units left idle in the last round,
units - tiles % units; the candidate with the fewest rounds, then the fewest
idle units, wins (a stable sort on those two keys: a full tie keeps the
earlier candidate).

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
        tiles = (tgN * (max_padded + bm - 1)) // bm
        rounds = -(-tiles // units)
        idle = units - tiles % units
        scored.append((rounds, idle, bm))
    return sorted(scored, key=lambda r: r[:2])[0][2]


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


# ---------------------------------------------------------------------------
# GB300 analogues used by the library's planner for the swap-AB (decode) kernels, restated
# here from their definitions (the page's two rules with this GPU's tiles and SM count):
#
#  * block size: get_block_size_M's choice (fewest rounds, then fewest idle units, a full tie
#    keeping the earlier candidate) over {16, 32, 64, 128} ({16, 32, 64} for MXFP4) with the
#    swap kernels' stage-1 tile count, experts_that_can_hold_a_slot * inter_dim / 128, which
#    does not depend on the block size;
#  * stage-2 K split: get_ksplit's split_max = ceil(units / tiles) when the stage-2 tiles
#    (experts * ceil(model_dim / 256)) leave units idle, taking the smallest divisor of the
#    K blocks (up to 16) that reaches it, else the largest divisor up to 16; no split when the
#    tiles already cover the units.


def swap_block_m(tokens: int, topk: int, experts: int, inter_dim: int, units: int, mxfp4: bool = False) -> int:
    e_act = min(tokens * topk, experts)
    scored = []
    for bm in ((16, 32, 64) if mxfp4 else (16, 32, 64, 128)):
        tiles = e_act * (inter_dim // 128)
        scored.append(((tiles + units - 1) // units, units - tiles % units, bm))
    return sorted(scored, key=lambda r: r[:2])[0][2]


def swap_split_k(tokens: int, topk: int, experts: int, model_dim: int, kblocks: int, units: int) -> int:
    tiles = min(tokens * topk, experts) * (-(-model_dim // 256))
    if tiles >= units:
        return 1
    need = -(-units // tiles)
    divisors = [d for d in range(2, min(16, kblocks) + 1) if kblocks % d == 0]
    reaching = [d for d in divisors if d >= need]
    if reaching:
        return reaching[0]
    return divisors[-1] if divisors else 1
