"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every function include/moe.h declares, the host-only helpers
(buffer sizes, the pages' block-size and K-split rules, the planner) agree
with the oracle's restatement and the pages' worked sizes, and invalid
calls are rejected before anything touches CUDA."""
import os
import re

import pytest

from mixture_experts_grouped_moe_gb300 import build as moe_build
from oracle import heuristics
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def moe():
    moe_build.build()
    from mixture_experts_grouped_moe_gb300 import moe as m
    m.load()
    return m


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_symbols_exported(moe):
    names = _declared_functions()
    assert len(names) >= 15
    lib = moe.load()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.EXPORTED) == names


def test_status_strings(moe):
    assert moe.status_string(0) == "ok"
    assert "workspace" in moe.status_string(moe.MOE_ERR_WORKSPACE)
    assert moe.status_string(-99) == "unknown status"
    assert moe.moe_version() >= 100


def test_align_sort_sizes_match_pages(moe):
    for (T, k, E, B) in [(16, 2, 4, 16), (8192, 2, 8, 128), (4096, 8, 256, 128), (1, 1, 1, 1), (0, 2, 8, 16)]:
        assert moe.moe_align_sort_sizes(T, k, E, B) == oracle.align_sort_sizes(T, k, E, B)
    with pytest.raises(moe.MoEError):
        moe.moe_align_sort_sizes(4, 0, 8, 16)


@pytest.mark.parametrize("units", [80, 148, 152, 160, 304])
def test_heuristics_match_restatement(moe, units):
    shapes = [(16, 2, 4, 256, 128), (32, 2, 8, 14336, 4096), (8192, 2, 8, 14336, 4096),
              (4096, 2, 8, 14336, 4096), (4096, 8, 256, 2048, 7168), (1, 1, 8, 14336, 4096),
              (2, 2, 8, 256, 4096), (3, 1, 16, 1024, 2048)]
    for token, topk, expert, inter, model in shapes:
        assert moe.moe_block_size_m_heuristic(token, topk, expert, inter, units) == \
            heuristics.block_size_m(token, topk, expert, inter, units)
        for bm in (16, 32, 64, 128):
            assert moe.moe_ksplit_heuristic(token, topk, expert, inter, model, units, bm) == \
                heuristics.ksplit(token, topk, expert, inter, model, units, bm)


def test_plan_without_gpu(moe):
    p = moe.moe_plan(moe.MOE_BF16, 32, 4096, 14336, 8, 2, num_sms=152)
    assert p.mode == moe.MOE_MODE_SWAP and p.block_m == 16
    assert p.split_k2 > 1 and (14336 // 64) % p.split_k2 == 0
    assert (p.max_padded, p.max_blocks) == oracle.align_sort_sizes(32, 2, 8, 16)
    p = moe.moe_plan(moe.MOE_BF16, 8192, 4096, 14336, 8, 2, num_sms=152)
    assert p.mode == moe.MOE_MODE_GROUPED and p.block_m == 128 and p.split_k2 == 1
    assert p.workspace_bytes > 17406 * (4096 + 14336) * 2
    p = moe.moe_plan(moe.MOE_FP8_BLOCK128, 4096, 4096, 14336, 8, 2, num_sms=152)
    assert p.mode == moe.MOE_MODE_GROUPED
    p = moe.moe_plan(moe.MOE_FP8_TOKEN, 32, 4096, 14336, 8, 2, num_sms=152)
    assert p.mode == moe.MOE_MODE_SWAP and (14336 // 128) % p.split_k2 == 0 and p.split_k2 > 1
    p = moe.moe_plan(moe.MOE_MXFP4, 32, 4096, 14336, 8, 2, num_sms=152)
    assert p.mode == moe.MOE_MODE_SWAP and p.block_m == 16 and (14336 // 256) % p.split_k2 == 0
    with pytest.raises(moe.MoEError):
        moe.moe_plan(moe.MOE_MXFP4, 32, 4096, 14336, 8, 2, block_m=128, num_sms=152)  # segments above 64 rows
    p = moe.moe_plan(moe.MOE_MXFP4, 65, 4096, 14336, 8, 2, num_sms=152)
    assert p.mode == moe.MOE_MODE_GROUPED and p.block_m == 128 and p.split_k2 == 1
    p = moe.moe_plan(moe.MOE_FP8_TOKEN, 4096, 4096, 14336, 8, 2, num_sms=152)
    assert p.mode == moe.MOE_MODE_GROUPED and p.block_m == 128
    p = moe.moe_plan(moe.MOE_BF16, 128, 256, 256, 4, 2, block_m=32, split_k=2, num_sms=152)
    assert p.mode == moe.MOE_MODE_SWAP and p.block_m == 32 and p.split_k2 == 2
    p = moe.moe_plan(moe.MOE_BF16, 129, 256, 256, 4, 2, num_sms=152)
    assert p.mode == moe.MOE_MODE_GROUPED


@pytest.mark.parametrize("args,status", [
    ((0, 16, 100, 256, 4, 2), -2),      # H not a multiple of 128
    ((0, 16, 128, 200, 4, 2), -2),      # I not a multiple of 128
    ((0, 16, 128, 256, 4, 5), -2),      # k > E
    ((0, 16, 128, 256, 2000, 2), -2),   # E > 1024
    ((0, 16, 128, 256, 64, 33), -2),    # k > 32
    ((4, 16, 128, 256, 4, 2), -1),      # unknown dtype
    ((3, 16, 128, 256, 4, 2), -2),      # MXFP4: H not a multiple of 256
    ((0, -1, 128, 256, 4, 2), -1),      # negative T
])
def test_plan_rejects_invalid(moe, args, status):
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan(*args, num_sms=152)
    assert ei.value.status == status


@pytest.mark.parametrize("units", [80, 148, 152, 304])
def test_swap_planner_follows_the_gb300_rules(moe, units):
    """moe_plan's automatic block size and stage-2 split in swap mode equal the restated GB300
    analogues of the page's get_block_size_M and get_ksplit (oracle/heuristics.py)."""
    for dtype, kgran, tmax in ((moe.MOE_BF16, 64, 128), (moe.MOE_FP8_TOKEN, 128, 128), (moe.MOE_MXFP4, 256, 64)):
        for T in (1, 2, 3, 8, 17, 32, 64, tmax):
            for (H, I, E, k) in ((4096, 14336, 8, 2), (7168, 2048, 256, 8), (1024, 768, 16, 4), (512, 256, 3, 3)):
                if dtype == moe.MOE_MXFP4 and (H % 256 or I % 256):
                    continue
                p = moe.moe_plan(dtype, T, H, I, E, k, num_sms=units)
                assert p.mode == moe.MOE_MODE_SWAP
                assert p.block_m == heuristics.swap_block_m(T, k, E, I, units, dtype == moe.MOE_MXFP4)
                assert p.split_k2 == heuristics.swap_split_k(T, k, E, H, I // kgran, units), (dtype, T, H, I, E, k)
    # the measured choices for the Mixtral decode shapes on 152 SMs
    if units == 152:
        assert moe.moe_plan(moe.MOE_BF16, 32, 4096, 14336, 8, 2, num_sms=152).split_k2 == 2
        assert moe.moe_plan(moe.MOE_BF16, 1, 4096, 14336, 8, 2, num_sms=152).split_k2 == 7
        assert moe.moe_plan(moe.MOE_BF16, 32, 4096, 14336, 8, 2, num_sms=152).block_m == 16


def test_plan_rejects_bad_options(moe):
    with pytest.raises(moe.MoEError):   # grouped mode supports block 128 only
        moe.moe_plan(moe.MOE_BF16, 512, 256, 256, 4, 2, block_m=64, num_sms=152)
    with pytest.raises(moe.MoEError):   # swap mode: block must be a multiple of 16
        moe.moe_plan(moe.MOE_BF16, 16, 256, 256, 4, 2, block_m=24, num_sms=152)
    with pytest.raises(moe.MoEError):   # split must divide I/64
        moe.moe_plan(moe.MOE_BF16, 16, 256, 256, 4, 2, split_k=3, num_sms=152)


def test_entry_points_reject_null_before_cuda(moe):
    lib = moe.load()
    # null required pointers: rejected on the host, nothing launched
    assert lib.moe_fused_forward(0, None, None, None, None, None, None, None, 16, 128, 256, 4, 2, 0, 0,
                                 None, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_fused_forward(1, 16, 16, None, 16, None, 16, None, 16, 128, 256, 4, 2, 0, 0,
                                 16, 256, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG  # FP8 needs scales
    assert lib.moe_route_topk(None, None, None, 4, 128, 4, 2, 1, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk(16, 16, None, 4, 12, 4, 2, 1, 16, 16, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk(16, 16, None, 4, 128, 4, 2, 2, 16, 16, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_align_sort(None, None, 4, 2, 4, 16, None, None, None, None, None, None, 0, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_fp8_act(None, 4, 128, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_fp8_weights(16, 100, 128, 16, 16, None) == moe.MOE_ERR_INVALID_ARG
    # T = 0 is a no-op
    assert lib.moe_fused_forward(0, 16, 16, None, 16, None, 16, None, 0, 128, 256, 4, 2, 0, 0,
                                 16, 256, 0, None) == moe.MOE_OK
    # misaligned workspace
    assert lib.moe_fused_forward(0, 16, 16, None, 16, None, 16, None, 4, 128, 256, 4, 2, 0, 0,
                                 16, 264, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG


def test_options_defaults_and_validation(moe):
    """Per-call options: the defaults, and out-of-range values rejected on the host before any CUDA call."""
    o = moe.Options()
    assert (o.gemm_pair, o.one_stage, o.pdl_mask, o.h_wait_limit_us, o.unsatisfiable_h_wait) == (-1, 1, -1, 0, 0)
    assert o.c.stage_events is None
    lib = moe.load()
    assert lib.moe_options_init(None) == moe.MOE_ERR_INVALID_ARG
    args = (0, 16, 16, None, 16, None, 16, None, 4, 128, 256, 4, 2, 0, 0, 16, 256, 1 << 30)
    for bad in (dict(gemm_pair=2), dict(gemm_pair=-2), dict(one_stage=2), dict(pdl_mask=0x80), dict(pdl_mask=-2),
                dict(unsatisfiable_h_wait=2)):
        opt = moe.Options(**bad)
        assert lib.moe_fused_forward_ex(*args, moe._opt(opt), None) == moe.MOE_ERR_INVALID_ARG, bad
        assert lib.moe_fused_forward_train(16, 16, None, 16, 16, 4, 128, 256, 4, 2, 16, 256, 1 << 30,
                                           moe._opt(opt), None) == moe.MOE_ERR_INVALID_ARG, bad


def test_no_environment_knobs_or_process_switches(moe):
    """The library reads no environment variables and exports no process-wide switches."""
    import subprocess
    lib_path = moe.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    assert "moe_set_gemm_pair" not in out and "moe_set_one_stage" not in out and "moe_set_stage_events" not in out
    und = subprocess.run(["nm", "-D", "--undefined-only", lib_path], capture_output=True, text=True).stdout
    assert "getenv" not in und


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from mixture_experts_grouped_moe_gb300 import moe as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        m.load()
