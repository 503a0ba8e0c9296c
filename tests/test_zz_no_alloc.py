"""moe_align_sort_noalloc, the token sort for callers that cannot allocate
device memory (a host framework that owns every allocation, a fixed memory
budget, or a hot path that cannot take cudaMalloc's synchronisation): it
must give exactly what moe_align_sort gives with a caller workspace, on two
calls in a row (the shared scratch keeps the previous call's contents), and
reject shapes whose scratch does not fit its fixed array.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test already.
"""
import numpy as np
import pytest
import torch


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_grouped_moe_gb300 import build
    build.build()
    from mixture_experts_grouped_moe_gb300 import moe as m
    m.load()
    return m


def _routing(T, k, E, seed):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(E, 0.3))
    if k == 1:
        ids = rng.choice(E, size=(T, 1), p=p).astype(np.int32)
    else:
        ids = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return ids, rng.random((T, k)).astype(np.float32)


def _outputs(P, NB, E, fill):
    return (torch.full((P,), fill, dtype=torch.int32, device="cuda"),
            torch.full((P,), float(fill), dtype=torch.float32, device="cuda"),
            torch.full((NB,), fill, dtype=torch.int32, device="cuda"),
            torch.full((1,), fill, dtype=torch.int32, device="cuda"),
            torch.full((E,), fill, dtype=torch.int32, device="cuda"))


# the largest shape whose scratch fits: E = 1024 experts and 254 chunks of 1024 slots
# (254 * 1024 histogram words, then 1025 offsets: 261,121 of the 262,144 words)
LIMIT_T = 254 * 1024


@pytest.mark.gpu
def test_noalloc_sort_matches_workspace_sort_twice(moe):
    # Calls in a row that all use the shared scratch (the chunked three-launch sort): a large
    # sort, then one with another chunk count and expert count, so the offsets sit elsewhere in
    # the array and the second must not read the first's leftovers; then the largest shape that
    # fits; then the first shape again.
    for (T, k, E, B, seed) in [(4096, 8, 256, 128, 1), (700, 2, 64, 64, 2), (LIMIT_T, 1, 1024, 128, 3),
                               (4096, 8, 256, 128, 4)]:
        assert T * k > 1024   # more than one CTA's worth of slots: the path that uses the scratch
        ids, w = _routing(T, k, E, seed)
        d_ids, d_w = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
        P, NB = moe.moe_align_sort_sizes(T, k, E, B)
        ref = _outputs(P, NB, E, -7)
        wsb = moe.moe_align_sort_workspace_size(T, k, E)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        moe.moe_align_sort(d_ids, d_w, T, k, E, B, *ref, ws, wsb)
        got = _outputs(P, NB, E, -9)
        moe.moe_align_sort_noalloc(d_ids, d_w, T, k, E, B, *got)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert int(got[3].item()) > 0


def test_noalloc_sort_rejects_oversize(moe):
    # rejected on the host before any launch (the pointers are never touched)
    lib = moe.load()
    rc = lib.moe_align_sort_noalloc(16, 16, 1 << 20, 1, 1024, 128, 16, 16, 16, 16, None, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    # one chunk more than the largest shape that fits
    rc = lib.moe_align_sort_noalloc(16, 16, LIMIT_T + 1, 1, 1024, 128, 16, 16, 16, 16, None, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
