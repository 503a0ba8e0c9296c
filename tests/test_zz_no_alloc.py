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
    ids = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return ids, rng.random((T, k)).astype(np.float32)


def _outputs(P, NB, E, fill):
    return (torch.full((P,), fill, dtype=torch.int32, device="cuda"),
            torch.full((P,), float(fill), dtype=torch.float32, device="cuda"),
            torch.full((NB,), fill, dtype=torch.int32, device="cuda"),
            torch.full((1,), fill, dtype=torch.int32, device="cuda"),
            torch.full((E,), fill, dtype=torch.int32, device="cuda"))


@pytest.mark.gpu
def test_noalloc_sort_matches_workspace_sort_twice(moe):
    # a large sort first, then a small one: the second must not see the first's leftovers
    for (T, k, E, B, seed) in [(4096, 8, 256, 128, 1), (100, 2, 8, 16, 2)]:
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


def test_noalloc_sort_rejects_oversize(moe):
    # 1 MiB of scratch: 1024 experts x 1024 chunks of slots cannot fit; rejected before any launch
    lib = moe.load()
    rc = lib.moe_align_sort_noalloc(16, 16, 1 << 20, 1, 1024, 128, 16, 16, 16, 16, None, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
