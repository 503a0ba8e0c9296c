"""Shared checks for the tests: properties every correct result has."""
import numpy as np

import oracle


def check_sort_invariants(ids, E, B, sorted_ids, sorted_eids, npp, counts):
    """Properties any correct align-sort output has (used for oracle and GPU)."""
    T, k = ids.shape
    S = T * k
    P, NB = oracle.align_sort_sizes(T, k, E, B)
    assert sorted_ids.shape == (P,) and sorted_eids.shape == (NB,)
    assert counts.sum() == S
    assert npp % B == 0 and npp <= P
    real = sorted_ids[sorted_ids != S]
    assert np.array_equal(np.sort(real), np.arange(S))
    assert np.all(sorted_ids[npp:] == S)
    used = sorted_eids[: npp // B]
    assert np.all(np.diff(used) >= 0)
    assert np.all(sorted_eids[npp // B:] == -1)
    pos = 0
    for e in range(E):
        c = int(counts[e])
        pad = -(-c // B) * B
        seg = sorted_ids[pos:pos + pad]
        assert np.all(ids.flat[seg[:c]] == e)
        assert np.all(np.diff(seg[:c]) > 0)
        assert np.all(seg[c:] == S)
        assert np.all(sorted_eids[pos // B:(pos + pad) // B] == e)
        pos += pad
    assert pos == npp


def rel_l2(got, ref) -> float:
    """||got - ref|| / ||ref|| in fp64 over the whole compared tensor."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
