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


def parity_tokens(ids, E, block_m, n_random=512, tail_slots=512, seed=1234):
    """Tokens whose full-size outputs are compared with the oracle.

    - n_random seeded tokens;
    - one seeded real row of every block_m-row block of the expert-sorted order (so every
      (expert, M-block) tile row of the grouped GEMMs has a compared token);
    - the last real row of every expert (its ragged tail block);
    - every token of the least-loaded non-empty experts, taken in increasing load, at most 8
      experts, while their slots add up to at most tail_slots (this bounds the oracle's work
      where even the least-loaded experts hold thousands of slots).
    Returns a sorted int64 array of token indices.
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    rng = np.random.default_rng(seed)
    toks = set(rng.choice(T, size=min(n_random, T), replace=False).tolist())
    sorted_ids, _, npp, counts = oracle.align_sort(ids, E, block_m)
    S = T * k
    for b0 in range(0, npp, block_m):
        real = sorted_ids[b0:b0 + block_m]
        real = real[real < S]
        if len(real):
            toks.add(int(real[rng.integers(len(real))]) // k)
    pos = 0
    for e in range(E):
        c = int(counts[e])
        if c:
            toks.add(int(sorted_ids[pos + c - 1]) // k)
        pos += -(-c // block_m) * block_m
    taken = 0
    for n, e in enumerate(e for e in np.argsort(counts, kind="stable") if counts[e] > 0):
        if n >= 8 or taken + counts[e] > tail_slots:
            break
        taken += int(counts[e])
        toks.update(np.nonzero((ids == e).any(1))[0].tolist())
    return np.array(sorted(toks), np.int64)


def check_rows(got, ref, tol, row_factor=4.0, label=""):
    """Whole-tensor relL2 <= tol and every row's relL2 <= row_factor * tol (localises errors a
    whole-tensor norm would average away).  Returns (relL2, worst row relL2, its row index)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    err = rel_l2(got, ref)
    rows = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-300)
    worst = int(np.argmax(rows))
    print(f"{label}: relL2 {err:.3e} over {got.shape[0]} rows, worst row {rows[worst]:.3e} (row {worst})")
    assert err <= tol, f"{label}: relL2 {err:.3e} > {tol}"
    assert rows[worst] <= row_factor * tol, f"{label}: row {worst} relL2 {rows[worst]:.3e} > {row_factor * tol}"
    return err, float(rows[worst]), worst


E4M3_LEADERS = (1.3 * 2.0 ** -126, 1e-30, 0.7, 3.1, 57.0, 672.0, 2e30, 1.3 * 2.0 ** 120)


def every_bf16_below(leaders, C, group):
    """bf16 rows for exhaustive quantiser checks: per group of `group` columns a leader (the group's
    largest magnitude, so it fixes the group's scale), then every finite bf16 value v with
    leader * 2^-21 <= |v| <= leader, both signs, spread over the row's groups in ascending bit
    order, the rest zero.  One row per leader; group = C gives one scale per row."""
    import torch
    vals = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    rows = []
    for lead in leaders:
        lead = torch.tensor(lead).to(torch.bfloat16).float().item()
        v = vals[torch.isfinite(vals) & (vals.abs() <= lead) & (vals.abs() >= lead * 2.0 ** -21)]
        ng, per = C // group, group - 1
        assert len(v) <= ng * per
        v = torch.cat([v, torch.zeros(ng * per - len(v))]).view(ng, per)
        rows.append(torch.cat([torch.full((ng, 1), lead), v], 1).reshape(-1))
    return torch.stack(rows).to(torch.bfloat16)
