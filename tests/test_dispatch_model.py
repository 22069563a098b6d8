"""Host model of the single-launch dispatch (no GPU).

The fused dispatch kernel runs as one cluster of C CTAs (16 where the GPU
can schedule a 16-CTA cluster, else 8; the GB300 always takes 16, so the
8-CTA form is exercised here only). CTA c owns a contiguous share of the N
pairs, each of its 32 warps a contiguous sub-share rounded to whole rows of
32; every warp counts its experts, the CTAs exchange their per-expert counts,
and each pair's position is

    off[e] + (pairs of e in earlier CTAs) + (pairs of e in earlier warps of
    this CTA) + (pairs of e in earlier rows of this warp) + (lanes of this
    row before it with the same expert).

This model restates that arithmetic in NumPy and checks, for both cluster
sizes and ragged N, that it is the oracle's stable counting sort (LLEP Sec.
2.1 re-index; Alg. 4 sort of the flattened ids).
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle

WARPS = 32  # 1024 threads per CTA


def model_dispatch(ids: np.ndarray, E: int, nctas: int):
    N = ids.shape[0]
    per_cta = -(-N // nctas)
    per_warp = ((-(-per_cta // WARPS)) + 31) // 32 * 32
    # the pairs each (CTA, warp) owns
    owners = []
    for c in range(nctas):
        c_lo, c_hi = c * per_cta, min(N, c * per_cta + per_cta)
        for w in range(WARPS):
            w_lo = min(c_hi, c_lo + w * per_warp)
            w_hi = min(c_hi, w_lo + per_warp)
            owners.append((c, w, w_lo, w_hi))
    # per-warp counts, then per-CTA counts
    wcnt = np.zeros((nctas, WARPS, E), dtype=np.int64)
    for c, w, lo, hi in owners:
        np.add.at(wcnt[c, w], ids[lo:hi], 1)
    cta_cnt = wcnt.sum(axis=1)
    counts = cta_cnt.sum(axis=0)
    off = np.concatenate([[0], np.cumsum(counts)])
    perm = np.full(N, -1, dtype=np.int64)
    inv = np.full(N, -1, dtype=np.int64)
    for c, w, lo, hi in owners:
        base = off[:E] + cta_cnt[:c].sum(axis=0) + wcnt[c, :w].sum(axis=0)
        run = np.zeros(E, dtype=np.int64)
        for b in range(lo, hi, 32):  # rows of 32 lanes, in order
            row = ids[b:min(b + 32, hi)]
            for lane, e in enumerate(row):
                pos = base[e] + run[e] + int(np.sum(row[:lane] == e))
                perm[pos] = b + lane
                inv[b + lane] = pos
            np.add.at(run, row, 1)
    return perm, inv, counts, off


@pytest.mark.parametrize("nctas", [8, 16])
@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (37, 2, 5), (300, 8, 128), (1111, 4, 256)])
def test_model_equals_the_oracle_dispatch(nctas, T, K, E):
    rng = np.random.default_rng(T * 1000 + E)
    # skewed routing: a few experts hold most pairs, some none
    w = 1.0 / np.arange(1, E + 1) ** 1.3
    ids = np.stack([rng.choice(E, size=K, replace=False, p=w / w.sum()) if K <= E
                    else rng.integers(0, E, K) for _ in range(T)]).reshape(-1)
    perm, inv, counts, off = model_dispatch(ids, E, nctas)
    r_perm, r_inv, r_counts, r_off = oracle.dispatch_permute(ids.reshape(T, K), E)
    assert np.array_equal(perm, r_perm)
    assert np.array_equal(inv, r_inv)
    assert np.array_equal(counts, r_counts)
    assert np.array_equal(off, r_off)


def test_every_pair_lands_once_when_ctas_own_nothing():
    # fewer pairs than CTAs x rows: most CTAs and warps own empty ranges
    ids = np.array([3, 0, 3, 1, 3], dtype=np.int64)
    for nctas in (8, 16):
        perm, inv, counts, off = model_dispatch(ids, 4, nctas)
        assert sorted(perm.tolist()) == list(range(5))
        assert np.array_equal(perm[inv], np.arange(5))
        assert perm.tolist() == [1, 3, 0, 2, 4]
