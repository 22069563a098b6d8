"""Host model of the selection kernel's radix select (no GPU).

The CUDA selection finds each expert's q-th largest score with an 8-bit
radix select over the scores' IEEE bit patterns (non-negative floats order
like their bits): the first pass counts the top byte of every key; if the
bucket holding the q-th key fits a candidate buffer, the later passes look
only at that bucket's keys; the passes stop as soon as the bucket holding the
q-th key is kept whole, and the keep rule then compares keys on the bits
decided so far. This model restates those steps in NumPy and checks them
against the oracle's selector (sort by score descending, ties to the lower
pair index; LRMoE Sec. 7.2 Prop. 7.1) on segments built to reach every
branch: heavy ties, one shared top byte, a candidate buffer too small, early
stops after each pass, and the extreme quotas.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle


def _find(keys, prefix, mask, remaining, shift):
    """Bin (descending) holding the remaining-th largest key among those
    matching prefix under mask: (new prefix, remaining inside it, bin size)."""
    sub = keys[(keys & mask) == prefix]
    hist = np.bincount((sub >> shift) & 255, minlength=256)
    acc = 0
    for d in range(255, -1, -1):
        c = int(hist[d])
        if acc + c >= remaining:
            return prefix | (d << shift), remaining - acc, c
        acc += c
    raise AssertionError("remaining exceeds the matching keys")


def model_select(scores_f32, q, cand_cap):
    """Keep flags of one segment as the kernel computes them, and the number
    of radix passes it ran."""
    keys = np.asarray(scores_f32, dtype=np.float32).view(np.uint32).astype(np.int64)
    n = keys.shape[0]
    if q == n:
        return np.ones(n, dtype=bool), 0
    if q == 0:
        return np.zeros(n, dtype=bool), 0
    prefix, remaining, bucket = _find(keys, 0, 0, q, 24)
    mask, passes = 0xFF000000, 1
    done = bucket == remaining
    cur = keys
    if not done and bucket <= cand_cap:
        cur = keys[(keys >> 24) == (prefix >> 24)]
        assert cur.shape[0] == bucket
    for shift in (16, 8, 0):
        if done:
            break
        prefix, remaining, bucket = _find(cur, prefix, mask, remaining, shift)
        mask |= 0xFF << shift
        passes += 1
        done = bucket == remaining
    km = keys & mask
    kept = km > prefix
    eq = np.nonzero(km == prefix)[0]
    kept[eq[:remaining]] = True
    return kept, passes


def oracle_keep(scores_f32, q):
    n = len(scores_f32)
    keep, _, _ = oracle.select_quota(np.asarray(scores_f32, dtype=np.float32).astype(np.float64),
                                     np.array([0, n]), np.array([q]), np.arange(n))
    return keep.astype(bool)


def _segments():
    rng = np.random.default_rng(7)
    yield "lognormal", rng.lognormal(0.0, 2.0, 3000).astype(np.float32)
    yield "few distinct", rng.integers(0, 5, 2000).astype(np.float32) * 0.25
    yield "all equal", np.full(777, 3.5, dtype=np.float32)
    # one top byte: values in [1, 2) share sign and exponent
    yield "one top byte", (1.0 + rng.random(4096)).astype(np.float32)
    # one 16-bit prefix: the first two passes cannot split them
    yield "one 16-bit prefix", (1.0 + rng.integers(0, 2 ** 15, 1500) * 2.0 ** -23).astype(np.float32)
    yield "zeros and ones", (rng.random(999) < 0.3).astype(np.float32)
    yield "with zeros", np.where(rng.random(2500) < 0.5, 0.0,
                                 rng.lognormal(0, 1, 2500)).astype(np.float32)
    yield "single", np.array([2.0], dtype=np.float32)


@pytest.mark.parametrize("cand_cap", [0, 64, 1 << 20])
def test_model_matches_the_oracle_selector(cand_cap):
    for name, s in _segments():
        n = len(s)
        for q in sorted({0, 1, n // 3, n // 2, n - 1, n} & set(range(n + 1))):
            got, _ = model_select(s, q, cand_cap)
            want = oracle_keep(s, q)
            assert got.sum() == q, (name, q)
            assert np.array_equal(got, want), (name, q, cand_cap)


def test_every_branch_is_reached():
    """Early stops after one to four passes, with and without candidates."""
    rng = np.random.default_rng(3)
    passes = set()
    for _ in range(200):
        n = int(rng.integers(2, 400))
        kind = int(rng.integers(0, 3))
        if kind == 0:
            s = rng.lognormal(0, 3, n)
        elif kind == 1:
            s = rng.integers(0, 4, n) * 1.5
        else:
            s = 1.0 + rng.integers(0, 2 ** 12, n) * 2.0 ** -23
        s = s.astype(np.float32)
        q = int(rng.integers(1, n))
        for cap in (0, n):
            got, p = model_select(s, q, cap)
            passes.add(p)
            assert np.array_equal(got, oracle_keep(s, q))
    assert {1, 2, 3, 4} <= passes


def test_a_planted_keep_rule_mistake_is_caught():
    """Keeping the LAST equal keys instead of the first breaks the tie rule."""
    s = np.array([1.0, 2.0, 2.0, 2.0, 0.5], dtype=np.float32)
    kept, _ = model_select(s, 2, 1 << 20)
    assert np.array_equal(kept, [False, True, True, False, False])
    wrong = np.array([False, False, True, True, False])
    assert not np.array_equal(wrong, oracle_keep(s, 2))
