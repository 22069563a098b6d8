"""Host models of two grouped-GEMM protocols (no GPU).

1. Accumulator hand-over. The MMA warp and the epilogue warps share two
   256-column tensor-memory accumulators, each with a 'full' barrier (the MMA
   warp's commit) and an 'empty' barrier (the epilogue's arrival), waited on by
   parity. A 256-column tile uses one accumulator, alternating; a wide tile
   (256 x 512 on a CTA pair) uses both. The model plays both sides' sequences
   of (barrier, parity) waits and arrivals under random interleavings and checks
   that every wait passes on the phase it was meant for (never on an older one)
   and that the two sides agree on which accumulator holds which columns.

2. Tile queue tickets. One 64-bit counter holds the takes from the head of the
   longest-first list in its low word and from the tail in its high word; a
   take whose two counts already sum to the tile count finds the list empty.
   Under random interleavings of head and tail takers every position is handed
   out exactly once.
"""

import random

import pytest


def _mma_side(tiles, wide):
    """The MMA warp's sequence: per tile, the (accumulator, parity) pairs it
    waits 'empty' on, then the accumulators it commits 'full' for."""
    acc, ph, out = 0, 0, []
    for _ in range(tiles):
        accs = [0, 1] if wide else [acc]
        out.append(("wait_empty", [(a, ph ^ 1) for a in accs]))
        out.append(("commit_full", accs))
        if wide:
            ph ^= 1
        else:
            acc ^= 1
            if acc == 0:
                ph ^= 1
    return out


def _epi_side(tiles, wide):
    """The epilogue's sequence: per accumulator it drains, the (accumulator,
    parity) it waits 'full' on and the column offset it stores, then its
    arrival on 'empty'."""
    acc, ph, out = 0, 0, []
    for t in range(tiles):
        for half in range(2 if wide else 1):
            out.append(("wait_full", acc, ph, (t, 256 * half)))
            out.append(("arrive_empty", acc))
            acc ^= 1
            if acc == 0:
                ph ^= 1
    return out


def _run_handover(tiles, wide, seed):
    rnd = random.Random(seed)
    full_c = [0, 0]   # completed phases of each 'full' barrier
    empty_c = [0, 0]  # completed phases of each 'empty' barrier
    uses_m = [0, 0]   # MMA warp: waits passed on each 'empty' so far
    uses_e = [0, 0]   # epilogue: waits passed on each 'full' so far
    held = {0: None, 1: None}  # what the accumulator holds: (tile, column offset)
    mma, epi = _mma_side(tiles, wide), _epi_side(tiles, wide)
    i = j = 0
    t_mma = 0
    bad = []

    def can_m():
        if i >= len(mma):
            return False
        kind, arg = mma[i]
        return kind != "wait_empty" or all((empty_c[a] & 1) != p for a, p in arg)

    def can_e():
        if j >= len(epi):
            return False
        ev = epi[j]
        return ev[0] != "wait_full" or (full_c[ev[1]] & 1) != ev[2]

    while i < len(mma) or j < len(epi):
        ready = [s for s, ok in (("m", can_m()), ("e", can_e())) if ok]
        if not ready:
            bad.append(("deadlock", i, j))
            break
        side = rnd.choice(ready)
        if side == "m":
            kind, arg = mma[i]
            if kind == "wait_empty":
                # a parity wait passes when the barrier's completed-phase count
                # has the other parity; the n-th use of an accumulator must see
                # exactly n completed 'empty' phases (the epilogue drained it n times)
                if all((empty_c[a] & 1) != p for a, p in arg):
                    for a, _ in arg:
                        if empty_c[a] != uses_m[a]:
                            bad.append(("empty aliased", a, empty_c[a], uses_m[a]))
                        uses_m[a] += 1
                    i += 1
            else:
                for half, a in enumerate(arg):
                    held[a] = (t_mma, 256 * half)
                    full_c[a] += 1
                t_mma += 1
                i += 1
        else:
            ev = epi[j]
            if ev[0] == "wait_full":
                _, a, p, want = ev
                if (full_c[a] & 1) != p:
                    # the n-th drain of an accumulator must see exactly n + 1 commits
                    if full_c[a] != uses_e[a] + 1:
                        bad.append(("full aliased", a, full_c[a], uses_e[a]))
                    elif held[a] != want:
                        bad.append(("columns", a, held[a], want))
                    uses_e[a] += 1
                    j += 1
            else:
                empty_c[ev[1]] += 1
                j += 1
    return bad


def test_the_model_catches_a_parity_slip():
    # plant a mistake on the MMA side: a wide tile that flips the phase twice
    # (as a narrow tile would per accumulator pair) lets the next waits pass early
    def slipped(tiles):
        acc, ph, out = 0, 0, []
        for _ in range(tiles):
            out.append(("wait_empty", [(0, ph ^ 1), (1, ph ^ 1)]))
            out.append(("commit_full", [0, 1]))
            ph ^= 1
            ph ^= 1
        return out
    global _mma_side
    orig = _mma_side
    try:
        _mma_side = lambda tiles, wide: slipped(tiles)
        assert any(_run_handover(6, True, seed) for seed in range(50))
    finally:
        _mma_side = orig


@pytest.mark.parametrize("wide", [False, True])
def test_accumulator_handover_matches_on_both_sides(wide):
    for seed in range(200):
        assert _run_handover(9, wide, seed) == []


def test_wide_epilogue_sequence_is_the_narrow_one():
    # the epilogue's (accumulator, parity) sequence does not depend on the tile
    # width: a wide tile is two consecutive narrow hand-overs
    nar = [e[1:3] for e in _epi_side(8, False) if e[0] == "wait_full"]
    wid = [e[1:3] for e in _epi_side(4, True) if e[0] == "wait_full"]
    assert nar == wid


def _take(counter, total, from_tail):
    old = counter[0]
    counter[0] += (1 << 32) if from_tail else 1
    h, t = old & 0xFFFFFFFF, old >> 32
    if h + t >= total:
        return None
    return total - 1 - t if from_tail else h


@pytest.mark.parametrize("total,takers", [(1, 2), (7, 3), (100, 8), (513, 152)])
def test_queue_tickets_hand_out_every_position_once(total, takers):
    for seed in range(40):
        rnd = random.Random(seed)
        counter = [0]
        tails = [rnd.random() < 0.5 for _ in range(takers)]
        live = list(range(takers))
        got = []
        while live:
            k = rnd.choice(live)
            pos = _take(counter, total, tails[k])
            if pos is None:
                live.remove(k)
            else:
                got.append(pos)
        assert sorted(got) == list(range(total))


def test_queue_tickets_from_the_head_only_keep_the_order():
    counter = [0]
    got = [_take(counter, 5, False) for _ in range(7)]
    assert got == [0, 1, 2, 3, 4, None, None]


def test_a_queue_that_did_not_start_at_zero_skips_positions():
    # the kernel's check: tiles handed out != tile count flags LRM_DEVERR_QUEUE
    counter = [3]
    got = []
    while (pos := _take(counter, 10, False)) is not None:
        got.append(pos)
    assert len(got) == 7 and got == list(range(3, 10))
