"""Host model of the weight-gradient tile queue's ring of tile ids (no GPU).

The copy lane of every CTA takes the next position of the longest-first tile
list with an atomic add and publishes its tile id in a ring of kTQ slots,
each with a 'full' mbarrier (the copy lane's arrival) and an 'empty' one
(one arrival per consumer warp: MMA, epilogue and gather warps). The copy
lane reuses a slot only after every consumer has read its previous id. This
replays the ring under random interleavings: every consumer sees every tile
once, in the copy lane's order, then the end mark, and no consumer ever
finds a slot more than one lap ahead (a parity wait could not tell).
"""

import random

import pytest


def _ring_run(total, consumers, kTQ=8, seed=0):
    rnd = random.Random(seed)
    full = [0] * kTQ     # completed phases of tq_full[slot]
    empty = [0] * kTQ    # completed phases of tq_empty[slot]
    arrived = [0] * kTQ  # consumer arrivals in the current empty phase
    ids = [None] * kTQ
    r_prod = 0
    seen = [[] for _ in range(consumers)]
    r_cons = [0] * consumers
    done_prod = False
    order = list(range(total))
    while not (done_prod and all(s and s[-1] == total for s in seen)):
        actors = (["p"] if not done_prod else []) + [c for c in range(consumers)
                                                     if not (seen[c] and seen[c][-1] == total)]
        a = rnd.choice(actors)
        if a == "p":
            slot = r_prod % kTQ
            if empty[slot] < r_prod // kTQ:  # parity wait: the slot's previous use not read by all
                continue
            ids[slot] = order[r_prod] if r_prod < total else total
            full[slot] += 1
            done_prod = r_prod >= total
            r_prod += 1
        else:
            r = r_cons[a]
            slot = r % kTQ
            if full[slot] <= r // kTQ:  # not yet published for this lap
                continue
            assert full[slot] == r // kTQ + 1  # never more than one lap ahead
            seen[a].append(ids[slot])
            arrived[slot] += 1
            if arrived[slot] == consumers:
                arrived[slot] = 0
                empty[slot] += 1
            r_cons[a] += 1
    return seen


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("consumers", [9, 13])
def test_ring_of_tile_ids_delivers_every_tile_once_in_order(seed, consumers):
    total = 97
    seen = _ring_run(total, consumers, seed=seed)
    for s in seen:
        assert s == list(range(total)) + [total]
