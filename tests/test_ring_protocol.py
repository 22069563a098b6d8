"""Host model of the grouped-GEMM operand ring when several gather warps fill
it (no GPU).

The ring has S stages, each with a 'full' and an 'empty' mbarrier. An
in-order copy thread and ng gather warps (warp g fills K blocks g, g+ng, ...)
wait on 'empty' with a parity wait, which passes when the barrier's
completion count has the other parity; the MMA consumer takes K blocks in
order and completes 'empty'. A parity wait is only sound while the barrier is
at most one phase behind the one awaited. The kernel runs min(4, S) gather
warps; this model checks that no wait passes on an aliased phase under random
interleavings, and that the rule is needed (four warps on a 3-stage ring do
alias).
"""

import random

import pytest


def _aliased_waits(S, ng, n=300, seed=0):
    rnd = random.Random(seed)
    empty_c = [0] * S
    arrivals = [0] * n  # copy thread + the block's gather warp
    prod = 0
    gw = list(range(ng))
    mma = 0
    bad = 0

    def wait(it):
        nonlocal bad
        s = it % S
        parity = ((it // S) & 1) ^ 1
        passes = (empty_c[s] & 1) != parity
        if passes and empty_c[s] != it // S:
            bad += 1
        return passes

    while mma < n:
        actors = ["m"] + (["p"] if prod < n else []) + [g for g in range(ng) if gw[g] < n]
        a = rnd.choice(actors)
        if a == "m":
            if arrivals[mma] == 2:
                empty_c[mma % S] += 1
                mma += 1
        elif a == "p":
            if wait(prod):
                arrivals[prod] += 1
                prod += 1
        elif wait(gw[a]):
            arrivals[gw[a]] += 1
            gw[a] += ng
    return bad


@pytest.mark.parametrize("S", [3, 4, 5, 6])
def test_gather_warps_never_wait_on_an_aliased_phase(S):
    ng = min(4, S)
    assert sum(_aliased_waits(S, ng, seed=k) for k in range(50)) == 0


def test_more_gather_warps_than_stages_would_alias():
    assert sum(_aliased_waits(3, 4, seed=k) for k in range(50)) > 0
