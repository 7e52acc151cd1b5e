"""The on-chip merge layout of the decode kernel's clustered instance, checked on the CPU.

A sequence held by p CTAs of an 8-CTA cluster has head group g (of 8) merged by the
(g mod p)-th of them, and part k of head group g lands in that CTA's receive slot
k * ceil(8 / p) + g // p.  The kernel reserves 14 slots per receive area; these tests check
that every (part, head group) pair of one sequence gets its own slot, within the 14, and
that every head group has exactly one merging CTA.
"""
import math

import pytest

CLUSTER, GROUPS, SLOTS = 8, 8, 14


def slot_of(p: int, k: int, g: int) -> tuple[int, int]:
    """(receiving CTA index among the p, slot) of part k of head group g."""
    qmax = math.ceil(GROUPS / p)
    return g % p, k * qmax + g // p


@pytest.mark.parametrize("p", range(1, CLUSTER + 1))
def test_receive_slots_are_distinct_and_fit(p):
    used = {}
    for k in range(p):
        for g in range(GROUPS):
            recv, slot = slot_of(p, k, g)
            assert 0 <= recv < p
            assert 0 <= slot < SLOTS
            key = (recv, slot)
            assert key not in used, (p, k, g, used[key])
            used[key] = (k, g)
    # every receiving CTA gets all p parts of each of its head groups
    for recv in range(p):
        groups = [g for g in range(GROUPS) if g % p == recv]
        assert sum(1 for (r, _s) in used if r == recv) == p * len(groups)


def test_fourteen_slots_is_the_most_any_cluster_needs():
    assert max(p * math.ceil(GROUPS / p) for p in range(1, CLUSTER + 1)) == SLOTS
