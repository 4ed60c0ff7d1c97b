"""The balanced split-KV schedule, restated in Python (CPU only).

The partition kernel's producer warps cut the concatenated stream of units
(sequence, kv head, head group) into equal position ranges, one per CTA; a unit
costs UNIT_COST positions plus one per ring stage.  This model checks, for random
length mixes and grid sizes, the properties the kernel relies on:
  * every block of every unit is streamed by exactly one CTA;
  * a unit seen whole by one CTA is written directly, otherwise each CTA touching it
    writes one partial into a slot (2c if the unit began in an earlier CTA, else
    2c + 1) that no other partial uses;
  * the merge set a CTA derives (c_first, nparts, skipping CTAs with empty ranges)
    is exactly the set of partials written for that unit;
  * every empty unit is owned by exactly one CTA (it writes zeros).
"""
import random

import pytest

UNIT_COST = 2   # positions charged per unit (kUnitCost in the kernel)


def cta_of(x, total, G):
    return ((x + 1) * G - 1) // total


def walk(lens, units, bs, bps, G, cta):
    """Items of CTA `cta`: (seq, unit, j0, j1, partial, slot, c_first, nparts)."""
    nss = [((t + bs - 1) // bs + bps - 1) // bps for t in lens]
    total = sum(units * (UNIT_COST + ns) for ns in nss)
    s_c, e_c = cta * total // G, (cta + 1) * total // G
    items = []
    if s_c >= e_c:
        return items, total
    base = 0
    for s, ns in enumerate(nss):
        span = UNIT_COST + ns
        if base + units * span <= s_c:
            base += units * span
            continue
        if base >= e_c:
            break
        nb = (lens[s] + bs - 1) // bs
        for u in range(units):
            a = base + u * span
            ra, rb = a + UNIT_COST, a + UNIT_COST + ns
            if ns == 0:
                if s_c <= a < e_c:
                    items.append((s, u, 0, 0, False, None, None, None))
                continue
            lo, hi = max(ra, s_c), min(rb, e_c)
            if lo >= hi:
                continue
            partial = not (lo == ra and hi == rb)
            slot = 2 * cta + (0 if ra < s_c else 1)
            cf = nparts = None
            if partial:
                cf, cl = cta_of(ra, total, G), cta_of(rb - 1, total, G)
                nparts = 1 + sum(1 for c in range(cf + 1, cl + 1)
                                 if c * total // G < (c + 1) * total // G)
            items.append((s, u, (lo - ra) * bps, min((hi - ra) * bps, nb), partial, slot, cf, nparts))
        base += units * span
    return items, total


def merge_slots(cf, nparts, total, G):
    slots, cc = [2 * cf + 1], cf
    for _ in range(nparts - 1):
        cc += 1
        while cc * total // G >= (cc + 1) * total // G:
            cc += 1
        slots.append(2 * cc)
    return slots


def check(lens, units, bs, bps, G):
    cover, written, zero_owner, merges = {}, {}, {}, {}
    for c in range(G):
        items, total = walk(lens, units, bs, bps, G, c)
        for (s, u, j0, j1, partial, slot, cf, nparts) in items:
            if j0 == j1:
                assert (s, u) not in zero_owner
                zero_owner[(s, u)] = c
                continue
            for j in range(j0, j1):
                assert (s, u, j) not in cover
                cover[(s, u, j)] = c
            if partial:
                assert slot not in written, "two partials in one slot"
                written[slot] = (s, u)
                merges.setdefault((s, u), set()).add((cf, nparts))
    for s, t in enumerate(lens):
        nb = (t + bs - 1) // bs
        for u in range(units):
            if nb == 0:
                assert (s, u) in zero_owner
            for j in range(nb):
                assert (s, u, j) in cover, (s, u, j)
    for (s, u), sets in merges.items():
        assert len(sets) == 1, "CTAs disagree on the merge set"
        cf, nparts = sets.pop()
        slots = merge_slots(cf, nparts, total, G)
        assert sorted(slots) == sorted(k for k, v in written.items() if v == (s, u))


@pytest.mark.parametrize("seed", range(40))
def test_balanced_schedule_invariants(seed):
    rng = random.Random(seed)
    S = rng.randint(1, 30)
    lens = [rng.choice([0, 1, 5, 16, 17, 33, 100, 700, 3000]) for _ in range(S)]
    units = rng.choice([1, 2, 8, 40])
    bs = rng.choice([16, 32])
    bps = 32 // bs if rng.random() < 0.7 else 1
    G = rng.choice([1, 2, 7, 152, 304, 608])
    check(lens, units, bs, bps, G)


def test_single_long_sequence_spreads_over_every_cta():
    check([60000], 1, 16, 2, 304)


def test_more_ctas_than_positions():
    check([1, 0, 3], 2, 16, 2, 608)
