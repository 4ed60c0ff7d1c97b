"""The balanced split-KV schedule, restated in Python (CPU only).

The partition kernel's producer warps cut the concatenated stream of units
(sequence, kv head, head group) -- for the own blocks of a batch with shared
prefixes, (kv head, head group, sequence) -- into equal position ranges, one per
CTA; a unit
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

UNIT_COST = 4   # positions charged per unit (kUnitCost in the kernel)


def cta_of(x, total, G):
    return ((x + 1) * G - 1) // total


def walk(lens, units, bs, bps, G, cta):
    """Items of CTA `cta`: (seq, unit, j0, j1, partial, slot, c_first, nparts)."""
    su = [(units, 0, (t + bs - 1) // bs) for t in lens]
    return walk_units(su, bps, G, cta)


def walk_units(su, bps, G, cta):
    """Like walk, for per-sequence units: su[s] = (units, first block, end block)."""
    nss = [(nb - start + bps - 1) // bps if n else 0 for (n, start, nb) in su]
    total = sum(n * (UNIT_COST + ns) for (n, _, _), ns in zip(su, nss))
    s_c, e_c = cta * total // G, (cta + 1) * total // G
    items = []
    if s_c >= e_c:
        return items, total
    base = 0
    for s, ((units, start, nb), ns) in enumerate(zip(su, nss)):
        span = UNIT_COST + ns
        if base + units * span <= s_c:
            base += units * span
            continue
        if base >= e_c:
            break
        for u in range(units):
            a = base + u * span
            ra, rb = a + UNIT_COST, a + UNIT_COST + ns
            if ns == 0:
                if s_c <= a < e_c:
                    items.append((s, u, start, start, False, None, None, None))
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
            items.append((s, u, start + (lo - ra) * bps, min(start + (hi - ra) * bps, nb), partial,
                          slot, cf, nparts))
        base += units * span
    return items, total


def walk_units_unit_major(su, bps, G, cta):
    """The (unit, sequence) order of the own-block pass of a batch with shared
    prefixes: unit 0 of every sequence, then unit 1, ...  Every sequence has the
    same number of units there."""
    nss = [(nb - start + bps - 1) // bps if n else 0 for (n, start, nb) in su]
    U = su[0][0]
    assert all(n == U for n, _, _ in su)
    spans = [UNIT_COST + ns for ns in nss]
    W = sum(spans)
    total = U * W
    s_c, e_c = cta * total // G, (cta + 1) * total // G
    items = []
    if s_c >= e_c:
        return items, total
    for u in range(s_c // W, U):
        base = u * W
        if base >= e_c:
            break
        for s, ((_, start, nb), ns) in enumerate(zip(su, nss)):
            a = base
            base += spans[s]
            if a >= e_c:
                break
            ra, rb = a + UNIT_COST, a + UNIT_COST + ns
            if ns == 0:
                if s_c <= a < e_c:
                    items.append((s, u, start, start, False, None, None, None))
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
            items.append((s, u, start + (lo - ra) * bps, min(start + (hi - ra) * bps, nb), partial,
                          slot, cf, nparts))
    return items, total


def walk_pass(su, bps, G, cta):
    """The kernel's choice: (unit, sequence) order once some unit starts after
    shared leading blocks, else (sequence, unit)."""
    if any(n and start > 0 for (n, start, _) in su):
        return walk_units_unit_major(su, bps, G, cta)
    return walk_units(su, bps, G, cta)


def merge_slots(cf, nparts, total, G):
    slots, cc = [2 * cf + 1], cf
    for _ in range(nparts - 1):
        cc += 1
        while cc * total // G >= (cc + 1) * total // G:
            cc += 1
        slots.append(2 * cc)
    return slots


def check(lens, units, bs, bps, G, starts=None):
    """starts[s]: first block of sequence s's units (shared leading blocks before
    it), which selects the (unit, sequence) order; None: all 0."""
    cover, written, zero_owner, merges = {}, {}, {}, {}
    for c in range(G):
        if starts is None:
            items, total = walk(lens, units, bs, bps, G, c)
        else:
            su = [(units, min(p, (t + bs - 1) // bs), (t + bs - 1) // bs)
                  for t, p in zip(lens, starts)]
            items, total = walk_pass(su, bps, G, c)
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
        first = 0 if starts is None else min(starts[s], nb)
        for u in range(units):
            if nb == first:
                assert (s, u) in zero_owner
            for j in range(first, nb):
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


@pytest.mark.parametrize("seed", range(40))
def test_unit_major_schedule_invariants(seed):
    """The own-block pass of a batch with shared prefixes: (unit, sequence) order."""
    rng = random.Random(500 + seed)
    S = rng.randint(1, 30)
    lens = [rng.choice([0, 1, 5, 16, 17, 33, 100, 700, 3000]) for _ in range(S)]
    bs = rng.choice([16, 32])
    starts = [rng.choice([0, 0, 1, 2, 40]) for _ in range(S)]
    starts[rng.randrange(S)] = 1 + rng.randrange(3)
    units = rng.choice([1, 2, 8, 40])
    bps = 32 // bs if rng.random() < 0.7 else 1
    G = rng.choice([1, 2, 7, 152, 304, 608])
    check(lens, units, bs, bps, G, starts)


def test_unit_major_gives_each_cta_a_mix_of_sequences():
    # 128 sequences x 40 units of own parts of 0 .. 16 stages over 304 CTAs: in
    # (sequence, unit) order a CTA sees one or two sequences, in (unit, sequence)
    # order about 17
    lens = [1024 + (i * 37) % 513 for i in range(128)]
    su = [(40, 64, (t + 15) // 16) for t in lens]
    seq_major = [len({it[0] for it in walk_units(su, 2, 304, c)[0]}) for c in range(304)]
    unit_major = [len({it[0] for it in walk_pass(su, 2, 304, c)[0]}) for c in range(304)]
    assert max(seq_major) <= 3
    assert min(unit_major) >= 10


def test_single_long_sequence_spreads_over_every_cta():
    check([60000], 1, 16, 2, 304)


def test_more_ctas_than_positions():
    check([1, 0, 3], 2, 16, 2, 608)


# ---------------------------------------------------------------------------
# Shared-prefix decode: pass 1 streams each group's P shared blocks once per kv
# head and member group (the query rows of up to 8 // group members for groups
# of at most 8 heads, else 16 // group), pass 0
# every sequence's blocks P .. nb.  Together they must cover every (sequence,
# query head, block) exactly once.
# ---------------------------------------------------------------------------
HEADS_PER_ITEM = 16
NARROW_ROWS = 8


def members_per_item(group):
    return (NARROW_ROWS if group <= NARROW_ROWS else HEADS_PER_ITEM) // group


def shared_units(lens, share, Hkv, group, bs, pass_):
    hg = (group + HEADS_PER_ITEM - 1) // HEADS_PER_ITEM
    out = []
    S = len(lens)
    for s in range(S):
        nb = (lens[s] + bs - 1) // bs
        P = share[s][1] if share[s][0] >= 0 else 0
        if pass_ == 0:
            out.append((Hkv * hg, min(P, nb), nb))
            continue
        if share[s][0] != s or P <= 0:
            out.append((0, 0, 0))
            continue
        m = 1
        while s + m < S and share[s + m][0] == s:
            m += 1
        mpi = members_per_item(group)
        out.append((Hkv * ((m + mpi - 1) // mpi), 0, P))
    return out


def rows_of(pass_, s, u, share, lens, Hkv, group):
    """(sequence, query head) pairs of unit u of sequence s."""
    if pass_ == 1:
        S = len(lens)
        m = 1
        while s + m < S and share[s + m][0] == s:
            m += 1
        mpi = members_per_item(group)
        mgroups = (m + mpi - 1) // mpi
        kvh, mg = divmod(u, mgroups)
        members = range(s + mg * mpi, s + min(m, (mg + 1) * mpi))
        return [(x, kvh * group + r) for x in members for r in range(group)]
    hg = (group + HEADS_PER_ITEM - 1) // HEADS_PER_ITEM
    kvh, h = divmod(u, hg)
    rows = min(HEADS_PER_ITEM, group - h * HEADS_PER_ITEM)
    return [(s, kvh * group + h * HEADS_PER_ITEM + r) for r in range(rows)]


def check_shared(lens, share, Hkv, group, bs, bps, G):
    cover = {}
    for pass_ in (1, 0):
        su = shared_units(lens, share, Hkv, group, bs, pass_)
        for c in range(G):
            items, _ = walk_pass(su, bps, G, c)
            for (s, u, j0, j1, _, _, _, _) in items:
                rows = rows_of(pass_, s, u, share, lens, Hkv, group)
                # the kernel sizes an item's accumulators for this many rows
                assert len(rows) <= (NARROW_ROWS if group <= NARROW_ROWS else HEADS_PER_ITEM)
                for j in range(j0, j1):
                    for (x, h) in rows:
                        key = (x, h, j)
                        assert key not in cover, (pass_, key)
                        cover[key] = pass_
    for s, t in enumerate(lens):
        nb = (t + bs - 1) // bs
        for h in range(Hkv * group):
            for j in range(nb):
                assert (s, h, j) in cover, (s, h, j)
                P = share[s][1] if share[s][0] >= 0 else 0
                assert cover[(s, h, j)] == (1 if j < P else 0)
    assert len(cover) == sum((t + bs - 1) // bs for t in lens) * Hkv * group


def random_shared_batch(rng, bs):
    lens, share = [], []
    while len(lens) < rng.randint(1, 40):
        m = rng.choice([1, 1, 2, 3, 8, 17, 33])
        P = rng.choice([0, 1, 2, 5, 40])
        first = len(lens)
        for _ in range(m):
            lens.append(P * bs + rng.randint(1, 3 * bs))
            share.append((first, P) if (m > 1 and P > 0) else (-1, 0))
    return lens, share


@pytest.mark.parametrize("seed", range(30))
def test_shared_prefix_passes_cover_every_block_once(seed):
    rng = random.Random(1000 + seed)
    bs = rng.choice([16, 32])
    bps = 32 // bs
    group = rng.choice([1, 2, 4, 5, 8, 16])
    Hkv = rng.choice([1, 2, 3])
    lens, share = random_shared_batch(rng, bs)
    G = rng.choice([1, 3, 152, 304])
    check_shared(lens, share, Hkv, group, bs, bps, G)


def test_shared_prefix_workload_shape():
    # 16 prompts x 8 samples, MHA 40 heads: pass 1 has 16 * 40 units of 8-row items
    # (all 8 samples); pass 0 has 128 * 40 units of the private blocks
    lens = [1024 + 1 + (i * 37) % 513 for i in range(128)]
    share = [(8 * (i // 8), 64) for i in range(128)]
    su1 = shared_units(lens, share, 40, 1, 16, 1)
    assert sum(n for n, _, _ in su1) == 16 * 40
    check_shared(lens[:24], share[:24], 2, 1, 16, 2, 152)
