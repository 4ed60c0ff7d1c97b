"""pa_decode_shared_plan (host only) against the shared-prefix walks restated in Python.

For each of the two launches the plan must hold, per CTA of the persistent grid,
what that launch's walk derives before its first item: the stream total, the
positions per CTA, the number of CTAs, the CTA's range, the sequence holding its
first position with that position's base, the sequence's units as the launch
counts them (shared launch: the group's members and shared blocks; own launch: the
first own block and whether the (unit, sequence) order applies), and the first
16 block ids of the first item the walk emits."""
import random

import numpy as np
import pytest

import paged_kv_cache_79_gb300 as P
from tests.test_schedule_model import (UNIT_COST, random_shared_batch, shared_units, walk_pass)

MIN_POSITIONS = 4
PLAN_INTS = 32
AUX_MASK = (1 << 29) - 1
AUX_UNIT_MAJOR = 1 << 29
AUX_SHARE_ERR = 1 << 30


def field64(e, f):
    return int(np.uint32(e[f])) | (int(e[f + 1]) << 32)


def divisor(total, units):
    avg = (total + units - 1) // units if units else 1
    return avg if (avg <= 8 and avg > MIN_POSITIONS) else MIN_POSITIONS


def check_pass(entries, su, bps, grid, bt, lens, aux_of, len_of, unit_major):
    nss = [(nb - start + bps - 1) // bps if n else 0 for (n, start, nb) in su]
    spans = [UNIT_COST + ns for ns in nss]
    total = sum(n * sp for (n, _, _), sp in zip(su, spans))
    units = sum(n for n, _, _ in su)
    div = divisor(total, units)
    G = min(grid, max(1, (total + div - 1) // div)) if su else 0
    starts = np.concatenate([[0], np.cumsum([n * sp for (n, _, _), sp in zip(su, spans)])]).tolist()
    cum = np.concatenate([[0], np.cumsum(spans)]).tolist()
    Wtab = bt.shape[1]
    for c in range(grid):
        e = entries[c]
        assert field64(e, 4) == total and e[6] == div and e[7] == G and e[8] == grid
        assert e[14] == len(su)
        if c >= G:
            assert e[0] == -1
            continue
        s_c, e_c = c * total // G, (c + 1) * total // G
        if total == 0:              # nothing to stream (no group shares blocks)
            assert e[0] == -1
            continue
        assert (field64(e, 9), field64(e, 11)) == (s_c, e_c)
        s, base = int(e[0]), field64(e, 1)
        if unit_major:
            Wrow = total // su[0][0]
            u, inner = s_c // Wrow, s_c - (s_c // Wrow) * Wrow
            assert cum[s] <= inner < cum[s + 1]
            assert base == u * Wrow + cum[s]
        else:
            assert starts[s] <= s_c < starts[s + 1] and base == starts[s]
        assert e[3] == len_of(s) and e[15] == aux_of(s)
        # the first item the walk emits: where the plan's unit is that item, its
        # first block agrees; the window is the sequence's table row from j0
        items, tot = walk_pass(su, bps, G, c)
        assert tot == total
        j0 = int(e[13])
        u_plan = s_c // (total // su[0][0]) if unit_major else \
            ((s_c - base) // spans[s] if s_c > base else 0)
        if items and items[0][:2] == (s, u_plan):
            assert j0 == items[0][2]
        want = [int(bt[s, j]) if j < Wtab else -1 for j in range(j0, j0 + 16)]
        assert e[16:32].tolist() == want


CASES = []
rng = random.Random(77)
for i in range(40):
    bs = rng.choice([16, 32])
    dtype = rng.choice(["f32", "f16", "bf16"])
    group = rng.choice([1, 2, 4, 5, 8, 16])
    hkv = rng.choice([1, 2, 3, 8])
    lens, share = random_shared_batch(rng, bs)
    grid = rng.choice([16, 152, 304])
    CASES.append((bs, dtype, group, hkv, lens, share, grid))


def run_case(bs, dtype, group, hkv, lens, share, grid, W=None):
    hq = hkv * group
    nbs = [(t + bs - 1) // bs for t in lens]
    W = W or max(1, max(nbs)) + 1
    r = np.random.default_rng(len(lens) + grid)
    bt = r.integers(0, 10 ** 6, size=(len(lens), W)).astype(np.int32)
    cl = np.array(lens, dtype=np.int32)
    sh = np.array(share, dtype=np.int32).reshape(-1, 2)
    plan = P.pa_decode_shared_plan(bt, cl, sh, hq, hkv, 128, bs, dtype,
                                   plan_bytes=2 * grid * PLAN_INTS * 4).reshape(2, grid, PLAN_INTS)
    return plan, bt


@pytest.mark.parametrize("bs,dtype,group,hkv,lens,share,grid", CASES, ids=[str(i) for i in range(len(CASES))])
def test_shared_plan_matches_the_walks(bs, dtype, group, hkv, lens, share, grid):
    plan, bt = run_case(bs, dtype, group, hkv, lens, share, grid)
    bps = 1 if (dtype == "f32" or bs >= 32) else 32 // bs
    su1 = shared_units(lens, share, hkv, group, bs, 1)
    su0 = shared_units(lens, share, hkv, group, bs, 0)
    S = len(lens)

    def members(s):
        m = 1
        while s + m < S and share[s + m][0] == s:
            m += 1
        return m

    check_pass(plan[0], su1, bps, grid, bt, lens, aux_of=members, len_of=lambda s: su1[s][2],
               unit_major=False)
    unit_major = any(n and start > 0 for (n, start, _) in su0)
    check_pass(plan[1], su0, bps, grid, bt, lens,
               aux_of=lambda s: su0[s][1] | (AUX_UNIT_MAJOR if unit_major else 0),
               len_of=lambda s: lens[s], unit_major=unit_major)


def test_member_ending_inside_shared_blocks_is_flagged():
    """A member whose context ends inside its group's shared blocks decodes all its
    blocks in the own launch (first own block 0) and its entry carries the flag the
    device raises PA_DEVERR_SHARE from."""
    bs = 16
    lens = [5 * bs + 3, 5 * bs, 5 * bs + 9, 40]     # member 1 ends inside the 5 shared blocks
    share = [(0, 5), (0, 5), (0, 5), (-1, 0)]
    grid = 8
    plan, bt = run_case(bs, "f16", 1, 2, lens, share, grid)
    flagged = [e for e in plan[1] if e[0] == 1]
    assert flagged, "no CTA starts at sequence 1"
    for e in flagged:
        assert e[15] & AUX_SHARE_ERR and (e[15] & AUX_MASK) == 0
    for e in plan[1]:
        if e[0] in (0, 2):
            assert not e[15] & AUX_SHARE_ERR and (e[15] & AUX_MASK) == 5


def test_shared_plan_argument_errors():
    bt = np.zeros((2, 4), dtype=np.int32)
    cl = np.array([3, 40], dtype=np.int32)
    sh = np.array([[-1, 0], [-1, 0]], dtype=np.int32)
    with pytest.raises(P.PagedKVError):
        P.pa_decode_shared_plan(bt, cl, sh, 8, 3, 128, 16, "bf16", plan_bytes=2 * 304 * 128)  # 8 % 3
    with pytest.raises(P.PagedKVError):
        P.pa_decode_shared_plan(bt, cl, sh, 8, 8, 128, 16, "bf16", plan_bytes=128)           # one pass
    with pytest.raises(P.PagedKVError):
        P.pa_decode_shared_plan(bt, cl, sh, 34, 2, 128, 16, "bf16", plan_bytes=256)          # group 17


def test_empty_batch_shared_plan():
    plan = P.pa_decode_shared_plan(np.zeros((0, 1), np.int32), np.zeros(0, np.int32), np.zeros((0, 2), np.int32),
                                   8, 8, 64, 16, "f16", plan_bytes=2 * 4 * 128).reshape(2, 4, PLAN_INTS)
    assert (plan[:, :, 0] == -1).all() and (plan[:, :, 7] == 0).all()
