"""pa_decode_plan (host only) against the balanced split restated in Python.

The plan must hold, for every CTA of the persistent grid, exactly what the
device's walk derives before its first item: the stream total, the positions per
CTA, the number of CTAs, the CTA's range, the sequence holding its first position
with that sequence's first position and clamped length; and, for the first item
the walk emits, its first block and the block ids that follow it in the table."""
import random

import numpy as np
import pytest

import paged_kv_cache_79_gb300 as P
from tests.test_schedule_model import UNIT_COST, walk

HEADS_PER_ITEM = 16
MIN_POSITIONS = 4
PLAN_INTS = 32


def field64(e, f):
    return int(np.uint32(e[f])) | (int(e[f + 1]) << 32)


def expected_schedule(lens, W, B, bps, units_per_seq, grid):
    cl = [min(max(t, 0), W * B) for t in lens]
    ns = [((t + B - 1) // B + bps - 1) // bps for t in cl]
    pos = [units_per_seq * (UNIT_COST + n) for n in ns]
    total = sum(pos)
    units = len(lens) * units_per_seq
    avg = (total + units - 1) // units if units else 1
    div = avg if (avg <= 8 and avg > MIN_POSITIONS) else MIN_POSITIONS
    G = min(grid, max(1, (total + div - 1) // div))
    starts = np.concatenate([[0], np.cumsum(pos)]).tolist()
    return cl, total, div, G, starts


CASES = []
rng = random.Random(5)
for i in range(40):
    B = rng.choice([16, 32])
    dtype = rng.choice(["f32", "f16", "bf16"])
    hkv = rng.choice([1, 2, 8, 40])
    G_q = rng.choice([1, 4, 8, 20])
    S = rng.choice([1, 3, 8, 64, 257])
    lens = [rng.choice([0, 1, rng.randint(1, 40), rng.randint(1, 3000), rng.randint(1, 70000)]) for _ in range(S)]
    grid = rng.choice([16, 152, 304, 608])
    CASES.append((B, dtype, hkv, G_q, lens, grid))


@pytest.mark.parametrize("B,dtype,hkv,G_q,lens,grid", CASES, ids=[str(i) for i in range(len(CASES))])
def test_plan_matches_the_walk(B, dtype, hkv, G_q, lens, grid):
    hq = hkv * G_q
    nbs = [(t + B - 1) // B for t in lens]
    W = max(1, max(nbs)) + 1
    r = np.random.default_rng(len(lens) + grid)
    bt = r.integers(0, 10 ** 6, size=(len(lens), W)).astype(np.int32)
    cl = np.array(lens, dtype=np.int32)
    plan = P.pa_decode_plan(bt, cl, hq, hkv, 128, B, dtype, plan_bytes=grid * PLAN_INTS * 4).reshape(grid, PLAN_INTS)
    bps = 1 if (dtype == "f32" or B >= 32) else 32 // B
    units_per_seq = hkv * ((G_q + HEADS_PER_ITEM - 1) // HEADS_PER_ITEM)
    clamped, total, div, G, starts = expected_schedule(lens, W, B, bps, units_per_seq, grid)
    for c in range(grid):
        e = plan[c]
        assert field64(e, 4) == total and e[6] == div and e[7] == G and e[8] == grid and e[14] == len(lens)
        if c >= G:
            assert e[0] == -1
            continue
        s_c, e_c = c * total // G, (c + 1) * total // G
        assert (field64(e, 9), field64(e, 11)) == (s_c, e_c)
        s = int(e[0])
        assert starts[s] <= s_c < starts[s + 1]
        assert field64(e, 1) == starts[s] and e[3] == clamped[s]
        # the first item the walk emits: where the plan's guess is its unit, the
        # first block must agree, and the window must be the table's next entries
        items, tot = walk(lens, units_per_seq, B, bps, G, c)
        assert tot == total
        span = UNIT_COST + ((clamped[s] + B - 1) // B + bps - 1) // bps
        u_guess = (s_c - starts[s]) // span if s_c > starts[s] else 0
        first = items[0] if items else None
        if first is not None and first[0] == s and first[1] == u_guess:
            assert e[13] == first[2]
        j0 = int(e[13])
        want = [int(bt[s, j]) if j < W else -1 for j in range(j0, j0 + 16)]
        assert e[16:32].tolist() == want


def test_plan_argument_errors():
    bt = np.zeros((2, 4), dtype=np.int32)
    cl = np.array([3, 40], dtype=np.int32)
    with pytest.raises(P.PagedKVError):
        P.pa_decode_plan(bt, cl, 8, 3, 128, 16, "bf16", plan_bytes=304 * 128)     # 8 % 3 != 0
    with pytest.raises(P.PagedKVError):
        P.pa_decode_plan(bt, cl, 8, 8, 128, 16, "bf16", plan_bytes=100)           # not a multiple of 128
    with pytest.raises(P.PagedKVError):
        P.pa_decode_plan(bt, cl, 8, 8, 96, 16, "bf16", plan_bytes=128)            # head_dim 96


def test_empty_batch_plan():
    plan = P.pa_decode_plan(np.zeros((0, 1), np.int32), np.zeros(0, np.int32), 8, 8, 64, 16, "f16",
                            plan_bytes=4 * 128).reshape(4, PLAN_INTS)
    assert (plan[:, 0] == -1).all() and (plan[:, 7] == 0).all()
