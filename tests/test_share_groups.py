"""Shared-prefix groups derived from block tables (pa_share_groups, host only).

The groups feed pa_decode_shared, whose result must equal the plain decode; the
decode is only correct if every declared group really shares its leading blocks
and no member's newest token lies in them.  These tests check those conditions,
that the groups are as large as the rule allows, and the groups of the
parallel-sampling and multi-turn workloads (prompt blocks shared by all samples
of a prompt, "Memory sharing" of the PagedAttention paper summary)."""
import random

import numpy as np
import pytest

import paged_kv_cache_79_gb300 as P
import workloads as W
from paged_kv_cache_79_gb300 import runner


def check_valid_and_maximal(bt, cl, B, share):
    S = len(cl)
    cap = [max(0, (int(t) - 1) // B) if t > 0 else 0 for t in cl]
    s = 0
    while s < S:
        e = s + 1
        while e < S and bt[s, 0] >= 0 and bt[e, 0] == bt[s, 0]:
            e += 1
        first, Pb = share[s]
        if first >= 0:
            assert first == s and Pb >= 1 and e - s >= 2
            for m in range(s, e):
                assert tuple(share[m]) == (s, Pb)
                assert Pb <= cap[m], "a member's newest token would sit in a shared block"
                assert np.array_equal(bt[m, :Pb], bt[s, :Pb])
            # maximal: one more block would break the sharing or the cap
            if all(Pb + 1 <= cap[m] for m in range(s, e)):
                assert any(bt[m, Pb] != bt[s, Pb] for m in range(s, e))
        else:
            for m in range(s, e):
                assert tuple(share[m]) == (-1, 0)
            if e - s >= 2:
                # the run agrees on entry 0, so only the cap can forbid sharing it
                assert min(cap[s:e]) == 0
        s = e


@pytest.mark.parametrize("seed", range(20))
def test_random_fork_trees(seed):
    rng = random.Random(seed)
    B = rng.choice([2, 4, 16])
    a = P.BlockAllocator(4000, B)
    seqs = []
    for _ in range(rng.randint(1, 6)):
        root = a.new_seq()
        a.append_n(root, rng.randint(0, 6 * B))
        seqs.append(root)
        for _ in range(rng.randint(0, 5)):
            c = a.fork(rng.choice(seqs[-1:] + [root]))
            seqs.append(c)
    for s in seqs:
        for _ in range(rng.randint(0, 2 * B)):
            a.append(s)
    bt, cl = runner.tables_for(a, seqs)
    share = P.share_groups(bt, cl, B)
    check_valid_and_maximal(bt, cl, B, share)


def test_min_shared_blocks_and_degenerate_cases():
    bt = np.array([[5, 6, 7], [5, 6, 9], [5, 8, -1], [3, -1, -1]], dtype=np.int32)
    cl = np.array([40, 40, 30, 5], dtype=np.int32)
    # rows 0..2 start with block 5; common prefix 1 block (row 2 differs at entry 1)
    assert P.share_groups(bt, cl, 16).tolist() == [[0, 1], [0, 1], [0, 1], [-1, 0]]
    assert P.share_groups(bt, cl, 16, min_shared_blocks=2).tolist() == [[-1, 0]] * 4
    # the newest token of row 2 (T = 16) sits in block 0: nothing may be shared
    cl2 = np.array([40, 40, 16, 5], dtype=np.int32)
    assert P.share_groups(bt, cl2, 16).tolist() == [[-1, 0]] * 4
    # rows 0 and 1 alone share two blocks
    assert P.share_groups(bt[:2], cl[:2], 16).tolist() == [[0, 2], [0, 2]]
    assert P.share_groups(np.zeros((0, 1), np.int32), np.zeros(0, np.int32), 16).shape == (0, 2)
    with pytest.raises(P.PagedKVError):
        P.share_groups(bt, cl, 0)


@pytest.mark.parametrize("name,prompt_blocks", [("shared_prefix_fp16", 64),
                                                 ("shared_prefix_fp16_p1032", 64)])
def test_parallel_sampling_groups(name, prompt_blocks):
    w = W.by_name(name)
    a = P.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    for ev in w.events:
        k = type(ev).__name__
        if k == "NewSeq":
            a.new_seq()
        elif k == "Fork":
            a.fork(ev.parent)
        elif k == "Prefill":
            a.append_n(ev.seq, ev.n)
        elif k == "Step":
            for s in ev.seqs:
                a.append(s)
    bt, cl = runner.tables_for(a, w.decode_seqs)
    share = P.share_groups(bt, cl, w.block_size)
    assert share[:, 0].tolist() == [8 * (i // 8) for i in range(128)]
    assert set(share[:, 1].tolist()) == {prompt_blocks}
    check_valid_and_maximal(bt, cl, w.block_size, share)


def test_multiturn_groups():
    w = W.by_name("long_multiturn_bf16")
    a = P.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    for ev in w.events:
        k = type(ev).__name__
        if k == "NewSeq":
            a.new_seq()
        elif k == "Fork":
            a.fork(ev.parent)
        elif k == "Prefill":
            a.append_n(ev.seq, ev.n)
        elif k == "Step":
            for s in ev.seqs:
                a.append(s)
    bt, cl = runner.tables_for(a, w.decode_seqs)
    share = P.share_groups(bt, cl, w.block_size)
    check_valid_and_maximal(bt, cl, w.block_size, share)
    nbs = (cl + w.block_size - 1) // w.block_size
    for g in range(64):
        want = int(np.floor(0.6 * nbs[4 * g:4 * g + 4].min()))
        got = share[4 * g:4 * g + 4]
        if want > 0:
            assert got.tolist() == [[4 * g, want]] * 4
        else:
            assert got.tolist() == [[-1, 0]] * 4


def test_share_saving_counts_every_member_but_the_first():
    # two groups: 3 members x 4 shared blocks, 2 members x 1 block; one loner
    share = np.array([[0, 4], [0, 4], [0, 4], [3, 1], [3, 1], [-1, 0]], dtype=np.int32)
    cl = np.array([80, 70, 65, 20, 30, 16], dtype=np.int32)     # B = 16: 5+5+5+2+2+1 blocks
    assert P.share_saving(share, cl, 16) == pytest.approx((2 * 4 + 1 * 1) / 20)
    assert P.share_saving(np.full((2, 2), -1, np.int32), np.array([5, 9]), 16) == 0.0
