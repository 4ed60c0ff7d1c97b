"""Oracle allocator, reshape_and_cache and copy_blocks against the pages (CPU only)."""
import numpy as np
import pytest

import oracle
import workloads as W
from oracle import BlockAllocator, OracleOOM


def test_tutorial_workflow_allocation():
    """CSDN tutorial §4: 100 pages of 16 tokens, 50 appends.  §2.2 builds the free
    list as list(range(total_pages)) and pops from its end, so pages 99, 98, 97, 96
    are allocated at steps 0, 16, 32, 48 ('Step 16 ... a new page is allocated')."""
    a = BlockAllocator(100, 16)
    s = a.new_seq()
    slots = [a.append(s)[0] for _ in range(50)]
    assert a.block_table(s) == [99, 98, 97, 96]
    assert slots[0] == 99 * 16 and slots[15] == 99 * 16 + 15
    assert slots[16] == 98 * 16
    assert slots[49] == 96 * 16 + 1              # the fourth page holds 2 tokens
    assert a.num_free() == 96
    assert all(a.refcount(b) == 1 for b in (96, 97, 98, 99))


def test_oom_is_memory_error_and_changes_nothing():
    """Tutorial §2.2: allocate_page raises MemoryError on an empty free list."""
    a = BlockAllocator(2, 1, free_order=[1, 0])
    s = a.new_seq()
    a.append(s)
    a.append(s)
    snap = (a.free_list(), list(a.ref), a.block_table(s), a.seq_len(s))
    with pytest.raises(MemoryError):
        a.append(s)
    assert snap == (a.free_list(), list(a.ref), a.block_table(s), a.seq_len(s))


def test_oom_during_copy_on_write_changes_nothing():
    a = BlockAllocator(1, 4)
    p = a.new_seq()
    a.append(p)
    c = a.fork(p)
    snap = (a.free_list(), list(a.ref), a.block_table(p), a.block_table(c), a.seq_len(c))
    with pytest.raises(OracleOOM):
        a.append(c)
    assert snap == (a.free_list(), list(a.ref), a.block_table(p), a.block_table(c), a.seq_len(c))


def test_fork_shares_and_counts_references():
    """Tutorial §5.1 clone_sequence: the clone copies the table, ref_count += 1."""
    a = BlockAllocator(10, 4, free_order=list(range(10)))
    p = a.new_seq()
    for _ in range(6):
        a.append(p)
    c = a.fork(p)
    assert a.block_table(c) == a.block_table(p) == [9, 8]
    assert a.refcount(9) == 2 and a.refcount(8) == 2
    assert a.seq_len(c) == 6


def test_free_returns_blocks_at_refcount_zero():
    """Tutorial §2.2 free_page: decrement; back on the free list at 0."""
    a = BlockAllocator(6, 2, free_order=list(range(6)))
    p = a.new_seq()
    for _ in range(4):
        a.append(p)                               # blocks 5, 4
    c = a.fork(p)
    a.free_seq(p)
    assert a.free_list() == [0, 1, 2, 3]
    assert a.refcount(5) == 1 and a.refcount(4) == 1
    a.free_seq(c)
    assert a.free_list() == [0, 1, 2, 3, 5, 4]   # table order, appended at the end


def test_copy_on_write_copies_only_the_shared_partial_block():
    """azimuth.plus summary, 'Memory sharing': writing into a shared block copies
    that block only and changes only the writer's table; the last holder writes in
    place."""
    a = BlockAllocator(8, 4, free_order=list(range(8)))
    p = a.new_seq()
    for _ in range(6):                            # blocks 7 (full), 6 (2 of 4 rows)
        a.append(p)
    c = a.fork(p)
    slot, cow = a.append(c)
    assert cow == (6, 5)
    assert a.block_table(c) == [7, 5] and a.block_table(p) == [7, 6]
    assert slot == 5 * 4 + 2
    assert a.refcount(6) == 1 and a.refcount(5) == 1 and a.refcount(7) == 2
    slot, cow = a.append(p)                       # parent is now the only holder of 6
    assert cow is None and slot == 6 * 4 + 2


def test_block_aligned_fork_never_copies():
    a = BlockAllocator(8, 4)
    p = a.new_seq()
    for _ in range(8):
        a.append(p)
    c = a.fork(p)
    _, cow = a.append(c)
    assert cow is None and a.block_table(c)[:2] == a.block_table(p)


def _check_conservation(a: BlockAllocator):
    used = {}
    for t in a.tables.values():
        for b in t:
            used[b] = used.get(b, 0) + 1
    assert len(a.free) + len(used) == a.num_blocks
    assert not (set(a.free) & set(used))
    for b in range(a.num_blocks):
        assert a.refcount(b) == used.get(b, 0)
    for s, t in a.tables.items():
        assert len(t) == (a.seq_len(s) + a.block_size - 1) // a.block_size


@pytest.mark.parametrize("seed", range(6))
def test_random_traces_conserve_blocks_and_references(seed):
    rng = np.random.default_rng(seed)
    a = BlockAllocator(64, 4, free_order=rng.permutation(64))
    live = []
    for _ in range(400):
        r = rng.random()
        try:
            if r < 0.1 or not live:
                live.append(a.new_seq())
            elif r < 0.2:
                live.append(a.fork(live[rng.integers(len(live))]))
            elif r < 0.27:
                a.free_seq(live.pop(rng.integers(len(live))))
            else:
                a.append(live[rng.integers(len(live))])
        except MemoryError:
            pass
        _check_conservation(a)


def test_reshape_and_cache_round_trip():
    """Appending T tokens, then gathering rows through the table, returns them in order."""
    rng = np.random.default_rng(3)
    B, H, d, T = 4, 2, 8, 19
    a = BlockAllocator(9, B, free_order=rng.permutation(9))
    s = a.new_seq()
    k = rng.standard_normal((T, H, d)).astype(np.float32)
    v = rng.standard_normal((T, H, d)).astype(np.float32)
    kc = np.full((9, B, H, d), np.nan, np.float32)
    vc = np.full((9, B, H, d), np.nan, np.float32)
    slots = np.array([a.append(s)[0] for _ in range(T)])
    oracle.reshape_and_cache(k, v, kc, vc, slots, B)
    tab = a.block_table(s)
    back_k = np.stack([kc[tab[t // B], t % B] for t in range(T)])
    back_v = np.stack([vc[tab[t // B], t % B] for t in range(T)])
    assert np.array_equal(back_k, k) and np.array_equal(back_v, v)
    assert np.isnan(kc[tab[-1], T % B:]).all()            # rows past T untouched


def test_reshape_and_cache_negative_slot_skips():
    kc = np.zeros((2, 2, 1, 2), np.float32)
    vc = np.zeros((2, 2, 1, 2), np.float32)
    k = np.ones((2, 1, 2), np.float32)
    oracle.reshape_and_cache(k, 2 * k, kc, vc, np.array([-1, 3]), 2)
    assert kc[1, 1].tolist() == [[1.0, 1.0]] and vc[1, 1].tolist() == [[2.0, 2.0]]
    assert np.count_nonzero(kc) == 2 and np.count_nonzero(vc) == 2


def test_copy_blocks_copies_whole_blocks_only():
    rng = np.random.default_rng(4)
    kc = rng.standard_normal((6, 4, 2, 8)).astype(np.float16)
    vc = rng.standard_normal((6, 4, 2, 8)).astype(np.float16)
    k0, v0 = kc.copy(), vc.copy()
    oracle.copy_blocks(kc, vc, [(1, 4), (2, 0)])
    assert np.array_equal(kc[4], k0[1]) and np.array_equal(vc[4], v0[1])
    assert np.array_equal(kc[0], k0[2]) and np.array_equal(vc[0], v0[2])
    for b in (1, 2, 3, 5):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])


def test_script_with_cow_keeps_prefix_shared_in_data():
    """After copy-on-write, a forked sample still sees the prompt's K/V rows."""
    w = W.shared_prefix_fp16(prompts=2, samples=3, prompt_len=20, max_cont=6)
    kc = np.zeros((w.num_blocks, 16, 1, 2), np.float32)
    vc = np.zeros_like(kc)
    # tag every row with its (block, row) so copies are traceable
    for b in range(w.num_blocks):
        for r in range(16):
            kc[b, r] = b * 100 + r
    vc[:] = kc
    alloc, recs = oracle.run_script(w.events, w.num_blocks, 16, w.free_order, kc, vc,
                                    step_kv=lambda ev: (np.full((len(ev.seqs), 1, 2), -1, np.float32),) * 2)
    pairs = [p for _, _, ps in recs for p in ps]
    assert len(pairs) == 2 * 2                     # per prompt: samples 0..1 copy, the last writes in place
    for s in w.decode_seqs:
        tab = alloc.block_table(s)
        assert kc[tab[1], :4].tolist() == kc[alloc.block_table(0 if s < 3 else 3)[1], :4].tolist()
    _check_conservation(alloc)
