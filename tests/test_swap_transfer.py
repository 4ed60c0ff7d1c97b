"""Swap space and KV-transfer staging on the host (no GPU).

Oracle pins: the azimuth.plus summary, section "vLLM", fixes what swapping must
preserve -- a preempted request resumes with the same keys and values -- and the
block manager's bookkeeping (reference counts, free list) must stay consistent.
The spke.com article on bidirectional KV transfer, section "KV recompute
threshold", fixes the transfer-or-recompute rule (64 tokens by default).  Then the
library's C++ allocator must agree with the oracle's, move for move."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_79_gb300 as P
from oracle import BlockAllocator, OracleOOM


def tokens_of(a, seq, kc, host_kc):
    """A sequence's key rows in order, read through its table from the pool it is in."""
    pool = host_kc if a.is_swapped(seq) else kc
    B = a.block_size
    T = a.seq_len(seq)
    tab = a.block_table(seq)
    return np.stack([pool[tab[t // B], t % B] for t in range(T)]) if T else np.zeros((0,) + kc.shape[2:])


def conserved(a, live):
    """References equal table entries; free lists hold exactly the unreferenced blocks."""
    dev = [0] * a.num_blocks
    host = [0] * len(a.host_ref)
    for s in live:
        for b in a.block_table(s):
            (host if a.is_swapped(s) else dev)[b] += 1
    assert dev == [a.refcount(b) for b in range(a.num_blocks)]
    assert host == [a.host_refcount(b) for b in range(len(a.host_ref))]
    assert sorted(a.free_list()) == [b for b in range(a.num_blocks) if dev[b] == 0]
    assert sorted(a.host_free_list()) == [b for b in range(len(a.host_ref)) if host[b] == 0]


def test_swap_round_trip_keeps_every_token():
    rng = np.random.default_rng(1)
    a = BlockAllocator(12, 4, free_order=rng.permutation(12))
    a.set_host_pool(10)
    kc = np.zeros((12, 4, 1, 2))
    hk = np.full((10, 4, 1, 2), np.nan)
    s0 = a.new_seq()
    for t in range(9):
        slot, _ = a.append(s0)
        kc[slot // 4, slot % 4] = [t, -t]
    s1 = a.fork(s0)
    slot, cow = a.append(s1)                    # s1 writes into the shared partial block
    oracle.copy_blocks(kc, kc.copy(), [cow])
    kc[slot // 4, slot % 4] = [100, 100]
    before = {s: tokens_of(a, s, kc, hk).copy() for s in (s0, s1)}
    pairs = a.swap_out([s0, s1])
    hv = hk.copy()
    oracle.swap_blocks(kc, kc, hk, hv, pairs)
    # distinct blocks copied once: 2 shared full blocks + 2 private partial blocks
    assert len(pairs) == 4 and a.num_free() == 12
    assert all(a.is_swapped(s) for s in (s0, s1))
    conserved(a, [s0, s1])
    kc[:] = np.nan                               # the device blocks are reused by others
    for s in (s0, s1):
        assert np.array_equal(tokens_of(a, s, kc, hk), before[s])
    back = a.swap_in([s1, s0])
    oracle.swap_blocks(hk, hv, kc, kc.copy(), back)
    conserved(a, [s0, s1])
    for s in (s0, s1):
        assert not a.is_swapped(s)
        assert np.array_equal(tokens_of(a, s, kc, hk), before[s])
    # the two shared blocks are still shared after the round trip
    assert a.block_table(s0)[:2] == a.block_table(s1)[:2]
    assert a.refcount(a.block_table(s0)[0]) == 2


def test_swapping_one_sharer_copies_the_shared_block():
    a = BlockAllocator(8, 2)
    a.set_host_pool(8)
    s0 = a.new_seq()
    for _ in range(4):
        a.append(s0)
    s1 = a.fork(s0)
    pairs = a.swap_out([s1])
    assert [d for d, _ in pairs] == a.block_table(s0)       # both shared blocks copied
    assert all(a.refcount(b) == 1 for b in a.block_table(s0))
    assert all(a.host_refcount(h) == 1 for h in a.block_table(s1))
    conserved(a, [s0, s1])


def test_swap_errors_change_nothing():
    a = BlockAllocator(6, 2)
    a.set_host_pool(1)
    s = a.new_seq()
    for _ in range(4):
        a.append(s)
    snap = (a.block_table(s), a.free_list(), a.host_free_list())
    with pytest.raises(OracleOOM):
        a.swap_out([s])                          # two blocks, one host block
    assert (a.block_table(s), a.free_list(), a.host_free_list()) == snap
    with pytest.raises(ValueError):
        a.swap_in([s])                           # not swapped out
    with pytest.raises(ValueError):
        a.swap_out([s, s])
    a.set_host_pool(4)
    a.swap_out([s])
    with pytest.raises(ValueError):
        a.append(s)
    with pytest.raises(ValueError):
        a.fork(s)
    a.free_seq(s)                                # releases the host blocks
    assert a.num_free_host() == 4 and a.num_free() == 6


@pytest.mark.parametrize("seed", range(6))
def test_random_traces_with_swaps_conserve_references(seed):
    rng = np.random.default_rng(40 + seed)
    a = BlockAllocator(30, 4, free_order=rng.permutation(30))
    a.set_host_pool(30)
    live = []
    for _ in range(400):
        r = rng.random()
        try:
            if r < 0.1 or not live:
                live.append(a.new_seq())
            elif r < 0.18:
                p = live[rng.integers(len(live))]
                if not a.is_swapped(p):
                    live.append(a.fork(p))
            elif r < 0.24:
                a.free_seq(live.pop(rng.integers(len(live))))
            elif r < 0.32:
                pick = sorted(set(rng.choice(live, size=min(len(live), 3)).tolist()))
                if all(not a.is_swapped(q) for q in pick):
                    a.swap_out(pick)
            elif r < 0.40:
                pick = [q for q in live if a.is_swapped(q)][:3]
                if pick:
                    a.swap_in(pick)
            else:
                q = live[rng.integers(len(live))]
                if not a.is_swapped(q):
                    a.append(q)
        except OracleOOM:
            pass
        conserved(a, live)


def test_staging_round_trip_moves_a_sequence_between_pools():
    rng = np.random.default_rng(3)
    src = BlockAllocator(20, 4, free_order=rng.permutation(20))
    kc = rng.standard_normal((20, 4, 2, 3))
    vc = rng.standard_normal((20, 4, 2, 3))
    s = src.new_seq()
    for _ in range(13):
        src.append(s)
    ks, vs = oracle.gather_blocks(kc, vc, src.block_table(s))
    dst = BlockAllocator(9, 4)
    d = dst.new_seq()
    for _ in range(13):
        dst.append(d)
    k2 = np.zeros((9, 4, 2, 3))
    v2 = np.zeros_like(k2)
    oracle.scatter_blocks(ks, vs, k2, v2, dst.block_table(d))
    for t in range(13):
        b0, b1 = src.block_table(s)[t // 4], dst.block_table(d)[t // 4]
        assert np.array_equal(kc[b0, t % 4], k2[b1, t % 4])
        assert np.array_equal(vc[b0, t % 4], v2[b1, t % 4])


def test_recompute_threshold_of_the_article():
    """Below the threshold (default 64) the prefill side recomputes; at or above it
    fetches the KV."""
    assert not oracle.kv_transfer_worthwhile(63)
    assert oracle.kv_transfer_worthwhile(64)
    assert oracle.kv_transfer_worthwhile(5000)
    assert not oracle.kv_transfer_worthwhile(0, threshold=0)
    for n in (-1, 0, 1, 63, 64, 65, 10 ** 6):
        for th in (0, 1, 64, 128):
            assert P.pa_kv_transfer_worthwhile(n, th) == oracle.kv_transfer_worthwhile(n, th)


# ---------------------------------------------------------------------------
# the library's allocator against the oracle's
# ---------------------------------------------------------------------------
def _state(a, seqs):
    return ([a.block_table(s) for s in seqs], [a.seq_len(s) for s in seqs],
            [a.is_swapped(s) for s in seqs],
            [a.refcount(b) for b in range(a.num_blocks)], a.free_list(),
            [a.host_refcount(b) for b in range(a.num_host_blocks)], a.host_free_list())


@pytest.mark.parametrize("seed", range(10))
def test_library_allocator_swaps_like_the_oracle(seed):
    rng = np.random.default_rng(500 + seed)
    nb, bs, hb = int(rng.integers(6, 40)), int(rng.choice([1, 2, 4, 16])), int(rng.integers(0, 40))
    order = rng.permutation(nb)
    lib_a = P.BlockAllocator(nb, bs, order)
    ora_a = BlockAllocator(nb, bs, order)
    lib_a.set_host_pool(hb)
    ora_a.set_host_pool(hb)
    ora_a.num_host_blocks = hb
    live = []
    for _ in range(400):
        r = rng.random()
        if r < 0.1 or not live:
            assert lib_a.new_seq() == ora_a.new_seq()
            live.append(ora_a._next_id - 1)
            continue
        q = live[rng.integers(len(live))]
        if r < 0.17:
            if ora_a.is_swapped(q):
                with pytest.raises(P.PagedKVError):
                    lib_a.fork(q)
                continue
            assert lib_a.fork(q) == ora_a.fork(q)
            live.append(ora_a._next_id - 1)
        elif r < 0.23:
            live.remove(q)
            lib_a.free_seq(q)
            ora_a.free_seq(q)
        elif r < 0.35:
            pick = sorted(set(rng.choice(live, size=min(len(live), int(rng.integers(1, 4)))).tolist()))
            out = not ora_a.is_swapped(pick[0])
            try:
                want = ora_a.swap_out(pick) if out else ora_a.swap_in(pick)
            except OracleOOM:
                with pytest.raises(MemoryError):
                    lib_a.swap_out(pick) if out else lib_a.swap_in(pick)
            except ValueError:
                with pytest.raises(P.PagedKVError):
                    lib_a.swap_out(pick) if out else lib_a.swap_in(pick)
            else:
                got = lib_a.swap_out(pick) if out else lib_a.swap_in(pick)
                assert [tuple(x) for x in got.tolist()] == want
        else:
            if ora_a.is_swapped(q):
                with pytest.raises(P.PagedKVError):
                    lib_a.append(q)
                continue
            try:
                want = ora_a.append(q)
            except MemoryError:
                with pytest.raises(MemoryError):
                    lib_a.append(q)
            else:
                assert lib_a.append(q) == want
        assert _state(lib_a, live) == _state(ora_a, live)
