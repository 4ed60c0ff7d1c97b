"""Block moves on the GPU through the C ABI: swap to pinned host memory and back,
staging for a KV transfer.  Bit-exact against the oracle's byte copies, and a
decode after the round trip equals the decode before it bit for bit (the decode
depends on the data and the lengths, not on which physical blocks hold them)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_79_gb300 as P
import workloads as W
from paged_kv_cache_79_gb300 import runner
from tests.gpu_harness import raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("direction", ["d2h", "h2d", "d2d"])
def test_swap_blocks_bit_exact(dtype, direction):
    rng = np.random.default_rng(7)
    nb_src, nb_dst, shape = 40, 25, (16, 4, 64)
    src_k = W.randn((nb_src,) + shape, dtype, 11)
    src_v = W.randn((nb_src,) + shape, dtype, 12)
    dst_k = W.randn((nb_dst,) + shape, dtype, 13)
    dst_v = W.randn((nb_dst,) + shape, dtype, 14)
    pairs = np.stack([rng.permutation(nb_src)[:20], rng.permutation(nb_dst)[:20]], 1).astype(np.int32)
    pairs[3] = (nb_src + 5, 1)                   # out of range: skipped
    pairs[4] = (2, -1)
    want_k, want_v = raw(dst_k).copy(), raw(dst_v).copy()
    oracle.swap_blocks(raw(src_k), raw(src_v), want_k, want_v, [tuple(p) for p in pairs.tolist()])
    on_dev = {"d2h": (True, False), "h2d": (False, True), "d2d": (True, True)}[direction]
    place = lambda t, d: t.to(DEV) if d else t.pin_memory()
    sk, sv = place(src_k, on_dev[0]), place(src_v, on_dev[0])
    dk, dv = place(dst_k, on_dev[1]), place(dst_v, on_dev[1])
    P.pa_swap_blocks(sk, sv, dk, dv, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(raw(dk), want_k) and np.array_equal(raw(dv), want_v)


@pytest.mark.parametrize("pinned", [False, True])
def test_gather_scatter_bit_exact(pinned):
    rng = np.random.default_rng(9)
    kc = W.randn((30, 16, 8, 128), "bf16", 21).to(DEV)
    vc = W.randn((30, 16, 8, 128), "bf16", 22).to(DEV)
    ids = rng.permutation(30)[:11].astype(np.int32)
    ids_d = torch.from_numpy(ids).to(DEV)
    sk = torch.zeros((11, 16, 8, 128), dtype=torch.bfloat16)
    sv = torch.zeros_like(sk)
    if pinned:
        sk, sv = sk.pin_memory(), sv.pin_memory()
    else:
        sk, sv = sk.to(DEV), sv.to(DEV)
    P.pa_gather_blocks(kc, vc, ids_d, sk, sv)
    torch.cuda.synchronize()
    wk, wv = oracle.gather_blocks(raw(kc), raw(vc), ids.tolist())
    assert np.array_equal(raw(sk), wk) and np.array_equal(raw(sv), wv)
    k2 = torch.zeros_like(kc)
    v2 = torch.zeros_like(vc)
    dst_ids = rng.permutation(30)[:11].astype(np.int32)
    P.pa_scatter_blocks(sk, sv, k2, v2, torch.from_numpy(dst_ids).to(DEV))
    torch.cuda.synchronize()
    hk, hv = raw(k2).copy(), raw(v2).copy()
    hk[:] = 0
    hv[:] = 0
    oracle.scatter_blocks(wk, wv, hk, hv, dst_ids.tolist())
    assert np.array_equal(raw(k2), hk) and np.array_equal(raw(v2), hv)


def _decode(ds, bt, cl):
    out = torch.empty_like(ds.q)
    P.pa_decode(out, ds.q, ds.k_cache, ds.v_cache, torch.from_numpy(bt).to(DEV),
                torch.from_numpy(cl).to(DEV), ds.scale, ds.num_q_heads, ds.num_kv_heads, ds.head_dim,
                ds.block_size, 0)
    torch.cuda.synchronize()
    return out


def _replay(w, kc, vc):
    """Run the workload script; return (allocator, decode step)."""
    return runner.execute(w, kc, vc, lambda ev: W.step_tensors(w, ev, DEV),
                          lambda ev: W.query_tensor(w, ev.index, DEV))


def test_swap_out_and_in_restores_the_decode_bitwise():
    w = W.shared_prefix_fp16(prompts=4, prompt_len=1032)
    kc, vc = W.pool_tensors(w, DEV)
    alloc, ds = _replay(w, kc, vc)
    bt, cl = runner.tables_for(alloc, w.decode_seqs)
    before = _decode(ds, bt, cl)
    seqs = list(w.decode_seqs)
    out_seqs = seqs[4:20]                          # parts of three prompt groups
    n_host = sum(len(alloc.block_table(s)) for s in out_seqs)
    alloc.set_host_pool(n_host)
    host_k = torch.empty((n_host,) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    pairs = alloc.swap_out(out_seqs)
    P.pa_swap_blocks(kc, vc, host_k, host_v, torch.from_numpy(np.ascontiguousarray(pairs)).to(DEV))
    torch.cuda.synchronize()
    # freed device blocks are reused by someone else: scribble over every free block
    free = torch.tensor(alloc.free_list(), dtype=torch.long, device=DEV)
    kc.index_fill_(0, free, float("nan"))
    vc.index_fill_(0, free, float("nan"))
    back = alloc.swap_in(out_seqs)
    P.pa_swap_blocks(host_k, host_v, kc, vc, torch.from_numpy(np.ascontiguousarray(back)).to(DEV))
    bt2, cl2 = runner.tables_for(alloc, w.decode_seqs, width=bt.shape[1])
    assert np.array_equal(cl, cl2) and not np.array_equal(bt, bt2)
    after = _decode(ds, bt2, cl2)
    assert torch.equal(before, after)
    assert P.pa_device_errors() == 0


def test_kv_transfer_between_pools_keeps_the_decode_bitwise():
    """Gather one engine's sequences into a staging buffer (pinned host memory),
    scatter them into fresh blocks of another engine's pool, decode there."""
    w = W.mha_fp16()
    kc, vc = W.pool_tensors(w, DEV)
    alloc, ds = _replay(w, kc, vc)
    bt, cl = runner.tables_for(alloc, w.decode_seqs)
    before = _decode(ds, bt, cl)
    nbs = [(int(t) + w.block_size - 1) // w.block_size for t in cl]
    assert all(P.pa_kv_transfer_worthwhile(int(t)) == (t >= 64) for t in cl)
    ids = np.concatenate([bt[s, :nbs[s]] for s in range(len(cl))]).astype(np.int32)
    sk = torch.empty((len(ids),) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
    sv = torch.empty_like(sk).pin_memory()
    P.pa_gather_blocks(kc, vc, torch.from_numpy(ids).to(DEV), sk, sv)
    # the receiving engine: its own pool and allocator
    nb2 = len(ids) + 50
    recv = P.BlockAllocator(nb2, w.block_size, np.random.default_rng(5).permutation(nb2))
    for t in cl:
        s = recv.new_seq()
        recv.append_n(s, int(t))
    bt2, cl2 = runner.tables_for(recv, range(len(cl)), width=bt.shape[1])
    ids2 = np.concatenate([bt2[s, :nbs[s]] for s in range(len(cl))]).astype(np.int32)
    k2 = torch.full((nb2,) + tuple(kc.shape[1:]), float("nan"), dtype=kc.dtype, device=DEV)
    v2 = torch.full_like(k2, float("nan"))
    P.pa_scatter_blocks(sk, sv, k2, v2, torch.from_numpy(ids2).to(DEV))
    out = torch.empty_like(ds.q)
    P.pa_decode(out, ds.q, k2, v2, torch.from_numpy(bt2).to(DEV), torch.from_numpy(cl2).to(DEV), ds.scale,
                ds.num_q_heads, ds.num_kv_heads, ds.head_dim, ds.block_size, 0)
    torch.cuda.synchronize()
    assert torch.equal(before, out)


def test_pageable_host_memory_is_refused_before_any_launch():
    lib = P._load()
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.float16, device=DEV)
    pageable = np.zeros((4, 16, 2, 64), dtype=np.float16)
    pairs = torch.tensor([[0, 1]], dtype=torch.int32, device=DEV)
    st = lib.pa_swap_blocks(kc.data_ptr(), kc.data_ptr(), pageable.ctypes.data, pageable.ctypes.data,
                            pairs.data_ptr(), 1, 4, 4, 16 * 2 * 64 * 2, None)
    assert st == P.PA_ERR_INVALID
    assert not pageable.any()
