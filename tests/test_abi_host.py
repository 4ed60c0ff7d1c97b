"""The C ABI on the host (no GPU needed): exports, validation, allocator parity."""
import ctypes
import re
import subprocess

import numpy as np
import pytest

import oracle
import paged_kv_cache_79_gb300 as P
import workloads as W
from paged_kv_cache_79_gb300 import _lib, build as B

HEADER = B.INCLUDE + "/pagedkv.h"


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported():
    lib = _lib.load()
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    dyn = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (pa_[a-z0-9_]+)$", dyn, flags=re.M))
    assert set(names) <= exported, set(names) - exported


def test_binding_declares_every_function():
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_wait_limit_round_trip():
    """pa_set_wait_limit_ns returns the previous limit; 0 restores the 2 s default."""
    assert P.pa_set_wait_limit_ns(1000) == P.PA_WAIT_LIMIT_DEFAULT_NS
    assert P.pa_set_wait_limit_ns(0) == 1000
    assert P.pa_set_wait_limit_ns(0) == P.PA_WAIT_LIMIT_DEFAULT_NS


def test_status_strings():
    for s in range(6):
        assert P.pa_status_string(s)
    assert P.pa_status_string(99) == "unknown status"


FAKE = 1 << 20   # a 16-byte aligned non-null value; never dereferenced: validation fails first


def _decode(**kw):
    args = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, W=4, cl=FAKE, S=2, NB=8, scale=0.1, Hq=4,
                Hkv=2, D=128, B=16, dt=2, part=0, ws=None, wsb=0, st=None)
    args.update(kw)
    a = args
    return _lib.load().pa_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["W"], a["cl"], a["S"],
                                 a["NB"], a["scale"], a["Hq"], a["Hkv"], a["D"], a["B"], a["dt"],
                                 a["part"], a["ws"], a["wsb"], a["st"])


@pytest.mark.parametrize("kw,want", [
    (dict(out=None), P.PA_ERR_INVALID),
    (dict(q=FAKE + 2), P.PA_ERR_INVALID),
    (dict(k=FAKE + 8), P.PA_ERR_INVALID),
    (dict(Hq=5), P.PA_ERR_INVALID),
    (dict(Hkv=0), P.PA_ERR_INVALID),
    (dict(NB=0), P.PA_ERR_INVALID),
    (dict(W=0), P.PA_ERR_INVALID),
    (dict(part=24), P.PA_ERR_INVALID),
    (dict(part=-16), P.PA_ERR_INVALID),
    (dict(S=-1), P.PA_ERR_INVALID),
    (dict(D=96), P.PA_ERR_UNSUPPORTED),
    (dict(D=256), P.PA_ERR_UNSUPPORTED),
    (dict(B=8), P.PA_ERR_UNSUPPORTED),
    (dict(dt=7), P.PA_ERR_UNSUPPORTED),
    (dict(NB=1 << 28), P.PA_ERR_INVALID),
    (dict(S=0, out=None), P.PA_OK),
])
def test_decode_validation(kw, want):
    assert _decode(**kw) == want


def test_cache_op_validation():
    L = _lib.load()
    assert L.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 128, 16, 4, 2, None) == P.PA_OK
    assert L.pa_reshape_and_cache(None, FAKE, FAKE, FAKE, FAKE, 1, 8, 128, 16, 4, 2, None) == P.PA_ERR_INVALID
    assert L.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 1, 8, 128, 16, 4, 2, None) == P.PA_ERR_INVALID
    assert L.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 6, 16, 4, 2, None) == P.PA_ERR_UNSUPPORTED
    assert L.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 16, 4, 9, None) == P.PA_ERR_UNSUPPORTED
    assert L.pa_copy_blocks(FAKE, FAKE, FAKE, 0, 4, 64, None) == P.PA_OK
    assert L.pa_copy_blocks(FAKE, FAKE, FAKE, 2, 4, 24, None) == P.PA_ERR_INVALID
    assert L.pa_copy_blocks(None, FAKE, FAKE, 2, 4, 64, None) == P.PA_ERR_INVALID
    assert L.pa_copy_blocks(FAKE, FAKE, FAKE, -1, 4, 64, None) == P.PA_ERR_INVALID


def test_block_move_validation():
    # every check below returns before any CUDA call (nothing is launched)
    L = _lib.load()
    assert L.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 4, 64, None) == P.PA_OK
    assert L.pa_swap_blocks(None, FAKE, FAKE, FAKE, FAKE, 2, 4, 4, 64, None) == P.PA_ERR_INVALID
    assert L.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, None, 2, 4, 4, 64, None) == P.PA_ERR_INVALID
    assert L.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 4, 24, None) == P.PA_ERR_INVALID
    assert L.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 0, 4, 64, None) == P.PA_ERR_INVALID
    assert L.pa_swap_blocks(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 2, 4, 4, 64, None) == P.PA_ERR_INVALID
    assert L.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 4, 16 * 65536 * 1024 + 16, None) == \
        P.PA_ERR_UNSUPPORTED
    gather = lambda ids, n, nbytes: L.pa_gather_blocks(FAKE, FAKE, ids, n, 4, FAKE, FAKE, nbytes, None)
    scatter = lambda ids, n, nbytes: L.pa_scatter_blocks(FAKE, FAKE, FAKE, FAKE, ids, n, 4, nbytes, None)
    for fn in (gather, scatter):
        assert fn(FAKE, 0, 64) == P.PA_OK
        assert fn(None, 3, 64) == P.PA_ERR_INVALID
        assert fn(FAKE, -1, 64) == P.PA_ERR_INVALID
        assert fn(FAKE, 3, 40) == P.PA_ERR_INVALID
    assert L.pa_kv_transfer_worthwhile(64, 64) == 1 and L.pa_kv_transfer_worthwhile(63, 64) == 0


def test_shared_decode_validation():
    L = _lib.load()
    args = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, kn=None, vn=None, bt=FAKE, W=4, cl=FAKE, share=FAKE,
                S=2, NB=8, scale=0.1, hq=8, hkv=8, d=128, b=16, dt=1, ws=FAKE, wsb=1 << 30)

    def call(**kw):
        a = dict(args, **kw)
        return L.pa_decode_shared(a["out"], a["q"], a["kc"], a["vc"], a["kn"], a["vn"], a["bt"], a["W"],
                                  a["cl"], a["share"], a["S"], a["NB"], a["scale"], a["hq"], a["hkv"],
                                  a["d"], a["b"], a["dt"], a["ws"], a["wsb"], None)
    assert call(S=0) == P.PA_OK
    assert call(share=None) == P.PA_ERR_INVALID
    assert call(share=FAKE + 4) == P.PA_ERR_INVALID              # share needs 8-byte alignment
    assert call(kn=FAKE) == P.PA_ERR_INVALID                     # k_new without v_new
    assert call(hq=40, hkv=2) == P.PA_ERR_UNSUPPORTED            # 20 query heads per kv head
    assert P.pa_decode_shared_workspace_size(2, 8, 8, 128, 16, 4) > P.pa_decode_workspace_size(
        2, 8, 8, 128, 16, 4, 0)


def test_workspace_size_formula():
    # one partition: no workspace; several: fp32 partials + log-sum-exp per (seq, part, head)
    assert P.pa_decode_workspace_size(4, 8, 8, 64, 16, 4, 64) == 0
    n = P.pa_decode_workspace_size(4, 8, 2, 64, 16, 10, 64)   # 4 blocks per partition -> 3 parts
    rows = 4 * 3 * 8
    assert n == ((rows * 64 * 4 + 255) // 256) * 256 + rows * 4
    with pytest.raises(P.PagedKVError):
        P.pa_decode_workspace_size(4, 8, 3, 64, 16, 10, 64)


def test_partition_size_resolution():
    # 0 selects the balanced split; a fixed size is capped at the table capacity
    assert P.pa_decode_partition_size(8, 40, 40, 128, 16, 128, 0) == 0
    assert P.pa_decode_partition_size(8, 40, 40, 128, 16, 128, 512) == 512
    assert P.pa_decode_partition_size(8, 40, 40, 128, 16, 4, 512) == 64
    assert P.pa_decode_partition_size(8, 40, 40, 128, 16, 4, 24) == -1


def test_balanced_workspace_does_not_depend_on_lengths():
    a = P.pa_decode_workspace_size(8, 40, 40, 128, 16, 128, 0)
    b = P.pa_decode_workspace_size(256, 32, 8, 128, 32, 4096, 0)
    assert a == b > 0


def test_balanced_workspace_formula():
    # C = 4 CTAs per SM at most: C merge counters, then 2 * C * 16 fp32 rows of d
    # values and their log2-sum-exp
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 160
    C = 4 * sms
    rows = 2 * C * 16
    align = lambda n: (n + 255) // 256 * 256
    for d in (64, 128):
        assert P.pa_decode_workspace_size(3, 8, 8, d, 16, 7, 0) == align(C * 8) + align(rows * d * 4) + rows * 4


# ---------------------------------------------------------------------------
# allocator: the library's C++ allocator against the oracle's Python allocator
# ---------------------------------------------------------------------------
def _state(a, seqs):
    return ([a.block_table(s) for s in seqs], [a.seq_len(s) for s in seqs],
            [a.refcount(b) for b in range(a.num_blocks)], a.free_list())


@pytest.mark.parametrize("seed", range(8))
def test_allocator_matches_oracle_on_random_traces(seed):
    rng = np.random.default_rng(100 + seed)
    nb, bs = int(rng.integers(4, 40)), int(rng.choice([1, 2, 4, 16]))
    order = rng.permutation(nb)
    lib_a = P.BlockAllocator(nb, bs, order)
    ora_a = oracle.BlockAllocator(nb, bs, order)
    live = []
    for _ in range(300):
        r = rng.random()
        if r < 0.1 or not live:
            assert lib_a.new_seq() == ora_a.new_seq()
            live.append(ora_a._next_id - 1)
        elif r < 0.2:
            p = live[rng.integers(len(live))]
            assert lib_a.fork(p) == ora_a.fork(p)
            live.append(ora_a._next_id - 1)
        elif r < 0.27:
            s = live.pop(rng.integers(len(live)))
            lib_a.free_seq(s)
            ora_a.free_seq(s)
        else:
            s = live[rng.integers(len(live))]
            try:
                want = ora_a.append(s)
            except MemoryError:
                with pytest.raises(MemoryError):
                    lib_a.append(s)
            else:
                assert lib_a.append(s) == want
        assert _state(lib_a, live) == _state(ora_a, live)


@pytest.mark.parametrize("name", ["tiny", "mha_fp16", "shared_prefix_fp16", "shared_prefix_fp16_p1032"])
def test_allocator_matches_oracle_on_workload_scripts(name):
    from paged_kv_cache_79_gb300 import runner
    w = W.by_name(name)
    lib_a = P.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    lib_pairs = []
    for ev in w.events:
        k = type(ev).__name__
        if k == "NewSeq":
            lib_a.new_seq()
        elif k == "Fork":
            lib_a.fork(ev.parent)
        elif k == "Prefill":
            _, pr = lib_a.append_n(ev.seq, ev.n)
            lib_pairs += [tuple(x) for x in pr.tolist()]
        elif k == "Step":
            for s in ev.seqs:
                _, c = lib_a.append(s)
                if c:
                    lib_pairs.append(c)
    ora_a, recs = oracle.run_script(w.events, w.num_blocks, w.block_size, w.free_order)
    ora_pairs = [p for _, _, ps in recs for p in ps]
    assert lib_pairs == ora_pairs
    assert _state(lib_a, w.decode_seqs) == _state(ora_a, w.decode_seqs)
    bt, cl = runner.tables_for(lib_a, w.decode_seqs)
    bt2, cl2 = oracle.tables_for(ora_a, w.decode_seqs)
    assert np.array_equal(bt, bt2) and np.array_equal(cl, cl2)
    if name == "shared_prefix_fp16":
        assert lib_pairs == []            # block-aligned prompt: nothing to copy
    if name == "shared_prefix_fp16_p1032":
        assert len(lib_pairs) == 16 * 7   # every sample but the last holder copies


def test_allocator_append_n_oom_keeps_earlier_appends():
    a = P.BlockAllocator(2, 2)
    s = a.new_seq()
    with pytest.raises(MemoryError):
        a.append_n(s, 5)
    assert a.seq_len(s) == 4 and a.num_free() == 0


def test_allocator_rejects_bad_free_order():
    with pytest.raises(P.PagedKVError):
        P.BlockAllocator(3, 4, [0, 0, 1])
    with pytest.raises(P.PagedKVError):
        P.BlockAllocator(3, 4, [0, 1, 3])
