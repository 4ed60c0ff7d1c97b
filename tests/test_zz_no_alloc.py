"""pa_decode_noalloc: the decode entry point that allocates nothing.

It serves callers that may not allocate device memory while they run (an engine
plugin whose buffers were planned up front, an embedded runtime with a fixed
budget, a C caller without a device allocator): its split-KV scratch is a fixed
array inside the library instead of a caller workspace.  These tests call it
through the C ABI and check it against pa_decode with a caller workspace (bit for
bit) and the oracle, on calls in a row of different shapes, with fixed partitions
and with the balanced split (the second call must not see the first call's
leftovers).  The file is named to be collected last."""
import math

import pytest
import torch

import oracle
import paged_kv_cache_79_gb300 as P
from paged_kv_cache_79_gb300 import _lib
from tests.gpu_harness import assert_close, raw, small_case

pytestmark = pytest.mark.gpu
DEV = "cuda"
CAPACITY = 64 << 20   # PA_DECODE_NOALLOC_SCRATCH_BYTES in include/pagedkv.h


def _noalloc(out, q, kc, vc, bt, cl, scale, hq, hkv, d, b, part):
    lib = _lib.load()
    return lib.pa_decode_noalloc(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                 bt.data_ptr(), bt.shape[1], cl.data_ptr(), q.shape[0], kc.shape[0],
                                 scale, hq, hkv, d, b, {torch.float32: 0, torch.float16: 1,
                                                        torch.bfloat16: 2}[q.dtype], part,
                                 torch.cuda.current_stream().cuda_stream)


CALLS = [  # calls in a row with different shapes
    ("bf16", 128, 16, 16, 2, [3000, 17, 1500, 700], 256),      # fixed partitions + merge kernel
    ("f32", 64, 32, 8, 8, [900, 2, 333], 64),
    # balanced split: the split units' merge counters and partial rows live in the
    # fixed array and keep the previous call's contents; long units are cut over
    # many CTAs
    ("bf16", 128, 32, 32, 8, [20000, 129, 7], 0),
    ("f16", 128, 16, 40, 40, [1500, 33, 2048], 0),
]


def _case(i, dtype, D, B, hq, hkv, lens):
    return [t.to(DEV) for t in small_case(40 + i, dtype, D, B, hq, hkv, lens)]


def test_noalloc_matches_pa_decode_on_two_calls_in_a_row():
    """Each call equals pa_decode with a caller workspace bit for bit (same kernels,
    same schedule) and the oracle within tolerance; the calls alternate with
    pa_decode calls, so the array holds another shape's leftovers every time."""
    for i, (dtype, D, B, hq, hkv, lens, part) in enumerate(CALLS):
        q, kc, vc, bt, cl = _case(i, dtype, D, B, hq, hkv, lens)
        scale = 1.0 / math.sqrt(D)
        need = P.pa_decode_workspace_size(q.shape[0], hq, hkv, D, B, bt.shape[1], part)
        assert 0 < need <= CAPACITY
        ref = torch.empty_like(q)
        P.pa_decode(ref, q, kc, vc, bt, cl, scale, hq, hkv, D, B, partition_size=part)
        got = torch.full_like(q, float("nan"))
        assert _noalloc(got, q, kc, vc, bt, cl, scale, hq, hkv, D, B, part) == P.PA_OK
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {i}: differs from pa_decode"
        want = oracle.decode(raw(q), raw(kc), raw(vc), bt.cpu().numpy(), cl.cpu().numpy(), scale, dtype, hq,
                             hkv, D, B)
        assert_close(got, want, dtype, f"call {i}")
    assert P.pa_device_errors() == 0


def test_noalloc_back_to_back_balanced_calls():
    """Two balanced-split calls of different shapes enqueued back to back, with no
    synchronisation between them: the second reuses the array (and the counters
    the first left) right after the first, in stream order."""
    cases = [CALLS[2], CALLS[3]]
    ins, outs = [], []
    for i, (dtype, D, B, hq, hkv, lens, part) in enumerate(cases):
        ins.append(_case(10 + i, dtype, D, B, hq, hkv, lens))
    for i, (dtype, D, B, hq, hkv, lens, part) in enumerate(cases):
        q, kc, vc, bt, cl = ins[i]
        outs.append(torch.full_like(q, float("nan")))
        assert _noalloc(outs[i], q, kc, vc, bt, cl, 0.09, hq, hkv, D, B, part) == P.PA_OK
    torch.cuda.synchronize()
    for i, (dtype, D, B, hq, hkv, lens, part) in enumerate(cases):
        q, kc, vc, bt, cl = ins[i]
        ref = torch.empty_like(q)
        P.pa_decode(ref, q, kc, vc, bt, cl, 0.09, hq, hkv, D, B, partition_size=part)
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref), f"back-to-back call {i}"
    assert P.pa_device_errors() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    S, hq, hkv, D, B, W = 64, 64, 8, 128, 16, 4096
    need = P.pa_decode_workspace_size(S, hq, hkv, D, B, W, 256)
    assert need > CAPACITY
    x = torch.empty(16, dtype=torch.bfloat16, device=DEV)   # never read: rejected first
    i32 = torch.zeros(16, dtype=torch.int32, device=DEV)
    lib = _lib.load()
    st = lib.pa_decode_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), i32.data_ptr(), W,
                               i32.data_ptr(), S, 100, 0.1, hq, hkv, D, B, 2, 256,
                               torch.cuda.current_stream().cuda_stream)
    assert st == P.PA_ERR_UNSUPPORTED
