"""Device-side waits that run out.

Every wait inside the decode kernels is bounded.  With the wait limit cut to 1 ns
(pa_set_wait_limit_ns), any wait that lasts longer than a couple of the hardware's
try_wait suspend intervals runs out.  The balanced-split batches here carry 16384
empty sequences behind the real ones: every CTA's producer sums the stream over
all of them (hundreds of memory round trips, tens of microseconds) before it
publishes its first work item, so the consumers' first wait surely runs out.  The launch must then give up: the CTA stops issuing
copies, lets the copies it issued land, and returns.  The call returns, nothing
hangs or faults, pa_device_errors reports the timeout (PA_ERR_TIMEOUT from the C
call), and the next decode with the default limit matches the oracle.  Batches of
long contexts without the padding time out in mid-stream, with copies in flight,
when they time out at all; so do fixed partitions, whose CTAs find their first
items among the first sequences of the batch."""
import ctypes
import math

import pytest
import torch

import oracle
import paged_kv_cache_79_gb300 as P
from paged_kv_cache_79_gb300 import _lib
from tests.gpu_harness import assert_close, raw, small_case

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUTS = P.PA_DEVERR_TIMEOUT_FULL | P.PA_DEVERR_TIMEOUT_EMPTY

PAD = [0] * 16384    # empty sequences: a long walk before any work item

CASES = [
    # dtype, head_dim, block_size, Hq, Hkv, context lengths, partition size
    ("bf16", 128, 16, 64, 8, [30000, 5000, 17, 9000] + PAD, 0),   # tensor-core consumers, 8-row items
    ("f16", 128, 32, 32, 2, [20000, 3] + PAD, 0),                 # 16-row items
    ("f32", 64, 16, 8, 8, [6000, 40] + PAD, 0),                   # CUDA-core consumers
]
MIDSTREAM = [
    ("bf16", 128, 16, 64, 8, [30000, 5000, 17, 9000], 0),
    ("f16", 128, 16, 40, 40, [3000, 2048, 1500, 999, 1200, 64, 2000, 1800], 0),
    ("bf16", 128, 32, 32, 8, [9000, 129], 512),                   # fixed partitions + merge kernel
    ("bf16", 128, 32, 32, 8, [9000, 129] + PAD, 512),
]


def _oracle(q, kc, vc, bt, cl, scale, dtype, hq, hkv, d, b):
    return oracle.decode(raw(q), raw(kc), raw(vc), bt.cpu().numpy(), cl.cpu().numpy(), scale, dtype, hq,
                         hkv, d, b)


def _status_and_flags():
    flags = ctypes.c_uint(0)
    st = _lib.load().pa_device_errors(ctypes.byref(flags), torch.cuda.current_stream().cuda_stream)
    return st, flags.value


@pytest.mark.parametrize("dtype,D,B,hq,hkv,lens,part", CASES, ids=lambda v: str(v).replace(" ", ""))
def test_wait_limit_runs_out_and_the_next_call_is_correct(dtype, D, B, hq, hkv, lens, part):
    flags = _short_limit_then_default(dtype, D, B, hq, hkv, lens, part)
    assert flags & TIMEOUTS, f"no timeout reported (flags {flags:#x})"


@pytest.mark.parametrize("dtype,D,B,hq,hkv,lens,part", MIDSTREAM, ids=lambda v: str(v).replace(" ", ""))
def test_wait_limit_in_mid_stream(dtype, D, B, hq, hkv, lens, part):
    """Long contexts, no padding: a wait that runs out does so while the CTA's
    copies are in flight (or none runs out); either way the launch returns, the
    status matches the flags, and the next call is correct."""
    flags = _short_limit_then_default(dtype, D, B, hq, hkv, lens, part)
    print(f"\n[timeout] {dtype} {lens[:4]} part {part}: flags {flags:#x}")


def _short_limit_then_default(dtype, D, B, hq, hkv, lens, part):
    q, kc, vc, bt, cl = [t.to(DEV) for t in small_case(60 + len(lens), dtype, D, B, hq, hkv, lens)]
    scale = 1.0 / math.sqrt(D)
    assert P.pa_device_errors() == 0
    out = torch.empty_like(q)
    prev = P.pa_set_wait_limit_ns(1)
    try:
        P.pa_decode(out, q, kc, vc, bt, cl, scale, hq, hkv, D, B, partition_size=part)
        st, flags = _status_and_flags()       # waits for the launch: it returned
    finally:
        P.pa_set_wait_limit_ns(0)
    assert prev == P.PA_WAIT_LIMIT_DEFAULT_NS
    assert flags & ~TIMEOUTS == 0
    assert st == (P.PA_ERR_TIMEOUT if flags else P.PA_OK)
    assert _status_and_flags() == (P.PA_OK, 0)       # reading cleared the flags
    # the default limit again: a full, correct decode
    out2 = torch.full_like(q, float("nan"))
    P.pa_decode(out2, q, kc, vc, bt, cl, scale, hq, hkv, D, B, partition_size=part)
    torch.cuda.synchronize()
    assert P.pa_device_errors() == 0
    assert_close(out2, _oracle(q, kc, vc, bt, cl, scale, dtype, hq, hkv, D, B), dtype, "after a timeout")
    return flags


def test_shared_prefix_decode_gives_up_too():
    """The shared-prefix decode's two launches (the second streams while the first
    ends, and stages prefix rows with per-thread asynchronous copies) give up the
    same way, with the newest tokens' append inside the second."""
    import numpy as np
    dtype, D, B, hq, hkv = "f16", 128, 16, 8, 8
    P_shared, members = 40, 6
    rng = np.random.default_rng(3)
    lens = [P_shared * B + int(x) for x in rng.integers(1, 300, size=members)]
    q, kc, vc, bt, cl = [t.to(DEV) for t in small_case(71, dtype, D, B, hq, hkv, lens + PAD, stale=0.0)]
    bt[:members, :P_shared] = bt[0, :P_shared]          # the members share their first blocks
    share = torch.tensor([[0, P_shared]] * members + [[-1, 0]] * len(PAD), dtype=torch.int32, device=DEV)
    n = len(lens + PAD)
    k_new = torch.randn(n, hkv, D, device=DEV).to(q.dtype)
    v_new = torch.randn(n, hkv, D, device=DEV).to(q.dtype)
    kc0, vc0 = kc.clone(), vc.clone()
    out = torch.empty_like(q)
    P.pa_set_wait_limit_ns(1)
    try:
        P.pa_decode_shared(out, q, kc, vc, bt, cl, share, 0.1, hq, hkv, D, B, k_new=k_new, v_new=v_new)
        st, flags = _status_and_flags()
    finally:
        P.pa_set_wait_limit_ns(0)
    assert flags & TIMEOUTS and st == P.PA_ERR_TIMEOUT
    kc.copy_(kc0)
    vc.copy_(vc0)
    out2 = torch.empty_like(q)
    P.pa_decode_shared(out2, q, kc, vc, bt, cl, share, 0.1, hq, hkv, D, B, k_new=k_new, v_new=v_new)
    ref = torch.empty_like(q)
    kr, vr = kc0.clone(), vc0.clone()
    bth, clh = bt.cpu(), cl.cpu()
    slots = torch.tensor([int(bth[s, (int(clh[s]) - 1) // B]) * B + (int(clh[s]) - 1) % B if clh[s] > 0 else -1
                          for s in range(n)], dtype=torch.int64, device=DEV)
    P.pa_reshape_and_cache(k_new, v_new, kr, vr, slots)
    P.pa_decode(ref, q, kr, vr, bt, cl, 0.1, hq, hkv, D, B)
    torch.cuda.synchronize()
    assert P.pa_device_errors() == 0
    assert torch.equal(kc, kr) and torch.equal(vc, vr)
    assert_close(out2, _oracle(q, kr, vr, bt, cl, 0.1, dtype, hq, hkv, D, B), dtype, "shared, after a timeout")
