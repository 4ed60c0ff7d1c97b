"""K and V cache placement: one copy per block, or one per cache.

When v_cache lies above k_cache (both halves of one [2][num_blocks][B][Hkv][d]
buffer, as the workloads allocate them), one tensor map spans both caches and a
single copy brings a block's K and V tiles into the stage; otherwise each cache
has its own map and copy.  Both land the tiles in the same place, so every decode
must give the same bits either way (and match the oracle), including the fused
append, the planned start and the shared-prefix passes."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_79_gb300 as P
from tests.gpu_harness import assert_close, raw, small_case
from tests.test_gpu_shared import lens_for, shared_case

pytestmark = pytest.mark.gpu
DEV = "cuda"


def placed(kc, vc, v_above):
    """Device copies of kc, vc inside one buffer: V in the upper half (joint map)
    or in the lower half (one map per cache)."""
    buf = torch.empty((2,) + tuple(kc.shape), dtype=kc.dtype, device=DEV)
    k, v = (buf[0], buf[1]) if v_above else (buf[1], buf[0])
    k.copy_(kc.to(DEV))
    v.copy_(vc.to(DEV))
    return buf, k, v


CASES = []
for dtype in ("f32", "f16", "bf16"):
    for D in (64, 128):
        for B in (16, 32):
            CASES.append((dtype, D, B, 8, 2, [1, B - 1, B + 1, 2 * B, 777]))
CASES.append(("bf16", 128, 16, 64, 4, [5, 300, 2049]))        # 16-row (wide) items
CASES.append(("f16", 128, 16, 40, 40, [3000, 17, 1, 513]))    # MHA, two blocks per stage


@pytest.mark.parametrize("dtype,D,B,hq,hkv,lens", CASES, ids=lambda v: str(v).replace(" ", ""))
def test_placements_agree_bitwise(dtype, D, B, hq, hkv, lens):
    q, kc, vc, bt, cl = small_case(sum(lens) % 613 + 5, dtype, D, B, hq, hkv, lens)
    scale = 1.0 / math.sqrt(D)
    qd, btd, cld = q.to(DEV), bt.to(DEV), cl.to(DEV)
    outs = []
    for v_above in (True, False):
        _, k, v = placed(kc, vc, v_above)
        for part in (0, 4 * B):
            out = torch.full_like(qd, float("nan"))
            P.pa_decode(out, qd, k, v, btd, cld, scale, hq, hkv, D, B, partition_size=part)
            outs.append(out)
        plan = torch.from_numpy(P.pa_decode_plan(bt.numpy(), cl.numpy(), hq, hkv, D, B, dtype)).to(DEV)
        out = torch.full_like(qd, float("nan"))
        P.pa_decode_planned(out, qd, k, v, btd, cld, plan, scale, hq, hkv, D, B)
        outs.append(out)
    torch.cuda.synchronize()
    assert P.pa_device_errors() == 0
    for a, b in zip(outs[:3], outs[3:]):
        assert torch.equal(a, b)
    assert torch.equal(outs[0], outs[2])       # planned start: the same items as the walk
    want = oracle.decode(raw(q), raw(kc), raw(vc), bt.numpy(), cl.numpy(), scale, dtype, hq, hkv, D, B)
    assert_close(outs[0], want, dtype, "joint placement")
    assert_close(outs[1], want, dtype, "joint placement, fixed partitions")


@pytest.mark.parametrize("dtype,D,B,hq,hkv,lens", [
    ("bf16", 128, 16, 16, 4, [1, 16, 17, 500, 3001]),
    ("f16", 64, 32, 8, 8, [2, 33, 64, 1000]),
    ("f32", 128, 16, 4, 1, [3, 40, 700]),
], ids=lambda v: str(v).replace(" ", ""))
def test_fused_append_agrees_across_placements(dtype, D, B, hq, hkv, lens):
    q, kc, vc, bt, cl = small_case(sum(lens) % 517 + 9, dtype, D, B, hq, hkv, lens, stale=0.0)
    g = torch.Generator().manual_seed(21)
    k_new = torch.randn(len(lens), hkv, D, generator=g).to(q.dtype).to(DEV)
    v_new = torch.randn(len(lens), hkv, D, generator=g).to(q.dtype).to(DEV)
    qd, btd, cld = q.to(DEV), bt.to(DEV), cl.to(DEV)
    res = []
    for v_above in (True, False):
        _, k, v = placed(kc, vc, v_above)
        out = torch.empty_like(qd)
        P.pa_decode_append(out, qd, k, v, k_new, v_new, btd, cld, 0.1, hq, hkv, D, B, 0)
        res.append((out, k.clone(), v.clone()))
    torch.cuda.synchronize()
    assert P.pa_device_errors() == 0
    (o1, k1, v1), (o2, k2, v2) = res
    assert torch.equal(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    want = oracle.decode(raw(q), raw(k1), raw(v1), bt.numpy(), cl.numpy(), 0.1, dtype, hq, hkv, D, B)
    assert_close(o1, want, dtype, "fused append, joint placement")


@pytest.mark.parametrize("dtype,D,B,hq,hkv,groups", [
    ("f16", 128, 16, 40, 40, [(lens_for(8, 8, 16, 31), 8), (lens_for(4, 3, 16, 32), 3)]),
    ("bf16", 128, 32, 32, 8, [(lens_for(4, 30, 32, 33, 40), 30), ([70, 5], 0)]),
    ("f32", 64, 16, 4, 2, [(lens_for(3, 7, 16, 34), 7)]),
], ids=lambda v: str(v)[:50].replace(" ", ""))
def test_shared_decode_agrees_across_placements(dtype, D, B, hq, hkv, groups):
    q, kc, vc, bt, cl, share = shared_case(41, dtype, D, B, hq, hkv, groups)
    qd, btd, cld, shd = q.to(DEV), bt.to(DEV), cl.to(DEV), torch.from_numpy(share).to(DEV)
    outs = []
    for v_above in (True, False):
        _, k, v = placed(kc, vc, v_above)
        out = torch.full_like(qd, float("nan"))
        P.pa_decode_shared(out, qd, k, v, btd, cld, shd, 0.1, hq, hkv, D, B)
        outs.append(out)
    torch.cuda.synchronize()
    assert P.pa_device_errors() == 0
    assert torch.equal(outs[0], outs[1])
    want = oracle.decode(raw(q), raw(kc), raw(vc), bt.numpy(), cl.numpy(), 0.1, dtype, hq, hkv, D, B)
    assert_close(outs[0], want, dtype, "shared decode, joint placement")


def test_separate_buffers_either_order():
    """Two separate allocations (the caller's usual case) decode like one buffer."""
    dtype, D, B, hq, hkv, lens = "bf16", 128, 16, 16, 2, [100, 2000, 33]
    q, kc, vc, bt, cl = small_case(77, dtype, D, B, hq, hkv, lens)
    qd, btd, cld = q.to(DEV), bt.to(DEV), cl.to(DEV)
    _, k, v = placed(kc, vc, True)
    ref = torch.empty_like(qd)
    P.pa_decode(ref, qd, k, v, btd, cld, 0.1, hq, hkv, D, B)
    a, b = kc.to(DEV), vc.to(DEV)
    for kk, vv in ((a, b), (a.clone(), b.clone())):
        out = torch.empty_like(qd)
        P.pa_decode(out, qd, kk, vv, btd, cld, 0.1, hq, hkv, D, B)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert P.pa_device_errors() == 0
