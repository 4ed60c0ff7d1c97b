"""pa_decode_planned: the balanced-split decode started from a host plan.

It must give the same output (and, with the fused append, the same caches) as the
unplanned call, bit for bit, and match the oracle.  A plan made from other
lengths must not make a launch touch memory outside its arguments or send the
appended rows anywhere but where the block table says."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_79_gb300 as P
import workloads as W
from paged_kv_cache_79_gb300 import runner
from tests.gpu_harness import assert_close, raw, small_case
from tests.test_gpu_parity import BALANCED_EDGES, SHAPES

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [(dt, D, B, hq, hkv, lens) for (dt, D, B, hq, hkv, lens, part) in SHAPES if part == 0]
CASES += [tuple(c) for c in BALANCED_EDGES]


def plan_for(bt, cl, hq, hkv, D, B, dtype):
    return torch.from_numpy(P.pa_decode_plan(bt.cpu().numpy(), cl.cpu().numpy(), hq, hkv, D, B, dtype)).to(DEV)


@pytest.mark.parametrize("dtype,D,B,hq,hkv,lens", CASES, ids=lambda v: str(v)[:40].replace(" ", ""))
def test_planned_equals_unplanned(dtype, D, B, hq, hkv, lens):
    q, kc, vc, bt, cl = [t.to(DEV) for t in small_case(sum(lens) % 991 + 3, dtype, D, B, hq, hkv, lens)]
    scale = 1.0 / math.sqrt(D)
    ref = torch.empty_like(q)
    P.pa_decode(ref, q, kc, vc, bt, cl, scale, hq, hkv, D, B, partition_size=0)
    got = torch.full_like(q, float("nan"))
    P.pa_decode_planned(got, q, kc, vc, bt, cl, plan_for(bt, cl, hq, hkv, D, B, dtype), scale, hq, hkv, D, B)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    want = oracle.decode(raw(q), raw(kc), raw(vc), bt.cpu().numpy(), cl.cpu().numpy(), scale, dtype, hq, hkv,
                         D, B)
    assert_close(got, want, dtype)
    assert P.pa_device_errors() == 0


@pytest.mark.parametrize("dtype,D,B,hq,hkv,lens", [
    ("bf16", 128, 16, 8, 2, [1, 16, 17, 31, 32, 33, 500]),
    ("f16", 128, 32, 40, 40, [7, 64, 65, 1000]),
    ("f32", 64, 16, 4, 2, [1, 2, 40, 300]),
    ("bf16", 128, 32, 32, 8, [1, 32, 33, 777, 20000, 20001]),
    ("f16", 128, 16, 12, 3, [0, 5, 3000, 0]),
], ids=lambda v: str(v)[:40].replace(" ", ""))
def test_planned_append_equals_unplanned(dtype, D, B, hq, hkv, lens):
    q, kc, vc, bt, cl = small_case(sum(lens) % 997 + 7, dtype, D, B, hq, hkv, lens, stale=0.0)
    g = torch.Generator().manual_seed(11)
    k_new = torch.randn(len(lens), hkv, D, generator=g).to(q.dtype).to(DEV)
    v_new = torch.randn(len(lens), hkv, D, generator=g).to(q.dtype).to(DEV)
    q, bt_d, cl_d = q.to(DEV), bt.to(DEV), cl.to(DEV)
    k1, v1 = kc.to(DEV), vc.to(DEV)
    k2, v2 = k1.clone(), v1.clone()
    ref = torch.empty_like(q)
    P.pa_decode_append(ref, q, k1, v1, k_new, v_new, bt_d, cl_d, 0.1, hq, hkv, D, B, 0)
    got = torch.empty_like(q)
    P.pa_decode_planned(got, q, k2, v2, bt_d, cl_d, plan_for(bt, cl, hq, hkv, D, B, dtype), 0.1, hq, hkv, D, B,
                        k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert torch.equal(k1, k2) and torch.equal(v1, v2) and torch.equal(got, ref)
    assert P.pa_device_errors() == 0


@pytest.mark.parametrize("name", ["tiny", "mha_fp16", "gqa_bf16"])
def test_planned_workload_step(name):
    """The bench's planned step on a full-size workload equals the unplanned one."""
    w = W.by_name(name)
    kc, vc = W.pool_tensors(w, DEV)
    alloc, ds = runner.execute(w, kc, vc, lambda ev: W.step_tensors(w, ev, DEV),
                               lambda ev: W.query_tensor(w, ev.index, DEV))
    assert ds.plan is not None and ds.partition_size == 0
    k0, v0 = kc.clone(), vc.clone()
    ds.run_fused()
    torch.cuda.synchronize()
    ref, k1, v1 = ds.out.clone(), kc.clone(), vc.clone()
    kc.copy_(k0)
    vc.copy_(v0)
    ds.out.fill_(float("nan"))
    ds.run_planned()
    torch.cuda.synchronize()
    assert torch.equal(ds.out, ref) and torch.equal(kc, k1) and torch.equal(vc, v1)
    assert P.pa_device_errors() == 0


def test_stale_plan_stays_inside_its_arguments():
    """A plan made for other lengths: the launch returns, writes no cache row
    outside the appended slots the table names, and the next planned call with the
    right plan is exact."""
    dtype, D, B, hq, hkv = "bf16", 128, 16, 16, 4
    lens = [3000, 40, 999, 5000, 1]
    q, kc, vc, bt, cl = small_case(17, dtype, D, B, hq, hkv, lens, stale=0.0)
    other = torch.tensor([1, 5000, 17, 30, 2999], dtype=torch.int32)
    bt_other = bt.clone()
    bt_other[:, :] = torch.from_numpy(np.random.default_rng(3).integers(0, kc.shape[0], size=bt.shape)).int()
    stale = plan_for(bt_other, other, hq, hkv, D, B, dtype)
    g = torch.Generator().manual_seed(12)
    k_new = torch.randn(len(lens), hkv, D, generator=g).to(q.dtype).to(DEV)
    v_new = torch.randn(len(lens), hkv, D, generator=g).to(q.dtype).to(DEV)
    q, bt_d, cl_d, kd, vd = q.to(DEV), bt.to(DEV), cl.to(DEV), kc.to(DEV), vc.to(DEV)
    kr, vr = kd.clone(), vd.clone()
    slots = torch.tensor([int(bt[s, (t - 1) // B]) * B + (t - 1) % B for s, t in enumerate(lens)],
                         dtype=torch.int64, device=DEV)
    P.pa_reshape_and_cache(k_new, v_new, kr, vr, slots)
    out = torch.empty_like(q)
    P.pa_decode_planned(out, q, kd, vd, bt_d, cl_d, stale, 0.1, hq, hkv, D, B, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert P.pa_device_errors() & ~P.PA_DEVERR_PLAN == 0
    # every cache row that changed is an appended slot the table names, holding
    # its new row (a stale walk may skip some appends, never misplace one)
    k0 = kc.to(DEV)
    changed = ((kd != k0).flatten(2).any(-1) | (vd != vc.to(DEV)).flatten(2).any(-1)).flatten()
    allowed = torch.zeros_like(changed)
    allowed[slots] = True
    assert not (changed & ~allowed).any()
    rows = changed.nonzero().flatten()
    assert torch.equal(kd.flatten(0, 1)[rows], kr.flatten(0, 1)[rows])
    assert torch.equal(vd.flatten(0, 1)[rows], vr.flatten(0, 1)[rows])
    kd.copy_(kr)
    vd.copy_(vr)
    ref = torch.empty_like(q)
    P.pa_decode(ref, q, kr, vr, bt_d, cl_d, 0.1, hq, hkv, D, B, partition_size=0)
    got = torch.empty_like(q)
    P.pa_decode_planned(got, q, kd, vd, bt_d, cl_d, plan_for(bt, cl, hq, hkv, D, B, dtype), 0.1, hq, hkv, D, B)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert P.pa_device_errors() == 0


def test_plan_of_another_size_is_rejected():
    q, kc, vc, bt, cl = [t.to(DEV) for t in small_case(19, "f16", 128, 16, 8, 8, [100, 7])]
    plan = plan_for(bt, cl, 8, 8, 128, 16, "f16")
    out = torch.empty_like(q)
    with pytest.raises(P.PagedKVError):
        P.pa_decode_planned(out, q, kc, vc, bt, cl, plan[:-32], 0.1, 8, 8, 128, 16)
