"""pa_decode_shared_planned: both shared-prefix launches started from a host plan.

It must give the same output (and, with the fused append, the same caches) as the
unplanned pa_decode_shared, bit for bit, and match the oracle.  A plan made from
other inputs must not make a launch touch memory outside its arguments or send the
appended rows anywhere but where the block table says."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_79_gb300 as P
import workloads as W
from paged_kv_cache_79_gb300 import runner
from tests.gpu_harness import assert_close, raw
from tests.test_gpu_shared import CASES, lens_for, ora, shared_case

pytestmark = pytest.mark.gpu
DEV = "cuda"


def plan_for(bt, cl, share, hq, hkv, D, B, dtype):
    return torch.from_numpy(P.pa_decode_shared_plan(bt.cpu().numpy(), cl.cpu().numpy(), np.asarray(share),
                                                    hq, hkv, D, B, dtype)).to(DEV)


def plannable(S, hq, hkv, D, B, W, dtype):
    """Whether both launches share a grid (every fp16/bf16 shape; fp32 kernels sized
    for different item widths may not), else the plan size is reported as invalid."""
    try:
        P.pa_decode_shared_plan_bytes(S, hq, hkv, D, B, W, dtype)
        return True
    except P.PagedKVError:
        assert dtype == "f32"
        return False


def both(q, kc, vc, bt, cl, share, scale, hq, hkv, D, B, dtype, k_new=None, v_new=None):
    """(unplanned, planned) outputs and caches for the same inputs."""
    res = []
    for planned in (False, True):
        k, v = kc.to(DEV).clone(), vc.to(DEV).clone()
        out = torch.full(q.shape, float("nan"), dtype=q.dtype, device=DEV)
        args = (out, q.to(DEV), k, v, bt.to(DEV), cl.to(DEV), torch.from_numpy(share).to(DEV))
        if planned:
            P.pa_decode_shared_planned(*args, plan_for(bt, cl, share, hq, hkv, D, B, dtype), scale, hq, hkv,
                                       D, B, k_new=k_new, v_new=v_new)
        else:
            P.pa_decode_shared(*args, scale, hq, hkv, D, B, k_new=k_new, v_new=v_new)
        torch.cuda.synchronize()
        res.append((out, k, v))
    return res


@pytest.mark.parametrize("dtype,D,B,Hq,Hkv,groups", CASES, ids=lambda v: str(v)[:50].replace(" ", ""))
def test_planned_equals_unplanned(dtype, D, B, Hq, Hkv, groups):
    q, kc, vc, bt, cl, share = shared_case(23, dtype, D, B, Hq, Hkv, groups)
    if not plannable(cl.shape[0], Hq, Hkv, D, B, bt.shape[1], dtype):
        pytest.skip("the two fp32 launches run on different grids: no shared plan")
    (o0, _, _), (o1, _, _) = both(q, kc, vc, bt, cl, share, 0.1, Hq, Hkv, D, B, dtype)
    assert P.pa_device_errors() == 0
    assert torch.equal(o0, o1)
    assert_close(o1, ora(q, kc, vc, bt, cl, 0.1, dtype, Hq, Hkv, D, B), dtype)


@pytest.mark.parametrize("dtype,Hq,Hkv,B", [("bf16", 8, 2, 16), ("f16", 40, 40, 16), ("f32", 4, 4, 32),
                                            ("bf16", 32, 8, 32)])
def test_planned_append_equals_unplanned(dtype, Hq, Hkv, B):
    D = 128
    groups = [(lens_for(8, 6, B, 51), 6), ([B * 2 + 1], 0), (lens_for(3, 2, B, 52, 1), 2),
              ([2 * B + 1, 2 * B + 1, 2 * B + 2], 2)]
    q, kc, vc, bt, cl, share = shared_case(51, dtype, D, B, Hq, Hkv, groups, stale=0.0)
    S = cl.shape[0]
    if not plannable(S, Hq, Hkv, D, B, bt.shape[1], dtype):
        pytest.skip("the two fp32 launches run on different grids: no shared plan")
    g = torch.Generator().manual_seed(53)
    k_new = torch.randn(S, Hkv, D, generator=g).to(q.dtype).to(DEV)
    v_new = torch.randn(S, Hkv, D, generator=g).to(q.dtype).to(DEV)
    (o0, k0, v0), (o1, k1, v1) = both(q, kc, vc, bt, cl, share, 0.08, Hq, Hkv, D, B, dtype, k_new, v_new)
    assert P.pa_device_errors() == 0
    assert torch.equal(o0, o1) and torch.equal(k0, k1) and torch.equal(v0, v1)
    want = oracle.decode(raw(q), raw(k1), raw(v1), bt.numpy(), cl.numpy(), 0.08, dtype, Hq, Hkv, D, B)
    assert_close(o1, want, dtype)


@pytest.mark.parametrize("name", ["shared_prefix_fp16", "shared_prefix_fp16_p1032", "long_multiturn_bf16"])
def test_planned_workload_step(name):
    """The bench's shared-prefix step on a full-size workload, planned and walked."""
    w = W.by_name(name)
    kc, vc = W.pool_tensors(w, DEV)
    alloc, ds = runner.execute(w, kc, vc, lambda ev: W.step_tensors(w, ev, DEV),
                               lambda ev: W.query_tensor(w, ev.index, DEV))
    assert ds.share is not None and ds.shared_plan is not None
    k0, v0 = kc.clone(), vc.clone()
    ds.run_shared(planned=False)
    torch.cuda.synchronize()
    ref, k1, v1 = ds.out.clone(), kc.clone(), vc.clone()
    kc.copy_(k0)
    vc.copy_(v0)
    ds.out.fill_(float("nan"))
    ds.run_shared(planned=True)
    torch.cuda.synchronize()
    assert torch.equal(ds.out, ref) and torch.equal(kc, k1) and torch.equal(vc, v1)
    assert P.pa_device_errors() == 0


def test_stale_plan_stays_inside_its_arguments():
    """A plan made for other lengths and groups: the launches return, write no cache
    row outside the appended slots the table names, and the right plan is exact."""
    dtype, D, B, Hq, Hkv = "bf16", 128, 16, 16, 4
    groups = [(lens_for(6, 10, B, 61), 10), ([700], 0), (lens_for(3, 30, B, 62), 30)]
    q, kc, vc, bt, cl, share = shared_case(61, dtype, D, B, Hq, Hkv, groups, stale=0.0)
    S = cl.shape[0]
    other_cl = cl.clone()
    other_cl[:] = torch.from_numpy(np.random.default_rng(5).integers(1, 40 * B, size=S)).int()
    other_share = share.copy()
    other_share[:, 0] = np.where(np.arange(S) % 3 == 0, -1, 0)
    other_share[:, 1] = np.random.default_rng(6).integers(0, 50, size=S)
    bt_other = torch.from_numpy(np.random.default_rng(7).integers(0, kc.shape[0], size=bt.shape)).int()
    stale = plan_for(bt_other, other_cl, other_share, Hq, Hkv, D, B, dtype)
    g = torch.Generator().manual_seed(63)
    k_new = torch.randn(S, Hkv, D, generator=g).to(q.dtype).to(DEV)
    v_new = torch.randn(S, Hkv, D, generator=g).to(q.dtype).to(DEV)
    qd, btd, cld, shd = q.to(DEV), bt.to(DEV), cl.to(DEV), torch.from_numpy(share).to(DEV)
    kd, vd = kc.to(DEV), vc.to(DEV)
    kr, vr = kd.clone(), vd.clone()
    slots = torch.tensor([int(bt[s, (int(t) - 1) // B]) * B + (int(t) - 1) % B for s, t in enumerate(cl.tolist())],
                         dtype=torch.int64, device=DEV)
    P.pa_reshape_and_cache(k_new, v_new, kr, vr, slots)
    out = torch.empty_like(qd)
    P.pa_decode_shared_planned(out, qd, kd, vd, btd, cld, shd, stale, 0.1, Hq, Hkv, D, B,
                               k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert P.pa_device_errors() & ~(P.PA_DEVERR_PLAN | P.PA_DEVERR_SHARE) == 0
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
    ref = torch.empty_like(qd)
    P.pa_decode_shared(ref, qd, kr, vr, btd, cld, shd, 0.1, Hq, Hkv, D, B)
    got = torch.empty_like(qd)
    P.pa_decode_shared_planned(got, qd, kd, vd, btd, cld, shd, plan_for(bt, cl, share, Hq, Hkv, D, B, dtype),
                               0.1, Hq, Hkv, D, B)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert P.pa_device_errors() == 0


def test_member_ending_inside_shared_blocks_is_flagged_planned():
    dtype, D, B, Hq, Hkv, Pb = "bf16", 128, 16, 16, 4, 20
    lens = lens_for(5, Pb, B, 9)
    q, kc, vc, bt, cl, share = shared_case(31, dtype, D, B, Hq, Hkv, [(lens, Pb)], stale=0.0)
    cl[2] = 20 * 16 - 5
    bt[2, (int(cl[2]) + B - 1) // B:] = -1
    assert P.pa_device_errors() == 0
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    P.pa_decode_shared_planned(out, q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), cl.to(DEV),
                               torch.from_numpy(share).to(DEV), plan_for(bt, cl, share, Hq, Hkv, D, B, dtype),
                               0.09, Hq, Hkv, D, B)
    torch.cuda.synchronize()
    assert P.pa_device_errors() == P.PA_DEVERR_SHARE
    assert_close(out, ora(q, kc, vc, bt, cl, 0.09, dtype, Hq, Hkv, D, B), dtype)


def test_plan_of_another_size_is_rejected():
    groups = [(lens_for(3, 4, 16, 71), 4)]
    q, kc, vc, bt, cl, share = shared_case(71, "f16", 128, 16, 8, 8, groups)
    plan = plan_for(bt, cl, share, 8, 8, 128, 16, "f16")
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    with pytest.raises(P.PagedKVError):
        P.pa_decode_shared_planned(out, q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), cl.to(DEV),
                                   torch.from_numpy(share).to(DEV), plan[:-32], 0.1, 8, 8, 128, 16)


def test_planned_without_groups_equals_plain_decode_bitwise():
    """No group shares a block: the shared blocks' launch has an empty stream and the
    own blocks' launch walks in (sequence, unit) order from its plan."""
    groups = [([300], 0), ([17], 0), ([1000], 0), ([1], 0)]
    q, kc, vc, bt, cl, share = shared_case(5, "bf16", 128, 16, 32, 8, groups)
    plan = P.pa_decode_shared_plan(bt.numpy(), cl.numpy(), share, 32, 8, 128, 16, "bf16")
    assert (plan.reshape(2, -1, 32)[0, :, 0] == -1).all()
    got = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    P.pa_decode_shared_planned(got, q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), cl.to(DEV),
                               torch.from_numpy(share).to(DEV), torch.from_numpy(plan).to(DEV), 0.09,
                               32, 8, 128, 16)
    out = torch.empty_like(got)
    P.pa_decode(out, q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), cl.to(DEV), 0.09, 32, 8, 128, 16,
                partition_size=0)
    torch.cuda.synchronize()
    assert torch.equal(got, out)
    assert P.pa_device_errors() == 0
