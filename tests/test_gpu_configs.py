"""The five synthetic workloads end to end: allocator script, copy-on-write,
appends and decode on the GPU path, against the oracle's own execution of the
same script (allocator, cache ops and fp64 attention)."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_79_gb300 as P
import workloads as W
from paged_kv_cache_79_gb300 import runner
from tests.gpu_harness import TOL_16, assert_close, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gpu_tensors(w):
    kc, vc = W.pool_tensors(w, DEV)
    return kc, vc


def _step_kv(w):
    return lambda ev: W.step_tensors(w, ev, DEV)


def _query(w):
    return lambda ev: W.query_tensor(w, ev.index, DEV)


def test_tiny_fifty_appends_each_decoded():
    """The tutorial's workflow: 50 appends to one sequence, decode after each."""
    w = W.tiny()
    kc, vc = _gpu_tensors(w)
    kh, vh = raw(kc).copy(), raw(vc).copy()
    outs = []

    def on_step(ev, alloc, ds):
        outs.append((ds.decode().clone(), raw(ds.q), alloc.block_table(0), alloc.seq_len(0)))

    alloc, _ = runner.execute(w, kc, vc, _step_kv(w), _query(w), on_step=on_step)
    torch.cuda.synchronize()
    assert alloc.block_table(0) == oracle.run_script(w.events, w.num_blocks, w.block_size,
                                                     w.free_order)[0].block_table(0)
    oalloc = oracle.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    oalloc.new_seq()
    worst = 0.0
    for i, (out, q, table, T) in enumerate(outs):
        slot, _ = oalloc.append(0)
        k, v = W.step_tensors(w, W.Step((0,), i), DEV)
        oracle.reshape_and_cache(raw(k), raw(v), kh, vh, np.array([slot]), w.block_size)
        assert table == oalloc.block_table(0) and T == i + 1
        bt = np.array([table], dtype=np.int32)
        want = oracle.decode(q, kh, vh, bt, np.array([T], np.int32), w.softmax_scale, "f32", 8, 8, 64, 16)
        err, rel = assert_close(out, want, "f32", f"step {i}")
        worst = max(worst, err)
    print(f"\n[parity] tiny: max abs err over 50 decodes {worst:.3e}")
    assert np.array_equal(raw(kc), kh) and np.array_equal(raw(vc), vh)


def _check_workload(w, sample=None, min_seqs=0, shared=False):
    """Run `w` on both sides; compare allocator state, caches and sampled outputs
    (of pa_decode_shared over the groups the tables share, when `shared`)."""
    kc, vc = _gpu_tensors(w)
    kh, vh = raw(kc).copy(), raw(vc).copy()
    alloc, ds = runner.execute(w, kc, vc, _step_kv(w), _query(w))
    if shared:
        assert ds.share is not None
        out = ds.decode_shared()
    else:
        out = ds.decode()
    torch.cuda.synchronize()

    def step_kv_host(ev):
        k, v = W.step_tensors(w, ev, DEV)
        return raw(k), raw(v)

    oalloc, recs = oracle.run_script(w.events, w.num_blocks, w.block_size, w.free_order, kh, vh,
                                     step_kv=step_kv_host)
    bt, cl = runner.tables_for(alloc, w.decode_seqs)
    obt, ocl = oracle.tables_for(oalloc, w.decode_seqs)
    assert np.array_equal(bt, obt) and np.array_equal(cl, ocl)
    assert alloc.free_list() == oalloc.free_list()
    # caches bit-exact after every copy-on-write and append
    assert np.array_equal(raw(kc), kh) and np.array_equal(raw(vc), vh)
    seqs = list(range(len(w.decode_seqs))) if sample is None else sample(cl)
    q = raw(ds.q)
    want = oracle.decode(q[seqs], kh, vh, obt[seqs], ocl[seqs], w.softmax_scale, w.dtype, w.num_q_heads,
                         w.num_kv_heads, w.head_dim, w.block_size)
    err, rel = assert_close(out[seqs], want, w.dtype, w.name)
    if w.dtype != "f32":
        # the plain max-abs bound too: every full-size configuration meets it
        assert err <= TOL_16, f"{w.name}: max abs err {err:.3e} > {TOL_16}"
    print(f"\n[parity] {w.name}{' shared' if shared else ''}: {len(seqs)} sequences, "
          f"max abs err {err:.3e}, normwise rel {rel:.3e}")
    assert P.pa_device_errors() == 0
    return out, ds


def _sample(k, seed):
    def pick(cl):
        rng = np.random.default_rng(seed)
        longest = int(np.argmax(cl))
        rest = rng.choice(len(cl), size=min(k, len(cl)), replace=False).tolist()
        return sorted(set(rest + [longest, int(np.argmin(cl))]))
    return pick


def test_mha_fp16():
    _check_workload(W.mha_fp16())


def test_gqa_bf16():
    _check_workload(W.gqa_bf16())


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("prompt", [1024, 1032])
def test_shared_prefix_fp16(prompt, shared):
    _check_workload(W.shared_prefix_fp16(prompt_len=prompt), shared=shared)


def test_long_multiturn_bf16():
    """Full-size pool (~19 GB on the device); oracle on sampled sequences whose
    blocks are gathered to the host (block permutation invariance is pinned).
    Four decodes of the step are checked: the workload's fixed 512-token
    partitions (partition kernel + merge kernel), the two-pass shared-prefix decode,
    the step the bench times -- the two-pass shared-prefix decode with the newest
    tokens appended inside its second launch (the groups save 580 MB of reads) --
    and the same step on the plain balanced split (pa_decode_append, partition
    size 0), which the bench times with --no-share."""
    import dataclasses
    w = W.long_multiturn_bf16()
    kc, vc = _gpu_tensors(w)
    alloc, ds = runner.execute(w, kc, vc, _step_kv(w), _query(w))
    out = ds.decode()
    torch.cuda.synchronize()
    oalloc, _ = oracle.run_script(w.events, w.num_blocks, w.block_size, w.free_order)
    bt, cl = runner.tables_for(alloc, w.decode_seqs)
    obt, ocl = oracle.tables_for(oalloc, w.decode_seqs)
    assert np.array_equal(bt, obt) and np.array_equal(cl, ocl)
    seqs = _sample(32, 5)(cl)      # at least 32 sequences, the longest among them
    assert len(seqs) >= 32 and int(np.argmax(cl)) in seqs
    used = sorted({int(b) for s in seqs for b in obt[s, :(ocl[s] + w.block_size - 1) // w.block_size]})
    remap = {b: i for i, b in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=DEV)
    ks, vs = raw(kc.index_select(0, idx)), raw(vc.index_select(0, idx))
    sbt = np.full((len(seqs), obt.shape[1]), -1, dtype=np.int32)
    for i, s in enumerate(seqs):
        n = (ocl[s] + w.block_size - 1) // w.block_size
        sbt[i, :n] = [remap[int(b)] for b in obt[s, :n]]
    want = oracle.decode(raw(ds.q)[seqs], ks, vs, sbt, ocl[seqs], w.softmax_scale, "bf16", 32, 8, 128, 32)
    err, rel = assert_close(out[seqs], want, "bf16", w.name)
    assert err <= TOL_16
    print(f"\n[parity] {w.name}: {len(seqs)} sampled sequences, max abs err {err:.3e}, normwise rel {rel:.3e}")
    # the turns of a group share their leading blocks: the two-pass decode agrees too
    assert ds.share is not None
    out_s = ds.decode_shared().clone()
    torch.cuda.synchronize()
    err, _ = assert_close(out_s[seqs], want, "bf16", w.name + " shared")
    assert err <= TOL_16
    # the benched step: copy-on-write pairs (none here), then the shared-prefix
    # decode with every sequence's newest token appended in its own-block launch.
    # The rows it appends are the ones the script already wrote, so the caches do
    # not change.
    assert ds.fusable and ds.pairs.shape[0] == 0 and ds.share_pays
    dss = dataclasses.replace(ds, out=torch.full_like(ds.out, float("nan")))
    dss.run_shared()
    torch.cuda.synchronize()
    err, rel = assert_close(dss.out[seqs], want, "bf16", w.name + " benched step")
    assert err <= TOL_16
    print(f"[parity] {w.name} benched step (shared prefixes, fused append): max abs err {err:.3e}, "
          f"normwise rel {rel:.3e}")
    # the same step without prefix sharing: append fused with the balanced split
    ws0 = P.alloc_workspace(len(cl), w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                            bt.shape[1], 0, DEV)
    dsb = dataclasses.replace(ds, partition_size=0, workspace=ws0, out=torch.full_like(ds.out, float("nan")))
    dsb.run_fused()
    torch.cuda.synchronize()
    err, rel = assert_close(dsb.out[seqs], want, "bf16", w.name + " plain step")
    assert err <= TOL_16
    print(f"[parity] {w.name} step without sharing (fused append, balanced split): max abs err {err:.3e}, "
          f"normwise rel {rel:.3e}")
    # the step's appended rows are where the oracle's allocator put them, bit for bit
    k_new, v_new = W.step_tensors(w, w.step_events()[-1], DEV)
    slots = ds.slots.cpu().numpy()
    kflat = kc.view(-1, w.num_kv_heads, w.head_dim)
    vflat = vc.view(-1, w.num_kv_heads, w.head_dim)
    sl = torch.from_numpy(slots).to(DEV)
    assert torch.equal(kflat[sl], k_new) and torch.equal(vflat[sl], v_new)
    del kc, vc, kflat, vflat
    torch.cuda.empty_cache()
    assert P.pa_device_errors() == 0


@pytest.mark.parametrize("name", ["mha_fp16", "shared_prefix_fp16_p1032"])
def test_fused_step_equals_separate_step(name):
    """Replaying a workload's last step with the fused append (one launch) gives the
    same caches and output, bit for bit, as append then decode."""
    w = W.by_name(name, **({"prompts": 4} if name.startswith("shared") else {}))
    kc, vc = _gpu_tensors(w)
    alloc, ds = runner.execute(w, kc, vc, _step_kv(w), _query(w))
    assert ds.fusable
    k0, v0 = kc.clone(), vc.clone()
    ds.run()
    torch.cuda.synchronize()
    out1, k1, v1 = ds.out.clone(), kc.clone(), vc.clone()
    kc.copy_(k0)
    vc.copy_(v0)
    ds.run_fused()
    torch.cuda.synchronize()
    assert torch.equal(kc, k1) and torch.equal(vc, v1)
    assert torch.equal(ds.out, out1)


def test_shared_step_equals_separate_step():
    """The shared-prefix step (copy-on-write, then one launch per pass with the
    append fused into the second) leaves the caches bit-identical to append then
    decode, and its output matches the oracle on every sequence."""
    w = W.shared_prefix_fp16(prompt_len=1032, prompts=4)
    kc, vc = _gpu_tensors(w)
    kh, vh = raw(kc).copy(), raw(vc).copy()
    alloc, ds = runner.execute(w, kc, vc, _step_kv(w), _query(w))
    assert ds.fusable and ds.share is not None
    k0, v0 = kc.clone(), vc.clone()
    ds.run()
    torch.cuda.synchronize()
    k1, v1 = kc.clone(), vc.clone()
    kc.copy_(k0)
    vc.copy_(v0)
    ds.run_shared()
    torch.cuda.synchronize()
    assert torch.equal(kc, k1) and torch.equal(vc, v1)

    def step_kv_host(ev):
        k, v = W.step_tensors(w, ev, DEV)
        return raw(k), raw(v)

    oalloc, _ = oracle.run_script(w.events, w.num_blocks, w.block_size, w.free_order, kh, vh,
                                  step_kv=step_kv_host)
    obt, ocl = oracle.tables_for(oalloc, w.decode_seqs)
    want = oracle.decode(raw(ds.q), kh, vh, obt, ocl, w.softmax_scale, w.dtype, w.num_q_heads,
                         w.num_kv_heads, w.head_dim, w.block_size)
    assert_close(ds.out, want, w.dtype, "shared step")
    assert P.pa_device_errors() == 0


def test_packed_inputs_step_equals_the_plain_step():
    """The step run on inputs uploaded in one packed copy gives the same caches and
    output, bit for bit, as the step on the original device tensors."""
    import dataclasses
    w = W.mha_fp16()
    kc, vc = _gpu_tensors(w)
    alloc, ds = runner.execute(w, kc, vc, _step_kv(w), _query(w))
    k0, v0 = kc.clone(), vc.clone()
    ds.run_fused()
    torch.cuda.synchronize()
    out1, k1, v1 = ds.out.clone(), kc.clone(), vc.clone()
    kc.copy_(k0)
    vc.copy_(v0)
    names = ["q", "step_k", "step_v", "slots", "pairs", "block_tables", "context_lens"]
    packed = runner.PackedInputs({n: getattr(ds, n).cpu() for n in names}, DEV)
    packed.upload()
    dsv = dataclasses.replace(ds, out=torch.empty_like(ds.out), **packed.views)
    dsv.run_fused()
    torch.cuda.synchronize()
    assert torch.equal(kc, k1) and torch.equal(vc, v1) and torch.equal(dsv.out, out1)
