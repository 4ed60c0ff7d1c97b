"""pa_decode_shared (shared-prefix decode in two passes) against the fp64 oracle.

Groups of sequences share their first P physical blocks ("Memory sharing" of the
PagedAttention paper summary: parallel samples of one prompt point at the same
prompt blocks).  The oracle knows nothing of sharing: it gathers every
sequence's blocks through its table and runs dense softmax attention, so any
block read twice, skipped, or merged with the wrong weight shows up here."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_79_gb300 as P
import workloads as W
from tests.gpu_harness import assert_close, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


def shared_case(seed, dtype, D, B, Hq, Hkv, groups, stale=float("nan"), extra=7):
    """groups: list of (member context lengths, P shared blocks).  Returns CPU
    tensors q, kc, vc, bt, cl and the share array the groups declare."""
    rng = np.random.default_rng(seed)
    lens, rows = [], []
    need = extra
    for (ml, Pb) in groups:
        assert all(t >= Pb * B + 1 for t in ml) or Pb == 0
        need += Pb + sum((t + B - 1) // B - Pb for t in ml)
    perm = rng.permutation(need).astype(np.int32)
    nxt = 0
    share = []
    for (ml, Pb) in groups:
        pre = perm[nxt:nxt + Pb]
        nxt += Pb
        first = len(lens)
        for t in ml:
            nb = (t + B - 1) // B
            own = perm[nxt:nxt + nb - Pb]
            nxt += nb - Pb
            rows.append(np.concatenate([pre, own]))
            lens.append(t)
            share.append((first, Pb) if (len(ml) > 1 and Pb > 0) else (-1, 0))
    W_ = max(1, max(len(r) for r in rows)) + 1
    bt = np.full((len(lens), W_), -1, dtype=np.int32)
    for s, r in enumerate(rows):
        bt[s, :len(r)] = r
    kc = W.randn((need, B, Hkv, D), "f32", seed * 11 + 1)
    vc = W.randn((need, B, Hkv, D), "f32", seed * 11 + 2)
    used = np.zeros((need, B), dtype=bool)
    for s, t in enumerate(lens):
        for tok in range(t):
            used[bt[s, tok // B], tok % B] = True
    m = torch.from_numpy(~used)
    kc[m] = stale
    vc[m] = stale
    q = W.randn((len(lens), Hq, D), "f32", seed * 11 + 3)
    td = W.torch_dtype(dtype)
    return (q.to(td), kc.to(td), vc.to(td), torch.from_numpy(bt), torch.tensor(lens, dtype=torch.int32),
            np.array(share, dtype=np.int32).reshape(-1, 2))


def shared_decode(q, kc, vc, bt, cl, share, scale, Hq, Hkv, D, B, k_new=None, v_new=None):
    out = torch.empty_like(q, device=DEV)
    P.pa_decode_shared(out, q.to(DEV), kc, vc, bt.to(DEV), cl.to(DEV), torch.from_numpy(share).to(DEV),
                       scale, Hq, Hkv, D, B, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    return out


def ora(q, kc, vc, bt, cl, scale, dtype, Hq, Hkv, D, B):
    return oracle.decode(raw(q), raw(kc), raw(vc), bt.numpy(), cl.numpy(), scale, dtype, Hq, Hkv, D, B)


def lens_for(n, Pb, B, seed, spread=3):
    r = np.random.default_rng(seed)
    return [int(Pb * B + 1 + r.integers(0, spread * B)) for _ in range(n)]


CASES = [
    # dtype, D, B, Hq, Hkv, groups
    ("f16", 128, 16, 8, 8, [(lens_for(8, 64, 16, 1), 64), (lens_for(8, 64, 16, 2), 64)]),
    ("bf16", 128, 16, 16, 4, [(lens_for(5, 10, 16, 3), 10), ([40], 0), (lens_for(3, 2, 16, 4), 2)]),
    ("bf16", 128, 32, 32, 8, [(lens_for(4, 30, 32, 5, 40), 30), (lens_for(4, 1, 32, 6), 1)]),
    ("f32", 64, 16, 4, 2, [(lens_for(3, 7, 16, 7), 7), (lens_for(2, 3, 16, 8), 3)]),
    ("f16", 64, 32, 16, 1, [(lens_for(2, 20, 32, 9), 20), ([1, 33], 0)]),           # G = 16
    ("f16", 128, 16, 4, 4, [(lens_for(33, 5, 16, 10), 5)]),                          # G = 1: 3 member groups
    ("bf16", 128, 16, 12, 3, [(lens_for(9, 4, 16, 11), 4), (lens_for(2, 200, 16, 12), 200)]),   # G = 4
    ("f16", 128, 16, 40, 40, [(lens_for(8, 8, 16, 13), 8)] * 2 + [([17, 1], 0)]),
    ("bf16", 128, 16, 8, 1, [(lens_for(2, 3000, 16, 14), 3000)]),                   # long prefix over many CTAs
    ("f32", 128, 16, 8, 8, [([16 * 3 + 1, 16 * 3 + 1], 3)]),                          # own part = 1 token
    # 322 sequences: the own-block launch's (kv head, sequence) walk over many batches
    # of 32 sequences, with own parts of 1 to 48 tokens
    ("f16", 64, 16, 4, 4, [(lens_for(8, 2, 16, 100 + i), 2) for i in range(40)] + [([5, 70], 0)]),
]


@pytest.mark.parametrize("dtype,D,B,Hq,Hkv,groups", CASES, ids=lambda v: str(v)[:50].replace(" ", ""))
def test_shared_decode_matches_oracle(dtype, D, B, Hq, Hkv, groups):
    seed = (D * 7 + B * 3 + Hq + Hkv + len(groups)) % 997
    q, kc, vc, bt, cl, share = shared_case(seed, dtype, D, B, Hq, Hkv, groups)
    assert np.array_equal(P.share_groups(bt.numpy(), cl.numpy(), B), share)
    scale = 1.0 / math.sqrt(D)
    got = shared_decode(q, kc.to(DEV), vc.to(DEV), bt, cl, share, scale, Hq, Hkv, D, B)
    want = ora(q, kc, vc, bt, cl, scale, dtype, Hq, Hkv, D, B)
    assert_close(got, want, dtype, f"{dtype} D{D} B{B} G{Hq // Hkv}")
    assert P.pa_device_errors() == 0


def test_without_groups_equals_plain_decode_bitwise():
    groups = [([300], 0), ([17], 0), ([1000], 0), ([1], 0)]
    q, kc, vc, bt, cl, share = shared_case(5, "bf16", 128, 16, 32, 8, groups)
    got = shared_decode(q, kc.to(DEV), vc.to(DEV), bt, cl, share, 0.09, 32, 8, 128, 16)
    out = torch.empty_like(q, device=DEV)
    P.pa_decode(out, q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), cl.to(DEV), 0.09, 32, 8, 128, 16,
                partition_size=0)
    torch.cuda.synchronize()
    assert torch.equal(got, out)


def test_repeated_calls_are_identical():
    groups = [(lens_for(8, 40, 16, 21), 40), (lens_for(3, 9, 16, 22), 9)]
    q, kc, vc, bt, cl, share = shared_case(21, "f16", 128, 16, 16, 2, groups)
    kd, vd = kc.to(DEV), vc.to(DEV)
    a = shared_decode(q, kd, vd, bt, cl, share, 0.1, 16, 2, 128, 16)
    b = shared_decode(q, kd, vd, bt, cl, share, 0.1, 16, 2, 128, 16)
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,Hq,Hkv,B", [("bf16", 8, 2, 16), ("f16", 40, 40, 16), ("f32", 4, 4, 32),
                                            ("bf16", 32, 8, 32)])
def test_shared_decode_with_fused_append(dtype, Hq, Hkv, B):
    """pa_decode_shared(k_new, v_new) == pa_reshape_and_cache(newest tokens) + oracle."""
    D = 128
    groups = [(lens_for(8, 6, B, 31), 6), ([B * 2 + 1], 0), (lens_for(3, 2, B, 32, 1), 2)]
    # include members whose newest token is the first row of their first own block
    groups.append(([2 * B + 1, 2 * B + 1, 2 * B + 2], 2))
    q, kc, vc, bt, cl, share = shared_case(31, dtype, D, B, Hq, Hkv, groups, stale=0.0)
    S = cl.shape[0]
    g = torch.Generator().manual_seed(33)
    k_new = torch.randn(S, Hkv, D, generator=g).to(q.dtype)
    v_new = torch.randn(S, Hkv, D, generator=g).to(q.dtype)
    slots = [int(bt[s, (int(t) - 1) // B]) * B + (int(t) - 1) % B for s, t in enumerate(cl.tolist())]
    k2, v2 = kc.to(DEV), vc.to(DEV)
    got = shared_decode(q, k2, v2, bt, cl, share, 0.08, Hq, Hkv, D, B, k_new.to(DEV), v_new.to(DEV))
    kh, vh = raw(kc).copy(), raw(vc).copy()
    oracle.reshape_and_cache(raw(k_new), raw(v_new), kh, vh, np.array(slots), B)
    assert np.array_equal(raw(k2), kh) and np.array_equal(raw(v2), vh)
    want = oracle.decode(raw(q), kh, vh, bt.numpy(), cl.numpy(), 0.08, dtype, Hq, Hkv, D, B)
    assert_close(got, want, dtype)
    assert P.pa_device_errors() == 0


def test_group_wider_than_an_item_is_unsupported():
    groups = [(lens_for(2, 2, 16, 41), 2)]
    q, kc, vc, bt, cl, share = shared_case(41, "bf16", 64, 16, 40, 2, groups)
    with pytest.raises(P.PagedKVError):
        shared_decode(q, kc.to(DEV), vc.to(DEV), bt, cl, share, 0.1, 40, 2, 64, 16)


def test_empty_batch():
    q = torch.empty(0, 8, 64, dtype=torch.float16, device=DEV)
    kc = torch.zeros(4, 16, 8, 64, dtype=torch.float16, device=DEV)
    out = torch.empty_like(q)
    P.pa_decode_shared(out, q, kc, kc.clone(), torch.zeros(0, 1, dtype=torch.int32, device=DEV),
                       torch.zeros(0, dtype=torch.int32, device=DEV),
                       torch.zeros(0, 2, dtype=torch.int32, device=DEV), 0.1, 8, 8, 64, 16)
    torch.cuda.synchronize()


@pytest.mark.parametrize("short", [1, 20 * 16, 20 * 16 - 5])
def test_member_ending_inside_the_shared_blocks_is_flagged_and_decoded_alone(short):
    """A member whose context does not extend past its group's shared blocks breaks
    the decode's precondition: the device reports PA_DEVERR_SHARE, and the member
    is decoded as if it shared nothing, so every output still matches the oracle."""
    dtype, D, B, Hq, Hkv, Pb = "bf16", 128, 16, 16, 4, 20
    lens = lens_for(5, Pb, B, 9)
    q, kc, vc, bt, cl, share = shared_case(31, dtype, D, B, Hq, Hkv, [(lens, Pb)], stale=0.0)
    cl[2] = short                      # member 2 now ends inside the 20 shared blocks
    bt[2, (short + B - 1) // B:] = -1
    assert share[2, 0] == 0 and share[2, 1] == Pb
    assert P.pa_device_errors() == 0
    got = shared_decode(q, kc.to(DEV), vc.to(DEV), bt, cl, share, 0.09, Hq, Hkv, D, B)
    assert P.pa_device_errors() == P.PA_DEVERR_SHARE
    assert_close(got, ora(q, kc, vc, bt, cl, 0.09, dtype, Hq, Hkv, D, B), dtype, f"member of {short} tokens")
