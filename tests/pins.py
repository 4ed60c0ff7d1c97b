"""Pins for the oracle: checks against what the pages and the mathematics fix.

Each pin takes the decode function under test (same signature as oracle.decode),
so the mutation test can run the same pins against oracle builds with planted
mistakes.  Nothing here reuses the oracle's own formula: the brute force works on
contiguous (un-paged) keys with numpy's textbook softmax attention, the other pins
are closed forms, invariants and hand-evaluated examples.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# storage helpers (library conversions: numpy float16, torch bfloat16)
# ----------------------------------------------------------------------------
def to_raw(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64/32 values to the storage dtype; return raw storage bits."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(x, dtype=np.float16).view(np.uint16)
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def from_raw(r: np.ndarray, dtype: str) -> np.ndarray:
    """Exact value of raw storage as float64 (numpy / torch conversions)."""
    if dtype == "f32":
        return r.astype(np.float64)
    if dtype == "f16":
        return r.view(np.float16).astype(np.float64)
    t = torch.from_numpy(r.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def brute_force(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """Dense softmax attention on contiguous keys: softmax(scale * K q) V per head.

    q [Hq, d]; keys/values [T, Hkv, d] (float64); q heads grouped contiguously over
    kv heads.  Written with numpy's max-shifted softmax, the textbook routine."""
    hq, d = q.shape
    T, hkv, _ = keys.shape
    out = np.zeros((hq, d))
    if T == 0:
        return out
    g = hq // hkv
    for h in range(hq):
        K = keys[:, h // g, :]
        V = values[:, h // g, :]
        s = scale * (K @ q[h])
        w = np.exp(s - s.max())
        w /= w.sum()
        out[h] = w @ V
    return out


def scatter_to_pool(rng, seqs_kv, num_blocks, block_size, dtype, junk=np.nan):
    """Place each sequence's contiguous keys/values into random physical blocks.

    seqs_kv: list of (keys, values) float arrays [T, Hkv, d].  Returns raw pools,
    block tables (int32, -1 padded) and lengths.  Every unused row holds `junk`."""
    hkv, d = seqs_kv[0][0].shape[1:]
    kp = np.full((num_blocks, block_size, hkv, d), junk, dtype=np.float64)
    vp = np.full((num_blocks, block_size, hkv, d), junk, dtype=np.float64)
    nbs = [(k.shape[0] + block_size - 1) // block_size for k, _ in seqs_kv]
    perm = rng.permutation(num_blocks)
    width = max(1, max(nbs) + 1)
    tab = np.full((len(seqs_kv), width), -1, dtype=np.int32)
    c = 0
    for s, (k, v) in enumerate(seqs_kv):
        for j in range(nbs[s]):
            p = perm[c]
            c += 1
            tab[s, j] = p
            rows = k[j * block_size:(j + 1) * block_size]
            kp[p, :rows.shape[0]] = rows
            vp[p, :rows.shape[0]] = v[j * block_size:(j + 1) * block_size]
    lens = np.array([k.shape[0] for k, _ in seqs_kv], dtype=np.int32)
    with np.errstate(invalid="ignore", over="ignore"):
        return to_raw(kp, dtype), to_raw(vp, dtype), tab, lens


def _case(dec, rng, S, Hq, Hkv, d, B, dtype, lens, scale, junk=np.nan, nb_extra=3):
    seqs = []
    for T in lens:
        k = from_raw(to_raw(rng.standard_normal((T, Hkv, d)), dtype), dtype)
        v = from_raw(to_raw(rng.standard_normal((T, Hkv, d)), dtype), dtype)
        seqs.append((k, v))
    nb = sum((T + B - 1) // B for T in lens) + nb_extra
    kp, vp, tab, L = scatter_to_pool(rng, seqs, nb, B, dtype, junk)
    qraw = to_raw(rng.standard_normal((S, Hq, d)), dtype)
    qv = from_raw(qraw, dtype)
    got = dec(qraw, kp, vp, tab, L, scale, dtype, Hq, Hkv, d, B)
    want = np.stack([brute_force(qv[s], seqs[s][0], seqs[s][1], scale) for s in range(S)])
    return got, want


# ----------------------------------------------------------------------------
# attention pins
# ----------------------------------------------------------------------------
def pin_golden_two_block(dec):
    """Hand-evaluated example of the block-wise equation (tests/golden)."""
    with open(os.path.join(GOLDEN, "two_block_example.json")) as f:
        g = json.load(f)
    B, hkv, d, nb = g["block_size"], g["num_kv_heads"], g["head_dim"], g["num_blocks"]
    kp = np.full((nb, B, hkv, d), np.nan)
    vp = np.full((nb, B, hkv, d), np.nan)
    keys = np.array(g["keys_logical"])
    vals = np.array(g["values_logical"])
    for j, p in enumerate(g["block_table"]):
        kp[p, :, 0] = keys[j * B:(j + 1) * B]
        vp[p, :, 0] = vals[j * B:(j + 1) * B]
    tab = np.array([g["block_table"]], dtype=np.int32)
    q = np.array([[g["q"]]], dtype=np.float32)
    for case in g["cases"]:
        T = case["context_len"]
        kk, vv = kp.copy(), vp.copy()
        # rows at or beyond T are stale: make them poisonous
        for t in range(T, len(g["block_table"]) * B):
            p = g["block_table"][t // B]
            kk[p, t % B] = 1e30
            vv[p, t % B] = np.nan
        out = dec(q, kk.astype(np.float32), vv.astype(np.float32), tab, np.array([T], np.int32),
                  g["scale"], "f32", 1, 1, d, B)
        assert np.allclose(out[0, 0], case["expected"], rtol=0, atol=g["tolerance"]), (T, out[0, 0])


def pin_brute_force(dec):
    """Paged oracle == dense softmax attention on the same keys, several shapes."""
    rng = np.random.default_rng(11)
    shapes = [
        (1, 1, 1, 4, 2, "f32", [5], 0.5),
        (2, 4, 2, 8, 4, "f32", [13, 1], 1 / math.sqrt(8)),
        (2, 6, 3, 16, 16, "f16", [40, 17], 1 / 4),
        (1, 8, 1, 8, 4, "bf16", [9], 0.3),
        (2, 2, 2, 4, 3, "bf16", [7, 12], 1.7),
        (1, 5, 5, 8, 16, "f16", [16], -0.4),
    ]
    for (S, Hq, Hkv, d, B, dtype, lens, scale) in shapes:
        got, want = _case(dec, rng, S, Hq, Hkv, d, B, dtype, lens, scale)
        err = np.max(np.abs(got - want))
        assert err <= 1e-12 * max(1.0, np.max(np.abs(want))), (S, Hq, Hkv, d, B, dtype, lens, err)


def pin_single_token_is_value(dec):
    """T = 1: the only weight is 1, so out = V_0 exactly."""
    rng = np.random.default_rng(12)
    for dtype in ("f32", "f16", "bf16"):
        got, want = _case(dec, rng, 2, 4, 2, 8, 4, dtype, [1, 1], 0.7)
        assert np.array_equal(got, want), dtype


def pin_identical_keys_mean(dec):
    """All keys equal: every weight is 1/T and out = mean of the valid values."""
    rng = np.random.default_rng(13)
    T, hkv, d, B = 11, 2, 8, 4
    k = np.tile(rng.standard_normal((1, hkv, d)), (T, 1, 1))
    v = rng.standard_normal((T, hkv, d))
    kp, vp, tab, L = scatter_to_pool(rng, [(k, v)], 6, B, "f32")
    q = to_raw(rng.standard_normal((1, 4, d)), "f32")
    out = dec(q, kp, vp, tab, L, 0.9, "f32", 4, hkv, d, B)
    v32 = from_raw(to_raw(v, "f32"), "f32")
    for h in range(4):
        assert np.allclose(out[0, h], v32[:, h // 2].mean(axis=0), rtol=0, atol=1e-12)


def pin_zero_scale_mean(dec):
    """scale = 0: uniform weights regardless of the keys."""
    rng = np.random.default_rng(14)
    T, hkv, d, B = 9, 1, 4, 2
    k = rng.standard_normal((T, hkv, d)) * 10
    v = rng.standard_normal((T, hkv, d))
    kp, vp, tab, L = scatter_to_pool(rng, [(k, v)], 7, B, "f32")
    q = to_raw(rng.standard_normal((1, 1, d)), "f32")
    out = dec(q, kp, vp, tab, L, 0.0, "f32", 1, hkv, d, B)
    assert np.allclose(out[0, 0], from_raw(to_raw(v, "f32"), "f32")[:, 0].mean(axis=0), rtol=0, atol=1e-12)


def pin_weights_sum_to_one(dec):
    """V = 1 everywhere: out = sum_t p_t / sum_t p_t = 1."""
    rng = np.random.default_rng(15)
    T, hkv, d, B = 37, 2, 8, 16
    k = rng.standard_normal((T, hkv, d)) * 3
    v = np.ones((T, hkv, d))
    kp, vp, tab, L = scatter_to_pool(rng, [(k, v)], 5, B, "f32")
    q = to_raw(rng.standard_normal((1, 4, d)), "f32")
    out = dec(q, kp, vp, tab, L, 1.0, "f32", 4, hkv, d, B)
    assert np.max(np.abs(out - 1.0)) < 1e-14


def pin_block_permutation_invariance(dec):
    """Moving blocks to other physical ids (and remapping the table) changes nothing."""
    rng = np.random.default_rng(16)
    S, Hq, Hkv, d, B = 2, 4, 2, 8, 4
    lens = [14, 6]
    seqs = [(rng.standard_normal((T, Hkv, d)), rng.standard_normal((T, Hkv, d))) for T in lens]
    kp, vp, tab, L = scatter_to_pool(rng, seqs, 12, B, "f32")
    q = to_raw(rng.standard_normal((S, Hq, d)), "f32")
    a = dec(q, kp, vp, tab, L, 0.5, "f32", Hq, Hkv, d, B)
    perm = rng.permutation(12)           # new id of old block i is perm[i]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    tab2 = np.where(tab >= 0, perm[np.maximum(tab, 0)], -1).astype(np.int32)
    b = dec(q, kp2, vp2, tab2, L, 0.5, "f32", Hq, Hkv, d, B)
    assert np.max(np.abs(a - b)) <= 1e-12


def pin_stale_rows_ignored(dec):
    """Rows past T in the last block, and unreferenced blocks, never contribute."""
    rng = np.random.default_rng(17)
    clean, want = _case(dec, rng, 2, 2, 1, 8, 4, "f32", [10, 3], 0.6, junk=0.0)
    rng = np.random.default_rng(17)
    dirty, _ = _case(dec, rng, 2, 2, 1, 8, 4, "f32", [10, 3], 0.6, junk=np.nan)
    assert np.all(np.isfinite(dirty))
    assert np.array_equal(clean, dirty)
    rng = np.random.default_rng(17)
    big, _ = _case(dec, rng, 2, 2, 1, 8, 4, "f32", [10, 3], 0.6, junk=1e30)
    assert np.array_equal(clean, big)


def pin_empty_context_zeros(dec):
    """T = 0: the tutorial returns zeros_like(query)."""
    rng = np.random.default_rng(18)
    kp = to_raw(rng.standard_normal((3, 4, 1, 8)), "f32")
    vp = to_raw(rng.standard_normal((3, 4, 1, 8)), "f32")
    tab = np.array([[-1], [2]], dtype=np.int32)
    q = to_raw(rng.standard_normal((2, 2, 8)), "f32")
    out = dec(q, kp, vp, tab, np.array([0, 3], np.int32), 0.5, "f32", 2, 1, 8, 4)
    assert np.array_equal(out[0], np.zeros((2, 8)))
    assert np.all(np.abs(out[1]) > 0)


def pin_gqa_contiguous_groups(dec):
    """q head h reads kv head floor(h / G): value rows of kv head k are all k + 1."""
    rng = np.random.default_rng(19)
    Hq, Hkv, d, B, T = 12, 3, 4, 4, 7
    k = rng.standard_normal((T, Hkv, d))
    v = np.zeros((T, Hkv, d))
    for kv in range(Hkv):
        v[:, kv, :] = kv + 1
    kp, vp, tab, L = scatter_to_pool(rng, [(k, v)], 4, B, "f32")
    q = to_raw(rng.standard_normal((1, Hq, d)), "f32")
    out = dec(q, kp, vp, tab, L, 1.0, "f32", Hq, Hkv, d, B)
    for h in range(Hq):
        assert np.allclose(out[0, h], h // (Hq // Hkv) + 1, rtol=0, atol=1e-13), h


def pin_large_scores_stable(dec):
    """Scores near 1000 overflow exp() unless the maximum is subtracted first."""
    d, B = 2, 2
    kp = np.zeros((2, B, 1, d), np.float32)
    vp = np.zeros((2, B, 1, d), np.float32)
    kp[1, 0, 0] = [1000.0, 0.0]
    kp[1, 1, 0] = [1000.0 + math.log(3.0), 0.0]
    vp[1, 0, 0] = [4.0, 0.0]
    vp[1, 1, 0] = [0.0, 8.0]
    q = np.array([[[1.0, 0.0]]], np.float32)
    out = dec(q, kp, vp, np.array([[1]], np.int32), np.array([2], np.int32), 1.0, "f32", 1, 1, d, B)
    # weights 1:3 up to the float32 rounding of 1000 + ln 3 (spacing 2^-14 near 1000)
    w1 = 1.0 / (1.0 + math.exp(float(np.float32(1000.0 + math.log(3.0))) - 1000.0))
    assert np.allclose(out[0, 0], [4.0 * w1, 8.0 * (1 - w1)], rtol=0, atol=1e-9), out


ATTENTION_PINS = [pin_golden_two_block, pin_brute_force, pin_single_token_is_value,
                  pin_identical_keys_mean, pin_zero_scale_mean, pin_weights_sum_to_one,
                  pin_block_permutation_invariance, pin_stale_rows_ignored,
                  pin_empty_context_zeros, pin_gqa_contiguous_groups, pin_large_scores_stable]


# ----------------------------------------------------------------------------
# storage-decoding pins (all 65536 patterns against numpy / torch)
# ----------------------------------------------------------------------------
def pin_f16_all_patterns(conv):
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([conv(int(b)) for b in bits])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), bits[~same][:8]


def pin_bf16_all_patterns(conv):
    bits = np.arange(65536, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([conv(int(b)) for b in bits])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), bits[~same][:8]
