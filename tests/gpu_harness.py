"""Helpers for the GPU parity tests: raw storage views and tolerance checks.

Tolerances (stated for the attention output, fp32 accumulation):
  fp32 storage:        max |gpu - oracle| <= 1e-5
  fp16 / bf16 storage: "1e-2 (relative 1e-2)", read elementwise as
                       |gpu - oracle| <= 1e-2 * max(1, |oracle|)      and
                       max |gpu - oracle| / max |oracle| <= 1e-2      (normwise relative)
  A plain max-abs bound of 1e-2 would be finer than the output format: half a bf16
  ulp is 2^-9 |x|, more than 1e-2 once |x| > 2.56 (short contexts, where the output
  is an average of a few N(0,1) rows, reach |x| ~ 4).
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as W

TOL_F32 = 1e-5
TOL_16 = 1e-2


def raw(t: torch.Tensor) -> np.ndarray:
    """Storage bits of a tensor as numpy: float32 for fp32, uint16 for fp16/bf16."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def dtype_name(t: torch.Tensor) -> str:
    return {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[t.dtype]


def errors(got: torch.Tensor, want: np.ndarray):
    """(max abs error, normwise relative error, max of |error| / max(1, |ref|))."""
    g = got.detach().float().cpu().double().numpy()
    if not want.size:
        return 0.0, 0.0, 0.0
    d = np.abs(g - want)
    err = float(np.max(d))
    scale = float(np.max(np.abs(want)))
    mixed = float(np.max(d / np.maximum(1.0, np.abs(want))))
    return err, (err / scale if scale > 0 else err), mixed


def assert_close(got: torch.Tensor, want: np.ndarray, dtype: str, what: str = ""):
    assert np.all(np.isfinite(got.detach().float().cpu().numpy())), f"{what}: non-finite output"
    err, rel, mixed = errors(got, want)
    if dtype == "f32":
        assert err <= TOL_F32, f"{what}: max abs err {err:.3e} > {TOL_F32}"
    else:
        assert mixed <= TOL_16 and rel <= TOL_16, \
            f"{what}: max abs err {err:.3e}, elementwise {mixed:.3e}, normwise rel {rel:.3e}"
    return err, rel


def small_case(seed: int, dtype: str, D: int, B: int, Hq: int, Hkv: int, lens, extra_blocks: int = 5,
               stale=float("nan"), width_pad: int = 1):
    """Random pool + tables for the given context lengths (CPU tensors).

    Rows past each context and unreferenced blocks hold `stale`."""
    rng = np.random.default_rng(seed)
    nbs = [(t + B - 1) // B for t in lens]
    NB = sum(nbs) + extra_blocks
    bt, width = W.random_tables(rng, [max(t, 0) for t in lens], B, NB, pad=width_pad)
    kc = W.randn((NB, B, Hkv, D), "f32", seed * 7 + 1)
    vc = W.randn((NB, B, Hkv, D), "f32", seed * 7 + 2)
    used = np.zeros((NB, B), dtype=bool)
    for s, t in enumerate(lens):
        for tok in range(t):
            used[bt[s, tok // B], tok % B] = True
    m = torch.from_numpy(~used)
    kc[m] = stale
    vc[m] = stale
    q = W.randn((len(lens), Hq, D), "f32", seed * 7 + 3)
    td = W.torch_dtype(dtype)
    return (q.to(td), kc.to(td), vc.to(td), torch.from_numpy(bt), torch.tensor(lens, dtype=torch.int32))
