"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`
may import this package.  The library (`paged_kv_cache_79_gb300`) never imports it
and shares no code with it; both read their seeded inputs from `workloads`.

Contents
  decode(...)              fp64 attention by its plain definition (pa_oracle.c):
                           gather the T valid keys/values through the block table,
                           dense softmax attention.  Pages: azimuth.plus
                           PagedAttention summary, section "The PagedAttention
                           algorithm" (block-wise attention equation, identical to
                           standard attention); CSDN tutorial "PagedAttention实战"
                           §3.2 (gather valid rows, dense softmax, zeros if empty).
  reshape_and_cache(...)   write token t's K/V row at cache[slot // B][slot % B]
                           (tutorial §3.1: logical page pos // page_size, offset
                           pos % page_size); a negative slot skips the token.
  copy_blocks(...)         copy-on-write of whole blocks, pair by pair
                           (azimuth.plus summary, section "Memory sharing").
  swap_blocks(...)         block moves between two pools (summary, section "vLLM":
                           a preempted request's blocks go to CPU memory and back).
  gather_blocks(...),      pack blocks into a contiguous buffer and back (spke.com
  scatter_blocks(...)      article on bidirectional KV transfer, section
                           "Bidirectional KV transfer").
  kv_transfer_worthwhile   the same article's recompute threshold (section "KV
                           recompute threshold").
  BlockAllocator           reference allocator (oracle/allocator.py), swap included.
  run_script(...)          execute a workload's allocator script with the above.

Parity status: every function here is pinned by tests/test_oracle_*.py against
values the pages print or fix, closed forms, invariants and textbook routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from .allocator import BlockAllocator, OracleOOM

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpa_oracle.so")
_lib = None
_lock = threading.Lock()

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with the host C compiler (plain -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.oracle_decode.restype = ctypes.c_int
            L.oracle_decode.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_longlong, ctypes.c_double]
            L.oracle_f16_to_f64.restype = ctypes.c_double
            L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f64.restype = ctypes.c_double
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_num_threads.restype = ctypes.c_int
            L.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = L
        return _lib


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def _raw(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage bits as a C-contiguous array: float32 for fp32, uint16 for fp16/bf16."""
    want = np.float32 if dtype == "f32" else np.uint16
    if a.dtype == np.float16 and dtype == "f16":
        a = a.view(np.uint16)
    if a.dtype != want:
        raise TypeError(f"expected raw {want} storage for {dtype}, got {a.dtype}")
    return np.ascontiguousarray(a)


def decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_tables: np.ndarray,
           context_lens: np.ndarray, scale: float, dtype: str, num_q_heads: int, num_kv_heads: int,
           head_dim: int, block_size: int) -> np.ndarray:
    """fp64 paged decode attention; returns out[S, Hq, d] (float64).

    q: raw [S, Hq, d]; caches: raw [NB, B, Hkv, d]; block_tables int32 [S, W];
    context_lens int32 [S].  Raw = float32 for fp32, uint16 bit patterns otherwise."""
    q = _raw(q, dtype)
    k_cache = _raw(k_cache, dtype)
    v_cache = _raw(v_cache, dtype)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S = cl.shape[0]
    W = bt.shape[1] if bt.ndim == 2 else 0
    nb = k_cache.size // (block_size * num_kv_heads * head_dim)
    out = np.zeros((S, num_q_heads, head_dim), dtype=np.float64)
    rc = lib().oracle_decode(out.ctypes.data, q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
                             DTYPE_CODE[dtype], bt.ctypes.data, W, cl.ctypes.data, S, num_q_heads,
                             num_kv_heads, head_dim, block_size, nb, float(scale))
    if rc != 0:
        raise ValueError(f"oracle_decode rejected its inputs (code {rc})")
    return out


def f16_to_f64(bits: int) -> float:
    return lib().oracle_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    return lib().oracle_bf16_to_f64(bits)


def reshape_and_cache(k: np.ndarray, v: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                      slot_mapping: np.ndarray, block_size: int) -> None:
    """In place: cache[slot // B][slot % B] = row, token by token in order; slot < 0 skips."""
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        k_cache[blk, off] = k[t]
        v_cache[blk, off] = v[t]


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs: Sequence[Tuple[int, int]]) -> None:
    """In place: for each (src, dst) in order, the whole block dst becomes a copy of src."""
    for src, dst in pairs:
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]


def swap_blocks(src_k: np.ndarray, src_v: np.ndarray, dst_k: np.ndarray, dst_v: np.ndarray,
                pairs: Sequence[Tuple[int, int]]) -> None:
    """dst[dst_i] = src[src_i] for every pair: block moves between two pools
    (azimuth.plus summary, section "vLLM": blocks of a preempted request go to CPU
    memory and come back).  Pairs with an index outside a pool are skipped."""
    for s, d in pairs:
        if 0 <= s < src_k.shape[0] and 0 <= d < dst_k.shape[0]:
            dst_k[d] = src_k[s]
            dst_v[d] = src_v[s]


def gather_blocks(k_cache: np.ndarray, v_cache: np.ndarray, block_ids: Sequence[int]):
    """Contiguous copies of the listed blocks, in order (the sending half of a KV
    transfer; spke.com article, section "Bidirectional KV transfer").  Ids outside
    the pool give zero blocks."""
    ks = np.zeros((len(block_ids),) + k_cache.shape[1:], dtype=k_cache.dtype)
    vs = np.zeros_like(ks)
    for i, b in enumerate(block_ids):
        if 0 <= b < k_cache.shape[0]:
            ks[i] = k_cache[b]
            vs[i] = v_cache[b]
    return ks, vs


def scatter_blocks(staging_k: np.ndarray, staging_v: np.ndarray, k_cache: np.ndarray,
                   v_cache: np.ndarray, block_ids: Sequence[int]) -> None:
    """cache[block_ids[i]] = staging[i] (the receiving half)."""
    for i, b in enumerate(block_ids):
        if 0 <= b < k_cache.shape[0]:
            k_cache[b] = staging_k[i]
            v_cache[b] = staging_v[i]


def kv_transfer_worthwhile(reusable_tokens: int, threshold: int = 64) -> bool:
    """spke.com article, section "KV recompute threshold": the prefill side
    recomputes when fewer than `threshold` tokens could be reused and fetches the
    KV when that many or more can (default 64)."""
    return reusable_tokens > 0 and reusable_tokens >= threshold


def run_script(events, num_blocks: int, block_size: int, free_order,
               k_cache: Optional[np.ndarray] = None, v_cache: Optional[np.ndarray] = None,
               step_kv=None, on_step=None):
    """Execute an allocator script (workloads.NewSeq/Fork/Prefill/Step/FreeSeq).

    Copy-on-write pairs are applied to the caches (when given) before the step's
    K/V rows are written.  `step_kv(step)` returns raw (k, v) for a Step; `on_step`
    is called after each Step with (step, allocator).  Returns the allocator and
    the list of (event, slots, pairs) records."""
    import workloads as W
    alloc = BlockAllocator(num_blocks, block_size, free_order)
    records = []
    for ev in events:
        if isinstance(ev, W.NewSeq):
            alloc.new_seq()
        elif isinstance(ev, W.Fork):
            alloc.fork(ev.parent)
        elif isinstance(ev, W.FreeSeq):
            alloc.free_seq(ev.seq)
        elif isinstance(ev, (W.Prefill, W.Step)):
            seqs = [ev.seq] * ev.n if isinstance(ev, W.Prefill) else list(ev.seqs)
            slots, pairs = [], []
            for s in seqs:
                slot, cow = alloc.append(s)
                slots.append(slot)
                if cow is not None:
                    pairs.append(cow)
            if k_cache is not None and pairs:
                copy_blocks(k_cache, v_cache, pairs)
            if isinstance(ev, W.Step) and k_cache is not None and step_kv is not None:
                k, v = step_kv(ev)
                reshape_and_cache(k, v, k_cache, v_cache, np.array(slots, dtype=np.int64), block_size)
            records.append((ev, slots, pairs))
            if isinstance(ev, W.Step) and on_step is not None:
                on_step(ev, alloc)
        else:
            raise TypeError(f"unknown event {ev!r}")
    return alloc, records


def tables_for(alloc: BlockAllocator, seqs: Sequence[int], width: Optional[int] = None):
    """(block_tables int32 [S, width] padded with -1, context_lens int32 [S])."""
    tabs = [alloc.block_table(s) for s in seqs]
    w = width if width is not None else max(1, max(len(t) for t in tabs))
    bt = np.full((len(seqs), w), -1, dtype=np.int32)
    for i, t in enumerate(tabs):
        bt[i, :len(t)] = t
    cl = np.array([alloc.seq_len(s) for s in seqs], dtype=np.int32)
    return bt, cl


__all__ = ["decode", "reshape_and_cache", "copy_blocks", "BlockAllocator", "OracleOOM",
           "run_script", "tables_for", "build", "num_threads", "set_num_threads",
           "f16_to_f64", "bf16_to_f64"]
