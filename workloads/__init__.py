"""Seeded synthetic workloads for paged decode attention.

This module is shared by the CUDA path's tests and bench and by the CPU oracle's
tests.  It holds NO attention arithmetic and no allocator policy: only workload
shapes, seeded context lengths, seeded pool permutations, the allocator *scripts*
(which sequences are created, forked and grown, in which order) and seeded random
tensors.  Each side executes a script with its own allocator and its own cache
operations.

Workload shapes follow the five synthetic configurations of the paged-attention
decode benchmark:

  tiny                 1 sequence, T = 1..50 appended one token at a time, 8 heads
                       (MHA), head_dim 64, block_size 16, fp32, pool of 100 blocks.
                       Shape taken from the CSDN tutorial "PagedAttention实战" §4
                       (100 pages, page_size 16, 8 heads, head_dim 64, 50 steps).
  mha_fp16             8 sequences, 40/40 heads, head_dim 128, block_size 16,
                       T ~ U{1..2048}, pool of 8192 shuffled blocks.
  gqa_bf16             64 sequences, 64 q heads / 8 kv heads, head_dim 128,
                       block_size 16, T lognormal (median 4096, sigma 1.0) clipped
                       to [16, 32768], pool = ceil(1.1 x used blocks).
  shared_prefix_fp16   16 prompts x 8 samples, 40/40 heads, head_dim 128,
                       block_size 16, prompt 1024 tokens shared by the 8 samples
                       (variant: 1032 tokens, whose last prompt block is partial and
                       is copied on write), continuation U{0..512} per sample.
  long_multiturn_bf16  256 sequences in 64 groups of 4 "turns", 32 q / 8 kv heads,
                       head_dim 128, block_size 32, T log-uniform in [128, 131072],
                       each group sharing its first floor(0.6 * min nb) blocks,
                       split-KV partition 512 tokens.

Values of q, K and V are N(0, 1), drawn in fp32 with a seeded torch.Generator and
rounded to the storage dtype.  Structure (lengths, permutations) is drawn with
numpy's PCG64 seeded with 1000 + the configuration's index.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

import numpy as np

DTYPES = ("f32", "f16", "bf16")
DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2}

CONFIG_NAMES = ("tiny", "mha_fp16", "gqa_bf16", "shared_prefix_fp16", "long_multiturn_bf16")


# ----------------------------------------------------------------------------
# Allocator scripts.  An event names *what* happens to the sequences; how blocks
# are chosen, shared and copied is decided by whichever allocator runs it.
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class NewSeq:
    """Create an empty sequence; ids are handed out 0, 1, 2, ... in creation order."""


@dataclasses.dataclass(frozen=True)
class Fork:
    """Create a new sequence sharing every block of `parent` (parallel sampling)."""
    parent: int


@dataclasses.dataclass(frozen=True)
class Prefill:
    """Append `n` tokens to `seq` whose K/V already sit in the pool (no data write).

    Copy-on-write pairs that these appends produce must still be executed."""
    seq: int
    n: int


@dataclasses.dataclass(frozen=True)
class Step:
    """One decode step: append one token to each sequence of `seqs` (ascending id
    order), executing any copy-on-write pairs first, then writing the new tokens'
    K/V through the slot mapping.  `index` selects the random K/V of this step."""
    seqs: Tuple[int, ...]
    index: int


@dataclasses.dataclass(frozen=True)
class FreeSeq:
    """Release a sequence's blocks."""
    seq: int


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    num_blocks: int
    free_order: np.ndarray           # int32 permutation of 0..num_blocks-1 (initial free list)
    events: List[object]
    decode_seqs: List[int]           # the batch, in order, decoded after the script
    partition_size: int = 0          # 0: let the library choose
    scale: Optional[float] = None    # default 1/sqrt(head_dim)
    data_seed: int = 0
    note: str = ""

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def num_seqs(self) -> int:
        return len(self.decode_seqs)

    @property
    def elem_bytes(self) -> int:
        return DTYPE_BYTES[self.dtype]

    def step_events(self) -> List[Step]:
        return [e for e in self.events if isinstance(e, Step)]

    def total_steps(self) -> int:
        return len(self.step_events())


def _rng(index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(1000 + index))


def free_order(num_blocks: int, rng: np.random.Generator) -> np.ndarray:
    """A seeded shuffle of the pool ids (numpy's Fisher-Yates permutation)."""
    return rng.permutation(num_blocks).astype(np.int32)


def _blocks(t: int, b: int) -> int:
    return (t + b - 1) // b


# ----------------------------------------------------------------------------
# The five configurations
# ----------------------------------------------------------------------------
def tiny(steps: int = 50) -> Workload:
    rng = _rng(0)
    ev: List[object] = [NewSeq()]
    ev += [Step((0,), i) for i in range(steps)]
    return Workload("tiny", 8, 8, 64, 16, "f32", 100, free_order(100, rng), ev, [0],
                    data_seed=2000, note="CSDN tutorial §4 workflow: 50 appends, decode after each")


def mha_fp16(num_seqs: int = 8, max_len: int = 2048, pool: int = 8192) -> Workload:
    rng = _rng(1)
    lens = rng.integers(1, max_len + 1, size=num_seqs)
    ev: List[object] = []
    for s in range(num_seqs):
        ev.append(NewSeq())
        if lens[s] > 1:
            ev.append(Prefill(s, int(lens[s]) - 1))
    ev.append(Step(tuple(range(num_seqs)), 0))
    return Workload("mha_fp16", 40, 40, 128, 16, "f16", pool, free_order(pool, rng), ev,
                    list(range(num_seqs)), data_seed=2001)


def gqa_lengths(num_seqs: int, rng: np.random.Generator) -> np.ndarray:
    """Lognormal context lengths: median 4096, sigma 1.0 in log space, rounded, clipped to [16, 32768]."""
    t = np.exp(rng.normal(math.log(4096.0), 1.0, size=num_seqs))
    return np.clip(np.rint(t), 16, 32768).astype(np.int64)


def gqa_bf16(num_seqs: int = 64) -> Workload:
    rng = _rng(2)
    lens = gqa_lengths(num_seqs, rng)
    used = int(sum(_blocks(int(t), 16) for t in lens))
    pool = int(math.ceil(1.1 * used))
    ev: List[object] = []
    for s in range(num_seqs):
        ev.append(NewSeq())
        ev.append(Prefill(s, int(lens[s]) - 1))
    ev.append(Step(tuple(range(num_seqs)), 0))
    return Workload("gqa_bf16", 64, 8, 128, 16, "bf16", pool, free_order(pool, rng), ev,
                    list(range(num_seqs)), data_seed=2002)


def shared_prefix_fp16(prompts: int = 16, samples: int = 8, prompt_len: int = 1024,
                       max_cont: int = 512, decode_steps: int = 1) -> Workload:
    """Parallel sampling: each prompt is prefilled once, forked into `samples`
    sequences, and every sample then grows by its own continuation.

    The continuation of sample i is c_i ~ U{0..max_cont} tokens, prefilled; then
    `decode_steps` decode steps append one token to every sample.  With a prompt
    length that is not a multiple of the block size the first append of each sample
    lands in the shared partial prompt block (copy-on-write)."""
    rng = _rng(3)
    b = 16
    conts = rng.integers(0, max_cont + 1, size=(prompts, samples))
    ev: List[object] = []
    seq = 0
    order: List[int] = []
    groups = []
    for p in range(prompts):
        root = seq
        ev.append(NewSeq())
        ev.append(Prefill(root, prompt_len))
        seq += 1
        members = [root]
        for _ in range(samples - 1):
            ev.append(Fork(root))
            members.append(seq)
            seq += 1
        groups.append(members)
        order += members
    for p in range(prompts):
        for i, s in enumerate(groups[p]):
            if conts[p, i] > 0:
                ev.append(Prefill(s, int(conts[p, i])))
    for k in range(decode_steps):
        ev.append(Step(tuple(sorted(order)), k))
    # unique blocks: prompt blocks once per prompt + private blocks + copy-on-write slack
    tot = prompts * (_blocks(prompt_len, b) + samples * (_blocks(max_cont + decode_steps, b) + 2))
    pool = int(math.ceil(1.1 * tot))
    name = "shared_prefix_fp16" if prompt_len % b == 0 else f"shared_prefix_fp16_p{prompt_len}"
    return Workload(name, 40, 40, 128, b, "f16", pool, free_order(pool, rng), ev, sorted(order),
                    data_seed=2003)


def multiturn_lengths(groups: int, rng: np.random.Generator, lo: int = 128, hi: int = 131072) -> np.ndarray:
    """Log-uniform context lengths in [lo, hi], 4 per group, drawn independently."""
    t = np.exp(rng.uniform(math.log(lo), math.log(hi), size=(groups, 4)))
    return np.clip(np.rint(t), lo, hi).astype(np.int64)


def long_multiturn_bf16(groups: int = 64, lo: int = 128, hi: int = 131072) -> Workload:
    """Groups of 4 'turn' sequences.  The group's first P = floor(0.6 * min nb)
    blocks are prefilled once and shared (refcount 4); the rest is private."""
    rng = _rng(4)
    b = 32
    lens = multiturn_lengths(groups, rng, lo, hi)
    ev: List[object] = []
    seq = 0
    order: List[int] = []
    unique = 0
    for g in range(groups):
        nbs = [_blocks(int(t), b) for t in lens[g]]
        shared = int(math.floor(0.6 * min(nbs)))
        root = seq
        ev.append(NewSeq())
        seq += 1
        if shared > 0:
            ev.append(Prefill(root, shared * b))
        members = [root]
        for _ in range(3):
            ev.append(Fork(root))
            members.append(seq)
            seq += 1
        for i, s in enumerate(members):
            ev.append(Prefill(s, int(lens[g, i]) - shared * b - 1))
        order += members
        unique += shared + sum(n - shared for n in nbs)
    ev.append(Step(tuple(sorted(order)), 0))
    pool = unique + 64
    return Workload("long_multiturn_bf16", 32, 8, 128, b, "bf16", pool, free_order(pool, rng), ev,
                    sorted(order), partition_size=512, data_seed=2004)


def beam_search_fp16(beams: int = 4, prompt_len: int = 500, steps: int = 200, seed: int = 6,
                     pool: Optional[int] = None) -> Workload:
    """Beam search over one prompt (allocator trace; MHA fp16 shapes as in the
    parallel-sampling configuration).

    The prompt is prefilled once and forked into `beams` beams.  At every step each
    of the `beams` new beams picks its parent among the current beams (seeded,
    uniform, with replacement), is created as a fork of it, the previous beams are
    freed, and every new beam appends one token -- so beams that share a parent share
    its blocks and copy the partial last block on their first write."""
    rng = _rng(20 + seed)
    b = 16
    ev: List[object] = [NewSeq(), Prefill(0, prompt_len)]
    cur = [0]
    nxt = 1
    for _ in range(beams - 1):
        ev.append(Fork(0))
        cur.append(nxt)
        nxt += 1
    for k in range(steps):
        parents = rng.integers(0, beams, size=beams)
        new = []
        for p_ in parents:
            ev.append(Fork(cur[int(p_)]))
            new.append(nxt)
            nxt += 1
        for q in cur:
            ev.append(FreeSeq(q))
        cur = new
        ev.append(Step(tuple(cur), k))
    if pool is None:
        pool = 2 * beams * (_blocks(prompt_len + steps, b) + 2) + 8
    return Workload(f"beam_search_fp16_k{beams}", 40, 40, 128, b, "f16", pool, free_order(pool, rng), ev,
                    list(cur), data_seed=2006)


def by_name(name: str, **kw) -> Workload:
    table = {
        "tiny": tiny,
        "mha_fp16": mha_fp16,
        "gqa_bf16": gqa_bf16,
        "shared_prefix_fp16": shared_prefix_fp16,
        "shared_prefix_fp16_p1032": lambda **k: shared_prefix_fp16(prompt_len=1032, **k),
        "long_multiturn_bf16": long_multiturn_bf16,
        "beam_search_fp16": beam_search_fp16,
    }
    return table[name](**kw)


# ----------------------------------------------------------------------------
# Random tensors (torch; CPU or CUDA generator).  Plain value generation only.
# ----------------------------------------------------------------------------
def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def randn(shape, dtype: str, seed: int, device="cpu"):
    """N(0,1) drawn in fp32 with a seeded generator on `device`, rounded to `dtype`."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x.to(torch_dtype(dtype))


def cache_shape(w: Workload):
    """[num_blocks, block_size, num_kv_heads, head_dim]: the page layout of the
    CSDN tutorial's Page (keys/values of shape [page_size, num_heads, head_dim])."""
    return (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)


def pool_tensors(w: Workload, device="cpu"):
    """Initial K and V pools: every block holds N(0,1) data (prefilled or stale).

    Both are views of one [2, num_blocks, block_size, num_kv_heads, head_dim] buffer,
    V after K, the placement under which the decode fetches a block's K and V tiles
    with one copy.  The values are those of two separate seeded draws."""
    import torch
    shape = cache_shape(w)
    kv = torch.empty((2,) + shape, dtype=torch_dtype(w.dtype), device=device)
    kv[0].copy_(randn(shape, w.dtype, w.data_seed * 10 + 1, device))
    kv[1].copy_(randn(shape, w.dtype, w.data_seed * 10 + 2, device))
    return kv[0], kv[1]


def step_tensors(w: Workload, step: Step, device="cpu"):
    """New K, V for one decode step: [len(step.seqs), num_kv_heads, head_dim]."""
    n = len(step.seqs)
    base = w.data_seed * 1000 + 100 + 3 * step.index
    return (randn((n, w.num_kv_heads, w.head_dim), w.dtype, base, device),
            randn((n, w.num_kv_heads, w.head_dim), w.dtype, base + 1, device))


def query_tensor(w: Workload, step_index: int = 0, device="cpu"):
    """q: [num_seqs, num_q_heads, head_dim] for the decode after step `step_index`."""
    return randn((w.num_seqs, w.num_q_heads, w.head_dim), w.dtype,
                 w.data_seed * 1000 + 102 + 3 * step_index, device)


def random_tables(rng: np.random.Generator, lens, block_size: int, num_blocks: int,
                  pad: int = 0) -> Tuple[np.ndarray, int]:
    """Block tables drawn without replacement from a shuffled pool, padded with -1."""
    nbs = [_blocks(int(t), block_size) for t in lens]
    width = max(1, max(nbs) + pad)
    need = sum(nbs)
    if need > num_blocks:
        raise ValueError("pool too small")
    perm = rng.permutation(num_blocks)[:need]
    tab = np.full((len(lens), width), -1, dtype=np.int32)
    k = 0
    for s, n in enumerate(nbs):
        tab[s, :n] = perm[k:k + n]
        k += n
    return tab, width
