"""Execute an allocator script on the GPU path and prepare decode-step inputs.

A script is a list of events (new sequence, fork, prefill n tokens, decode step,
free).  The host allocator (pa_alloc_*) decides slots and copy-on-write pairs;
pa_copy_blocks and pa_reshape_and_cache apply them to the device caches.  The
last decode step's inputs are kept as a `DecodeStep`, which can be replayed: a
replay re-applies the same copy pairs and rows and recomputes the same decode.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional

import numpy as np

from . import (BlockAllocator, PagedKVError, alloc_workspace, pa_copy_blocks, pa_decode, pa_decode_append,
               pa_decode_plan, pa_decode_planned, pa_decode_shared, pa_decode_shared_plan,
               pa_decode_shared_planned, pa_decode_shared_workspace_size, pa_reshape_and_cache,
               share_groups, share_pays)


def _kind(ev) -> str:
    return type(ev).__name__


def tables_for(alloc: BlockAllocator, seqs, width: Optional[int] = None):
    """(block_tables int32 [S, width], -1 padded; context_lens int32 [S]) as numpy."""
    tabs = [alloc.block_table(s) for s in seqs]
    w = width if width is not None else max(1, max(len(t) for t in tabs))
    bt = np.full((len(seqs), w), -1, dtype=np.int32)
    for i, t in enumerate(tabs):
        bt[i, :len(t)] = t
    cl = np.array([alloc.seq_len(s) for s in seqs], dtype=np.int32)
    return bt, cl


@dataclasses.dataclass
class DecodeStep:
    """Device-resident inputs of one decode step (all CUDA tensors)."""
    q: "object"
    k_cache: "object"
    v_cache: "object"
    step_k: "object"
    step_v: "object"
    slots: "object"            # int64 [n_tok]
    pairs: "object"            # int32 [n_pairs, 2]
    block_tables: "object"     # int32 [S, W]
    context_lens: "object"     # int32 [S]
    out: "object"
    workspace: "object"
    scale: float
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    partition_size: int = 0
    fusable: bool = True        # step rows are the batch's newest tokens, in batch order
    share: "object" = None      # int32 [S, 2] shared-prefix groups, None if none share
    share_pays: bool = False    # the groups save enough reads for pa_decode_shared (share_pays)
    plan: "object" = None       # int32 device copy of pa_decode_plan for these tables and lengths
    shared_plan: "object" = None  # int32 device copy of pa_decode_shared_plan (with share)

    def run_planned(self, stream=None):
        """copy-on-write pairs, then the balanced-split decode with its CTAs starting
        where the host plan says (pa_decode_planned), the new tokens appended in the
        launch when the step is fusable, else before it."""
        if self.pairs.shape[0]:
            pa_copy_blocks(self.k_cache, self.v_cache, self.pairs, stream)
        if not self.fusable:
            pa_reshape_and_cache(self.step_k, self.step_v, self.k_cache, self.v_cache, self.slots, stream)
        return pa_decode_planned(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                 self.context_lens, self.plan, self.scale, self.num_q_heads,
                                 self.num_kv_heads, self.head_dim, self.block_size,
                                 k_new=self.step_k if self.fusable else None,
                                 v_new=self.step_v if self.fusable else None,
                                 workspace=self.workspace, stream=stream)

    def run_shared(self, stream=None, planned=True):
        """copy-on-write pairs, then the shared-prefix decode (which also appends the new
        tokens when the step is fusable), its CTAs starting from the host plan when
        there is one."""
        if self.pairs.shape[0]:
            pa_copy_blocks(self.k_cache, self.v_cache, self.pairs, stream)
        if not self.fusable:
            pa_reshape_and_cache(self.step_k, self.step_v, self.k_cache, self.v_cache, self.slots, stream)
        return self.decode_shared(stream, append=self.fusable, planned=planned)

    def decode_shared(self, stream=None, append=False, planned=True):
        kw = dict(k_new=self.step_k if append else None, v_new=self.step_v if append else None,
                  workspace=self.workspace, stream=stream)
        if planned and self.shared_plan is not None:
            return pa_decode_shared_planned(self.out, self.q, self.k_cache, self.v_cache,
                                            self.block_tables, self.context_lens, self.share,
                                            self.shared_plan, self.scale, self.num_q_heads,
                                            self.num_kv_heads, self.head_dim, self.block_size, **kw)
        return pa_decode_shared(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                self.context_lens, self.share, self.scale, self.num_q_heads,
                                self.num_kv_heads, self.head_dim, self.block_size, **kw)

    def run(self, stream=None):
        """copy-on-write pairs, then the new tokens' K/V, then decode."""
        if self.pairs.shape[0]:
            pa_copy_blocks(self.k_cache, self.v_cache, self.pairs, stream)
        pa_reshape_and_cache(self.step_k, self.step_v, self.k_cache, self.v_cache, self.slots, stream)
        return self.decode(stream)

    def run_fused(self, stream=None):
        """copy-on-write pairs, then one launch that appends the new tokens and decodes
        (step_k/step_v rows are the decoded sequences' newest tokens, in batch order)."""
        if self.pairs.shape[0]:
            pa_copy_blocks(self.k_cache, self.v_cache, self.pairs, stream)
        return pa_decode_append(self.out, self.q, self.k_cache, self.v_cache, self.step_k, self.step_v,
                                self.block_tables, self.context_lens, self.scale, self.num_q_heads,
                                self.num_kv_heads, self.head_dim, self.block_size, self.partition_size,
                                self.workspace, stream)

    def decode(self, stream=None):
        return pa_decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                         self.context_lens, self.scale, self.num_q_heads, self.num_kv_heads,
                         self.head_dim, self.block_size, self.partition_size, self.workspace,
                         stream)


class PackedInputs:
    """The inputs of a step packed at 256-byte aligned offsets into one pinned host
    buffer and one device buffer, so that they cross the bus in a single copy
    (each separate copy has a fixed cost of its own).  `views` are device tensors
    aliasing the device buffer; `host` tensors alias the host buffer."""

    def __init__(self, tensors, device):
        import torch
        offs, total = {}, 0
        for name, t in tensors.items():
            n = t.numel() * t.element_size()
            offs[name] = (total, n)
            total += (n + 255) // 256 * 256
        total = max(total, 256)
        self.host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.dev_buf = torch.empty(total, dtype=torch.uint8, device=device)
        self.views, self.host = {}, {}
        for name, t in tensors.items():
            o, n = offs[name]
            self.host[name] = self.host_buf[o:o + n].view(t.dtype).view(t.shape)
            self.views[name] = self.dev_buf[o:o + n].view(t.dtype).view(t.shape)
            self.host[name].copy_(t)

    def upload(self, stream=None):
        """One host-to-device copy of every input (on the current stream)."""
        self.dev_buf.copy_(self.host_buf, non_blocking=True)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.host.values())


def _shared_plan(bt, cl, share, w, dtype, dev):
    """Device copy of pa_decode_shared_plan for the step, or None where the two
    launches have no common grid (some fp32 shapes): they then walk from scratch."""
    import torch
    try:
        plan = pa_decode_shared_plan(bt, cl, share, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                     w.block_size, dtype)
    except PagedKVError:
        return None
    return torch.from_numpy(plan).to(dev)


def execute(w, k_cache, v_cache, step_kv: Callable, query: Callable,
            on_step: Optional[Callable] = None, stream=None, width: Optional[int] = None):
    """Run workload `w`'s script on the device caches.

    step_kv(step) -> (k, v) CUDA tensors of the step's new tokens; query(step) ->
    q [S, Hq, d].  After each step, `on_step(step, alloc, decode_step)` (if given) is
    called with a DecodeStep holding that step's inputs; the step's copies and
    writes have been enqueued, its decode has not.  Returns (alloc, last DecodeStep)."""
    import torch
    dev = k_cache.device
    alloc = BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    last = None
    for ev in w.events:
        kind = _kind(ev)
        if kind == "NewSeq":
            alloc.new_seq()
        elif kind == "Fork":
            alloc.fork(ev.parent)
        elif kind == "FreeSeq":
            alloc.free_seq(ev.seq)
        elif kind == "Prefill":
            if ev.n <= 0:
                continue
            _, pairs = alloc.append_n(ev.seq, ev.n)
            if len(pairs):
                pa_copy_blocks(k_cache, v_cache, torch.from_numpy(pairs).to(dev), stream)
        elif kind == "Step":
            slots, pairs = [], []
            for s in ev.seqs:
                slot, cow = alloc.append(s)
                slots.append(slot)
                if cow is not None:
                    pairs.append(cow)
            k, v = step_kv(ev)
            # the fused append pairs row i of the step's K/V with batch sequence i
            fusable = list(ev.seqs) == list(w.decode_seqs)
            bt, cl = tables_for(alloc, w.decode_seqs, width)
            S = len(w.decode_seqs)
            q = query(ev)
            share = share_groups(bt, cl, w.block_size)
            has_share = bool(np.any(share[:, 0] >= 0))
            ws = alloc_workspace(S, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                 bt.shape[1], w.partition_size, dev)
            if has_share and w.num_q_heads // w.num_kv_heads <= 16:
                n = pa_decode_shared_workspace_size(S, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                    w.block_size, bt.shape[1])
                if ws is None or ws.numel() < n:
                    ws = torch.empty(n, dtype=torch.uint8, device=dev)
            else:
                has_share = False
            ds = DecodeStep(
                q=q, k_cache=k_cache, v_cache=v_cache, step_k=k, step_v=v,
                slots=torch.tensor(slots, dtype=torch.int64, device=dev),
                pairs=torch.tensor(np.array(pairs, dtype=np.int32).reshape(-1, 2), device=dev),
                block_tables=torch.from_numpy(bt).to(dev), context_lens=torch.from_numpy(cl).to(dev),
                out=torch.empty_like(q),
                workspace=ws,
                scale=w.softmax_scale, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                head_dim=w.head_dim, block_size=w.block_size, partition_size=w.partition_size,
                fusable=fusable,
                share=torch.from_numpy(share).to(dev) if has_share else None,
                shared_plan=_shared_plan(bt, cl, share, w, k_cache.dtype, dev) if has_share else None,
                plan=torch.from_numpy(pa_decode_plan(bt, cl, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                     w.block_size, k_cache.dtype)).to(dev),
                share_pays=has_share and share_pays(
                    share, cl, w.block_size,
                    2 * w.block_size * w.num_kv_heads * w.head_dim * k_cache.element_size()))
            if ds.pairs.shape[0]:
                pa_copy_blocks(k_cache, v_cache, ds.pairs, stream)
            pa_reshape_and_cache(k, v, k_cache, v_cache, ds.slots, stream)
            if on_step is not None:
                on_step(ev, alloc, ds)
            last = ds
        else:
            raise TypeError(f"unknown event {ev!r}")
    return alloc, last


def replay_usage(w, host_blocks: int = 0):
    """Run `w`'s allocator script on the host only (no device data) and return the
    device-pool accounting (BlockAllocator.usage) after every decode step."""
    alloc = BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    out = []
    for ev in w.events:
        kind = _kind(ev)
        if kind == "NewSeq":
            alloc.new_seq()
        elif kind == "Fork":
            alloc.fork(ev.parent)
        elif kind == "FreeSeq":
            alloc.free_seq(ev.seq)
        elif kind == "Prefill":
            if ev.n > 0:
                alloc.append_n(ev.seq, ev.n)
        elif kind == "Step":
            for q in ev.seqs:
                alloc.append(q)
            out.append(alloc.usage())
        else:
            raise TypeError(f"unknown event {ev!r}")
    return out
