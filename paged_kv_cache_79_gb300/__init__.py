"""GB300-native paged decode attention: Python binding of libpagedkv.so.

Functions carry the names of the C ABI in include/pagedkv.h and only marshal
arguments (torch tensors -> device pointers and sizes, current stream); every step
of the computation runs in the library's CUDA kernels.  There is no CPU path:
calls on tensors that are not CUDA tensors raise.

    pa_decode               paged single-query attention (partition + merge kernels)
    pa_decode_append        the newest tokens' append fused with the decode
    pa_decode_plan /        the balanced split's CTA starts computed on the host, and
      pa_decode_planned       the decode (and append) that starts from them
    pa_decode_shared        decode reading each shared prefix block once per group
    pa_reshape_and_cache    write new tokens' K/V rows through a slot mapping
    pa_copy_blocks          copy-on-write block copies
    pa_swap_blocks          block moves between the device pool and pinned host memory
    pa_gather_blocks /      pack blocks into a contiguous staging buffer and back
      pa_scatter_blocks       (the local halves of a KV transfer)
    BlockAllocator          host ref-counted block allocator (pa_alloc_*)
"""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

from ._lib import load as _load, library_path  # noqa: F401

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_OOM, PA_ERR_TIMEOUT = range(6)
PA_F32, PA_F16, PA_BF16 = 0, 1, 2


class PagedKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _load()
        msg = lib.pa_status_string(status).decode()
        if status == PA_ERR_CUDA:
            msg += f" (cudaError {lib.pa_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")
        self.status = status


class OutOfBlocks(PagedKVError, MemoryError):
    pass


def _check(status: int, where: str) -> None:
    if status == PA_ERR_OOM:
        raise OutOfBlocks(status, where)
    if status != PA_OK:
        raise PagedKVError(status, where)


def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _cuda(t, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _dev_ptr(t, name: str):
    """Pointer of a CUDA tensor or of a pinned host tensor (device-accessible)."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def _torch_stream(stream, device):
    """`stream` (None: torch's current stream; a torch stream; or a raw cudaStream_t)
    as a torch stream object."""
    import torch
    if stream is None:
        return torch.cuda.current_stream(device)
    if hasattr(stream, "cuda_stream"):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


def _launch_scratch(nbytes: int, device, stream):
    """A uint8 workspace for a launch on `stream`, taken from torch's caching
    allocator on that stream.  The tensor is dropped when the call returns, while
    the launch may still be running; allocated on the launch's own stream, its
    block is handed out again only to later work on that stream, which runs after
    the launch."""
    import torch
    with torch.cuda.stream(_torch_stream(stream, device)):
        return torch.empty(nbytes, dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------
def pa_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_blocks_per_seq, partition_size=0) -> int:
    return _load().pa_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                            max_blocks_per_seq, partition_size)


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_blocks_per_seq, partition_size=0) -> int:
    n = _load().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                         max_blocks_per_seq, partition_size)
    if n == ctypes.c_size_t(-1).value:
        raise PagedKVError(PA_ERR_INVALID, "pa_decode_workspace_size")
    return n


def alloc_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                    partition_size=0, device="cuda", stream=None):
    """A caller-owned workspace tensor of the size pa_decode needs (None if 0),
    allocated on `stream` (default: torch's current stream)."""
    n = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_blocks_per_seq, partition_size)
    return _launch_scratch(n, device, stream) if n > 0 else None


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
              num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
              partition_size: int = 0, workspace=None, stream=None):
    """out[S, Hq, d] <- paged decode attention (see pa_decode in include/pagedkv.h).

    q/out [S, Hq, d]; caches [num_blocks, B, Hkv, d]; block_tables int32 [S, W];
    context_lens int32 [S]; workspace: uint8 CUDA tensor or None (allocated here)."""
    import torch
    S = q.shape[0]
    W = block_tables.shape[1]
    if workspace is None:
        workspace = alloc_workspace(S, num_q_heads, num_kv_heads, head_dim, block_size, W,
                                    partition_size, q.device, stream)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    st = _load().pa_decode(_cuda(out, "out"), _cuda(q, "q"), _cuda(k_cache, "k_cache"),
                           _cuda(v_cache, "v_cache"), _cuda(block_tables, "block_tables"), W,
                           _cuda(context_lens, "context_lens"), S, k_cache.shape[0], float(scale),
                           num_q_heads, num_kv_heads, head_dim, block_size, _dtype_code(q),
                           partition_size, ws_ptr, ws_bytes, _stream(stream))
    _check(st, "pa_decode")
    return out


def pa_decode_append(out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                     scale: float, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     block_size: int, partition_size: int = 0, workspace=None, stream=None):
    """Append each sequence's newest token (k_new/v_new [S, Hkv, d], position
    context_lens[s] - 1) to the caches and decode, in one launch; the same result as
    pa_reshape_and_cache followed by pa_decode."""
    import torch
    S = q.shape[0]
    W = block_tables.shape[1]
    if workspace is None:
        workspace = alloc_workspace(S, num_q_heads, num_kv_heads, head_dim, block_size, W,
                                    partition_size, q.device, stream)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    st = _load().pa_decode_append(_cuda(out, "out"), _cuda(q, "q"), _cuda(k_cache, "k_cache"),
                                  _cuda(v_cache, "v_cache"), _cuda(k_new, "k_new"),
                                  _cuda(v_new, "v_new"), _cuda(block_tables, "block_tables"), W,
                                  _cuda(context_lens, "context_lens"), S, k_cache.shape[0],
                                  float(scale), num_q_heads, num_kv_heads, head_dim, block_size,
                                  _dtype_code(q), partition_size, ws_ptr, ws_bytes, _stream(stream))
    _check(st, "pa_decode_append")
    return out


_DTYPE_NAMES = {"f32": PA_F32, "f16": PA_F16, "bf16": PA_BF16}


def _dtype_arg(dtype) -> int:
    """A pa_dtype code from a code, a name ('f32', 'f16', 'bf16') or a torch dtype."""
    if isinstance(dtype, int):
        return dtype
    if isinstance(dtype, str):
        return _DTYPE_NAMES[dtype]
    import torch
    return {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}[dtype]


def pa_decode_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                         dtype) -> int:
    """Size of a pa_decode_plan for these arguments on the current device."""
    n = _load().pa_decode_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                     max_blocks_per_seq, _dtype_arg(dtype))
    if n == ctypes.c_size_t(-1).value:
        raise PagedKVError(PA_ERR_INVALID, "pa_decode_plan_bytes")
    return n


def pa_decode_plan(block_tables, context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   block_size: int, dtype, plan_bytes: Optional[int] = None):
    """Host-side schedule of the balanced-split decode (see pa_decode_plan in
    include/pagedkv.h): int32 numpy array of plan_bytes / 4 entries, from HOST block
    tables [S, W] and context lengths [S] (numpy arrays or CPU tensors).  plan_bytes
    defaults to pa_decode_plan_bytes(...) on the current device."""
    import numpy as np
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    cl = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    S = cl.shape[0]
    W = bt.shape[1] if bt.ndim == 2 else 1
    if plan_bytes is None:
        plan_bytes = pa_decode_plan_bytes(S, num_q_heads, num_kv_heads, head_dim, block_size, W, dtype)
    plan = np.empty(plan_bytes // 4, dtype=np.int32)
    st = _load().pa_decode_plan(plan.ctypes.data, plan_bytes, bt.ctypes.data if S else None, W,
                                cl.ctypes.data if S else None, S, num_q_heads, num_kv_heads, head_dim,
                                block_size, _dtype_arg(dtype))
    _check(st, "pa_decode_plan")
    return plan


def pa_decode_planned(out, q, k_cache, v_cache, block_tables, context_lens, plan, scale: float,
                      num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                      k_new=None, v_new=None, workspace=None, stream=None):
    """pa_decode (balanced split), or with k_new/v_new pa_decode_append, whose CTAs
    start where `plan` (a CUDA int32 copy of pa_decode_plan's output for the same
    lengths and tables) says; bit-identical to the unplanned call."""
    import torch
    S = q.shape[0]
    W = block_tables.shape[1]
    if workspace is None:
        workspace = alloc_workspace(S, num_q_heads, num_kv_heads, head_dim, block_size, W, 0, q.device,
                                    stream)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or plan.dtype != torch.int32:
        raise TypeError("block_tables, context_lens and plan must be int32")
    st = _load().pa_decode_planned(_cuda(out, "out"), _cuda(q, "q"), _cuda(k_cache, "k_cache"),
                                   _cuda(v_cache, "v_cache"),
                                   _cuda(k_new, "k_new") if k_new is not None else None,
                                   _cuda(v_new, "v_new") if v_new is not None else None,
                                   _cuda(block_tables, "block_tables"), W,
                                   _cuda(context_lens, "context_lens"), S, k_cache.shape[0], float(scale),
                                   num_q_heads, num_kv_heads, head_dim, block_size, _dtype_code(q),
                                   _cuda(plan, "plan"), plan.numel() * 4,
                                   _cuda(workspace, "workspace") if workspace is not None else None,
                                   workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(st, "pa_decode_planned")
    return out


def pa_decode_shared_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                    max_blocks_per_seq) -> int:
    n = _load().pa_decode_shared_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                block_size, max_blocks_per_seq)
    if n == ctypes.c_size_t(-1).value:
        raise PagedKVError(PA_ERR_INVALID, "pa_decode_shared_workspace_size")
    return n


def pa_decode_shared(out, q, k_cache, v_cache, block_tables, context_lens, share, scale: float,
                     num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                     k_new=None, v_new=None, workspace=None, stream=None):
    """Decode a batch whose sequence groups share leading blocks, reading each shared
    block once per group; share: int32 [S, 2] = (first member of the group or -1,
    shared leading blocks).  With k_new/v_new, also appends the newest tokens."""
    import torch
    S = q.shape[0]
    W = block_tables.shape[1]
    if workspace is None:
        n = pa_decode_shared_workspace_size(S, num_q_heads, num_kv_heads, head_dim, block_size, W)
        workspace = _launch_scratch(n, q.device, stream)
    if share.dtype != torch.int32 or block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("share, block_tables and context_lens must be int32")
    st = _load().pa_decode_shared(_cuda(out, "out"), _cuda(q, "q"), _cuda(k_cache, "k_cache"),
                                  _cuda(v_cache, "v_cache"),
                                  _cuda(k_new, "k_new") if k_new is not None else None,
                                  _cuda(v_new, "v_new") if v_new is not None else None,
                                  _cuda(block_tables, "block_tables"), W,
                                  _cuda(context_lens, "context_lens"), _cuda(share, "share"), S,
                                  k_cache.shape[0], float(scale), num_q_heads, num_kv_heads, head_dim,
                                  block_size, _dtype_code(q), _cuda(workspace, "workspace"),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_decode_shared")
    return out


def pa_decode_shared_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, dtype) -> int:
    """Size of a pa_decode_shared_plan for these arguments on the current device."""
    n = _load().pa_decode_shared_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                            max_blocks_per_seq, _dtype_arg(dtype))
    if n == ctypes.c_size_t(-1).value:
        raise PagedKVError(PA_ERR_INVALID, "pa_decode_shared_plan_bytes")
    return n


def pa_decode_shared_plan(block_tables, context_lens, share, num_q_heads: int, num_kv_heads: int,
                          head_dim: int, block_size: int, dtype, plan_bytes: Optional[int] = None):
    """Host-side schedule of both launches of the shared-prefix decode (see
    pa_decode_shared_plan in include/pagedkv.h): int32 numpy array, from HOST block
    tables [S, W], context lengths [S] and share entries [S, 2].  plan_bytes defaults
    to pa_decode_shared_plan_bytes(...) on the current device."""
    import numpy as np
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    cl = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    sh = np.ascontiguousarray(np.asarray(share, dtype=np.int32))
    S = cl.shape[0]
    W = bt.shape[1] if bt.ndim == 2 else 1
    if plan_bytes is None:
        plan_bytes = pa_decode_shared_plan_bytes(S, num_q_heads, num_kv_heads, head_dim, block_size, W,
                                                 dtype)
    plan = np.empty(plan_bytes // 4, dtype=np.int32)
    st = _load().pa_decode_shared_plan(plan.ctypes.data, plan_bytes, bt.ctypes.data if S else None, W,
                                       cl.ctypes.data if S else None, sh.ctypes.data if S else None, S,
                                       num_q_heads, num_kv_heads, head_dim, block_size, _dtype_arg(dtype))
    _check(st, "pa_decode_shared_plan")
    return plan


def pa_decode_shared_planned(out, q, k_cache, v_cache, block_tables, context_lens, share, plan,
                             scale: float, num_q_heads: int, num_kv_heads: int, head_dim: int,
                             block_size: int, k_new=None, v_new=None, workspace=None, stream=None):
    """pa_decode_shared whose CTAs, in both launches, start where `plan` (a CUDA int32
    copy of pa_decode_shared_plan's output for the same inputs) says; bit-identical
    to the unplanned call."""
    import torch
    S = q.shape[0]
    W = block_tables.shape[1]
    if workspace is None:
        n = pa_decode_shared_workspace_size(S, num_q_heads, num_kv_heads, head_dim, block_size, W)
        workspace = _launch_scratch(n, q.device, stream)
    if (share.dtype != torch.int32 or block_tables.dtype != torch.int32 or
            context_lens.dtype != torch.int32 or plan.dtype != torch.int32):
        raise TypeError("share, block_tables, context_lens and plan must be int32")
    st = _load().pa_decode_shared_planned(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache"),
        _cuda(k_new, "k_new") if k_new is not None else None,
        _cuda(v_new, "v_new") if v_new is not None else None,
        _cuda(block_tables, "block_tables"), W, _cuda(context_lens, "context_lens"), _cuda(share, "share"),
        S, k_cache.shape[0], float(scale), num_q_heads, num_kv_heads, head_dim, block_size, _dtype_code(q),
        _cuda(plan, "plan"), plan.numel() * 4, _cuda(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_decode_shared_planned")
    return out


def share_groups(block_tables, context_lens, block_size: int, min_shared_blocks: int = 1):
    """share int32 [S, 2] for pa_decode_shared, from host block tables [S, W] and
    context lengths [S] (numpy or CPU tensors); see pa_share_groups."""
    import numpy as np
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    cl = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    S = cl.shape[0]
    share = np.empty((S, 2), dtype=np.int32)
    W = bt.shape[1] if bt.ndim == 2 else 0
    st = _load().pa_share_groups(bt.ctypes.data if S else None, S, W, cl.ctypes.data if S else None,
                                 block_size, min_shared_blocks, share.ctypes.data if S else None)
    _check(st, "pa_share_groups")
    return share


def share_saving(share, context_lens, block_size: int) -> float:
    """Fraction of the batch's block reads that pa_decode_shared saves over pa_decode:
    each group of m members sharing P blocks reads (m - 1) * P blocks fewer (when
    one item holds all m members' query rows)."""
    import numpy as np
    share = np.asarray(share)
    cl = np.asarray(context_lens).astype(np.int64)
    logical = int(((cl + block_size - 1) // block_size).sum())
    saved = 0
    for s in range(share.shape[0]):
        if share[s, 0] >= 0 and share[s, 0] != s:      # every member but the first
            saved += int(share[s, 1])
    return saved / logical if logical else 0.0


# pa_decode_shared pays for its second launch and its merges (a fixed ~10-15 us)
# once the groups save 10% of the block reads, or 256 MB of them (~37 us at
# 7 TB/s) on a large batch: the long multi-turn batch saves 2.7%, 580 MB, and
# decodes ~1% faster shared.
SHARE_MIN_SAVING = 0.10
SHARE_MIN_BYTES = 256 << 20


def share_pays(share, context_lens, block_size: int, block_bytes: int) -> bool:
    """Whether pa_decode_shared is expected to beat pa_decode on this batch.
    block_bytes: bytes of one block of K and V over all kv heads."""
    import numpy as np
    f = share_saving(share, context_lens, block_size)
    cl = np.asarray(context_lens).astype(np.int64)
    logical = int(((cl + block_size - 1) // block_size).sum()) * int(block_bytes)
    return f >= SHARE_MIN_SAVING or f * logical >= SHARE_MIN_BYTES


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                      num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                      partition_size: int = 0, stream=None):
    """pa_decode for callers that cannot allocate device memory: the split-KV
    scratch is the library's fixed device array (PA_DECODE_NOALLOC_SCRATCH_BYTES,
    shared by every call; calls overlapping on the GPU race).  Sizes needing more
    scratch raise PagedKVError (PA_ERR_UNSUPPORTED)."""
    import torch
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    st = _load().pa_decode_noalloc(_cuda(out, "out"), _cuda(q, "q"), _cuda(k_cache, "k_cache"),
                                   _cuda(v_cache, "v_cache"), _cuda(block_tables, "block_tables"),
                                   block_tables.shape[1], _cuda(context_lens, "context_lens"),
                                   q.shape[0], k_cache.shape[0], float(scale), num_q_heads,
                                   num_kv_heads, head_dim, block_size, _dtype_code(q), partition_size,
                                   _stream(stream))
    _check(st, "pa_decode_noalloc")
    return out


# ----------------------------------------------------------------------------
# cache writes
# ----------------------------------------------------------------------------
def pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """k_cache[slot // B][slot % B] = k[t] (and v) for every token t with slot >= 0."""
    import torch
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    n = slot_mapping.shape[0]
    if n == 0:
        return
    nb, B, hkv, d = k_cache.shape
    st = _load().pa_reshape_and_cache(_cuda(k, "k"), _cuda(v, "v"), _cuda(k_cache, "k_cache"),
                                      _cuda(v_cache, "v_cache"), _cuda(slot_mapping, "slot_mapping"),
                                      n, hkv, d, B, nb, _dtype_code(k_cache), _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_copy_blocks(k_cache, v_cache, src_dst_pairs, stream=None):
    """k_cache[dst] = k_cache[src] (and v) for every (src, dst) row of the int32 [n, 2] pairs."""
    import torch
    if src_dst_pairs.dtype != torch.int32:
        raise TypeError("src_dst_pairs must be int32")
    n = src_dst_pairs.shape[0]
    if n == 0:
        return
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    st = _load().pa_copy_blocks(_cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache"),
                                _cuda(src_dst_pairs, "src_dst_pairs"), n, k_cache.shape[0],
                                block_bytes, _stream(stream))
    _check(st, "pa_copy_blocks")


def pa_device_errors(stream=None) -> int:
    """The device-side error flags (PA_DEVERR_*) raised since the last read, after
    `stream` drains; reading clears them.  Set flags are returned, not raised (the
    C call's PA_ERR_TIMEOUT / PA_ERR_INVALID status); a CUDA failure raises."""
    flags = ctypes.c_uint(0)
    st = _load().pa_device_errors(ctypes.byref(flags), _stream(stream))
    if st not in (PA_ERR_TIMEOUT, PA_ERR_INVALID) or flags.value == 0:
        _check(st, "pa_device_errors")
    return flags.value


PA_DEVERR_TIMEOUT_FULL, PA_DEVERR_TIMEOUT_EMPTY, PA_DEVERR_SHARE, PA_DEVERR_PLAN = 1, 2, 4, 8
PLAN_BYTES_PER_CTA = 128
PA_WAIT_LIMIT_DEFAULT_NS = 2_000_000_000


def pa_set_wait_limit_ns(ns: int) -> int:
    """Limit (ns) of the device-side waits of decode launches enqueued from now on
    (0: the default, 2 s); returns the previous limit."""
    return int(_load().pa_set_wait_limit_ns(int(ns)))


def pa_status_string(status: int) -> str:
    return _load().pa_status_string(status).decode()


# ----------------------------------------------------------------------------
# host allocator
# ----------------------------------------------------------------------------
class BlockAllocator:
    """Ref-counted block allocator (pa_alloc_* of include/pagedkv.h); host only."""

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        import numpy as np
        self._lib = _load()
        self._h = ctypes.c_void_p()
        self.num_blocks = num_blocks
        self.block_size = block_size
        ptr = None
        if free_order is not None:
            self._order = np.ascontiguousarray(free_order, dtype=np.int32)
            if self._order.shape != (num_blocks,):
                raise ValueError("free_order must have num_blocks entries")
            ptr = self._order.ctypes.data
        _check(self._lib.pa_alloc_create(ctypes.byref(self._h), num_blocks, block_size, ptr),
               "pa_alloc_create")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pa_alloc_destroy(h)
            self._h = None

    def new_seq(self) -> int:
        sid = ctypes.c_int()
        _check(self._lib.pa_alloc_new_seq(self._h, ctypes.byref(sid)), "pa_alloc_new_seq")
        return sid.value

    def fork(self, parent: int) -> int:
        sid = ctypes.c_int()
        _check(self._lib.pa_alloc_fork(self._h, parent, ctypes.byref(sid)), "pa_alloc_fork")
        return sid.value

    def append(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        slot = ctypes.c_int64()
        src = ctypes.c_int32()
        dst = ctypes.c_int32()
        _check(self._lib.pa_alloc_append(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                         ctypes.byref(dst)), "pa_alloc_append")
        return slot.value, ((src.value, dst.value) if src.value >= 0 else None)

    def append_n(self, seq: int, n: int):
        """n appends: (slots int64 [n], cow pairs int32 [k, 2])."""
        import numpy as np
        slots = np.empty(max(n, 1), dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int32)
        k = ctypes.c_int()
        _check(self._lib.pa_alloc_append_n(self._h, seq, n, slots.ctypes.data, pairs.ctypes.data,
                                           ctypes.byref(k), None), "pa_alloc_append_n")
        return slots[:n], pairs[:k.value]

    def free_seq(self, seq: int) -> None:
        _check(self._lib.pa_alloc_free_seq(self._h, seq), "pa_alloc_free_seq")

    def block_table(self, seq: int) -> List[int]:
        import numpy as np
        n = ctypes.c_int()
        _check(self._lib.pa_alloc_block_table(self._h, seq, None, 0, ctypes.byref(n)), "pa_alloc_block_table")
        out = np.empty(max(n.value, 1), dtype=np.int32)
        _check(self._lib.pa_alloc_block_table(self._h, seq, out.ctypes.data, n.value, ctypes.byref(n)),
               "pa_alloc_block_table")
        return out[:n.value].tolist()

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int()
        _check(self._lib.pa_alloc_seq_len(self._h, seq, ctypes.byref(n)), "pa_alloc_seq_len")
        return n.value

    def refcount(self, block: int) -> int:
        return self._lib.pa_alloc_refcount(self._h, block)

    def num_free(self) -> int:
        return self._lib.pa_alloc_num_free(self._h)

    def free_list(self) -> List[int]:
        import numpy as np
        n = ctypes.c_int()
        _check(self._lib.pa_alloc_free_list(self._h, None, 0, ctypes.byref(n)), "pa_alloc_free_list")
        out = np.empty(max(n.value, 1), dtype=np.int32)
        _check(self._lib.pa_alloc_free_list(self._h, out.ctypes.data, n.value, ctypes.byref(n)),
               "pa_alloc_free_list")
        return out[:n.value].tolist()

    def usage(self) -> dict:
        """Device-pool accounting (pa_alloc_usage_stats) plus the derived waste and
        sharing-saving fractions."""
        class _Usage(ctypes.Structure):
            _fields_ = [(n, ctypes.c_int64) for n in ("used_blocks", "logical_blocks", "token_slots",
                                                       "tokens", "resident_seqs", "swapped_seqs")]
        u = _Usage()
        _check(self._lib.pa_alloc_usage_stats(self._h, ctypes.byref(u)), "pa_alloc_usage_stats")
        d = {n: getattr(u, n) for n, _ in _Usage._fields_}
        d["waste"] = 1.0 - d["tokens"] / d["token_slots"] if d["token_slots"] else 0.0
        d["sharing_saving"] = 1.0 - d["used_blocks"] / d["logical_blocks"] if d["logical_blocks"] else 0.0
        return d

    # swap space in host memory -------------------------------------------------
    def set_host_pool(self, num_host_blocks: int) -> None:
        _check(self._lib.pa_alloc_set_host_pool(self._h, num_host_blocks), "pa_alloc_set_host_pool")
        self.num_host_blocks = num_host_blocks

    def _move(self, fn, name, seqs):
        import numpy as np
        ids = np.ascontiguousarray(list(seqs), dtype=np.int32).reshape(-1)
        n = ctypes.c_int()
        cap = max(1, sum(len(self.block_table(q)) for q in ids.tolist())) if ids.size else 1
        pairs = np.empty((cap, 2), dtype=np.int32)
        _check(fn(self._h, ids.ctypes.data if ids.size else None, int(ids.size), pairs.ctypes.data, cap,
                  ctypes.byref(n)), name)
        return pairs[:n.value]

    def swap_out(self, seqs) -> "object":
        """Move `seqs` to the host pool: int32 [k, 2] (device block, host block) pairs."""
        return self._move(self._lib.pa_alloc_swap_out, "pa_alloc_swap_out", seqs)

    def swap_in(self, seqs) -> "object":
        """Move `seqs` back to the device pool: int32 [k, 2] (host block, device block) pairs."""
        return self._move(self._lib.pa_alloc_swap_in, "pa_alloc_swap_in", seqs)

    def is_swapped(self, seq: int) -> bool:
        v = self._lib.pa_alloc_is_swapped(self._h, seq)
        if v < 0:
            raise PagedKVError(PA_ERR_INVALID, "pa_alloc_is_swapped")
        return bool(v)

    def host_refcount(self, block: int) -> int:
        return self._lib.pa_alloc_host_refcount(self._h, block)

    def num_free_host(self) -> int:
        return self._lib.pa_alloc_num_free_host(self._h)

    def host_free_list(self) -> List[int]:
        import numpy as np
        n = ctypes.c_int()
        _check(self._lib.pa_alloc_host_free_list(self._h, None, 0, ctypes.byref(n)), "pa_alloc_host_free_list")
        out = np.empty(max(n.value, 1), dtype=np.int32)
        _check(self._lib.pa_alloc_host_free_list(self._h, out.ctypes.data, n.value, ctypes.byref(n)),
               "pa_alloc_host_free_list")
        return out[:n.value].tolist()


def _block_bytes(cache) -> int:
    return cache[0].numel() * cache.element_size()


def pa_swap_blocks(src_k, src_v, dst_k, dst_v, src_dst_pairs, stream=None):
    """dst pool blocks <- src pool blocks for each (src, dst) pair; pools are [NB, ...]
    tensors on the device or in pinned host memory (pairs likewise)."""
    if src_dst_pairs.shape[0] == 0:
        return
    st = _load().pa_swap_blocks(_dev_ptr(src_k, "src_k"), _dev_ptr(src_v, "src_v"), _dev_ptr(dst_k, "dst_k"),
                                _dev_ptr(dst_v, "dst_v"), _dev_ptr(src_dst_pairs, "src_dst_pairs"),
                                int(src_dst_pairs.shape[0]), int(src_k.shape[0]), int(dst_k.shape[0]),
                                _block_bytes(src_k), _stream(stream))
    _check(st, "pa_swap_blocks")


def pa_gather_blocks(k_cache, v_cache, block_ids, staging_k, staging_v, stream=None):
    """staging[i] <- cache[block_ids[i]] (staging: [n, ...] device or pinned host tensors)."""
    if block_ids.shape[0] == 0:
        return
    st = _load().pa_gather_blocks(_dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
                                  _dev_ptr(block_ids, "block_ids"), int(block_ids.shape[0]),
                                  int(k_cache.shape[0]), _dev_ptr(staging_k, "staging_k"),
                                  _dev_ptr(staging_v, "staging_v"), _block_bytes(k_cache), _stream(stream))
    _check(st, "pa_gather_blocks")


def pa_scatter_blocks(staging_k, staging_v, k_cache, v_cache, block_ids, stream=None):
    """cache[block_ids[i]] <- staging[i]."""
    if block_ids.shape[0] == 0:
        return
    st = _load().pa_scatter_blocks(_dev_ptr(staging_k, "staging_k"), _dev_ptr(staging_v, "staging_v"),
                                   _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
                                   _dev_ptr(block_ids, "block_ids"), int(block_ids.shape[0]),
                                   int(k_cache.shape[0]), _block_bytes(k_cache), _stream(stream))
    _check(st, "pa_scatter_blocks")


def pa_kv_transfer_worthwhile(reusable_tokens: int, threshold_tokens: int = 64) -> bool:
    """Fetch another engine's KV for a prefix (True) or recompute it (False)."""
    return bool(_load().pa_kv_transfer_worthwhile(int(reusable_tokens), int(threshold_tokens)))


__all__ = ["pa_decode", "pa_decode_append", "pa_decode_plan_bytes", "pa_decode_plan", "pa_decode_planned",
           "pa_decode_shared_plan_bytes", "pa_decode_shared_plan", "pa_decode_shared_planned",
           "PA_DEVERR_PLAN", "PLAN_BYTES_PER_CTA",
           "pa_decode_shared", "pa_decode_shared_workspace_size",
           "share_groups", "share_saving", "share_pays", "SHARE_MIN_SAVING", "SHARE_MIN_BYTES",
           "pa_decode_noalloc", "pa_decode_workspace_size", "pa_decode_partition_size", "alloc_workspace",
           "pa_reshape_and_cache", "pa_copy_blocks", "pa_swap_blocks", "pa_gather_blocks",
           "pa_scatter_blocks", "pa_kv_transfer_worthwhile", "pa_device_errors", "pa_set_wait_limit_ns",
           "PA_DEVERR_TIMEOUT_FULL", "PA_DEVERR_TIMEOUT_EMPTY", "PA_DEVERR_SHARE", "PA_WAIT_LIMIT_DEFAULT_NS", "pa_status_string",
           "BlockAllocator", "PagedKVError", "OutOfBlocks", "library_path"]
