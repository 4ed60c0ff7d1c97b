"""Decodes launched on a stream other than torch's current one.

When the binding allocates the workspace itself (workspace=None), the tensor is
dropped as the call returns, while the launch is still running on the caller's
stream.  It is allocated on that stream, so torch's caching allocator hands the
block only to later work on the same stream.  Here the current stream allocates
and overwrites memory right after each call; the side-stream decodes must still
equal the reference bit for bit."""
import math

import pytest
import torch

import paged_kv_cache_79_gb300 as P
from tests.gpu_harness import small_case

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("part", [0, 256])
def test_side_stream_decode_with_its_own_workspace(part):
    dtype, D, B, hq, hkv = "bf16", 128, 16, 32, 4
    lens = [30000, 20000, 7000, 513]
    q, kc, vc, bt, cl = [t.to(DEV) for t in small_case(81, dtype, D, B, hq, hkv, lens)]
    scale = 1.0 / math.sqrt(D)
    ref = torch.empty_like(q)
    P.pa_decode(ref, q, kc, vc, bt, cl, scale, hq, hkv, D, B, partition_size=part)
    torch.cuda.synchronize()
    nbytes = P.pa_decode_workspace_size(len(lens), hq, hkv, D, B, bt.shape[1], part)
    side = torch.cuda.Stream()
    for trial in range(4):
        out = torch.full_like(q, float("nan"))
        side.wait_stream(torch.cuda.current_stream())
        P.pa_decode(out, q, kc, vc, bt, cl, scale, hq, hkv, D, B, partition_size=part, stream=side)
        # the current stream takes and scribbles over blocks of the workspace's size
        junk = [torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV) for _ in range(4)]
        del junk
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"trial {trial}"
    assert P.pa_device_errors() == 0


def test_shared_decode_on_a_side_stream():
    """pa_decode_shared on a side stream with its workspace allocated by the binding."""
    dtype, D, B, hq, hkv = "f16", 128, 16, 8, 8
    shared_blocks, members = 32, 5
    lens = [shared_blocks * B + 100 * (i + 1) for i in range(members)]
    q, kc, vc, bt, cl = [t.to(DEV) for t in small_case(82, dtype, D, B, hq, hkv, lens, stale=0.0)]
    bt[:, :shared_blocks] = bt[0, :shared_blocks]
    share = torch.tensor([[0, shared_blocks]] * members, dtype=torch.int32, device=DEV)
    ref = torch.empty_like(q)
    P.pa_decode_shared(ref, q, kc, vc, bt, cl, share, 0.1, hq, hkv, D, B)
    torch.cuda.synchronize()
    n = P.pa_decode_shared_workspace_size(members, hq, hkv, D, B, bt.shape[1])
    side = torch.cuda.Stream()
    for trial in range(3):
        out = torch.full_like(q, float("nan"))
        side.wait_stream(torch.cuda.current_stream())
        P.pa_decode_shared(out, q, kc, vc, bt, cl, share, 0.1, hq, hkv, D, B, stream=side)
        junk = [torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV) for _ in range(4)]
        del junk
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"trial {trial}"
    assert P.pa_device_errors() == 0
