"""The decode entry points captured in a CUDA graph and replayed.

A serving loop captures its decode step once and replays it with new inputs in the
same buffers.  Every replay reuses the captured launch parameters, so anything the
kernels keep between launches (the balanced split's merge counters) must tell one
launch from the next on the device.  Each replay must give exactly what a direct
call gives on the same inputs."""
import math

import pytest
import torch

import paged_kv_cache_79_gb300 as P
from tests.gpu_harness import small_case

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(dtype, Hq, Hkv, lens, seed=5):
    D, B = 128, 16
    q, kc, vc, bt, cl = small_case(seed, dtype, D, B, Hq, Hkv, lens, stale=0.0)
    return [t.to(DEV) for t in (q, kc, vc, bt, cl)] + [D, B]


@pytest.mark.parametrize("dtype,Hq,Hkv,lens", [
    ("bf16", 64, 8, [3000, 17, 4096, 2222, 1, 700, 5000, 90]),   # many units cut between CTAs
    ("f16", 40, 40, [2048, 1500, 900, 64, 1, 1999]),
    ("f32", 8, 8, [50, 700]),
])
def test_decode_graph_replays_match_direct_calls(dtype, Hq, Hkv, lens):
    q, kc, vc, bt, cl, D, B = _case(dtype, Hq, Hkv, lens)
    W = bt.shape[1]
    scale = 1.0 / math.sqrt(D)
    ws = P.alloc_workspace(len(lens), Hq, Hkv, D, B, W, 0, DEV)
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        P.pa_decode(out, q, kc, vc, bt, cl, scale, Hq, Hkv, D, B, workspace=ws)   # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        P.pa_decode(out, q, kc, vc, bt, cl, scale, Hq, Hkv, D, B, workspace=ws)
    gen = torch.Generator(device=DEV).manual_seed(11)
    for _ in range(4):
        q.copy_(torch.randn(q.shape, device=DEV, generator=gen).to(q.dtype))
        g.replay()
        torch.cuda.synchronize()
        want = torch.empty_like(q)
        P.pa_decode(want, q, kc, vc, bt, cl, scale, Hq, Hkv, D, B)   # own workspace
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    assert P.pa_device_errors() == 0


def test_shared_decode_graph_replays_match_direct_calls():
    # two launches per step (shared prefixes, then own blocks); the second waits for
    # the first only where it reads its rows
    Hq = Hkv = 8
    D, B = 128, 16
    P_blocks, members = 20, 4
    lens = [P_blocks * B + 1 + 37 * i for i in range(members)] + [900, 33]
    q, kc, vc, bt, cl, D, B = _case("f16", Hq, Hkv, lens, seed=9)
    btc = bt.cpu()
    for i in range(1, members):                  # members share the first member's blocks
        btc[i, :P_blocks] = btc[0, :P_blocks]
    bt = btc.to(DEV)
    share = torch.tensor([[0, P_blocks]] * members + [[-1, 0], [-1, 0]], dtype=torch.int32,
                         device=DEV)
    W = bt.shape[1]
    scale = 1.0 / math.sqrt(D)
    nbytes = P.pa_decode_shared_workspace_size(len(lens), Hq, Hkv, D, B, W)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        P.pa_decode_shared(out, q, kc, vc, bt, cl, share, scale, Hq, Hkv, D, B, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        P.pa_decode_shared(out, q, kc, vc, bt, cl, share, scale, Hq, Hkv, D, B, workspace=ws)
    gen = torch.Generator(device=DEV).manual_seed(12)
    for _ in range(4):
        q.copy_(torch.randn(q.shape, device=DEV, generator=gen).to(q.dtype))
        g.replay()
        torch.cuda.synchronize()
        want = torch.empty_like(q)
        ws2 = torch.empty_like(ws)
        P.pa_decode_shared(want, q, kc, vc, bt, cl, share, scale, Hq, Hkv, D, B, workspace=ws2)
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    assert P.pa_device_errors() == 0
