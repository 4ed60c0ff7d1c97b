"""The multi-process (N > 1) bookkeeping of bench.py on CPU: gloo, world size 2.

Each rank decodes its own batch, so the only cross-rank step is the time: the job
takes as long as its slowest rank, and the whole-job value adds every rank's
bytes.  The reference arm runs on rank 0 alone."""
import argparse
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 3.0], "cpu")
    ref = bench.run_reference(argparse.Namespace(workload="tiny", steps=1, warmup=3, cpu_budget=1.0,
                                                 gpus=world))
    q.put((rank, got, ref is None))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_rank0_reference_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, got, ref_none in res:
        assert got == [2.0, 5.0, 3.0]
        assert ref_none == (rank != 0)     # only rank 0 runs (and prints) the reference arm


def test_job_value_adds_the_ranks_bytes():
    import bench
    assert bench.job_gbs(1e9, 1.0, 1) == pytest.approx(1000.0)
    assert bench.job_gbs(1e9, 2.0, 4) == pytest.approx(2000.0)
    assert bench.max_over_ranks([3.0, 1.0]) == [3.0, 1.0]      # outside torch.distributed


def test_cpu_baseline_one_core_restores_the_thread_count():
    """The one-core oracle timing runs on one thread and leaves the oracle's thread
    count as it found it."""
    import types
    import torch
    import bench
    import oracle
    import workloads as W
    w = W.by_name("tiny")
    oalloc, _ = oracle.run_script(w.events, w.num_blocks, w.block_size, w.free_order)
    bt, cl = oracle.tables_for(oalloc, w.decode_seqs)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    ds = types.SimpleNamespace(k_cache=W.randn(shape, w.dtype, 1), v_cache=W.randn(shape, w.dtype, 2),
                               q=W.query_tensor(w, 0))
    before = oracle.num_threads()
    reps, el, cores = bench.cpu_baseline(w, ds, bt, cl, budget_s=0.05, threads=1)
    assert cores == 1 and reps >= 1 and el > 0
    assert oracle.num_threads() == before
    reps, el, cores = bench.cpu_baseline(w, ds, bt, cl, budget_s=0.05)
    assert cores == before


def test_traffic_counters_follow_code_not_comments(tmp_path, monkeypatch):
    """The committed DRAM counters are reported while the decode sources' code is the
    one they were taken on: comment edits keep them, code edits drop them."""
    import bench
    assert bench.strip_comments("int a; // x\n/* y\n z */ int  b;") == "int a; int b;"
    src = tmp_path / "paged_kv_cache_79_gb300" / "csrc"
    src.mkdir(parents=True)
    for n in bench.DECODE_SOURCES:
        (src / n).write_text("int f() { return 1; } // v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.decode_source_hash()
    (src / bench.DECODE_SOURCES[0]).write_text("/* new comment */ int f() {  return 1; }\n")
    assert bench.decode_source_hash() == h
    (src / bench.DECODE_SOURCES[0]).write_text("int f() { return 2; }\n")
    assert bench.decode_source_hash() != h
