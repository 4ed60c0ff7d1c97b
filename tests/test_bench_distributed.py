"""The multi-process (N > 1) bookkeeping of bench.py on CPU: gloo, world size 2.

Each rank decodes its own batch, so the only cross-rank step is the time: the job
takes as long as its slowest rank, and the whole-job value adds every rank's
bytes.  The reference arm runs on rank 0 alone."""
import argparse
import json
import os
import socket
import subprocess
import sys

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
    reps, el, cores, nbytes, note = bench.cpu_baseline(w, ds, bt, cl, budget_s=0.05, threads=1)
    assert cores == 1 and reps >= 1 and el > 0
    assert nbytes == bench.step_bytes(w, bt, cl, 0, 0)["decode"] and "one sequence" in note
    assert oracle.num_threads() == before
    reps, el, cores, nbytes, note = bench.cpu_baseline(w, ds, bt, cl, budget_s=0.05)
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


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` outside torchrun starts the two ranks itself (here the
    reference arm, which needs no GPU): rank 0 prints the one line, whose n_gpus is
    the number of ranks that ran."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["impl"] == "reference"
    assert d["config"]["parallelism"].startswith("replica x2")
    assert d["cpu_baseline"]["cores"] == (os.cpu_count() or 1)


def test_gpus_flag_must_match_the_ranks_started(monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "0")
    with pytest.raises(SystemExit):
        bench.run_reference(argparse.Namespace(workload="tiny", steps=1, warmup=3, cpu_budget=1.0, gpus=3))


def test_oracle_legs_sample_the_long_workload():
    """The oracle legs decode every sequence of the workloads that fit, and a seeded
    sample of at least 32 sequences, the longest among them, of the long multi-turn
    batch; both arms' configs are the same dict."""
    import numpy as np
    import bench
    import oracle
    import workloads as W
    for name, full in (("mha_fp16", True), ("long_multiturn_bf16", False)):
        w = W.by_name(name)
        oalloc, _ = oracle.run_script(w.events, w.num_blocks, w.block_size, w.free_order)
        bt, cl = oracle.tables_for(oalloc, w.decode_seqs)
        seqs = bench.oracle_subset(w, bt, cl)
        if full:
            assert seqs == list(range(len(cl)))
        else:
            assert len(seqs) >= 32 and int(np.argmax(cl)) in seqs and seqs == sorted(set(seqs))
            assert seqs == bench.oracle_subset(w, bt, cl)          # seeded: the same every run
            used, sbt, scl = bench.subset_tables(w, bt, cl, seqs)
            assert sbt.max() == len(used) - 1 and np.array_equal(scl, cl[seqs])
            for i, s in enumerate(seqs):
                n = (int(cl[s]) + w.block_size - 1) // w.block_size
                assert [used[b] for b in sbt[i, :n]] == bt[s, :n].tolist()
        assert bench.workload_config(w, cl, 1) == bench.workload_config(w, cl.copy(), 1)
