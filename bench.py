#!/usr/bin/env python3
"""Paged decode attention benchmark: one JSON line on rank 0.

A step is one decode iteration of the whole hot path over one batch: the
copy-on-write block copies (pa_copy_blocks, when the step has any), then the new
tokens' K/V append fused with the decode attention (pa_decode_append: append +
partition kernel with the split-KV merge inside), on inputs already resident in
HBM.  The workload's allocator script (untimed) prepares the caches and tables.
The split is the balanced one (partition_size 0) unless --partition-size says
otherwise.  The default workload is the long-context multi-turn batch (256
sequences, 32 q / 8 kv heads, bf16, block size 32, contexts log-uniform in
[128, 131072], 20.6 GB of unique K/V per step): the largest configuration that
fits one GPU.  The step time reported is the median of the timed steps (the mean
is reported beside it).

Metric: KV GB/s (algorithmic bytes of the step / device time of the step); the
line also carries seq*layers/s (one pa_decode call = one layer), the roofline of
the decode kernel against the measured HBM copy bandwidth, the fp64 CPU oracle's
throughput on the host cores, and an end-to-end figure through the public API with
host buffers (pinned host -> device inputs, device -> host output inside the timed
region).  Before every timed step the L2 (129 MB) is flushed: a 512 MB buffer is
written, then a 1 GB buffer is read, so the flush's own dirty lines are written
back before the timed region instead of during it, and the step starts from a
cold, clean L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...     (the fp64 CPU oracle on the host cores)

With --gpus N > 1 outside torchrun, the script starts N ranks itself (one per GPU,
torch.distributed.run on 127.0.0.1) and rank 0 prints the line; every rank decodes
its own batch (replicas, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "long_multiturn_bf16"
METRIC = "paged decode attention KV GB/s and % of GB300 HBM peak; seq-layers/s at 1 GPU"
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ["pa_decode.cuh", "pa_device.cuh", "pa_api.cu", "pa_internal.h"]


# ----------------------------------------------------------------------------
# bytes accounting (algorithmic: each byte the step must move, counted once)
# ----------------------------------------------------------------------------
def step_bytes(w, bt, cl, n_tok, n_pairs):
    import numpy as np
    es = w.elem_bytes
    row = w.num_kv_heads * w.head_dim * es          # one token's K (or V) row
    B = w.block_size
    S = len(cl)
    logical = int(np.sum(cl)) * row * 2
    # unique: each referenced physical block once, with its largest valid row count
    rows_of = {}
    for s in range(S):
        T = int(cl[s])
        nb = (T + B - 1) // B
        for j in range(nb):
            b = int(bt[s, j])
            r = min(B, T - j * B)
            if rows_of.get(b, 0) < r:
                rows_of[b] = r
    unique = sum(rows_of.values()) * row * 2
    nb_total = int(sum((int(t) + B - 1) // B for t in cl))
    io = 2 * S * w.num_q_heads * w.head_dim * es + 4 * nb_total + 4 * S
    decode = unique + io
    append = n_tok * row * 2 * 2 + 8 * n_tok
    block_bytes = B * row
    cow = n_pairs * block_bytes * 2 * 2 + 8 * n_pairs
    return dict(decode=decode, decode_logical=logical + io, kv_unique=unique, kv_logical=logical,
                append=append, cow=cow, step=decode + append + cow)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank space (string literals in these
    sources hold no comment markers)."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def decode_source_hash():
    """Hash of the decode sources' code (comments and spacing excluded): the traffic
    counters stay valid while only comments change."""
    h = hashlib.sha256()
    for n in DECODE_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_79_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload, launches=1):
    """DRAM bytes of one step's decode launches from the committed ncu summary, if
    it was taken on the current decode sources and on the same path (its number
    of decode launches per step: 2 for the shared-prefix decode); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_hash") == decode_source_hash() and e.get("launches_per_step", 1) == launches:
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def raw(t):
    """Storage bits as numpy (float32 for fp32, uint16 for fp16/bf16)."""
    import numpy as np
    import torch
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def workload_kw(args):
    """--workload-kw key=value pairs (integers): parameters of the workload's
    generator, for a smaller case of the same workload (profiling)."""
    kw = {}
    for item in getattr(args, "workload_kw", None) or []:
        k, v = item.split("=", 1)
        kw[k] = int(v)
    return kw


def prepare(name, device, seed_offset=0, partition_size=None, kw=None):
    import workloads as W
    from paged_kv_cache_79_gb300 import runner
    w = W.by_name(name, **(kw or {}))
    if partition_size is not None:
        w.partition_size = partition_size
    if seed_offset:
        w.data_seed += 97 * seed_offset
    kc, vc = W.pool_tensors(w, device)
    alloc, ds = runner.execute(w, kc, vc, lambda ev: W.step_tensors(w, ev, device),
                               lambda ev: W.query_tensor(w, ev.index, device))
    bt, cl = runner.tables_for(alloc, w.decode_seqs)
    return w, ds, bt, cl


# the workloads whose oracle is also timed on one host core (tiny, MHA, GQA)
ONE_CORE_WORKLOADS = ("tiny", "mha_fp16", "gqa_bf16")

# The oracle legs (cpu_baseline and the reference arm) decode every sequence of a
# workload whose unique K/V fits in ORACLE_FULL_BYTES; a larger one (the long
# multi-turn batch: 20.6 GB) is sampled: ORACLE_SAMPLE_SEQS seeded sequences plus
# the longest, with only the blocks they reference gathered to the host.
ORACLE_FULL_BYTES = 2 << 30
ORACLE_SAMPLE_SEQS = 32

L2_NOTE = ("GPU arm: the 129 MB L2 is flushed before every timed step (512 MB written, "
           "then 1 GB read)")


def workload_config(w, cl, world=1):
    """The JSON line's config: the workload and the job layout, the same in both arms."""
    import numpy as np
    return {"workload": w.name, "num_seqs": len(cl), "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
            "num_blocks": w.num_blocks, "context_tokens": int(np.sum(cl)),
            "max_context": int(np.max(cl)), "l2": L2_NOTE,
            "parallelism": f"replica x{world} (independent batches, one per GPU)"}


def oracle_subset(w, bt, cl):
    """Indices of the sequences the oracle legs decode: all of them, or (workloads
    whose unique K/V exceeds ORACLE_FULL_BYTES) a seeded sample of
    ORACLE_SAMPLE_SEQS plus the longest."""
    import numpy as np
    S = len(cl)
    if step_bytes(w, bt, cl, 0, 0)["kv_unique"] <= ORACLE_FULL_BYTES or S <= ORACLE_SAMPLE_SEQS:
        return list(range(S))
    rng = np.random.default_rng(w.data_seed)
    pick = set(rng.choice(S, size=ORACLE_SAMPLE_SEQS, replace=False).tolist())
    pick.add(int(np.argmax(cl)))
    return sorted(pick)


def subset_tables(w, bt, cl, seqs):
    """(blocks the sequences reference, sorted; their tables renumbered into that
    list; their context lengths)."""
    import numpy as np
    B = w.block_size
    bt = np.asarray(bt)[seqs]
    cl = np.asarray(cl)[seqs].astype(np.int32)
    nbs = [(int(t) + B - 1) // B for t in cl]
    used = sorted({int(bt[i, j]) for i in range(len(seqs)) for j in range(nbs[i])})
    remap = {b: i for i, b in enumerate(used)}
    sbt = np.full(bt.shape, -1, dtype=np.int32)
    for i in range(len(seqs)):
        sbt[i, :nbs[i]] = [remap[int(b)] for b in bt[i, :nbs[i]]]
    return used, sbt, cl


def cpu_baseline(w, ds, bt, cl, budget_s=10.0, threads=None):
    """Time the fp64 oracle (as it stands) on the host cores on a bounded sample:
    decodes of the oracle subset's sequences (every sequence unless the workload is
    too large, see oracle_subset) over their blocks, repeated until ~budget_s.
    threads: the oracle's thread count for this timing (None: all host cores).
    Returns (repetitions, seconds, threads used, bytes per repetition, sample note)."""
    import numpy as np
    import torch
    import oracle
    seqs = oracle_subset(w, bt, cl)
    used, sbt, scl = subset_tables(w, bt, cl, seqs)
    idx = torch.tensor(used, dtype=torch.long, device=ds.k_cache.device)
    kh, vh = raw(ds.k_cache.index_select(0, idx)), raw(ds.v_cache.index_select(0, idx))
    q = raw(ds.q)[seqs]
    nbytes = step_bytes(w, sbt, scl, 0, 0)["decode"]
    note = sample_text(w, seqs, len(cl), scl, nbytes)
    before = oracle.num_threads()
    if threads is not None:
        oracle.set_num_threads(threads)
    try:
        # bound the sample: whole decodes until ~budget_s of work (at least one)
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.decode(q, kh, vh, sbt, scl, w.softmax_scale, w.dtype, w.num_q_heads,
                          w.num_kv_heads, w.head_dim, w.block_size)
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
        used_threads = oracle.num_threads()
    finally:
        oracle.set_num_threads(before)
    return reps, el, used_threads, nbytes, note


def sample_text(w, seqs, S, scl, nbytes):
    """What one oracle repetition decodes, for the line's `sample` fields."""
    import numpy as np
    if len(seqs) == S:
        what = "the step's one sequence" if S == 1 else f"all {S} sequences of the step"
        return f"{what} ({int(np.sum(scl))} tokens, {nbytes / 1e9:.3f} GB)"
    return (f"a seeded sample of {len(seqs)} of the {S} sequences, the longest among them "
            f"({int(np.sum(scl))} tokens, {nbytes / 1e9:.2f} GB of K/V)")


class L2Flush:
    """Write 512 MB, then read 1 GB: evicts everything (the L2 is 129 MB) and leaves
    only clean lines, so no write-back of the flush lands in the timed region."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=device)
        self.r = torch.ones(256 << 20, dtype=torch.float32, device=device)
        self.sink = torch.empty(1, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.sink.copy_(self.r.sum().view(1))


def max_over_ranks(values, device="cpu"):
    """Each value's maximum over the ranks: the job takes as long as its slowest rank
    (identity outside torch.distributed or at world size 1)."""
    import torch
    import torch.distributed as dist
    values = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return values
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_gbs(bytes_per_rank, ms, world):
    """Whole-job GB/s: every rank moves bytes_per_rank in the slowest rank's time."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but {world} ranks were started")
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"

    from paged_kv_cache_79_gb300 import build as libbuild
    libbuild.build()
    w, ds, bt, cl = prepare(args.workload, device, seed_offset=rank, partition_size=args.partition_size,
                            kw=workload_kw(args))
    n_tok = int(ds.slots.shape[0])
    n_pairs = int(ds.pairs.shape[0])
    by = step_bytes(w, bt, cl, n_tok, n_pairs)
    S = len(cl)
    stream = torch.cuda.Stream(device)
    flush = L2Flush(device)
    import paged_kv_cache_79_gb300 as P
    parts = P.pa_decode_partition_size(S, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                       bt.shape[1], w.partition_size)
    # balanced split (0): one partition kernel (split units merge in it); fixed
    # partitions: plus the merge kernel when a table spans several partitions
    merge = parts > 0 and -(-bt.shape[1] // (parts // w.block_size)) > 1
    fused = ds.fusable
    # the shared-prefix decode where the groups save enough reads to pay for its
    # second launch (parallel sampling: 69% of the reads; the long multi-turn
    # batch: 2.7%, 580 MB)
    share_mode = "never" if getattr(args, "no_share", False) else getattr(args, "share", "auto")
    shared = ds.share is not None and (share_mode == "always" or (share_mode == "auto" and ds.share_pays))
    if shared:
        merge = False
        parts = 0
    # the plain balanced split starts each CTA from the host plan (pa_decode_plan)
    planned = (not shared and parts == 0 and ds.plan is not None and
               getattr(args, "plan", "auto") != "never")
    # ... and the shared-prefix decode's two launches from theirs (pa_decode_shared_plan)
    shared_planned = shared and ds.shared_plan is not None and getattr(args, "plan", "auto") != "never"

    launches_per_step = ((1 if n_pairs else 0) + (0 if fused or not n_tok else 1) +
                         (2 if shared else 1) + (1 if merge else 0))

    with torch.cuda.stream(stream):
        step = ((lambda st: ds.run_shared(st, planned=shared_planned)) if shared else
                ds.run_planned if planned else ds.run_fused if fused else ds.run)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        # the sampler starts first: warm-up runs right before the timed steps, so the
        # GPU does not idle (and drop its clocks) between them
        clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
        if clocks:
            clocks.start()
            time.sleep(0.3)
        for _ in range(args.warmup):
            flush()
            step(stream)
        torch.cuda.synchronize(device)
        if world > 1:
            dist.barrier()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush()                                         # evict the previous step from L2
            e0, e1, e2 = ev[i]
            e0.record(stream)
            if n_pairs:
                P.pa_copy_blocks(ds.k_cache, ds.v_cache, ds.pairs, stream)
            if not fused:
                P.pa_reshape_and_cache(ds.step_k, ds.step_v, ds.k_cache, ds.v_cache, ds.slots, stream)
            e1.record(stream)
            if shared:
                ds.decode_shared(stream, append=fused, planned=shared_planned)
            elif planned:
                P.pa_decode_planned(ds.out, ds.q, ds.k_cache, ds.v_cache, ds.block_tables,
                                    ds.context_lens, ds.plan, ds.scale, ds.num_q_heads,
                                    ds.num_kv_heads, ds.head_dim, ds.block_size,
                                    k_new=ds.step_k if fused else None,
                                    v_new=ds.step_v if fused else None,
                                    workspace=ds.workspace, stream=stream)
            elif fused:
                P.pa_decode_append(ds.out, ds.q, ds.k_cache, ds.v_cache, ds.step_k, ds.step_v,
                                   ds.block_tables, ds.context_lens, ds.scale, ds.num_q_heads,
                                   ds.num_kv_heads, ds.head_dim, ds.block_size, ds.partition_size,
                                   ds.workspace, stream)
            else:
                ds.decode(stream)
            e2.record(stream)
        torch.cuda.synchronize(device)
        wall = time.perf_counter() - t_wall
        if world > 1:
            dist.barrier()
        clk = clocks.stop() if clocks else None

    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    dec_ms = [b.elapsed_time(c) for a, b, c in ev]
    # the step time is the median of the timed steps; the decode launch's mean
    # duration gives the roofline
    t_step = statistics.median(step_ms)
    t_step_mean = sum(step_ms) / len(step_ms)
    t_dec = sum(dec_ms) / len(dec_ms)
    t_dec_med = statistics.median(dec_ms)

    # secondary: warm steps, back to back with no flush (whatever of the step the
    # 129 MB L2 still holds from the step before is read from there)
    with torch.cuda.stream(stream):
        for _ in range(2):
            step(stream)
        wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in wev:
            a.record(stream)
            step(stream)
            b.record(stream)
        torch.cuda.synchronize(device)
    t_warm = statistics.median([a.elapsed_time(b) for a, b in wev])
    t_step, t_step_mean, t_dec, t_dec_med, t_warm = max_over_ranks(
        [t_step, t_step_mean, t_dec, t_dec_med, t_warm], device)

    # end to end through the public API with host buffers
    e2e = run_e2e(ds, stream, device, args, by, shared, world, planned, shared_planned)

    if rank != 0:
        return None
    value = job_gbs(by["step"], t_step, world)
    peak, peak_kind = measured_peak()
    dec_bytes = by["decode"] + (by["append"] if fused else 0)
    achieved = dec_bytes / (t_dec * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) q/K/V; seeded allocator script)",
        "config": workload_config(w, cl, world),
        "path": {"split": "balanced" if parts == 0 else f"fixed partitions of {parts} tokens",
                 "append": "fused into the decode launch" if fused else "separate launch",
                 "prefix_sharing": (f"{int((ds.share[:, 0] >= 0).sum())} sequences in groups that "
                                    "read their shared leading blocks once (two-pass decode)"
                                    if shared else "not used (groups save too few reads)"
                                    if ds.share is not None and share_mode == "auto" else
                                    "not used (--share never)" if ds.share is not None else "none"),
                 "cta_starts": ("planned on the host (pa_decode_plan, uploaded with the tables)"
                                if planned else
                                "planned on the host for both launches (pa_decode_shared_plan, "
                                "uploaded with the tables)" if shared_planned else
                                "walked on the device"),
                 "appended_tokens": n_tok,
                 "cow_pairs": n_pairs},
        "ms_per_step_mean": round(t_step_mean, 5),
        "seq_layers_per_s": round(world * S / (t_step * 1e-3), 1),
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "decode_ms": round(t_dec, 5),
        "decode_ms_median": round(t_dec_med, 5),
        "bytes_per_step": by,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     # the profiled bytes are those of the workload at its own sizes
                     "traffic": (profiled_traffic(w.name, 2 if shared else 1)
                                 if not workload_kw(args) else None),
                     "kernel": (("pa_decode_shared_planned" if shared_planned else "pa_decode_shared") +
                                " (partition kernel twice: shared prefixes, then own "
                                "blocks" + (" + append" if fused else "") + ", merges inside)" if shared
                                else "pa_decode_planned (append + decode partition kernel from the host "
                                "plan, merge inside)" if planned and fused
                                else "pa_decode_append (append + decode partition kernel, merge inside)"
                                if fused else
                                "pa_decode (partition kernel; split-KV merge fused or second kernel)")},
        "e2e": e2e,
        "warm": {"ms_per_step": round(t_warm, 5), "value": round(job_gbs(by["step"], t_warm, world), 2),
                 "unit": "GB/s", "note": "secondary: steps back to back without the L2 flush"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }
    if world == 1 and not args.no_cpu_baseline:
        reps, el, cores, nbytes, note = cpu_baseline(w, ds, bt, cl, args.cpu_budget)
        line["cpu_baseline"] = {"value": round(reps * nbytes / el / 1e9, 4), "unit": "GB/s",
                                "cores": cores, "kind": "oracle",
                                "sample": f"{reps} decodes of {note}, fp64 C oracle, {el:.1f} s"}
        if w.name in ONE_CORE_WORKLOADS:
            reps, el, cores, nbytes, note = cpu_baseline(w, ds, bt, cl, args.cpu_budget / 2, threads=1)
            line["cpu_baseline_one_core"] = {
                "value": round(reps * nbytes / el / 1e9, 4), "unit": "GB/s", "cores": cores,
                "kind": "oracle",
                "sample": f"{reps} decodes of {note}, fp64 C oracle on one core, {el:.1f} s"}
    return line


def run_e2e(ds, stream, device, args, by, shared=False, world=1, planned=False, shared_planned=False):
    """Same step through the public API with inputs in pinned host memory: H2D of
    the step's inputs (packed into one buffer, one copy), the step, D2H of the
    output -- all inside the timed region."""
    import dataclasses
    import torch
    from paged_kv_cache_79_gb300 import runner
    names = ["q", "step_k", "step_v", "slots", "pairs", "block_tables", "context_lens"]
    if shared:
        names.append("share")
    if planned:
        names.append("plan")
    if shared_planned:
        names.append("shared_plan")
    packed = runner.PackedInputs({n: getattr(ds, n) for n in names}, device)
    dsv = dataclasses.replace(ds, **packed.views)
    out_h = torch.empty(ds.out.shape, dtype=ds.out.dtype).pin_memory()
    h2d = packed.nbytes
    d2h = out_h.numel() * out_h.element_size()
    flush = L2Flush(device)
    times = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            packed.upload(stream)
            if shared:
                dsv.run_shared(stream, planned=shared_planned)
            elif planned:
                dsv.run_planned(stream)
            else:
                dsv.run_fused(stream) if dsv.fusable else dsv.run(stream)
            out_h.copy_(dsv.out, non_blocking=True)
            b.record(stream)
            b.synchronize()
            if i >= args.warmup:
                times.append(a.elapsed_time(b))
    t = max_over_ranks([sum(times) / len(times)], device)[0]
    return {"value": round(job_gbs(by["step"], t, world), 2), "unit": "GB/s", "ms_per_step": round(t, 5),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": "step inputs packed into one pinned buffer: one H2D copy, then the step, then one D2H copy"}


# ----------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle on the host cores
# ----------------------------------------------------------------------------
def run_reference(args):
    """The oracle as the reference arm, on rank 0's host cores: each timed step
    decodes the oracle subset of the workload (every sequence, or for the long
    multi-turn batch a seeded sample of 32 plus the longest; see oracle_subset),
    over pool data generated on the host for the blocks those sequences use."""
    import numpy as np
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    if world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but {world} ranks were started")
    if rank != 0:
        return None
    import oracle
    import workloads as W
    w = W.by_name(args.workload, **workload_kw(args))
    # the oracle executes the workload's script with its own allocator; the pool
    # data is N(0,1) drawn on the CPU (same recipe, CPU generator) for the blocks
    # the decoded sequences reference
    oalloc, _ = oracle.run_script(w.events, w.num_blocks, w.block_size, w.free_order)
    bt, cl = oracle.tables_for(oalloc, w.decode_seqs)
    seqs = oracle_subset(w, bt, cl)
    used, sbt, scl = subset_tables(w, bt, cl, seqs)
    shape = (len(used), w.block_size, w.num_kv_heads, w.head_dim)
    kh = raw(W.randn(shape, w.dtype, w.data_seed * 10 + 1))
    vh = raw(W.randn(shape, w.dtype, w.data_seed * 10 + 2))
    q = raw(W.query_tensor(w, 0))[seqs]
    nbytes = step_bytes(w, sbt, scl, 0, 0)["decode"]
    note = sample_text(w, seqs, len(cl), scl, nbytes)
    # every host core (torch.distributed.run sets OMP_NUM_THREADS=1 for its ranks;
    # only rank 0 works here)
    before = oracle.num_threads()
    oracle.set_num_threads(os.cpu_count() or 1)
    times = []
    try:
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.decode(q, kh, vh, sbt, scl, w.softmax_scale, w.dtype, w.num_q_heads,
                          w.num_kv_heads, w.head_dim, w.block_size)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        cores = oracle.num_threads()
    finally:
        oracle.set_num_threads(before)
    t = statistics.median(times)
    value = nbytes / t / 1e9
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
            "ms_per_step_mean": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": workload_config(w, cl, world),
            "path": {"oracle": "fp64 C, plain definition (gather the valid rows, dense softmax "
                               "attention), OpenMP over (sequence, head)",
                     "sample": f"each step decodes {note}"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"each timed step decodes {note} (fp64 C oracle)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------
# secondary measurements (not the headline step): block moves and pool accounting
# ----------------------------------------------------------------------------
def run_blocks(args):
    """GB/s of the block-move kernels: swap between the device pool and pinned host
    memory, staging gathers/scatters on the device.  Bytes = blocks moved x block
    bytes x 2 (K and V), counted once per move."""
    import numpy as np
    import torch
    import paged_kv_cache_79_gb300 as P
    from paged_kv_cache_79_gb300 import build as libbuild
    libbuild.build()
    dev = "cuda:0"
    nb, n, shape = 4096, 2048, (16, 40, 128)      # MHA fp16 blocks of 160 KB
    g = torch.Generator(device=dev).manual_seed(7)
    kc = torch.randn((nb,) + shape, device=dev, generator=g).half()
    vc = torch.randn((nb,) + shape, device=dev, generator=g).half()
    hk = torch.empty((n,) + shape, dtype=torch.float16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    dk = torch.empty((n,) + shape, dtype=torch.float16, device=dev)
    dv = torch.empty_like(dk)
    ids = torch.from_numpy(np.random.default_rng(0).permutation(nb)[:n].astype(np.int32)).to(dev)
    seq = torch.arange(n, dtype=torch.int32, device=dev)
    p_out = torch.stack([ids, seq], 1).contiguous()
    p_in = torch.stack([seq, ids], 1).contiguous()
    moved = 2 * n * kc[0].numel() * kc.element_size()
    flush = L2Flush(dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(args.steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        ms = sorted(ts)[len(ts) // 2]
        return {"us": round(ms * 1000, 1), "GB/s": round(moved / (ms * 1e-3) / 1e9, 1)}

    res = {
        "swap_out_device_to_pinned_host": timed(lambda: P.pa_swap_blocks(kc, vc, hk, hv, p_out)),
        "swap_in_pinned_host_to_device": timed(lambda: P.pa_swap_blocks(hk, hv, kc, vc, p_in)),
        "gather_device_to_device": timed(lambda: P.pa_gather_blocks(kc, vc, ids, dk, dv)),
        "scatter_device_to_device": timed(lambda: P.pa_scatter_blocks(dk, dv, kc, vc, ids)),
        "copy_engine_device_to_pinned_host_contiguous": timed(
            lambda: (hk.copy_(dk, non_blocking=True), hv.copy_(dv, non_blocking=True))),
    }
    peak, kind = measured_peak()
    return {"op": "blocks", "blocks": n, "block_bytes": kc[0].numel() * kc.element_size(),
            "bytes_per_move": moved, "results": res,
            "device_copy_frac": round(2 * res["gather_device_to_device"]["GB/s"] / peak, 4),
            "device_copy_note": f"device-to-device moves read and write each byte: 2 x GB/s vs the "
                                f"{kind} copy bandwidth {peak} GB/s",
            "steps": args.steps, "warmup": args.warmup}


def run_memory(args):
    """Pool accounting on allocator traces (host only): waste of slots and the
    saving from shared blocks, after the last step of each trace."""
    import workloads as W
    from paged_kv_cache_79_gb300 import build as libbuild
    from paged_kv_cache_79_gb300 import runner
    libbuild.build()
    res = {}
    for name, kw in [("shared_prefix_fp16", {}), ("shared_prefix_fp16", {"prompt_len": 1032}),
                     ("beam_search_fp16", {"beams": 4}), ("beam_search_fp16", {"beams": 8}),
                     ("long_multiturn_bf16", {}), ("gqa_bf16", {})]:
        w = W.by_name(name, **kw)
        u = runner.replay_usage(w)
        last = u[-1]
        res[w.name] = {"used_blocks": last["used_blocks"], "logical_blocks": last["logical_blocks"],
                       "waste": round(last["waste"], 4), "sharing_saving": round(last["sharing_saving"], 4),
                       "mean_sharing_saving_over_steps": round(sum(x["sharing_saving"] for x in u) / len(u), 4)}
    return {"op": "memory", "data": "synthetic allocator traces", "results": res}


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_ranks(n: int, argv) -> int:
    """Run this script as n ranks on this node (torch.distributed.run, rendezvous on
    127.0.0.1, one process per GPU); rank 0 prints the line.  Returns the exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", f"--master-port={free_port()}",
           os.path.abspath(__file__)] + list(argv)
    return subprocess.run(cmd).returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--workload-kw", action="append", default=[], metavar="KEY=INT",
                    help="a parameter of the workload's generator (e.g. groups=4 for a 16-sequence "
                         "long_multiturn_bf16): a smaller case of the same workload, for profiling")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--partition-size", type=int, default=0,
                    help="0: balanced split (default); >0: fixed partitions of that many tokens")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--share", default="auto", choices=["auto", "always", "never"],
                    help="the two-pass shared-prefix decode for batches whose sequences share leading "
                         "blocks: where it saves enough reads (auto), always, or never")
    ap.add_argument("--no-share", action="store_true", help="the same as --share never")
    ap.add_argument("--plan", default="auto", choices=["auto", "never"],
                    help="start the plain balanced split's CTAs from a host plan (auto) or walk the "
                         "stream on the device (never)")
    ap.add_argument("--op", default="decode", choices=["decode", "blocks", "memory"],
                    help="decode: the headline step (default); blocks: block-move GB/s; "
                         "memory: pool accounting on allocator traces")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.op == "decode" and args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:]))
    if args.op == "blocks":
        line = run_blocks(args)
    elif args.op == "memory":
        line = run_memory(args)
    else:
        line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
