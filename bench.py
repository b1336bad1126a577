#!/usr/bin/env python3
"""Benchmark: one decode step of paged attention per iteration, on GB300.

A step is the whole hot path over one batch: each sequence's newest token is
written into its slot and attention runs over every sequence (the serving
order: the new token's K/V is in the cache before attention). By default the
step is pa_decode_append, which does both in one kernel; ``--step separate``
runs pa_reshape_and_cache then pa_decode. Default workload: Llama-3-8B-shaped GQA decode
(128 sequences, 32 query / 8 kv heads, head_dim 128, block size 16, lengths
uniform in [1024, 8192], bf16, random block placement, seed 0).

Prints one JSON line. ``value`` is effective GB/s: the algorithmic bytes of the
step (K/V rows of every valid token, table entries, lengths, q and out, plus
the cache write's reads and writes) divided by device time, with inputs
resident in HBM. Per step ~2.4 GB of K/V is read, far more than the 129 MB
L2, so no L2 flush is needed between steps.

``--impl reference`` times the float64 CPU oracle instead (on a bounded
sample of the same workload) and prints the same metric.

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(seed = rank): weak scaling, no data-path collective; the timing is the max
over ranks.
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

# the CPU oracle leg is timed single-threaded; say so instead of guessing BLAS threads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention: effective KV-read GB/s (% of HBM peak), tokens/s"
DEFAULT_WORKLOAD = "llama3_8b_gqa"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _decode_source_sha() -> str:
    """SHA-256 over the decode kernel's source and the header of its constants."""
    h = hashlib.sha256()
    for name in ("decode.cu", "internal.h"):
        h.update(open(os.path.join(ROOT, "paged_kv_cache_305_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def _traffic(workload: str, partition_tokens: int):
    """DRAM bytes per decode launch from a committed ncu capture, if the kernel and
    the partition length are those of the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(workload)
    if not rec:
        return None
    if _decode_source_sha() != rec.get("source_sha256"):
        return None
    if rec.get("partition_tokens") != partition_tokens:
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        busy = [x for x in sm if smax and x > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Multi-process timing: every rank times its own replica; the job's time is the
# slowest rank's, and value counts the units all ranks processed.
# ---------------------------------------------------------------------------
def max_over_ranks(times_ms, dist, device="cpu"):
    """Element-wise max of this rank's timings over all ranks (identity without dist)."""
    if dist is None:
        return [float(t) for t in times_ms]
    import torch
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(units_per_rank, world, max_ms):
    """Whole-job throughput: units of all ranks over the slowest rank's time (per second)."""
    return units_per_rank * world / (max_ms * 1e-3)


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def _pair_bytes(case, s):
    """Algorithmic bytes attributed to one (sequence, query head) of the decode."""
    L, B = int(case.seq_lens[s]), case.block_size
    seq = 2 * L * case.num_kv_heads * case.head_dim * 2 + 4 * ((L + B - 1) // B) + 4
    return seq / case.num_q_heads + 2 * case.head_dim * 2


def oracle_prepare(case):
    """The step's cache write, applied by the oracle to the host caches (in place)."""
    import oracle
    oracle.reshape_and_cache(case.new_key, case.new_value, case.key_cache, case.value_cache,
                             case.slot_mapping, case.block_size, in_place=True)


def time_oracle(case, budget_s: float, start: int = 0):
    """Run the float64 oracle over (sequence, query head) output rows of the batch,
    from row ``start`` on (wrapping), until ``budget_s`` is spent (at least one row).

    Returns (GB/s over the rows' share of the algorithmic bytes, seconds, rows done).
    """
    import oracle
    S, Hq = case.num_seqs, case.num_q_heads
    t0 = time.perf_counter()
    done, nbytes = 0, 0.0
    while True:
        i = (start + done) % (S * Hq)
        s, hq = i // Hq, i % Hq
        oracle.paged_decode_pairs(case.query, case.key_cache, case.value_cache, case.block_tables,
                                  case.seq_lens, case.block_size, case.scale, case.dtype, [(s, hq)])
        nbytes += _pair_bytes(case, s)
        done += 1
        if time.perf_counter() - t0 >= budget_s or done >= S * Hq:
            break
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, dt, done


def host_cores() -> int:
    """Cores this process may run on (the machine's host cores available to the run)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# Why the oracle runs on one thread: it is timed as it stands, a plain NumPy
# program whose work per output row is small matrix-vector products (a few
# heads against a few thousand keys), where extra BLAS threads add overhead
# rather than speed; rows are independent, so a run over all host cores would
# take about the one-thread time divided by the core count.
ONE_THREAD = ("the oracle as it stands is single-threaded NumPy (BLAS pinned to 1 thread: "
              "per output row it does small matrix-vector products); its rows are independent")


def cpu_baseline_block(case, budget_s):
    t0 = time.perf_counter()
    oracle_prepare(case)
    gbs, dt, done = time_oracle(case, budget_s)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "host_cores": host_cores(),
            "kind": "oracle", "why_one_thread": ONE_THREAD,
            "sample": f"float64 NumPy oracle (one thread): {done} of {case.num_seqs * case.num_q_heads} "
                      f"(sequence, query head) output rows of the same batch in {dt:.1f} s "
                      f"(after its cache write, {time.perf_counter() - t0 - dt:.1f} s)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    case = W.make_workload(args.workload, seed=0, block_size=args.block_size, num_seqs=args.num_seqs)
    oracle_prepare(case)
    # every step is a bounded sample, sized so that warm-up + steps take ~2 minutes
    per_step = max(0.002, min(args.ref_budget, 120.0 / max(1, args.steps + args.warmup)))
    pos = 0
    for _ in range(args.warmup):
        _, _, n = time_oracle(case, per_step, pos)
        pos += n
    tot_bytes, tot_s, rows = 0.0, 0.0, 0
    for _ in range(args.steps):
        gbs, dt, n = time_oracle(case, per_step, pos)
        pos += n
        rows += n
        tot_bytes += gbs * dt * 1e9
        tot_s += dt
    gbs = tot_bytes / tot_s / 1e9
    S_Hq = case.num_seqs * case.num_q_heads
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        # each timed step is a bounded sample of the step's output rows
        "ms_per_step": round(1e3 * tot_s / args.steps, 3),
        "ms_per_step_kind": f"sample: {rows / args.steps:.0f} of the step's {S_Hq} (sequence, "
                            f"query head) output rows per timed step; value = the sampled rows' "
                            f"algorithmic bytes / their time",
        "ms_per_whole_step_estimate": round(1e3 * tot_s / args.steps * S_Hq / max(1.0, rows / args.steps), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": case.dtype,
        "data": "synthetic", "config": _config(case, args),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1,
                         "host_cores": host_cores(), "kind": "oracle", "why_one_thread": ONE_THREAD,
                         "sample": f"float64 NumPy oracle (one thread): {rows} (sequence, query head) "
                                   f"output rows over {args.steps} steps of ~{per_step:.3f} s each"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(case, args):
    import paged_kv_cache_305_gb300 as pa
    pt = args.partition_tokens if args.partition_tokens is not None else case.partition_tokens
    return {"workload": case.name, "num_seqs": case.num_seqs, "num_q_heads": case.num_q_heads,
            "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
            "block_size": case.block_size, "seq_len_range": [int(case.seq_lens.min()),
                                                             int(case.seq_lens.max())],
            "mean_seq_len": round(float(case.seq_lens.mean()), 1),
            # the length the library resolves (0 asks for its default)
            "partition_tokens": pa.decode_partition_tokens(pt, case.block_size,
                                                           case.max_blocks_per_seq),
            "kv_bytes_per_step": case.kv_bytes(),
            "step": "write each sequence's newest K/V row into its slot, then decode attention "
                    "over every sequence",
            "cuda_graph": bool(getattr(args, "graph", False)),
            "l2": "no flush: inputs larger than L2 (KV read per step >> 129 MB)",
            "parallelism": "replicas (weak scaling, no collective)", "seed": 0}


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_cache_305_gb300 as pa
    from paged_kv_cache_305_gb300 import build as pbuild

    pbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    case = W.make_workload(args.workload, seed=rank, num_seqs=args.num_seqs,
                           block_size=args.block_size if args.workload == "shared_prefix" else None)
    pt = args.partition_tokens if args.partition_tokens is not None else case.partition_tokens
    tdt = {"fp16": torch.float16, "bf16": torch.bfloat16}[case.dtype]

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(tdt)

    q, kc, vc = up(case.query), up(case.key_cache), up(case.value_cache)
    nk, nv = up(case.new_key), up(case.new_value)
    bt = torch.from_numpy(case.block_tables).to(dev)
    sl = torch.from_numpy(case.seq_lens).to(dev)
    slots = torch.from_numpy(case.slot_mapping).to(dev)
    out = torch.empty_like(q)
    ws = pa.alloc_workspace(q, kc, bt, pt)
    stream = torch.cuda.current_stream(dev)
    # pa_decode_append's contract: each sequence's newest token sits in a block
    # of its own. A workload where some newest tokens sit in shared blocks (a
    # copy-on-write case the generator marks with slot -1) runs the separate step.
    fused_ok = bool((case.slot_mapping >= 0).all())
    fused = args.step == "fused" and fused_ok

    def step():
        if fused:  # cache write + attention in one kernel
            pa.decode_append(out, q, nk, nv, kc, vc, bt, sl, case.scale, pt, ws)
        else:
            pa.reshape_and_cache(nk, nv, kc, vc, slots)
            pa.decode(out, q, kc, vc, bt, sl, case.scale, pt, ws)

    W_steps = max(3, args.warmup)
    graph = None
    if args.graph:  # the step captured once, replayed every iteration (no host launch cost)
        for _ in range(W_steps):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()

    dec_bytes = case.algorithmic_bytes()
    # the step must also store each new K/V row once (its read is already in
    # dec_bytes as the newest token of its sequence)
    written = 2 * int((case.slot_mapping >= 0).sum()) * case.num_kv_heads * case.head_dim * 2
    step_bytes = dec_bytes + written
    # per-iteration events bracket the decode kernel alone, except in graph
    # mode, where they bracket the replayed step (the write included)
    kern_bytes = step_bytes if (fused or args.graph) else dec_bytes
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    gpu_index = (local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else
                 int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank]))
    with ClockSampler(gpu_index) as clk:
        if graph is None:
            # the warm-up steps right before the timed region, so the GPU is
            # busy (and at its clocks) when timing starts
            for _ in range(W_steps):
                step()
        torch.cuda.synchronize()
        # a short device-side wait before the start event (outside the timed
        # region): while it runs the host queues the first timed launches, so
        # the first launch's events do not include the host's launch latency
        torch.cuda._sleep(400000)
        start.record(stream)
        for i in range(K):
            if graph is not None:
                ev[i][0].record(stream)
                graph.replay()
                ev[i][1].record(stream)
            elif fused:
                ev[i][0].record(stream)
                pa.decode_append(out, q, nk, nv, kc, vc, bt, sl, case.scale, pt, ws)
                ev[i][1].record(stream)
            else:
                pa.reshape_and_cache(nk, nv, kc, vc, slots)
                ev[i][0].record(stream)
                pa.decode(out, q, kc, vc, bt, sl, case.scale, pt, ws)
                ev[i][1].record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = start.elapsed_time(stop)
    dec_ms = [a.elapsed_time(b) for a, b in ev]

    # end to end through the public API: pinned host inputs in, result out, every step
    h = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16) if v.dtype == np.uint16 else v)
         .pin_memory() for k, v in (("q", case.query), ("nk", case.new_key), ("nv", case.new_value),
                                    ("bt", case.block_tables), ("sl", case.seq_lens),
                                    ("slots", case.slot_mapping))}
    host_out = torch.empty(out.shape, dtype=torch.int16).pin_memory()
    d_in = {"q": q.view(torch.int16), "nk": nk.view(torch.int16), "nv": nv.view(torch.int16),
            "bt": bt, "sl": sl, "slots": slots}
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = host_out.numel() * host_out.element_size()

    if args.graph:  # copies in, the step and the copy out, captured together
        def e2e_once():
            for k in h:
                d_in[k].copy_(h[k], non_blocking=True)
            step()
            host_out.copy_(out.view(torch.int16), non_blocking=True)

        for _ in range(3):
            e2e_once()
        torch.cuda.synchronize()
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2):
            e2e_once()
        e2e_step = g2.replay
        e2e_start = e2e_finish = lambda: None
    else:
        # Pipelined as a serving loop would run it: two sets of device inputs
        # and outputs; step i's host-to-device copies (copy stream) overlap
        # step i-1's kernel, and its result goes back on a third stream while
        # step i+1 runs. Every copy of every step is inside the timed region.
        cs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ins = [d_in] + [{k: torch.empty_like(v) for k, v in d_in.items()}]
        outs = [out, torch.empty_like(out)]
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        ran = [torch.cuda.Event(), torch.cuda.Event()]
        read = [torch.cuda.Event(), torch.cuda.Event()]
        for e in read:
            e.record(stream)
        it = [0]

        def e2e_step():
            b = it[0] & 1
            it[0] += 1
            bi, bo = ins[b], outs[b]
            cs.wait_event(ran[b]) if it[0] > 2 else None  # set b's previous kernel is done with its inputs
            with torch.cuda.stream(cs):
                for k in h:
                    bi[k].copy_(h[k], non_blocking=True)
                copied[b].record(cs)
            stream.wait_event(copied[b])
            stream.wait_event(read[b])  # set b's previous result has been read back
            qd, nkd, nvd = (bi["q"].view(q.dtype), bi["nk"].view(nk.dtype), bi["nv"].view(nv.dtype))
            if fused:
                pa.decode_append(bo, qd, nkd, nvd, kc, vc, bi["bt"], bi["sl"], case.scale, pt, ws)
            else:
                pa.reshape_and_cache(nkd, nvd, kc, vc, bi["slots"])
                pa.decode(bo, qd, kc, vc, bi["bt"], bi["sl"], case.scale, pt, ws)
            ran[b].record(stream)
            ds.wait_event(ran[b])
            with torch.cuda.stream(ds):
                host_out.copy_(bo.view(torch.int16), non_blocking=True)
                read[b].record(ds)

        def e2e_start():  # no copy may begin before the timed region does
            cs.wait_stream(stream)

        def e2e_finish():  # the timed region ends after the last result is back
            stream.wait_stream(ds)
            stream.wait_stream(cs)

    for _ in range(3):
        e2e_step()
    e2e_finish()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    Ke = min(K, args.e2e_steps)
    e0.record(stream)
    e2e_start()
    for _ in range(Ke):
        e2e_step()
    e2e_finish()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dist, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peak, peak_kind = _peaks()
    dec_mean_ms = statistics.mean(dec_ms)
    achieved = kern_bytes / (dec_mean_ms * 1e-3) / 1e9
    value = job_throughput(step_bytes * K, world, ms) / 1e9
    cfg = _config(case, args)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W_steps, "ms_per_step": round(ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": case.dtype,
        "data": "synthetic",
        "config": cfg,
        "step_impl": "pa_decode_append (one kernel)" if fused else
                     "pa_reshape_and_cache + pa_decode" +
                     ("" if fused_ok or args.step != "fused" else
                      " (some newest tokens sit in shared blocks: the fused write does not apply)"),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        **({"unique_kv_bytes_per_step": case.unique_kv_bytes(),
            "unique_kv_GBps": round(case.unique_kv_bytes() * K * world / (ms * 1e-3) / 1e9, 2)}
           if case.name.startswith("shared_prefix") else {}),
        "tokens_per_s": round(case.num_seqs * K * world / (ms * 1e-3), 1),
        "kv_tokens_per_s": round(float(case.seq_lens.sum()) * K * world / (ms * 1e-3), 1),
        "roofline": {"kernel": "paged_decode_kernel" + (" (cache write fused)" if fused else ""),
                     "bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs (copy)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": _traffic(case.name, cfg["partition_tokens"]),
                     "algorithmic_bytes": kern_bytes,
                     "mean_launch_us": round(dec_mean_ms * 1e3, 2),
                     "median_launch_us": round(statistics.median(dec_ms) * 1e3, 2),
                     "min_launch_us": round(min(dec_ms) * 1e3, 2),
                     "p90_launch_us": round(sorted(dec_ms)[int(0.9 * (len(dec_ms) - 1))] * 1e3, 2),
                     "first_launches_us": [round(x * 1e3, 2) for x in dec_ms[:3]]},
        "e2e": {"value": round(step_bytes * Ke * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke},
        "gpu_launches": K if fused else 2 * K,
        "clocks": clk.summary(),
    }
    if not args.no_prefill:
        # measured after the decode's timed region, on the same GPU
        line["prefill"] = prefill_block(max(10, min(K, 50)), max(3, args.warmup), gpu_index)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_block(
            W.make_workload(args.workload, seed=0, block_size=args.block_size,
                            num_seqs=args.num_seqs), args.cpu_budget)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# Secondary measurements (one JSON line each; not the headline)
# ---------------------------------------------------------------------------
def _events(fn, steps, warmup):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_copy_blocks(args):
    """Block copies (the device half of copy-on-write): GB/s moved, HBM-bound."""
    import torch
    import paged_kv_cache_305_gb300 as pa
    from paged_kv_cache_305_gb300 import build as pbuild
    pbuild.build()
    NB, B, Hkv, d = 44188, 16, 8, 128  # the GQA workload's pool
    kc = torch.randn((NB, B, Hkv, d), device="cuda").to(torch.bfloat16)
    vc = torch.randn_like(kc)
    n = 4096
    perm = torch.randperm(NB, device="cuda").to(torch.int32)
    src, dst = perm[:n].contiguous(), perm[n:2 * n].contiguous()
    ms = _events(lambda: pa.copy_blocks(kc, vc, src, dst), args.steps, max(3, args.warmup))
    moved = 2 * 2 * n * B * Hkv * d * 2  # read + write, K and V
    peak, kind = _peaks()
    gbs = moved / (ms * 1e-3) / 1e9
    print(json.dumps({"op": "copy_blocks", "metric": "block copy GB/s (read + write)", "value": round(gbs, 1),
                      "unit": "GB/s", "frac_of_hbm_peak": round(gbs / peak, 4), "peak_kind": kind,
                      "ms_per_call": round(ms, 4), "steps": args.steps,
                      "config": {"copies": n, "block_bytes": B * Hkv * d * 2, "dtype": "bf16"}}))


def run_cache_write(args):
    """pa_reshape_and_cache on a full fill (every token of a Llama-3-8B-shaped GQA
    batch) and on a decode append (one token per sequence): GB/s = 4 T Hkv d e."""
    import torch
    import paged_kv_cache_305_gb300 as pa
    from paged_kv_cache_305_gb300 import build as pbuild
    pbuild.build()
    S, Hkv, d, B = 128, 8, 128, 16
    g = torch.Generator().manual_seed(0)
    L = torch.randint(1024, 8193, (S,), generator=g)
    nblk = (L + B - 1) // B
    pool = int(1.2 * int(nblk.sum()))
    perm = torch.randperm(pool, generator=g)
    boff = torch.cumsum(nblk, 0) - nblk
    seq = torch.repeat_interleave(torch.arange(S), L)
    t = torch.arange(int(L.sum())) - torch.repeat_interleave(torch.cumsum(L, 0) - L, L)
    slots = (perm[boff[seq] + t // B] * B + t % B).to(torch.int64).cuda()
    T = int(L.sum())
    kc = torch.zeros((pool, B, Hkv, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.randn((T, Hkv, d), device="cuda").to(torch.bfloat16)
    v = torch.randn_like(k)
    peak, kind = _peaks()
    res = {}
    last = (torch.cumsum(L, 0) - 1).cuda()  # each sequence's newest token
    for name, kk, vv, sl in (("fill", k, v, slots), ("append", k[last], v[last], slots[last])):
        n = kk.shape[0]
        ms = _events(lambda: pa.reshape_and_cache(kk, vv, kc, vc, sl), args.steps, max(3, args.warmup))
        moved = 4 * n * Hkv * d * 2
        res[name] = {"tokens": n, "ms_per_call": round(ms, 5), "GBps": round(moved / (ms * 1e-3) / 1e9, 1),
                     "frac_of_hbm_peak": round(moved / (ms * 1e-3) / 1e9 / peak, 4)}
    print(json.dumps({"op": "cache_write", "metric": "cache write GB/s (read + write of K and V)",
                      "value": res["fill"]["GBps"], "unit": "GB/s", "peak": peak, "peak_kind": kind,
                      "fill": res["fill"], "append": res["append"], "steps": args.steps,
                      "config": {"sequences": S, "num_kv_heads": Hkv, "head_dim": d, "block_size": B,
                                 "seq_len_range": [1024, 8192], "dtype": "bf16"}}))


def run_block_manager(args):
    """Host throughput of the native block manager's append (one token per sequence)."""
    import paged_kv_cache_305_gb300 as pa
    from paged_kv_cache_305_gb300 import build as pbuild
    pbuild.build()
    S, B = 128, 16
    bm = pa.BlockManager(200000, B, 1024)
    seqs = []
    for i in range(S // 4):
        p = bm.new_sequence()
        bm.append([(p, 1000 + 37 * i)])
        seqs.append(p)
        seqs.extend(bm.fork(p) for _ in range(3))  # 4 candidates share the prompt
    reqs = [(sq, 1) for sq in seqs]
    for _ in range(10):
        bm.append(reqs)
    n = max(100, args.steps)
    t0 = time.perf_counter()
    for _ in range(n):
        bm.append(reqs)
    dt = (time.perf_counter() - t0) / n
    tt = time.perf_counter()
    for _ in range(n):
        bm.block_tables(seqs)
    dtt = (time.perf_counter() - tt) / n
    print(json.dumps({"op": "block_manager", "metric": "block-manager appends per second (host)",
                      "value": round(S / dt, 1), "unit": "appends/s", "us_per_append_call": round(dt * 1e6, 2),
                      "us_per_table_export": round(dtt * 1e6, 2), "calls": n,
                      "config": {"sequences": S, "block_size": B, "candidates_per_prompt": 4,
                                 "binding": "ctypes (includes Python marshalling)"}}))


def run_serving_step(args):
    """One serving decode step through the native block manager: append one token
    per sequence (copy-on-write where candidates diverge), upload slots and
    tables, copy blocks, write the new K/V, decode."""
    import torch
    import paged_kv_cache_305_gb300 as pa
    from paged_kv_cache_305_gb300 import build as pbuild
    pbuild.build()
    rng = np.random.default_rng(0)
    S, Hq, Hkv, d, B = 128, 32, 8, 128, 16
    prompts = rng.integers(1024, 8193, size=S // 4)
    NB = int(1.3 * (sum(int(p) // B + 2 for p in prompts) + S * (args.steps + args.warmup + 16) // B + S))
    MB = 8192 // B + (args.steps + args.warmup) // B + 4
    bm = pa.BlockManager(NB, B, MB)
    dt = torch.bfloat16
    kc = torch.randn((NB, B, Hkv, d), device="cuda").to(dt)
    vc = torch.randn_like(kc)
    seqs = []
    for p in prompts:
        sid = bm.new_sequence()
        bm.append([(sid, int(p))])  # prompt K/V: the random pool contents stand in
        seqs.append(sid)
        seqs.extend(bm.fork(sid) for _ in range(3))
    q = torch.randn((S, Hq, d), device="cuda").to(dt)
    nk = torch.randn((S, Hkv, d), device="cuda").to(dt)
    nv = torch.randn_like(nk)
    out = torch.empty_like(q)
    reqs = [(sq, 1) for sq in seqs]
    ws = pa.alloc_workspace(q, kc, torch.empty((S, MB), dtype=torch.int32), 0)
    copies_seen = [0]
    bytes_seen = [0]

    def step():
        slots, copies = bm.append(reqs)
        tables, lens = bm.block_tables(seqs)
        slots_d = torch.from_numpy(slots).pin_memory().cuda(non_blocking=True)
        bt = torch.from_numpy(tables).pin_memory().cuda(non_blocking=True)
        sl = torch.from_numpy(lens).pin_memory().cuda(non_blocking=True)
        if copies:
            c = torch.tensor(copies, dtype=torch.int32).t().contiguous().cuda(non_blocking=True)
            pa.copy_blocks(kc, vc, c[0], c[1])
            copies_seen[0] += len(copies)
        pa.reshape_and_cache(nk, nv, kc, vc, slots_d)
        pa.decode(out, q, kc, vc, bt, sl, 1.0 / d ** 0.5, 0, ws)
        bytes_seen[0] += int(2 * lens.astype(np.int64).sum() * Hkv * d * 2)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    copies_seen[0], bytes_seen[0] = 0, 0
    t0 = time.perf_counter()
    steps = min(args.steps, 200)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    print(json.dumps({"op": "serving_step", "metric": "serving decode step through the block manager",
                      "value": round(S * steps / el, 1), "unit": "tokens/s",
                      "ms_per_step": round(1e3 * el / steps, 4),
                      "kv_GBps": round(bytes_seen[0] / el / 1e9, 1), "cow_copies": copies_seen[0],
                      "steps": steps, "timing": "wall clock, host and device",
                      "config": {"sequences": S, "prompts": S // 4, "candidates_per_prompt": 4,
                                 "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": d,
                                 "block_size": B, "prompt_len_range": [1024, 8192], "dtype": "bf16"}}))


def run_waste(args):
    """KV-memory waste of paged vs contiguous reservation on a synthetic trace."""
    from paged_kv_cache_305_gb300 import build as pbuild
    pbuild.build()
    from paged_kv_cache_305_gb300 import waste
    rows = {}
    for B in (1, 8, 16, 32, 64):
        r = waste.simulate(block_size=B)
        rows[str(B)] = {"paged_waste": round(r.paged_waste, 4), "contiguous_waste": round(r.contiguous_waste, 4),
                        "max_paged_waste_per_seq": r.max_paged_waste_per_seq}
    print(json.dumps({"op": "waste", "metric": "KV-memory waste fraction (time-averaged)",
                      "by_block_size": rows,
                      "config": {"max_len": 2048, "concurrent": 64, "requests": 512,
                                 "prompt_range": [16, 512], "output": "geometric, mean 200", "seed": 0}}))


def _bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured bf16_tflops (cuBLAS, burst)"
    return 1900.0, "fallback bf16 burst"


def measure_prefill(ctx, chunk, B, tname, steps, warmup, S=16, Hq=32, Hkv=8, d=128,
                    workspace=True):
    """Paged causal prefill of S sequences (Hq/Hkv heads, head_dim d, block size
    B): a chunk of `chunk` new tokens per sequence whose K/V are in the cache
    after ctx - chunk older tokens (ctx = chunk: whole prompts). Returns
    algorithmic TFLOP/s (4 * d * Hq flops per visible (query, key) pair) and
    the CUDA-event time per call."""
    import torch
    import paged_kv_cache_305_gb300 as pa
    case = W.random_case(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B,
                         len_range=(ctx, ctx), dtype=tname, seed=0)
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[tname]
    up = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda().view(dt)
    kc, vc = up(case.key_cache), up(case.value_cache)
    bt = torch.from_numpy(case.block_tables).cuda()
    sl = torch.from_numpy(case.seq_lens).cuda()
    starts = torch.arange(0, (S + 1) * chunk, chunk, dtype=torch.int32).cuda()
    q = torch.randn((S * chunk, Hq, d), device="cuda").to(dt)
    out = torch.empty_like(q)
    # bf16: with the workspace the call converts the value rows to fp16 first
    # (a second kernel, timed with it) and P.V is one product
    ws = pa.alloc_prefill_workspace(sl, kc, bt) if workspace else None
    pa.wait_timeout_count(clear=True)
    ms = _events(lambda: pa.prefill(out, q, kc, vc, bt, sl, starts, chunk, case.scale, ws),
                 steps, max(3, warmup))
    # a bounded in-kernel wait that gave up means a CTA wound down early: the
    # timing would not be of the whole computation
    timeouts = pa.wait_timeout_count(clear=True)
    if timeouts:
        raise RuntimeError(f"prefill: {timeouts} bounded waits gave up during the measurement")
    pairs = S * sum(ctx - chunk + j + 1 for j in range(chunk))
    tf = 4.0 * d * Hq * pairs / (ms * 1e-3) / 1e12
    peak, kind = _bf16_peak()
    ws_bytes = 0 if ws is None else ws.numel()
    del kc, vc, q, out, ws
    torch.cuda.empty_cache()
    return {"value": round(tf, 1), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
            "frac": round(tf / peak, 4), "tokens_per_s": round(S * chunk / (ms * 1e-3), 1),
            "launches_per_call": 2 if ws_bytes else 1,
            "config": {"sequences": S, "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": d,
                       "block_size": B, "context": ctx, "chunk": chunk, "dtype": tname,
                       "workspace_bytes": ws_bytes,
                       "p_v": "one fp16 product" if (tname == "fp16" or ws_bytes) else
                              "two bf16 products (weight head + remainder)"}}


def prefill_block(steps, warmup, gpu_index):
    """The prefill sub-object of the default line: 2048-token chunks after 2048
    cached tokens, and whole 2048-token prompts (bf16, block size 16)."""
    peak, kind = _bf16_peak()
    with ClockSampler(gpu_index) as clk:
        chunked = measure_prefill(4096, 2048, 16, "bf16", steps, warmup)
        whole = measure_prefill(2048, 2048, 16, "bf16", steps, warmup)
    return {"kernel": "paged_prefill_tc_kernel", "metric": "paged causal prefill TFLOP/s (algorithmic)",
            "bound": "tensor", "peak": peak, "peak_kind": kind, "chunked": chunked,
            "whole_prompt": whole, "steps": steps,
            "launches_timed": steps * (chunked["launches_per_call"] + whole["launches_per_call"]),
            "clocks": clk.summary()}


def run_prefill(args):
    """Paged causal prefill: algorithmic TFLOP/s (4 * d * Hq per causal pair)."""
    from paged_kv_cache_305_gb300 import build as pbuild
    pbuild.build()
    r = measure_prefill(args.prefill_context, args.prefill_chunk, args.prefill_block_size,
                        args.prefill_dtype, args.steps, args.warmup,
                        workspace=not args.prefill_no_workspace)
    peak, kind = _bf16_peak()
    print(json.dumps({"op": "prefill", "metric": "paged causal prefill TFLOP/s (algorithmic)",
                      "value": r["value"], "unit": "TFLOP/s", "ms_per_call": r["ms_per_call"],
                      "roofline": {"bound": "tensor", "achieved": r["value"], "peak": peak,
                                   "peak_kind": kind + "; fp16 has the same nominal rate",
                                   "frac": r["frac"]},
                      "tokens_per_s": r["tokens_per_s"], "steps": args.steps, "config": r["config"]}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(W.WORKLOADS) + ["shared_prefix"])
    ap.add_argument("--block-size", type=int, default=16, help="shared_prefix only")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="shrink the batch (small profiling captures only)")
    ap.add_argument("--partition-tokens", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--ref-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="leave the prefill sub-object out of the default line")
    ap.add_argument("--prefill-context", type=int, default=4096)
    ap.add_argument("--prefill-chunk", type=int, default=2048)
    ap.add_argument("--prefill-block-size", type=int, default=16)
    ap.add_argument("--prefill-dtype", default="bf16", choices=["bf16", "fp16"])
    ap.add_argument("--prefill-no-workspace", action="store_true",
                    help="bf16 prefill without its workspace (two P.V products, no fp16 copy of V)")
    ap.add_argument("--graph", action="store_true",
                    help="capture the step (and the end-to-end step) in CUDA graphs and replay them")
    ap.add_argument("--step", default="fused", choices=["fused", "separate"],
                    help="fused: pa_decode_append; separate: pa_reshape_and_cache then pa_decode")
    ap.add_argument("--op", default="decode_step",
                    choices=["decode_step", "copy_blocks", "block_manager", "serving_step", "waste",
                             "prefill", "cache_write"],
                    help="decode_step is the headline; the others print secondary measurements")
    args = ap.parse_args()
    if args.op != "decode_step":
        if int(os.environ.get("RANK", "0")) == 0:
            {"copy_blocks": run_copy_blocks, "block_manager": run_block_manager,
             "serving_step": run_serving_step, "waste": run_waste,
             "prefill": run_prefill, "cache_write": run_cache_write}[args.op](args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
