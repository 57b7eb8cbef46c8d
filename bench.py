#!/usr/bin/env python
"""Benchmark of one paged-KV attention step on GB300.

A step is the whole hot path over one batch: pkv_write of the step's new K/V
rows, then pkv_attention (plan, decode and prefill kernels) over the paged
cache.  The default workload is the pure MHA decode batch (256 requests, cached
lengths uniform in [512, 4096], Hq = Hkv = 32, head size 128, block size 16),
reported as KV GB/s: the K and V bytes every request's attention reads once
per KV head, divided by the step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...   # the float64 CPU oracle, same workload

With N > 1 (launched by torchrun, one process per GPU; a plain
``python bench.py --gpus N`` re-executes itself under torch.distributed.run)
every rank runs its own replica of the batch (the step shards by request with
no exchange), and the value is the total over ranks divided by the slowest
rank's time.  On one GPU the line also carries ``extra_configs``: the other
workloads (prefill, mixed, GQA and MQA decode, the trace step, and the int8
cache lines), each timed the same way.
"""
import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from paged_kv_attention_05_gb300 import workloads as W  # noqa: E402

DECODE_CONFIGS = {"mha_decode", "gqa_decode", "mqa_long_decode"}


def metric_of(spec):
    if spec.name in DECODE_CONFIGS:
        return "paged-attn decode KV GB/s", "GB/s"
    if spec.name == "large_prefill":
        return "paged-attn prefill TFLOP/s", "TFLOP/s"
    return "mixed-batch query tokens/s", "tokens/s"


def causal_flops(spec):
    """4 * head_size flops per (visible key, query row, query head)."""
    tot = 0
    for c, n in zip(spec.ctx, spec.q_len):
        tot += n * c + n * (n + 1) // 2
    return 4 * spec.head_size * spec.hq * tot


def metric_work(spec):
    """Units of the metric one step processes."""
    name, unit = metric_of(spec)
    if unit == "GB/s":
        return spec.kv_bytes() / 1e9
    if unit == "TFLOP/s":
        return causal_flops(spec) / 1e12
    return float(spec.num_tokens)


def decode_algorithmic_bytes(spec, kv_elem_bytes=2):
    """Algorithmic bytes of one decode-kernel launch: every decode request's
    K and V rows once per KV head (bf16, or int8 codes), its query rows read
    and output rows written (bf16)."""
    G = spec.hq // spec.hkv
    cap = 16 if G <= 16 else 32  # query rows of one decode unit
    b = 0
    for c, n in zip(spec.ctx, spec.q_len):
        if 0 < n and n * G <= cap:  # the requests the decode kernel serves
            b += (c + n) * spec.hkv * spec.head_size * kv_elem_bytes * 2
            b += 2 * n * spec.hq * spec.head_size * 2
    return b


def step_bytes(spec, kv_elem_bytes=2):
    """Algorithmic bytes of a whole step (write + attention): every request's
    K and V rows once per KV head, the query rows read and output rows
    written, and the write's new K/V rows read (bf16) and stored."""
    d = spec.head_size
    kv = sum(c + n for c, n in zip(spec.ctx, spec.q_len)) * spec.hkv * d * kv_elem_bytes * 2
    qo = 2 * spec.num_tokens * spec.hq * d * 2
    wr = spec.num_tokens * spec.hkv * d * 2 * (2 + kv_elem_bytes)
    return kv + qo + wr


L2_BYTES = 129e6  # GB300 L2


def l2_copies(footprint_bytes, factor=4):
    """How many copies of a step's inputs (cache, qkv, output) the timed loop
    rotates through so that what one step touches has left L2 before it is
    touched again: enough copies to make the rotation `factor` times the L2
    size, one when a single step already is."""
    return max(1, int(np.ceil(factor * L2_BYTES / max(footprint_bytes, 1))))


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, sources):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's
    source is unchanged since the counters were taken; else None."""
    path = os.path.join(ROOT, "profiles", "%s_%s.json" % (kernel, workload))
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != source_hash(sources):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0=None, t1=None):
        """Ends sampling; clocks and reasons from the samples taken between the
        host times t0 and t1 (the loaded window), all samples if none fall
        there."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]),
                                 {nm for nm, val in zip(names, parts[6:10])
                                  if val.lower().startswith("active")}))
                except ValueError:
                    continue
        os.unlink(self.path)
        loaded = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        use = loaded or rows
        reasons = set().union(*[r[3] for r in use]) if use else set()
        return {"sm_mhz": statistics.median([r[1] for r in use]) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": sorted(reasons), "samples": len(use),
                "window": ("the timed steps, the traced pass and at least 0.6 s more of the "
                           "same steps" if loaded else "whole run (no sample in the loaded window)")}


def max_over_ranks(x, dist, device):
    """The slowest rank's time: every rank's replica must finish for the
    whole-job throughput (all ranks' work / this time)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(work_per_rank, world, seconds_max):
    """Weak scaling: each rank processes one replica of the batch."""
    return work_per_rank * world / seconds_max


def cpu_baseline(step, sample_reqs=None, target_s=None):
    """The float64 oracle on the host cores over (a sample of) the same step:
    write + attention for the first sample_reqs requests (all by default),
    repeated until about target_s seconds of CPU work when that is given."""
    import oracle
    spec = step.spec
    R = spec.num_reqs if sample_reqs is None else min(sample_reqs, spec.num_reqs)
    kc, vc = step.key_cache, step.value_cache
    qsl = step.query_start_loc[:R + 1]
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.write(step.k, step.v, kc, vc, step.slot_mapping)
        oracle.attention(step.q, kc, vc, qsl, step.seq_lens[:R], step.block_table[:R], R,
                         step.scale)
        reps += 1
        dt = time.perf_counter() - t0
        if target_s is None or dt >= target_s:
            break
    sub = W.StepSpec(spec.name, spec.ctx[:R], spec.q_len[:R], spec.hq, spec.hkv,
                     spec.num_blocks, spec.seed)
    work = metric_work(sub) * reps
    return {"value": work / dt, "unit": metric_of(spec)[1], "cores": oracle.num_threads(),
            "kind": "oracle", "seconds_per_pass": dt / reps,
            "sample": "%d of %d requests, write + attention, %d pass%s, %.1f s" %
                      (R, spec.num_reqs, reps, "" if reps == 1 else "es", dt)}


def cpu_baseline_bounded(step, target_s=10.0):
    """cpu_baseline on a sample sized for about target_s seconds: the whole
    batch (repeated) when one pass is short, else the first requests."""
    spec = step.spec
    n_probe = min(2, spec.num_reqs)
    probe = cpu_baseline(step, sample_reqs=n_probe)
    per_req = float(probe["sample"].split(", ")[-1].rstrip(" s")) / n_probe
    reqs = max(1, min(spec.num_reqs, int(target_s / max(per_req, 1e-9))))
    return cpu_baseline(step, sample_reqs=reqs, target_s=target_s)


def l2_note(spec, int8):
    """How the timed steps keep K/V reads in HBM (stated in the line's config)."""
    n_copies = l2_copies(step_bytes(spec, 1 if int8 else 2))
    sb_mb = step_bytes(spec, 1 if int8 else 2) / 1e6
    if n_copies == 1:
        return "inputs larger than L2 (%.0f MB touched per step vs 129 MB)" % sb_mb
    return ("inputs larger than L2: %d copies of cache, qkv and output rotated, "
            "%.1f MB touched per step, %.0f MB per rotation vs 129 MB"
            % (n_copies, sb_mb, sb_mb * n_copies))


def config_of(spec, kv_dtype, with_prepare, world):
    """The workload a line measures; both arms print the same keys."""
    int8 = kv_dtype == "int8"
    return {"workload": spec.name, "requests": spec.num_reqs, "query_tokens": spec.num_tokens,
            "step": ("prepare + " if with_prepare else "") + "write + attention",
            "num_heads": spec.hq, "num_kv_heads": spec.hkv, "head_size": spec.head_size,
            "block_size": spec.block_size,
            "kv_bytes_per_step": spec.kv_bytes() // (2 if int8 else 1),
            "kv_dtype": kv_dtype, "l2": l2_note(spec, int8),
            "parallelism": "replica per GPU (dp%d)" % world}


def run_reference(args, spec, rank):
    """--impl reference: the float64 CPU oracle as it stands, same workload."""
    if rank != 0:
        return
    import oracle
    step = W.build(spec)
    name, unit = metric_of(spec)
    # size each step as a bounded sample of the workload (whole batch if cheap)
    probe = cpu_baseline(step, sample_reqs=min(8, spec.num_reqs))
    per_req = (metric_work(spec) / spec.num_reqs) / probe["value"]
    sample = max(1, min(spec.num_reqs, int(8.0 / max(per_req, 1e-9))))
    for _ in range(args.warmup if args.warmup < 1 else 1):
        cpu_baseline(step, sample)
    times = []
    for _ in range(args.steps):
        times.append(cpu_baseline(step, sample))
    vals = [t["value"] for t in times]
    value = statistics.median(vals)
    # a step here is the bounded sample: its wall time, median over the steps
    ms_step = statistics.median([t["seconds_per_pass"] for t in times]) * 1e3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rec = {"metric": name, "value": value, "unit": unit, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": config_of(spec, args.kv_dtype, args.with_prepare, world),
           "impl": "reference",
           "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": times[-1]["sample"],
                            "requests_per_step": sample},
           "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(rec))


def launch_check(args):
    """--gpus N must run N ranks: under torchrun WORLD_SIZE has to equal N;
    without it, N > 1 re-executes this script under torch.distributed.run
    (one process per GPU on this node) after checking that N GPUs exist.
    Returns only when this process is a rank of the right world."""
    world = os.environ.get("WORLD_SIZE")
    if world is not None:
        if int(world) != args.gpus:
            raise SystemExit("bench.py: --gpus %d but WORLD_SIZE=%s; launch one process per GPU"
                             % (args.gpus, world))
        return
    if args.gpus == 1:
        return
    if args.gpus < 1:
        raise SystemExit("bench.py: --gpus must be at least 1")
    if args.impl == "ours":
        import torch
        have = torch.cuda.device_count()
        if have < args.gpus:
            raise SystemExit("bench.py: --gpus %d but %d CUDA device(s) visible" %
                             (args.gpus, have))
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node=%d" % args.gpus, "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    sys.stdout.flush()
    os.execv(sys.executable, cmd)


class Workload:
    """Device buffers of one workload and its step: pkv_write + pkv_attention
    (int8 caches: pkv_write_int8 + pkv_attention_int8), optionally preceded by
    pkv_prepare_step.  Steps whose inputs fit in L2 rotate through copies of
    the cache, the qkv rows and the output (same contents, same block ids), so
    that every timed step reads its K/V from HBM as a serving step would."""

    KS = VS = 0.03  # int8 scales: codes saturate beyond about 3.8 sigma

    def __init__(self, spec, int8=False, with_prepare=False):
        import torch
        import paged_kv_attention_05_gb300 as pkv
        self.pkv, self.torch = pkv, torch
        self.spec, self.int8, self.with_prepare = spec, int8, with_prepare
        self.step = step = W.build(spec)
        s, d = spec, spec.head_size
        rows = step.qkv.shape[0]
        self.rows = rows
        self.n_copies = l2_copies(step_bytes(s, 1 if int8 else 2))
        qkv = self.dev(step.qkv)
        self.qkv = qkv
        self.qkvs = [self.split(t) for t in [qkv] + [qkv.clone() for _ in range(self.n_copies - 1)]]
        self.slot_mapping = torch.from_numpy(step.slot_mapping).cuda()
        self.qsl = torch.from_numpy(step.query_start_loc).cuda()
        self.seq_lens = torch.from_numpy(step.seq_lens).cuda()
        self.block_table = torch.from_numpy(step.block_table).cuda()
        self.outs = [torch.empty((rows, s.hq, d), dtype=torch.bfloat16, device="cuda")
                     for _ in range(self.n_copies)]
        self.stream = torch.cuda.current_stream()
        pkv.pkv_reserve_workspace(s.num_reqs, rows, step.block_table.shape[1], s.hq, s.hkv)
        key_cache, value_cache = self.dev(step.key_cache), self.dev(step.value_cache)
        if int8:
            # the history as int8 codes, quantised once by the library's own write
            nb = key_cache.shape[0]
            kc8 = torch.empty(key_cache.shape, dtype=torch.int8, device="cuda")
            vc8 = torch.empty_like(kc8)
            all_slots = torch.arange(nb * s.block_size, dtype=torch.int64, device="cuda")
            pkv.pkv_write_int8(key_cache.view(-1, s.hkv, d), value_cache.view(-1, s.hkv, d), kc8,
                               vc8, all_slots, self.KS, self.VS)
            pkv.pkv_get_error()
            key_cache = value_cache = all_slots = None  # the bf16 history is no longer needed
            self.caches = [(kc8, vc8)] + [(kc8.clone(), vc8.clone())
                                          for _ in range(self.n_copies - 1)]
        else:
            self.caches = [(key_cache, value_cache)] + [
                (key_cache.clone(), value_cache.clone()) for _ in range(self.n_copies - 1)]
        if with_prepare:
            self.num_computed = torch.tensor(s.ctx, dtype=torch.int32, device="cuda")
            self.persistent_bt = self.block_table.clone()
            self.positions = torch.empty(rows, dtype=torch.int64, device="cuda")

    def dev(self, bits):
        torch = self.torch
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).cuda()

    def split(self, t):
        s, d, rows = self.spec, self.spec.head_size, self.rows
        return (t[:, :s.hq * d].view(rows, s.hq, d),
                t[:, s.hq * d:(s.hq + s.hkv) * d].view(rows, s.hkv, d),
                t[:, (s.hq + s.hkv) * d:].view(rows, s.hkv, d))

    def one_step(self, i=0):
        pkv, s, st = self.pkv, self.spec, self.stream
        c = i % self.n_copies
        q, k, v = self.qkvs[c]
        kc, vc = self.caches[c]
        if self.with_prepare:
            pkv.pkv_prepare_step(self.qsl, self.num_computed, self.persistent_bt, s.num_reqs,
                                 self.rows, self.positions, self.seq_lens, self.slot_mapping,
                                 self.block_table, stream=st)
        if self.int8:
            pkv.pkv_write_int8(k, v, kc, vc, self.slot_mapping, self.KS, self.VS, stream=st)
            pkv.pkv_attention_int8(q, kc, vc, self.KS, self.VS, self.qsl, self.seq_lens,
                                   self.block_table, s.num_reqs, s.scale, self.outs[c], stream=st)
            return
        pkv.pkv_write(k, v, kc, vc, self.slot_mapping, stream=st)
        pkv.pkv_attention(q, kc, vc, self.qsl, self.seq_lens, self.block_table, s.num_reqs,
                          s.scale, self.outs[c], stream=st)


def time_steps(wl, steps, warmup, dist=None):
    """W warm-up steps, then K timed steps (CUDA events on the launch stream,
    barrier + synchronize on both sides, no per-launch events), then the same
    K steps again with the library's per-launch trace events, then the same
    steps for at least 0.6 s more so that the 200 ms clock samples see the
    GPU under this load.  Returns (timed ms, launches in the timed region,
    per-kernel trace, clocks)."""
    torch, pkv, stream = wl.torch, wl.pkv, wl.stream
    # the clock sampler starts before the warm-up, so that the GPU goes from
    # the warm-up steps straight into the timed ones (no idle gap)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    for i in range(max(warmup, 0)):
        wl.one_step(i)
    torch.cuda.synchronize()
    bits = pkv.pkv_get_error()
    if bits:
        clocks.stop()
        raise SystemExit("device error word %d after warm-up of %s" % (bits, wl.spec.name))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # the timed region: recording an event between two launches holds the
    # next one back by a few microseconds, which lengthens short steps by up
    # to a third, so only its two ends are recorded
    launches0 = pkv.pkv_launch_count()
    barrier()
    t_load0 = time.time()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        wl.one_step(i)
    e1.record(stream)
    barrier()
    launches = pkv.pkv_launch_count() - launches0
    # the per-kernel durations behind the roofline
    pkv.pkv_trace_read()
    pkv.pkv_trace_enable(True)
    barrier()
    for i in range(steps):
        wl.one_step(i)
    barrier()
    pkv.pkv_trace_enable(False)
    trace = pkv.pkv_trace_read()
    ms = e0.elapsed_time(e1)
    per = max(1, int(0.05 / max(ms / steps / 1e3, 1e-6)))
    i, t_soak = steps, time.time() + 0.6
    while time.time() < t_soak:
        for _ in range(per):
            wl.one_step(i)
            i += 1
        torch.cuda.synchronize()
    t_load1 = time.time()
    if pkv.pkv_get_error():
        clocks.stop()
        raise SystemExit("device error word set while timing %s" % wl.spec.name)
    return ms, launches, trace, clocks.stop(t_load0, t_load1)


PREFILL_SOURCES = ["paged_kv_attention_05_gb300/csrc/pkv_prefill.cu",
                   "paged_kv_attention_05_gb300/csrc/pkv_device.cuh",
                   "paged_kv_attention_05_gb300/csrc/pkv_internal.cuh",
                   "paged_kv_attention_05_gb300/csrc/pkv_combine.cuh"]


def kernel_sources(kind, int8):
    if kind == "prefill":
        return PREFILL_SOURCES
    kfile = "decode_i8" if (int8 and kind == "decode") else kind
    return ["paged_kv_attention_05_gb300/csrc/pkv_%s.cu" % kfile,
            "paged_kv_attention_05_gb300/csrc/pkv_device.cuh",
            "paged_kv_attention_05_gb300/csrc/pkv_internal.cuh"]


def write_bytes(spec, int8):
    """Algorithmic bytes of one cache-write launch: the new K and V rows read
    (bf16) and stored (bf16, or int8 codes)."""
    return 2 * spec.num_tokens * spec.hkv * spec.head_size * (2 + (1 if int8 else 2))


def rooflines(spec, trace, int8, peaks):
    """(dominant kernel's roofline, the cache write's roofline, the whole
    step's floor), from the live per-launch durations."""
    d = spec.head_size
    kinds = {k: v for k, v in trace.items() if v[1] > 0}
    dominant = max(kinds, key=lambda k: kinds[k][0]) if kinds else "decode"
    dom_ms, dom_n = trace.get(dominant, (0.0, 0))
    avg_ms = dom_ms / max(dom_n, 1)
    if dominant == "prefill":
        algo = causal_flops(spec)
        peak = peaks.get("bf16_tflops")
        roof = {"bound": "tensor", "achieved": algo / (avg_ms / 1e3) / 1e12,
                "peak": peak, "unit": "TFLOP/s", "peak_source": "measured" if peak else None}
    else:
        algo = decode_algorithmic_bytes(spec, 1 if int8 else 2) if dominant == "decode" else \
            write_bytes(spec, int8) if dominant == "write" else 0
        peak = peaks.get("hbm_gbs")
        roof = {"bound": "hbm", "achieved": algo / (avg_ms / 1e3) / 1e9,
                "peak": peak, "unit": "GB/s", "peak_source": "measured" if peak else None}
    if roof["peak"] is None:
        roof["peak"] = 1900.0 if roof["unit"] == "TFLOP/s" else 6800.0
        roof["peak_source"] = "fallback"
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dominant
    roof["avg_launch_ms"] = avg_ms
    roof["traffic"] = profiled_traffic(dominant, spec.name + ("_int8" if int8 else ""),
                                       kernel_sources(dominant, int8))
    bw = peaks.get("hbm_gbs") or 6800.0
    tf = peaks.get("bf16_tflops") or 1900.0
    w_ms, w_n = trace.get("write", (0.0, 0))
    wroof = None
    if w_n:
        w_avg = w_ms / w_n
        wb = write_bytes(spec, int8)
        wroof = {"bound": "hbm", "bytes": wb, "avg_launch_ms": w_avg,
                 "achieved": wb / (w_avg / 1e3) / 1e9, "peak": bw, "unit": "GB/s",
                 "frac": wb / (w_avg / 1e3) / 1e9 / bw,
                 "traffic": profiled_traffic("write", spec.name + ("_int8" if int8 else ""),
                                             kernel_sources("write", int8))}
    # the whole step against its own floor: max(bytes / copy bandwidth,
    # flops / bf16 peak), both algorithmic
    sb, sf = step_bytes(spec, 1 if int8 else 2), causal_flops(spec)
    floor_ms = max(sb / (bw * 1e9), sf / (tf * 1e12)) * 1e3
    step_roof = {"bytes": sb, "flops": sf, "floor_ms": floor_ms,
                 "bound": "hbm" if sb / (bw * 1e9) >= sf / (tf * 1e12) else "tensor"}
    return roof, wroof, step_roof


def metric_value(spec, int8, world, ms_per_step):
    name, unit = metric_of(spec)
    work = metric_work(spec)
    if int8:  # one byte per cached element instead of two
        name, work = name + " (int8 cache)", work / 2
    return name, unit, work, whole_job_value(work, world, ms_per_step / 1e3)


EXTRA_CONFIGS = [("large_prefill", "bf16"), ("mixed_chunked", "bf16"), ("gqa_decode", "bf16"),
                 ("mqa_long_decode", "bf16"), ("tiny_mixed", "bf16"), ("mha_decode", "int8"),
                 ("gqa_decode", "int8"), ("mqa_long_decode", "int8")]


def measure_extra(name, kv_dtype, args, peaks):
    """One extra workload, measured as the headline is (same timing, trace
    and clock rules) without the end-to-end and CPU-baseline legs."""
    import torch
    spec = W.spec(name)
    int8 = kv_dtype == "int8"
    wl = Workload(spec, int8=int8)
    ms, launches, trace, clk = time_steps(wl, args.steps, args.warmup)
    del wl
    torch.cuda.empty_cache()
    ms_per_step = ms / args.steps
    metric, unit, _, value = metric_value(spec, int8, 1, ms_per_step)
    roof, wroof, step_roof = rooflines(spec, trace, int8, peaks)
    step_roof["frac"] = step_roof["floor_ms"] / ms_per_step
    return {"metric": metric, "value": value, "unit": unit, "ms_per_step": ms_per_step,
            "dtype": "int8 cache, fp16 math" if int8 else "bf16",
            "config": config_of(spec, kv_dtype, False, 1), "gpu_launches": int(launches),
            "kernel_ms": {k: v[0] / max(v[1], 1) for k, v in trace.items() if v[1]},
            "roofline": roof, "write_roofline": wroof, "step_roofline": step_roof,
            "clocks": clk}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mha_decode", choices=W.CONFIG_NAMES)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip the other workloads (extra_configs of the line)")
    ap.add_argument("--with-prepare", action="store_true",
                    help="start each step with pkv_prepare_step (positions, seq_lens, slot "
                         "mapping and block table computed on the device)")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "int8"],
                    help="int8: the step writes and reads an int8 KV cache (one scale per "
                         "cache; decode workloads only)")
    ap.add_argument("--reqs", type=int, default=0,
                    help="first N requests of the workload only, with a pool sized for them "
                         "(a small case of the same kernel shapes, e.g. for profiling)")
    args = ap.parse_args()
    launch_check(args)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    spec = W.spec(args.config)
    if args.reqs:
        spec = W.subset(spec, args.reqs)
    int8 = args.kv_dtype == "int8"
    if int8 and any(n != 1 for n in spec.q_len):
        raise SystemExit("--kv-dtype int8 runs decode workloads only (mha_decode, gqa_decode, "
                         "mqa_long_decode)")
    if args.impl == "reference":
        run_reference(args, spec, rank)
        return

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = json.load(open(peaks_path)) if os.path.exists(peaks_path) else {}
    wl = Workload(spec, int8=int8, with_prepare=args.with_prepare)
    pkv, step, s, d = wl.pkv, wl.step, spec, spec.head_size
    ms, launches, trace, clk = time_steps(wl, args.steps, args.warmup, dist)
    ms = max_over_ranks(ms, dist, "cuda")
    ms_per_step = ms / args.steps
    name, unit, work, value = metric_value(spec, int8, world, ms_per_step)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # end to end through the public API with host buffers, as a serving loop
    # runs it: every step's inputs (fused qkv and metadata) copied in from
    # pinned host memory and its output copied back, double-buffered on two
    # copy streams so that step i+1's upload and step i-1's download overlap
    # step i's kernels (which run on the compute stream in step order, so the
    # shared cache sees each write before the next step's attention)
    e2e = None
    if not args.no_e2e:
        rows, stream = wl.rows, wl.stream
        KS, VS = wl.KS, wl.VS
        h_qkv = torch.from_numpy(step.qkv.view(np.int16)).pin_memory()
        h_slots = torch.from_numpy(step.slot_mapping).pin_memory()
        h_qsl = torch.from_numpy(step.query_start_loc).pin_memory()
        h_sl = torch.from_numpy(step.seq_lens).pin_memory()
        h_bt = torch.from_numpy(step.block_table).pin_memory()
        h_out = [torch.empty((rows, s.hq, d), dtype=torch.bfloat16).pin_memory()
                 for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in (h_qkv, h_slots, h_qsl, h_sl, h_bt))
        d2h = h_out[0].numel() * h_out[0].element_size()
        sets = []
        for _ in range(2):
            b_qkv = torch.empty_like(wl.qkv)
            sets.append({"qkv": b_qkv,
                         "q": b_qkv[:, :s.hq * d].view(rows, s.hq, d),
                         "k": b_qkv[:, s.hq * d:(s.hq + s.hkv) * d].view(rows, s.hkv, d),
                         "v": b_qkv[:, (s.hq + s.hkv) * d:].view(rows, s.hkv, d),
                         "slots": torch.empty_like(wl.slot_mapping),
                         "qsl": torch.empty_like(wl.qsl),
                         "sl": torch.empty_like(wl.seq_lens),
                         "bt": torch.empty_like(wl.block_table),
                         "out": torch.empty_like(wl.outs[0])})
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev = {n: [torch.cuda.Event() for _ in range(2)]
              for n in ("in_ready", "in_free", "out_ready", "out_free")}

        def upload(i):
            b, j = sets[i % 2], i % 2
            up.wait_event(ev["in_free"][j])  # step i-2 is done with these buffers
            with torch.cuda.stream(up):
                b["qkv"].view(torch.int16).copy_(h_qkv, non_blocking=True)
                b["slots"].copy_(h_slots, non_blocking=True)
                b["qsl"].copy_(h_qsl, non_blocking=True)
                b["sl"].copy_(h_sl, non_blocking=True)
                b["bt"].copy_(h_bt, non_blocking=True)
                ev["in_ready"][j].record(up)

        def compute(i):
            b, j = sets[i % 2], i % 2
            kc, vc = wl.caches[i % wl.n_copies]
            stream.wait_event(ev["in_ready"][j])
            stream.wait_event(ev["out_free"][j])  # step i-2's output is read back
            if int8:
                pkv.pkv_write_int8(b["k"], b["v"], kc, vc, b["slots"], KS, VS, stream=stream)
                pkv.pkv_attention_int8(b["q"], kc, vc, KS, VS, b["qsl"], b["sl"], b["bt"],
                                       s.num_reqs, s.scale, b["out"], stream=stream)
            else:
                pkv.pkv_write(b["k"], b["v"], kc, vc, b["slots"], stream=stream)
                pkv.pkv_attention(b["q"], kc, vc, b["qsl"], b["sl"], b["bt"],
                                  s.num_reqs, s.scale, b["out"], stream=stream)
            ev["in_free"][j].record(stream)
            ev["out_ready"][j].record(stream)

        def download(i):
            b, j = sets[i % 2], i % 2
            down.wait_event(ev["out_ready"][j])
            with torch.cuda.stream(down):
                h_out[j].copy_(b["out"], non_blocking=True)
                ev["out_free"][j].record(down)

        def run_e2e(n):
            upload(0)
            for i in range(n):
                if i + 1 < n:
                    upload(i + 1)
                compute(i)
                download(i)

        run_e2e(3)
        barrier()
        t0 = time.perf_counter()
        run_e2e(args.steps)
        barrier()
        e2e_s = (time.perf_counter() - t0) / args.steps
        e2e_s = max_over_ranks(e2e_s, dist, "cuda")
        e2e = {"value": work * world / e2e_s, "unit": unit,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_s * 1e3,
               "overlap": "double-buffered: step i+1's upload and step i-1's download on "
                          "copy streams during step i's kernels"}
        if pkv.pkv_get_error():
            raise SystemExit("device error word set in the end-to-end loop")

    roof, wroof, step_roof = rooflines(spec, trace, int8, peaks)
    step_roof["frac"] = step_roof["floor_ms"] / ms_per_step
    rec = {"metric": name, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None,
           "dtype": "int8 cache, fp16 math" if int8 else "bf16", "data": "synthetic",
           "config": config_of(spec, args.kv_dtype, args.with_prepare, world),
           "clocks": clk, "e2e": e2e, "gpu_launches": int(launches),
           "kernel_ms": {k: v[0] / max(v[1], 1) for k, v in trace.items() if v[1]},
           "kernel_timing": "CUDA events around each launch, in a second pass of the same K "
                            "steps right after the timed one (which records none)",
           "roofline": roof, "write_roofline": wroof, "step_roofline": step_roof}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not int8:
        rec["cpu_baseline"] = cpu_baseline_bounded(step)
    # the other workloads, each timed as the headline is (one GPU only: the
    # scaling runs carry the headline alone)
    if world == 1 and not args.no_extra_configs and not args.reqs:
        del wl, step
        torch.cuda.empty_cache()
        extra = {}
        for nm, kvd in EXTRA_CONFIGS:
            if nm == spec.name and kvd == args.kv_dtype:
                continue
            extra[nm if kvd == "bf16" else nm + "_int8"] = measure_extra(nm, kvd, args, peaks)
        rec["extra_configs"] = extra
    if rank == 0:
        print(json.dumps(rec))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
