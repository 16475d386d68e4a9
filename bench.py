#!/usr/bin/env python
"""Benchmark of single-query paged decode attention on one GB300 per rank.

One step = one call of the C ABI's pa_decode_v2 over a whole synthetic decode
batch (paged K/V gather, scores, online softmax per partition, cross-partition
combine, output).  Headline workload (default ``--config``): ``d256_fp16``,
the largest of the five benchmark configurations by bytes moved (256
sequences, 16 heads, head_size 256, block_size 16, lengths U[1, 2048],
partition_size 512).  The same JSON line carries ``per_config``: every one of
the five configurations (tiny_fp16, mha_fp16, gqa_bf16, long_skew_bf16,
d256_fp16) timed the same way.

Timing: after warm-up, K = ``--steps`` calls are timed with CUDA events on the
launching stream, bracketed by a barrier and a device synchronise on both
sides.  Short regions are repeated (each repetition K calls, bracketed the
same way) until the repetitions cover ``--min-seconds`` of GPU time; the
median repetition is reported.  Pools larger than L2 need no flush; a pool
smaller than L2 (tiny_fp16) is timed call by call with an L2-sized write
between calls, outside the events.

Prints one JSON line (rank 0):
  value      achieved HBM GB/s = algorithmic bytes of all ranks / max-over-ranks
             time of the K timed calls (inputs resident in HBM);
  e2e        the same metric through pa_decode_v2_host_io with the per-step
             inputs (query, block tables, sequence lengths) copied from pinned
             host memory and the output copied back, inside the timed region;
             the KV cache stays device-resident (it is the cache);
  roofline   achieved GB/s of one call (algorithmic bytes over the median
             call duration, CUDA events: the phase-1 kernel, which moves all
             the algorithmic bytes, plus the phase-2 combine and the header
             clear) against the measured HBM peak;
  per_config the five benchmark configurations, each with the same fields;
  cpu_baseline  the fp64 oracle on a bounded sample, on the host cores.
``--impl reference`` times that oracle alone (the CPU reference arm).
Multi-GPU: one process per GPU (torchrun); every rank decodes its own batch
(independent replicas, no collective on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
import dataclasses
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from decode_attention_paged_pa_gb300 import workloads  # noqa: E402

METRIC = "paged decode attention achieved HBM GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
HEADLINE = "d256_fp16"
BASE_CONFIGS = list(workloads.WORKLOAD_ORDER)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--config", choices=list(workloads.WORKLOADS), default=HEADLINE)
    ap.add_argument("--variant", choices=["auto", "simt", "mma"], default="auto")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the K-step timed region until it covers this much GPU time")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --config (no per_config block)")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="--impl reference: host seconds for all warm-up and timed steps together")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--seqs", type=int, default=0,
                    help="use only this many sequences of the workload (smaller case for profiling)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "decode_attention_paged_pa_gb300", "csrc", "*")))
    for p in files:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_file(config: str) -> str:
    return os.path.join(ROOT, "profiles", f"pa_decode_kernel_{config}.txt")


def profile_traffic(config: str):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel sources (else None)."""
    try:
        fields = {}
        with open(profile_file(config)) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_hash") != kernel_source_hash() or fields.get("workload") != config:
            return None
        return int(float(fields["dram_bytes_per_launch"]))
    except Exception:
        return None


def _hex(s: str) -> str:
    return "".join(c for c in str(s).lower() if c in "0123456789abcdef")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (every 100 ms) while running.

    Queries every GPU nvidia-smi sees (read-only) and keeps the rows of this
    process's device, matched by UUID (or the only GPU listed)."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.lines = []
        self.err = []
        self.threads = []
        try:
            self.uuid = _hex(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.uuid = ""

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
        except Exception as e:  # no nvidia-smi
            self.proc = None
            self.err.append(str(e))
            return
        for stream, sink in ((self.proc.stdout, self.lines), (self.proc.stderr, self.err)):
            t = threading.Thread(target=self._read, args=(stream, sink), daemon=True)
            t.start()
            self.threads.append(t)

    @staticmethod
    def _read(stream, sink):
        for line in stream:
            sink.append(line.strip())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            for t in self.threads:
                t.join(timeout=5)
        out = summarize_clocks(self.lines, self.uuid)
        if not out["samples"] and self.err:
            out["error"] = self.err[0][:200]
        return out


def summarize_clocks(lines, uuid: str) -> dict:
    """Median SM clock, maximum clock and the throttle reasons seen, from
    nvidia-smi CSV rows (ClockSampler.FIELDS), keeping the rows of GPU
    ``uuid`` (or of the only GPU listed)."""
    rows = [[p.strip() for p in line.split(",")] for line in lines]
    rows = [r for r in rows if len(r) >= 9]
    uuids = {_hex(r[0]) for r in rows}
    if uuid and _hex(uuid) in uuids:
        rows = [r for r in rows if _hex(r[0]) == _hex(uuid)]
    elif len(uuids) > 1:  # cannot tell which GPU is ours: report nothing rather than a wrong one
        rows = []
    sm, smax, reasons = [], [], set()
    for r in rows:
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
        except ValueError:
            continue
        for name, val in zip(ClockSampler.REASONS, r[5:9]):
            if val.lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


def sample_workload(w: workloads.Workload, seconds: float) -> workloads.Workload:
    """The first n sequences of ``w`` (same shapes and distributions), n the
    whole batch unless one fp64 oracle pass over it would take longer than
    ``seconds`` on this host (cost per token measured on a few sequences)."""
    import oracle

    def sample_of(n):
        n = max(1, min(n, w.num_seqs))
        forced = tuple((i, v) for i, v in w.forced_lens if i < n)
        lens = w.lens if w.lens_random else w.lens[:n]
        return dataclasses.replace(w, num_seqs=n, num_blocks=n * w.max_blocks_per_seq, lens=lens,
                                   forced_lens=forced, distinct_tables=False)

    probe = sample_of(min(w.num_seqs, 8))
    pin = workloads.make_inputs(probe)
    t0 = time.perf_counter()
    oracle_call(oracle, probe, pin)
    per_token = (time.perf_counter() - t0) / max(1, workloads.kv_tokens(pin["seq_lens"].tolist()))
    mean_len = (sum(w.lens) / 2.0) if w.lens_random else (sum(w.lens) / len(w.lens))
    return sample_of(max(1, int(seconds / max(per_token * mean_len * max(1, w.q_len), 1e-12))))


def oracle_sample(w: workloads.Workload, cpu_seconds: float):
    """Time the fp64 oracle on this host's cores on a bounded sample of
    workload ``w`` (:func:`sample_workload`), passed over repeatedly until
    ``cpu_seconds`` have gone by."""
    import oracle

    ws = sample_workload(w, cpu_seconds)
    inp = workloads.make_inputs(ws)
    lens = inp["seq_lens"].tolist()
    passes = 0
    t0 = time.perf_counter()
    while True:
        oracle_call(oracle, ws, inp)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= cpu_seconds or passes >= 10000:
            break
    nbytes = workloads.algorithmic_bytes(ws, lens) * passes
    return {
        "seconds": dt,
        "bytes": nbytes,
        "tokens": sum(lens) * passes,
        "gbs": nbytes / dt / 1e9,
        "cores": oracle.max_threads(),
        "sample": f"{ws.num_seqs} of {w.num_seqs} sequences of {w.name} (all {w.num_heads} heads, "
                  f"{sum(lens)} tokens) x {passes} passes in {dt:.1f} s, fp64 oracle",
        "workload": ws,
    }


def oracle_call(oracle, w: workloads.Workload, inp):
    """One oracle pass over a batch (multi-query batches through decode_mq, fp8
    caches through decode_fp8kv, fp32 through decode_fp32)."""
    if w.kv_dtype == "e4m3":
        return oracle.decode_fp8kv(inp["query"], inp["key_cache"], inp["value_cache"], inp["block_tables"],
                                   inp["seq_lens"], inp["scale"], w.k_scale, w.v_scale,
                                   workloads.DTYPE_CODES[w.dtype])
    if w.dtype == "fp32":
        return oracle.decode_fp32(inp["query"], inp["key_cache"], inp["value_cache"], inp["block_tables"],
                                  inp["seq_lens"], inp["scale"])
    args = (inp["query"], inp["key_cache"], inp["value_cache"], inp["block_tables"], inp["seq_lens"],
            inp["scale"], workloads.DTYPE_CODES[w.dtype])
    return oracle.decode_mq(*args) if w.q_len > 1 else oracle.decode(*args)


def expected_lens(w: workloads.Workload):
    """The workload's sequence lengths (drawn from its seeded CPU generator)."""
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    return workloads.draw_seq_lens(w, gen).tolist()


def config_of(w: workloads.Workload, world: int, variant: str, lens=None) -> dict:
    """The ``config`` object of a JSON line: the workload, by what it is."""
    lens = expected_lens(w) if lens is None else lens
    pool = 2 * w.num_blocks * w.num_kv_heads * w.head_size * w.block_size * (
        1 if w.kv_dtype == "e4m3" else workloads.DTYPES[w.dtype].itemsize)
    flush = (f"no flush: KV pool {pool / 1e9:.2f} GB per rank > L2 {L2_BYTES / 1e6:.0f} MB" if pool > L2_BYTES
             else f"L2 flushed between timed calls ({2 * L2_BYTES / 1e6:.0f} MB write): "
                  f"KV pool {pool / 1e6:.1f} MB < L2")
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
            "num_kv_heads": w.num_kv_heads, "head_size": w.head_size,
            "block_size": w.block_size, "partition_size": w.partition_size,
            "seq_lens": f"{min(lens)}..{max(lens)} (sum {sum(lens)})", "accumulate": "fp32",
            "q_len": w.q_len, "kv_dtype": w.kv_dtype or w.dtype, "variant": variant,
            "parallelism": f"replicas x{world}", "l2": flush}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, rank):
    """CPU reference arm: the fp64 oracle as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle

    w = workloads.WORKLOADS[args.config]
    # Each step is a sample of the workload sized so that all warm-up and
    # timed steps together take about --ref-seconds of host time.
    per_step = min(2.0, args.cpu_seconds, args.ref_seconds / max(1, args.steps + args.warmup))
    ws = sample_workload(w, per_step)
    inp = workloads.make_inputs(ws)
    lens = inp["seq_lens"].tolist()
    nbytes = workloads.algorithmic_bytes(ws, lens)

    def step():
        oracle_call(oracle, ws, inp)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    sample = (f"{ws.num_seqs} of {w.num_seqs} sequences of {w.name} per step ({sum(lens)} tokens, "
              f"all {w.num_heads} heads), fp64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(w, args.gpus, args.variant),
        "kv_tokens_per_s": sum(lens) * args.steps / dt,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- native arm
def replica_workload(w: workloads.Workload, rank: int) -> workloads.Workload:
    """Rank r's own batch: the same shapes and distributions, seed + 100 r
    (replicas share nothing, so the multi-GPU path has no exchange)."""
    return dataclasses.replace(w, seed=w.seed + 100 * rank)


def aggregate_over_ranks(dist, device, nbytes: float, tokens: float, ms: float):
    """Whole-job totals of the replicas: bytes and tokens summed over ranks,
    time the maximum over ranks.  ``dist`` None means one process."""
    if dist is None:
        return float(nbytes), float(tokens), float(ms)
    sums = torch.tensor([float(nbytes), float(tokens)], dtype=torch.float64, device=device)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(sums, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(sums[0].item()), float(sums[1].item()), float(t.item())


def repetitions_needed(first_ms: float, min_seconds: float, cap: int = 2000) -> int:
    """Repetitions of a K-step region (the first took ``first_ms``) that cover
    ``min_seconds`` of GPU time: at least 1, at most ``cap``."""
    if first_ms <= 0:
        return 1
    return max(1, min(cap, int(-(-min_seconds * 1e3 // first_ms))))


class Timer:
    """Times K calls of ``step`` on ``stream``: one CUDA event pair around the K
    back-to-back calls (an event between calls would stand between one call's
    last kernel and the next call's first, which otherwise overlap through
    programmatic dependent launch; the per-call time is the pair's time over
    K), or, with ``flush``, an event pair around each call and an L2-sized
    write between calls outside them.  Every repetition is bracketed by a
    barrier and a device synchronise on both sides."""

    def __init__(self, dev, stream, dist, flush: bool):
        self.dev, self.stream, self.dist = dev, stream, dist
        self.scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def region(self, step, k: int):
        """GPU milliseconds of k calls (this rank) and the per-call times."""
        if self.dist:
            self.dist.barrier()
        torch.cuda.synchronize(self.dev)
        if self.scrub is None:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            for _ in range(k):
                step()
            b.record(self.stream)
            torch.cuda.synchronize(self.dev)
            total = a.elapsed_time(b)
            per = [total / k] * k
        else:
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(k)]
            for a, b in pairs:
                self.scrub.zero_()
                a.record(self.stream)
                step()
                b.record(self.stream)
            torch.cuda.synchronize(self.dev)
            per = [a.elapsed_time(b) for a, b in pairs]
            total = sum(per)
        if self.dist:
            self.dist.barrier()
        return total, per


def measure(w0: workloads.Workload, args, dev, dist, rank, world, variant_name: str, clocks=None):
    """Time one workload: device-resident value, per-launch roofline and e2e."""
    from decode_attention_paged_pa_gb300 import binding

    w = replica_workload(w0, rank)   # each rank: its own replica batch
    inp = workloads.make_inputs(w, device=dev)
    lens = inp["seq_lens"].tolist()
    nbytes = workloads.algorithmic_bytes(w, lens)
    tokens = workloads.kv_tokens(lens)
    pool = inp["key_cache"].numel() * inp["key_cache"].element_size() * 2
    variant = {"auto": binding.PA_VARIANT_AUTO, "simt": binding.PA_VARIANT_SIMT,
               "mma": binding.PA_VARIANT_MMA}[variant_name]
    out = torch.empty_like(inp["query"])
    rows = w.num_seqs * w.q_len
    wsb = binding.workspace_bytes(rows, w.num_heads, w.num_kv_heads, w.head_size,
                                  w.max_blocks_per_seq, w.block_size, w.partition_size)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = binding.launches_per_call(
        w.num_seqs, w.q_len, -(-w.max_blocks_per_seq * w.block_size // w.partition_size))

    def step():
        if w.kv_dtype == "e4m3":
            binding.pa_decode_v2_fp8(out, inp["query"], inp["key_cache"], inp["value_cache"],
                                     inp["block_tables"], inp["seq_lens"], inp["scale"], w.k_scale,
                                     w.v_scale, partition_size=w.partition_size, workspace=ws, stream=stream)
        elif w.q_len > 1:
            binding.pa_decode_v2_mq(out, inp["query"], inp["key_cache"], inp["value_cache"],
                                    inp["block_tables"], inp["seq_lens"], inp["scale"],
                                    partition_size=w.partition_size, workspace=ws, stream=stream)
        else:
            binding.pa_decode_v2(out, inp["query"], inp["key_cache"], inp["value_cache"],
                                 inp["block_tables"], inp["seq_lens"], inp["scale"],
                                 partition_size=w.partition_size, workspace=ws, stream=stream,
                                 variant=variant)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if binding.device_status(ws, stream) != binding.PA_OK:
        raise SystemExit(f"bench.py: device-side error during warm-up of {w.name}")

    timer = Timer(dev, stream, dist, flush=pool <= L2_BYTES)
    k = args.steps
    first, per = timer.region(step, k)
    reps = [first]
    per_call = list(per)
    n_more = repetitions_needed(first, args.min_seconds, cap=max(1, 20000 // k)) - 1
    if dist:  # every rank runs the same number of repetitions
        t = torch.tensor([n_more], dtype=torch.int64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        n_more = int(t.item())
    for _ in range(n_more):
        total, per = timer.region(step, k)
        reps.append(total)
        per_call.extend(per)
    if binding.device_status(ws, stream) != binding.PA_OK:
        raise SystemExit(f"bench.py: device-side error in the timed region of {w.name}")
    rep_ms = statistics.median(reps)
    job_bytes, job_tokens, ms = aggregate_over_ranks(dist, dev, nbytes, tokens, rep_ms)
    seconds = ms / 1e3
    value = job_bytes * k / seconds / 1e9
    call_ms = statistics.median(per_call)
    achieved = nbytes / (call_ms / 1e3) / 1e9
    peak, peak_src = measured_peak()
    res = {
        "value": value, "unit": "GB/s", "ms_per_step": ms / k, "steps": k,
        "repetitions": len(reps), "timed_calls": len(reps) * k,
        "rep_ms_min": min(reps), "rep_ms_max": max(reps),
        "kv_tokens_per_s": job_tokens * k / seconds,
        "pct_of_measured_peak": 100.0 * value / world / peak,
        "frac_of_nominal_8000": value / world / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profile_traffic(w0.name),
                     "peak_source": f"{peak_src} hbm_gbs (copy)",
                     "algorithmic_bytes_per_call": nbytes, "launches_per_call": launches_per_step,
                     "call_us_median": call_ms * 1e3,
                     "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS},
        "gpu_launches": len(reps) * k * launches_per_step,
        "config": config_of(w0, world, variant_name, lens if rank == 0 else None),
        "e2e": None,
    }

    # ---- e2e: per-step inputs from pinned host memory, output back to host
    if not args.no_e2e and w.q_len == 1 and not w.kv_dtype:
        q_h = inp["query"].cpu().pin_memory()
        bt_h = inp["block_tables"].cpu().pin_memory()
        lens_h = inp["seq_lens"].cpu().pin_memory()
        out_h = torch.empty_like(q_h).pin_memory()
        wsh = torch.empty(binding.host_io_workspace_bytes(
            w.num_seqs, w.num_heads, w.num_kv_heads, w.head_size, w.max_blocks_per_seq,
            w.block_size, w.partition_size), dtype=torch.uint8, device=dev)

        def step_host():
            binding.pa_decode_v2_host_io(out_h, q_h, inp["key_cache"], inp["value_cache"], bt_h,
                                         lens_h, inp["scale"], w.partition_size, wsh, stream)

        for _ in range(max(3, args.warmup)):
            step_host()
        torch.cuda.synchronize(dev)
        hreps = [timer.region(step_host, k)[0] for _ in range(len(reps))]
        _, _, e2e_ms = aggregate_over_ranks(dist, dev, nbytes, tokens, statistics.median(hreps))
        if not torch.equal(out_h, out.cpu()):
            raise SystemExit(f"bench.py: host-I/O result differs from the device-resident result ({w.name})")
        res["e2e"] = {"value": job_bytes * k / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                      "ms_per_step": e2e_ms / k,
                      "h2d_bytes_per_step": q_h.numel() * q_h.element_size() + bt_h.numel() * 4
                      + lens_h.numel() * 4,
                      "d2h_bytes_per_step": out_h.numel() * out_h.element_size()}
        res["gpu_launches"] += len(hreps) * k * launches_per_step
        del q_h, bt_h, lens_h, out_h, wsh
    del inp, out, ws, timer
    torch.cuda.empty_cache()
    return res


def run_native(args, rank, world, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the native arm runs only on the GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", rank=rank, world_size=world, device_id=dev)

    w0 = workloads.WORKLOADS[args.config]
    if args.seqs > 0:
        w0 = dataclasses.replace(w0, num_seqs=min(args.seqs, w0.num_seqs),
                                 num_blocks=min(args.seqs, w0.num_seqs) * w0.max_blocks_per_seq,
                                 lens=w0.lens if w0.lens_random else w0.lens[:args.seqs],
                                 forced_lens=tuple((i, v) for i, v in w0.forced_lens if i < args.seqs),
                                 distinct_tables=False, name=f"{w0.name}[:{args.seqs}]")
    names = [] if (args.no_per_config or args.seqs > 0) else list(BASE_CONFIGS)
    clocks = ClockSampler(local)
    clocks.start()
    head = measure(w0, args, dev, dist, rank, world, args.variant)
    per_config = {}
    for name in names:
        if name == w0.name and args.variant == "auto":
            per_config[name] = head
        else:
            per_config[name] = measure(workloads.WORKLOADS[name], args, dev, dist, rank, world, "auto")
    clk = clocks.stop()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cs = oracle_sample(w0, args.cpu_seconds)
        cpu = {"value": cs["gbs"], "unit": "GB/s", "cores": cs["cores"], "kind": "oracle",
               "sample": cs["sample"], "seconds": cs["seconds"]}
    slim = {}
    for name, r in per_config.items():
        slim[name] = {"value": r["value"], "unit": "GB/s", "ms_per_step": r["ms_per_step"],
                      "roofline_frac": r["roofline"]["frac"],
                      "frac_of_nominal_8000": r["frac_of_nominal_8000"],
                      "kv_tokens_per_s": r["kv_tokens_per_s"],
                      "call_us_median": r["roofline"]["call_us_median"],
                      "repetitions": r["repetitions"], "timed_calls": r["timed_calls"],
                      "e2e": r["e2e"], "config": r["config"]}
    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w0.dtype, "data": "synthetic",
        "config": dict(head["config"], timing=(
            f"median of {head['repetitions']} repetitions of {args.steps} calls "
            f"(>= {args.min_seconds:g} s of GPU time)")),
        "kv_tokens_per_s": head["kv_tokens_per_s"],
        "pct_of_measured_peak": head["pct_of_measured_peak"],
        "pct_of_nominal_8000": 100.0 * head["frac_of_nominal_8000"],
        "roofline": head["roofline"],
        "cpu_baseline": cpu,
        "e2e": head["e2e"],
        "gpu_launches": sum(r["gpu_launches"] for n, r in per_config.items() if r is not head)
        + head["gpu_launches"],
        "clocks": clk,
        "per_config": slim,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        run_native(args, rank, world, local)


if __name__ == "__main__":
    main()
