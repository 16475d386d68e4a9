#!/usr/bin/env python
"""Benchmark of single-query paged decode attention on one GB300 per rank.

One step = one call of the C ABI's pa_decode_v2 over a whole synthetic decode
batch (paged K/V gather, scores, online softmax per partition, cross-partition
combine, output).  Default workload: ``mha_fp16`` (64 sequences, 32 heads,
head_size 128, block_size 16, lengths U[512, 4096], partition_size 512).

Prints one JSON line (rank 0):
  value      achieved HBM GB/s = algorithmic bytes of all ranks / max-over-ranks
             time of the timed steps (inputs resident in HBM);
  e2e        the same metric through pa_decode_v2_host_io with the per-step
             inputs (query, block tables, sequence lengths) copied from pinned
             host memory and the output copied back, inside the timed region;
             the KV cache stays device-resident (it is the cache);
  roofline   the decode kernel's achieved GB/s against the measured HBM peak;
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
PROFILE_FILE = os.path.join(ROOT, "profiles", "pa_decode_kernel_mha_fp16.txt")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--config", choices=list(workloads.WORKLOADS), default="mha_fp16")
    ap.add_argument("--variant", choices=["auto", "simt", "mma"], default="auto")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="--impl reference: host seconds for all warm-up and timed steps together")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--seqs", type=int, default=0,
                    help="use only this many sequences of the workload (smaller case for profiling)")
    return ap.parse_args()


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


def profile_traffic(config: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources and this workload (else None)."""
    try:
        fields = {}
        with open(PROFILE_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_hash") != kernel_source_hash() or fields.get("workload") != config:
            return None
        return int(float(fields["dram_bytes_per_launch"]))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (every 100 ms) while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.lines = []
        self.thread = None

    def _gpu_id(self):
        try:
            u = torch.cuda.get_device_properties(self.device).uuid
            s = str(u)
            return s if s.startswith("GPU-") else "GPU-" + s
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            if vis:
                return vis.split(",")[self.device]
            return str(self.device)

    def start(self):
        cmd = ["nvidia-smi", "-i", self._gpu_id(), f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_sample(w: workloads.Workload, cpu_seconds: float):
    """Time the fp64 oracle on a bounded sample of workload ``w`` (same shapes
    and distributions, fewer sequences) on this host's cores."""
    import oracle

    def sample_of(n):
        n = max(1, min(n, w.num_seqs))
        forced = tuple((i, v) for i, v in w.forced_lens if i < n)
        lens = w.lens if w.lens_random else w.lens[:n]
        return dataclasses.replace(w, num_seqs=n, num_blocks=n * w.max_blocks_per_seq, lens=lens,
                                   forced_lens=forced, distinct_tables=False)

    def run(ws):
        inp = workloads.make_inputs(ws)
        t0 = time.perf_counter()
        oracle_call(oracle, ws, inp)
        dt = time.perf_counter() - t0
        return dt, inp["seq_lens"].tolist()

    probe = sample_of(1)
    dt1, lens1 = run(probe)
    per_token = dt1 / max(1, sum(lens1))
    mean_len = (sum(w.lens) / 2.0) if w.lens_random else (sum(w.lens) / len(w.lens))
    n = int(cpu_seconds / max(per_token * mean_len, 1e-9))
    ws = sample_of(max(1, n))
    dt, lens = run(ws)
    nbytes = workloads.algorithmic_bytes(ws, lens)
    return {
        "seconds": dt,
        "bytes": nbytes,
        "tokens": sum(lens),
        "gbs": nbytes / dt / 1e9,
        "cores": oracle.max_threads(),
        "sample": f"{ws.num_seqs} of {w.num_seqs} sequences of {w.name} (all {w.num_heads} heads, "
                  f"{sum(lens)} tokens), fp64 oracle",
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


# ----------------------------------------------------------------------------- arms
def run_reference(args, rank):
    """CPU reference arm: the fp64 oracle as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle

    w = workloads.WORKLOADS[args.config]
    # Each step is a sample of the workload sized so that all warm-up and
    # timed steps together take about --ref-seconds of host time.
    per_step = min(2.0, args.cpu_seconds, args.ref_seconds / max(1, args.steps + args.warmup))
    calib = oracle_sample(w, cpu_seconds=per_step)
    ws = calib["workload"]
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
    sample = f"{ws.num_seqs} of {w.num_seqs} sequences of {w.name} per step ({sum(lens)} tokens)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "sample": sample},
        "kv_tokens_per_s": sum(lens) * args.steps / dt,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


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


def run_native(args, rank, world, local):
    from decode_attention_paged_pa_gb300 import binding

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
    w = replica_workload(w0, rank)   # each rank: its own replica batch
    inp = workloads.make_inputs(w, device=dev)
    lens = inp["seq_lens"].tolist()
    nbytes = workloads.algorithmic_bytes(w, lens)
    tokens = workloads.kv_tokens(lens)
    kv_bytes = 2 * inp["key_cache"].numel() * inp["key_cache"].element_size()
    variant = {"auto": binding.PA_VARIANT_AUTO, "simt": binding.PA_VARIANT_SIMT,
               "mma": binding.PA_VARIANT_MMA}[args.variant]
    out = torch.empty_like(inp["query"])
    rows = w.num_seqs * w.q_len
    wsb = binding.workspace_bytes(rows, w.num_heads, w.num_kv_heads, w.head_size,
                                  w.max_blocks_per_seq, w.block_size, w.partition_size)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = binding.launches_per_call(w.num_seqs, w.q_len)

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
        raise SystemExit("bench.py: device-side error during warm-up")

    # ---- timed region: K steps, CUDA events on the launching stream
    events = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    events[0].record(stream)
    for k in range(args.steps):
        step()
        events[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if dist:
        dist.barrier()
    per_step_ms = [events[k].elapsed_time(events[k + 1]) for k in range(args.steps)]
    job_bytes, job_tokens, total_ms = aggregate_over_ranks(dist, dev, nbytes, tokens,
                                                           events[0].elapsed_time(events[-1]))
    seconds = total_ms / 1e3
    value = job_bytes * args.steps / seconds / 1e9

    # ---- e2e: per-step inputs from pinned host memory, output back to host
    e2e = None
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
        if dist:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step_host()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        _, _, e2e_ms = aggregate_over_ranks(dist, dev, nbytes, tokens, e0.elapsed_time(e1))
        if not torch.equal(out_h, out.cpu()):
            raise SystemExit("bench.py: host-I/O result differs from the device-resident result")
        e2e = {"value": job_bytes * args.steps / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": q_h.numel() * q_h.element_size() + bt_h.numel() * 4 + lens_h.numel() * 4,
               "d2h_bytes_per_step": out_h.numel() * out_h.element_size()}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peak, peak_src = measured_peak()
    launch_ms = statistics.mean(per_step_ms) / launches_per_step
    achieved = nbytes / launches_per_step / (launch_ms / 1e3) / 1e9
    traffic = profile_traffic(w.name)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": nbytes // launches_per_step,
                "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cs = oracle_sample(w0, args.cpu_seconds)
        cpu = {"value": cs["gbs"], "unit": "GB/s", "cores": cs["cores"], "kind": "oracle",
               "sample": cs["sample"], "seconds": cs["seconds"]}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
                   "num_kv_heads": w.num_kv_heads, "head_size": w.head_size,
                   "block_size": w.block_size, "partition_size": w.partition_size,
                   "seq_lens": f"{min(lens)}..{max(lens)} (sum {tokens})", "accumulate": "fp32",
                   "q_len": w.q_len, "kv_dtype": w.kv_dtype or w.dtype, "variant": args.variant, "parallelism": f"replicas x{world}",
                   "l2": f"no flush: KV pool {kv_bytes / 1e9:.2f} GB per rank > L2 {L2_BYTES / 1e6:.0f} MB"},
        "kv_tokens_per_s": job_tokens * args.steps / seconds,
        "pct_of_measured_peak": 100.0 * value / world / peak,
        "pct_of_nominal_8000": 100.0 * value / world / NOMINAL_HBM_GBS,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk,
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
