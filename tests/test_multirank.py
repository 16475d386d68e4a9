"""The multi-GPU path of the bench on CPU: two gloo ranks (no GPU needed).

Replicas share nothing, so the only cross-rank step is the bench's own
bookkeeping: each rank draws its own batch (seed + 100 * rank) and the job's
totals are the bytes and tokens summed over ranks over the slowest rank's
time."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from decode_attention_paged_pa_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        w = bench.replica_workload(workloads.WORKLOADS["tiny_fp16"], rank)
        inp = workloads.make_inputs(w)
        lens = inp["seq_lens"].tolist()
        nbytes = workloads.algorithmic_bytes(w, lens)
        tokens = workloads.kv_tokens(lens)
        ms = 10.0 + 5.0 * rank            # the slower rank sets the job's time
        got = bench.aggregate_over_ranks(dist, torch.device("cpu"), nbytes, tokens, ms)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{nbytes} {tokens} {ms} {got[0]} {got[1]} {got[2]} {w.seed} {sum(lens)}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_replicas(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    rows = [list(map(float, open(tmp_path / f"rank{r}.txt").read().split())) for r in range(world)]
    total_bytes = sum(r[0] for r in rows)
    total_tokens = sum(r[1] for r in rows)
    for r in rows:
        assert r[3] == total_bytes and r[4] == total_tokens and r[5] == 15.0
    # Each rank decodes its own batch: different seeds, different lengths.
    assert rows[0][6] != rows[1][6] and rows[0][7] != rows[1][7]


def test_one_process_needs_no_collective():
    bench = _bench()
    assert bench.aggregate_over_ranks(None, None, 100, 7, 2.5) == (100.0, 7.0, 2.5)
    w = workloads.WORKLOADS["mha_fp16"]
    assert bench.replica_workload(w, 0) == w
