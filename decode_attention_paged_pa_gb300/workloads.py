"""Seeded synthetic inputs for paged decode attention, and their byte accounting.

This module holds no attention arithmetic: it draws random queries, key/value
caches, block tables and sequence lengths in the layouts of the page
"paged_attention_v2_triton.py -- Triton PagedAttention V2 for BI-V100" (phase-1
kernel argument comments), and it counts the bytes a call must move.  Both the
CUDA path's tests/bench and the fp64 oracle consume what it makes.

Layouts:
    query        [S, H, D]
    key_cache    [num_blocks, KH, D/x, BS, x]   x = 16 / sizeof(dtype): 8 (fp16/bf16), 4 (fp32)
    value_cache  [num_blocks, KH, D, BS]
    block_tables [S, MB] int32
    seq_lens     [S] int32
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

X_PACK = 8  # 16 bytes / sizeof(fp16 or bf16)

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}
DTYPE_CODES = {"fp16": 0, "bf16": 1, "fp32": 2}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode batch.  ``lens`` is either an explicit tuple or a
    (low, high) pair meaning ``randint(low, high + 1)`` per sequence."""

    name: str
    dtype: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    partition_size: int
    scale: float
    max_blocks_per_seq: int
    num_blocks: int
    lens: tuple
    lens_random: bool
    forced_lens: tuple = ()          # (index, value) pairs applied after drawing
    k_std: float = 1.0
    v_uniform: bool = False          # V ~ U(-1, 1) instead of N(0, 1)
    distinct_tables: bool = False    # per-seq randperm(num_blocks)[:MB] instead of one pool permutation
    seed: int = 0
    q_len: int = 1                   # query rows per sequence (multi-query decode when > 1)
    kv_dtype: str = ""               # "e4m3": fp8 caches (codes, key x = 16), else the query's dtype
    k_scale: float = 1.0             # fp8 caches: real keys / values are k_scale * K, v_scale * V
    v_scale: float = 1.0

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads


def _cfg(**kw) -> Workload:
    return Workload(**kw)


# The five configurations of the benchmark definition (seed = 1000 + index).
WORKLOADS: dict[str, Workload] = {
    "tiny_fp16": _cfg(
        name="tiny_fp16", dtype="fp16", num_seqs=4, num_heads=4, num_kv_heads=4, head_size=64,
        block_size=16, partition_size=512, scale=1.0 / 8.0, max_blocks_per_seq=19,
        num_blocks=128, lens=(1, 300), lens_random=True, distinct_tables=True, seed=1000),
    "mha_fp16": _cfg(
        name="mha_fp16", dtype="fp16", num_seqs=64, num_heads=32, num_kv_heads=32, head_size=128,
        block_size=16, partition_size=512, scale=1.0 / math.sqrt(128), max_blocks_per_seq=256,
        num_blocks=64 * 256, lens=(512, 4096), lens_random=True, seed=1001),
    "gqa_bf16": _cfg(
        name="gqa_bf16", dtype="bf16", num_seqs=128, num_heads=32, num_kv_heads=8, head_size=128,
        block_size=16, partition_size=512, scale=1.0 / math.sqrt(128), max_blocks_per_seq=512,
        num_blocks=128 * 512, lens=(2048, 8192), lens_random=True, seed=1002),
    "long_skew_bf16": _cfg(
        name="long_skew_bf16", dtype="bf16", num_seqs=8, num_heads=64, num_kv_heads=8, head_size=128,
        block_size=32, partition_size=512, scale=1.0 / math.sqrt(128), max_blocks_per_seq=4096,
        num_blocks=8 * 4096, lens=(131072, 16384, 8192, 4096, 2048, 1024, 1000, 17),
        lens_random=False, seed=1003),
    "d256_fp16": _cfg(
        name="d256_fp16", dtype="fp16", num_seqs=256, num_heads=16, num_kv_heads=16, head_size=256,
        block_size=16, partition_size=512, scale=1.0 / 16.0, max_blocks_per_seq=128,
        num_blocks=256 * 128, lens=(1, 2048), lens_random=True,
        forced_lens=((0, 1), (1, 2048), (2, 17)), k_std=2.0, v_uniform=True, seed=1004),
}
WORKLOAD_ORDER = ["tiny_fp16", "mha_fp16", "gqa_bf16", "long_skew_bf16", "d256_fp16"]

# Multi-query decode (speculative verification of 4 draft tokens) on the GQA
# batch's shapes and lengths: query [S, 4, H, D], each row causal.
WORKLOADS["spec4_gqa_bf16"] = _cfg(
    name="spec4_gqa_bf16", dtype="bf16", num_seqs=128, num_heads=32, num_kv_heads=8, head_size=128,
    block_size=16, partition_size=512, scale=1.0 / math.sqrt(128), max_blocks_per_seq=512,
    num_blocks=128 * 512, lens=(2048, 8192), lens_random=True, seed=1002, q_len=4)
# The GQA batch over an fp8 (E4M3) KV cache with per-tensor scales.
WORKLOADS["gqa_fp8kv_bf16"] = _cfg(
    name="gqa_fp8kv_bf16", dtype="bf16", num_seqs=128, num_heads=32, num_kv_heads=8, head_size=128,
    block_size=16, partition_size=512, scale=1.0 / math.sqrt(128), max_blocks_per_seq=512,
    num_blocks=128 * 512, lens=(2048, 8192), lens_random=True, seed=1002, kv_dtype="e4m3",
    k_scale=0.5, v_scale=1.5)
# Shapes beyond the benchmark definition's (head sizes 80 / 96 / 112, blocks
# of 8 or 64 tokens): the GQA batch's lengths with head size 112 in 8-token
# blocks, and the MHA batch's with head size 80 in 64-token blocks.
WORKLOADS["gqa_d112_bs8_bf16"] = _cfg(
    name="gqa_d112_bs8_bf16", dtype="bf16", num_seqs=128, num_heads=32, num_kv_heads=8, head_size=112,
    block_size=8, partition_size=512, scale=1.0 / math.sqrt(112), max_blocks_per_seq=1024,
    num_blocks=128 * 1024, lens=(2048, 8192), lens_random=True, seed=1005)
WORKLOADS["mha_d80_bs64_fp16"] = _cfg(
    name="mha_d80_bs64_fp16", dtype="fp16", num_seqs=64, num_heads=32, num_kv_heads=32, head_size=80,
    block_size=64, partition_size=512, scale=1.0 / math.sqrt(80), max_blocks_per_seq=64,
    num_blocks=64 * 64, lens=(512, 4096), lens_random=True, seed=1006)
# The MHA batch in fp32 (query, caches and output; key layout x = 4).
WORKLOADS["mha_fp32"] = _cfg(
    name="mha_fp32", dtype="fp32", num_seqs=64, num_heads=32, num_kv_heads=32, head_size=128,
    block_size=16, partition_size=512, scale=1.0 / math.sqrt(128), max_blocks_per_seq=256,
    num_blocks=64 * 256, lens=(512, 4096), lens_random=True, seed=1001)
# The same on the MHA batch's shapes: 4 row heads per kv head, one unit each.
WORKLOADS["spec4_mha_fp16"] = _cfg(
    name="spec4_mha_fp16", dtype="fp16", num_seqs=64, num_heads=32, num_kv_heads=32, head_size=128,
    block_size=16, partition_size=512, scale=1.0 / math.sqrt(128), max_blocks_per_seq=256,
    num_blocks=64 * 256, lens=(512, 4096), lens_random=True, seed=1001, q_len=4)


def custom(name="custom", dtype="fp16", num_seqs=2, num_heads=4, num_kv_heads=4, head_size=64,
           block_size=16, partition_size=512, scale=None, lens=(1, 64), lens_random=True,
           max_blocks_per_seq=None, num_blocks=None, k_std=1.0, v_uniform=False,
           distinct_tables=False, seed=0, forced_lens=()) -> Workload:
    """A workload of arbitrary shape (for parity and edge-case tests)."""
    if scale is None:
        scale = 1.0 / math.sqrt(head_size)
    max_len = max(lens) if lens else 0
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, -(-max_len // block_size))
    if num_blocks is None:
        num_blocks = num_seqs * max_blocks_per_seq
    return Workload(name=name, dtype=dtype, num_seqs=num_seqs, num_heads=num_heads,
                    num_kv_heads=num_kv_heads, head_size=head_size, block_size=block_size,
                    partition_size=partition_size, scale=float(scale),
                    max_blocks_per_seq=max_blocks_per_seq, num_blocks=num_blocks,
                    lens=tuple(lens), lens_random=lens_random, forced_lens=tuple(forced_lens),
                    k_std=k_std, v_uniform=v_uniform, distinct_tables=distinct_tables, seed=seed)


def draw_seq_lens(w: Workload, gen: torch.Generator) -> torch.Tensor:
    if w.lens_random:
        lo, hi = w.lens
        lens = torch.randint(lo, hi + 1, (w.num_seqs,), generator=gen, dtype=torch.int64)
    else:
        lens = torch.tensor(w.lens, dtype=torch.int64)
    for i, v in w.forced_lens:
        lens[i] = v
    return lens.to(torch.int32)


def draw_block_tables(w: Workload, gen: torch.Generator) -> torch.Tensor:
    S, MB, NB = w.num_seqs, w.max_blocks_per_seq, w.num_blocks
    if w.distinct_tables:
        rows = [torch.randperm(NB, generator=gen)[:MB] for _ in range(S)]
        return torch.stack(rows).to(torch.int32)
    if NB >= S * MB:
        return torch.randperm(NB, generator=gen)[: S * MB].view(S, MB).to(torch.int32)
    # smaller pool than S*MB: blocks repeat across sequences, distinct within one
    rows = [torch.randperm(NB, generator=gen)[:MB] for _ in range(S)]
    return torch.stack(rows).to(torch.int32)


def make_inputs(w: Workload, device: str | torch.device = "cpu",
                value_device: Optional[str | torch.device] = None) -> dict:
    """Draw one batch.  Table/lengths always come from a CPU generator (identical on
    every machine); the float tensors are drawn on ``value_device`` (default:
    ``device``) by a generator seeded with the workload's seed, then moved to
    ``device``."""
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    seq_lens = draw_seq_lens(w, gen)
    block_tables = draw_block_tables(w, gen)
    vdev = torch.device(value_device if value_device is not None else device)
    vgen = torch.Generator(device=vdev).manual_seed(w.seed + 7919)
    dt = DTYPES[w.dtype]
    S, H, KH, D, BS, NB = (w.num_seqs, w.num_heads, w.num_kv_heads, w.head_size,
                           w.block_size, w.num_blocks)
    qshape = (S, H, D) if w.q_len == 1 else (S, w.q_len, H, D)
    query = torch.randn(qshape, generator=vgen, device=vdev, dtype=torch.float32).to(dt)
    if w.kv_dtype == "e4m3":
        # E4M3 codes of N(0, k_std) / N(0, 1) draws (rounded by torch), key x = 16.
        def codes(shape, std):
            t = torch.empty(shape, device=vdev, dtype=torch.float32).normal_(0.0, std, generator=vgen)
            return t.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        key_cache = codes((NB, KH, D // 16, BS, 16), w.k_std)
        value_cache = codes((NB, KH, D, BS), 1.0)
    else:
        x = 16 // torch.empty((), dtype=dt).element_size()
        key_cache = torch.empty((NB, KH, D // x, BS, x), device=vdev, dtype=dt)
        key_cache.normal_(0.0, w.k_std, generator=vgen)
        value_cache = torch.empty((NB, KH, D, BS), device=vdev, dtype=dt)
        if w.v_uniform:
            value_cache.uniform_(-1.0, 1.0, generator=vgen)
        else:
            value_cache.normal_(0.0, 1.0, generator=vgen)
    dev = torch.device(device)
    return {
        "query": query.to(dev), "key_cache": key_cache.to(dev), "value_cache": value_cache.to(dev),
        "block_tables": block_tables.to(dev), "seq_lens": seq_lens.to(dev),
        "scale": float(w.scale), "workload": w,
    }


def algorithmic_bytes(w: Workload, seq_lens: Sequence[int]) -> int:
    """Bytes one call must move: K and V of every token once per kv head (all
    query heads of a group, and all query rows of a multi-query sequence, share
    them), q in, out, the block-table entries that cover the tokens, and
    seq_lens.  Workspace traffic is not counted."""
    esz = DTYPES[w.dtype].itemsize
    kv_esz = 1 if w.kv_dtype == "e4m3" else esz
    lens = [int(v) for v in seq_lens]
    kv = sum(lens) * w.num_kv_heads * w.head_size * 2 * kv_esz
    q_out = 2 * w.num_seqs * w.q_len * w.num_heads * w.head_size * esz
    tables = 4 * sum(-(-L // w.block_size) for L in lens)
    return kv + q_out + tables + 4 * w.num_seqs


def kv_tokens(seq_lens: Sequence[int]) -> int:
    return sum(int(v) for v in seq_lens)
