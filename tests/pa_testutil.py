"""Helpers shared by the tests: token-major views of the paged caches, a
numpy textbook attention, golden-file readers and the parity tolerance.

None of this is used by the CUDA library or by the oracle.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Elementwise parity bar for fp16/bf16 inputs against the fp64 oracle.
ATOL = 2e-3
RTOL = 1e-2


def within_tolerance(out, ref, atol=ATOL, rtol=RTOL):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(out - ref)
    bound = atol + rtol * np.abs(ref)
    ok = bool(np.all(err <= bound))
    worst = float(np.max(err - bound)) if err.size else 0.0
    return ok, worst


def token_views(key_cache: torch.Tensor, value_cache: torch.Tensor):
    """Token-major views of the pools, [num_blocks, BS, KH, D], obtained by
    permuting the cache tensors' axes:
    key_cache [nb, KH, D/x, BS, x] -> [nb, BS, KH, D/x, x] -> [nb, BS, KH, D];
    value_cache [nb, KH, D, BS] -> [nb, BS, KH, D]."""
    nb, KH, dx, BS, x = key_cache.shape
    k_tok = key_cache.permute(0, 3, 1, 2, 4).reshape(nb, BS, KH, dx * x)
    v_tok = value_cache.permute(0, 3, 1, 2)
    return k_tok, v_tok


def caches_from_tokens(k_tok: torch.Tensor, v_tok: torch.Tensor):
    """Inverse of :func:`token_views`: build the paged caches from token-major pools."""
    nb, BS, KH, D = k_tok.shape
    key_cache = k_tok.reshape(nb, BS, KH, D // 8, 8).permute(0, 2, 3, 1, 4).contiguous()
    value_cache = v_tok.permute(0, 2, 3, 1).contiguous()
    return key_cache, value_cache


def gather_sequence(key_cache, value_cache, block_tables, s: int, L: int):
    """K, V of sequence s as [L, KH, D] float64 numpy arrays (torch indexing)."""
    k_tok, v_tok = token_views(key_cache, value_cache)
    BS = key_cache.shape[3]
    t = torch.arange(L)
    b = block_tables[s].long()[t // BS]
    o = t % BS
    return (k_tok[b, o].to(torch.float64).numpy(), v_tok[b, o].to(torch.float64).numpy())


def textbook_decode(query, key_cache, value_cache, block_tables, seq_lens, scale):
    """softmax(scale * q K^T) V per (s, h) with numpy fp64; the kv head of query
    head h is found by repeating each kv head's K/V G times consecutively."""
    S, H, D = query.shape
    KH = key_cache.shape[1]
    G = H // KH
    out = np.zeros((S, H, D))
    q64 = query.to(torch.float64).numpy()
    sc = float(np.float32(scale))
    for s in range(S):
        L = int(seq_lens[s])
        if L == 0:
            continue
        K, V = gather_sequence(key_cache, value_cache, block_tables, s, L)
        K = np.repeat(K, G, axis=1)  # [L, H, D]
        V = np.repeat(V, G, axis=1)
        for h in range(H):
            z = sc * (K[:, h, :] @ q64[s, h])
            w = np.exp(z - z.max())
            w /= w.sum()
            out[s, h] = w @ V[:, h, :]
    return out


def read_golden(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def random_case(seed, S, H, KH, D, BS, lens, dtype=torch.float16, MB=None, num_blocks=None,
                k_std=1.0):
    """Small random inputs on the CPU with a random physical placement."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.tensor(lens, dtype=torch.int32)
    if MB is None:
        MB = max(1, math.ceil(max(int(v) for v in lens) / BS)) if len(lens) else 1
    if num_blocks is None:
        num_blocks = S * MB
    q = torch.randn((S, H, D), generator=g).to(dtype)
    kc = (torch.randn((num_blocks, KH, D // 8, BS, 8), generator=g) * k_std).to(dtype)
    vc = torch.randn((num_blocks, KH, D, BS), generator=g).to(dtype)
    if num_blocks >= S * MB:
        bt = torch.randperm(num_blocks, generator=g)[: S * MB].view(S, MB).to(torch.int32)
    else:
        bt = torch.stack([torch.randperm(num_blocks, generator=g)[:MB] for _ in range(S)]).to(torch.int32)
    return q, kc, vc, bt, lens


def compact_sequences(inputs: dict, seqs):
    """Inputs restricted to sequences ``seqs``: the physical blocks they use are
    copied into a compact pool (CPU) and their tables renumbered.  Plain data
    movement, so the oracle can check sampled outputs of a full-size batch."""
    q, kc, vc = inputs["query"], inputs["key_cache"], inputs["value_cache"]
    bt, lens = inputs["block_tables"], inputs["seq_lens"]
    BS = kc.shape[3]
    seqs = [int(s) for s in seqs]
    lens_cpu = lens.cpu()
    bt_cpu = bt.cpu()
    used = []
    for s in seqs:
        nb = -(-int(lens_cpu[s]) // BS)
        used.append(bt_cpu[s, :nb].long())
    allb = torch.unique(torch.cat(used)) if used else torch.zeros(0, dtype=torch.long)
    remap = {int(b): i for i, b in enumerate(allb.tolist())}
    MB = max(1, max((u.numel() for u in used), default=1))
    bt_sub = torch.zeros((len(seqs), MB), dtype=torch.int32)
    for i, u in enumerate(used):
        if u.numel():
            bt_sub[i, : u.numel()] = torch.tensor([remap[int(b)] for b in u.tolist()], dtype=torch.int32)
    idx = allb.to(kc.device)
    kc_sub = kc.index_select(0, idx).cpu() if allb.numel() else kc[:1].cpu()
    vc_sub = vc.index_select(0, idx).cpu() if allb.numel() else vc[:1].cpu()
    q_sub = q[torch.tensor(seqs, device=q.device)].cpu()
    lens_sub = lens_cpu[seqs].clone()
    return q_sub, kc_sub, vc_sub, bt_sub, lens_sub


def fp8_caches_from_tokens(k_tok: torch.Tensor, v_tok: torch.Tensor):
    """E4M3 code caches from token-major uint8 pools [nb, BS, KH, D]: key_cache
    [nb, KH, D/16, BS, 16] (x = 16 one-byte elements per 16-byte chunk) and
    value_cache [nb, KH, D, BS], by permuting axes."""
    nb, BS, KH, D = k_tok.shape
    key_cache = k_tok.reshape(nb, BS, KH, D // 16, 16).permute(0, 2, 3, 1, 4).contiguous()
    value_cache = v_tok.permute(0, 2, 3, 1).contiguous()
    return key_cache, value_cache


def fp8_random_case(seed, S, H, KH, D, BS, lens, qdtype=torch.float16, MB=None, num_blocks=None):
    """Random inputs with E4M3 code caches (values drawn from N(0, 1), rounded to
    E4M3 by torch; no NaN codes) and a random physical placement."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.tensor(lens, dtype=torch.int32)
    if MB is None:
        MB = max(1, math.ceil(max(int(v) for v in lens) / BS)) if len(lens) else 1
    if num_blocks is None:
        num_blocks = S * MB
    q = torch.randn((S, H, D), generator=g).to(qdtype)
    to_codes = lambda t: t.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    k_tok = to_codes(torch.randn((num_blocks, BS, KH, D), generator=g))
    v_tok = to_codes(torch.randn((num_blocks, BS, KH, D), generator=g))
    kc, vc = fp8_caches_from_tokens(k_tok, v_tok)
    if num_blocks >= S * MB:
        bt = torch.randperm(num_blocks, generator=g)[: S * MB].view(S, MB).to(torch.int32)
    else:
        bt = torch.stack([torch.randperm(num_blocks, generator=g)[:MB] for _ in range(S)]).to(torch.int32)
    return q, kc, vc, bt, lens


def f32_caches_from_tokens(k_tok: torch.Tensor, v_tok: torch.Tensor):
    """fp32 caches from token-major pools [nb, BS, KH, D]: key_cache
    [nb, KH, D/4, BS, 4] (x = 4 four-byte elements per 16-byte chunk) and
    value_cache [nb, KH, D, BS], by permuting axes."""
    nb, BS, KH, D = k_tok.shape
    key_cache = k_tok.reshape(nb, BS, KH, D // 4, 4).permute(0, 2, 3, 1, 4).contiguous()
    value_cache = v_tok.permute(0, 2, 3, 1).contiguous()
    return key_cache, value_cache


def f32_random_case(seed, S, H, KH, D, BS, lens, MB=None, num_blocks=None):
    """Random fp32 inputs (N(0, 1)) in the x = 4 layout with a random physical placement."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.tensor(lens, dtype=torch.int32)
    if MB is None:
        MB = max(1, math.ceil(max(int(v) for v in lens) / BS)) if len(lens) else 1
    if num_blocks is None:
        num_blocks = S * MB
    q = torch.randn((S, H, D), generator=g)
    kc, vc = f32_caches_from_tokens(torch.randn((num_blocks, BS, KH, D), generator=g),
                                    torch.randn((num_blocks, BS, KH, D), generator=g))
    if num_blocks >= S * MB:
        bt = torch.randperm(num_blocks, generator=g)[: S * MB].view(S, MB).to(torch.int32)
    else:
        bt = torch.stack([torch.randperm(num_blocks, generator=g)[:MB] for _ in range(S)]).to(torch.int32)
    return q, kc, vc, bt, lens
