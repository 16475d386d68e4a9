"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance for fp16/bf16 inputs: |out - ref| <= 2e-3 + 1e-2 |ref| elementwise.
Block-table indexing and partition bookkeeping are checked bit-exactly with
inputs whose exact answer is representable (needle, seq_len 1, sentinels,
placement permutation, determinism)."""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding, workloads
from pa_testutil import (caches_from_tokens, compact_sequences, random_case, token_views,
                         within_tolerance)

pytestmark = pytest.mark.gpu

DT_CODE = {torch.float16: oracle.DTYPE_FP16, torch.bfloat16: oracle.DTYPE_BF16}
SIMT, MMA = binding.PA_VARIANT_SIMT, binding.PA_VARIANT_MMA


def run_gpu(q, kc, vc, bt, lens, scale, P, variant=binding.PA_VARIANT_AUTO, max_ctas=0,
            expect_status=binding.PA_OK, num_blocks=None):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), kc.to(dev), vc.to(dev)
    btd, ld = bt.to(dev).contiguous(), lens.to(dev)
    out = torch.full_like(qd, float("nan"))
    ws = binding.pa_decode_v2(out, qd, kd, vd, btd, ld, scale, partition_size=P, variant=variant,
                              max_ctas=max_ctas)
    st = binding.device_status(ws)
    assert st == expect_status, binding.status_string(st)
    return out.cpu(), ws


def check_parity(q, kc, vc, bt, lens, scale, P, variant=binding.PA_VARIANT_AUTO, what=""):
    out, _ = run_gpu(q, kc, vc, bt, lens, scale, P, variant)
    ref = oracle.decode(q, kc, vc, bt, lens, scale, DT_CODE[q.dtype])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"{what}: worst excess {worst:.3e}"
    return out, ref


def test_tiny_workload_full_parity():
    inp = workloads.make_inputs(workloads.WORKLOADS["tiny_fp16"])
    w = inp["workload"]
    check_parity(inp["query"], inp["key_cache"], inp["value_cache"], inp["block_tables"],
                 inp["seq_lens"], inp["scale"], w.partition_size, what="tiny")


CASES = [(dt, D, BS, G, var)
         for dt in (torch.float16, torch.bfloat16)
         for D in (64, 128, 256)
         for BS in (16, 32)
         for G in (1, 2, 3, 4, 8)
         for var in (SIMT, MMA)]


@pytest.mark.parametrize("dt,D,BS,G,variant", CASES,
                         ids=[f"{str(c[0])[6:]}-D{c[1]}-BS{c[2]}-G{c[3]}-{'mma' if c[4] == MMA else 'simt'}"
                              for c in CASES])
def test_parity_small(dt, D, BS, G, variant):
    P = 64
    lens = [1, BS - 1, BS + 1, 2 * P - 1, 3 * P + 5]
    KH = 2
    q, kc, vc, bt, L = random_case(1000 + D + BS + G, S=len(lens), H=KH * G, KH=KH, D=D, BS=BS,
                                   lens=lens, dtype=dt)
    check_parity(q, kc, vc, bt, L, 1.0 / math.sqrt(D), P, variant, "small")


@pytest.mark.parametrize("P", [16, 32, 64, 512, 4096])
@pytest.mark.parametrize("variant", [SIMT, MMA])
def test_partition_size_invariance(P, variant):
    lens = [1, 700, 1500, 33, 512]
    q, kc, vc, bt, L = random_case(77, S=5, H=8, KH=2, D=128, BS=16, lens=lens, dtype=torch.bfloat16)
    check_parity(q, kc, vc, bt, L, 0.09, P, variant, f"P={P}")


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_long_sequences_two_level_combine(dt):
    """Sequences of 63-94 partitions with 8 query heads per kv head and
    head_size 256: combined per chunk of 16 partitions, then across chunks;
    both steps are large enough to be shared between the warps of a CTA."""
    lens = [1500, 700, 33, 1009]
    q, kc, vc, bt, L = random_case(78, S=4, H=16, KH=2, D=256, BS=16, lens=lens, dtype=dt)
    check_parity(q, kc, vc, bt, L, 1.0 / 16, 16, MMA, "two-level combine")
    check_parity(q, kc, vc, bt, L, 1.0 / 16, 16, SIMT, "two-level combine, SIMT")


@pytest.mark.parametrize("variant,G,BS", [(SIMT, 1, 16), (SIMT, 2, 32), (MMA, 4, 16), (MMA, 8, 32)])
def test_needle_bitexact(variant, G, BS):
    """q = 8 e_0, K[t*][0] = 200 and K[t][0] = 0 elsewhere: the weight of t* is
    exactly 1 and every other weight is exactly 0 in fp32, so out == V[t*]
    bitwise.  t* sweeps block and partition boundaries under a random table."""
    D, P, KH = 128, 64, 2
    L = 5 * P + 7
    q, kc, vc, bt, lens = random_case(5, S=1, H=KH * G, KH=KH, D=D, BS=BS, lens=[L])
    q.zero_()
    q[..., 0] = 8.0
    k_tok, v_tok = token_views(kc, vc)
    rng = np.random.default_rng(3)
    stars = sorted({0, BS - 1, BS, P - 1, P, P + 1, 2 * P + BS - 1, L - 2, L - 1,
                    *rng.integers(0, L, 6).tolist()})
    for t_star in stars:
        k2 = k_tok.clone()
        k2[..., 0] = 0.0
        b, o = int(bt[0, t_star // BS]), t_star % BS
        k2[b, o, :, 0] = 200.0
        kc2, _ = caches_from_tokens(k2, v_tok)
        out, _ = run_gpu(q, kc2, vc, bt, lens, 0.125, P, variant)
        for h in range(KH * G):
            want = v_tok[b, o, h // G]
            assert torch.equal(out[0, h], want), f"needle at {t_star}, head {h}"


@pytest.mark.parametrize("variant", [SIMT, MMA])
def test_seq_len_one_returns_v_bitexact(variant):
    q, kc, vc, bt, lens = random_case(8, S=6, H=8, KH=2, D=128, BS=16, lens=[1] * 6)
    out, _ = run_gpu(q, kc, vc, bt, lens, 0.1, 512, variant)
    _, v_tok = token_views(kc, vc)
    for s in range(6):
        for h in range(8):
            assert torch.equal(out[s, h], v_tok[int(bt[s, 0]), 0, h // 4])


@pytest.mark.parametrize("variant", [SIMT, MMA])
def test_placement_permutation_bitexact(variant):
    q, kc, vc, bt, lens = random_case(9, S=4, H=8, KH=2, D=128, BS=16, lens=[300, 1025, 17, 64],
                                      num_blocks=300, MB=65)
    perm = torch.randperm(300, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(300)
    a, _ = run_gpu(q, kc, vc, bt, lens, 0.1, 128, variant)
    b, _ = run_gpu(q, kc[perm].contiguous(), vc[perm].contiguous(), inv[bt.long()].to(torch.int32),
                   lens, 0.1, 128, variant)
    assert torch.equal(a, b)


@pytest.mark.parametrize("variant", [SIMT, MMA])
def test_deterministic_across_runs_and_grid_sizes(variant):
    q, kc, vc, bt, lens = random_case(10, S=9, H=16, KH=4, D=128, BS=16,
                                      lens=[4000, 1, 700, 2048, 513, 3000, 90, 1500, 2600])
    base, _ = run_gpu(q, kc, vc, bt, lens, 0.08, 256, variant)
    for ctas in (0, 1, 3, 17, 152):
        out, _ = run_gpu(q, kc, vc, bt, lens, 0.08, 256, variant, max_ctas=ctas)
        assert torch.equal(out, base), f"max_ctas={ctas}"


@pytest.mark.parametrize("variant,BS", [(SIMT, 16), (MMA, 16), (MMA, 32)])
def test_sequence_output_independent_of_batch(variant, BS):
    """Units run longest sequence first and each unit's work is split over the
    warps by its partition and head group only, so a sequence's output does
    not depend on the rest of the batch: each sequence decoded alone, and the
    batch in reverse order, give the batch's rows bit for bit."""
    lens = [700, 1, 3000, 513, 90, 2048, 0, 1500]
    q, kc, vc, bt, L = random_case(31, S=8, H=16, KH=4, D=128, BS=BS, lens=lens)
    base, _ = run_gpu(q, kc, vc, bt, L, 0.08, 256, variant)
    for s in range(len(lens)):
        one, _ = run_gpu(q[s:s + 1], kc, vc, bt[s:s + 1], L[s:s + 1], 0.08, 256, variant)
        assert torch.equal(one[0], base[s]), f"sequence {s} alone"
    rev = torch.arange(len(lens) - 1, -1, -1)
    r, _ = run_gpu(q[rev].contiguous(), kc, vc, bt[rev].contiguous(), L[rev].contiguous(), 0.08, 256, variant)
    assert torch.equal(r, base[rev])


@pytest.mark.parametrize("variant,KH,G,BS", [(SIMT, 16, 1, 16), (MMA, 16, 1, 16), (MMA, 8, 4, 32),
                                              (SIMT, 8, 1, 32)])
def test_repeatable_under_load(variant, KH, G, BS):
    """A busy batch (head_size 256, short and long sequences, many units per
    CTA) run 8 times: every output bit must repeat.  Consumer warps run at
    different speeds; a pipeline race would show up as run-to-run noise."""
    rng = np.random.default_rng(16)
    lens = rng.integers(1, 2049, 48).tolist()
    q, kc, vc, bt, L = random_case(16, S=48, H=KH * G, KH=KH, D=256, BS=BS, lens=lens)
    base, _ = run_gpu(q, kc, vc, bt, L, 1.0 / 16, 512, variant)
    ref = oracle.decode(q, kc, vc, bt, L, 1.0 / 16, oracle.DTYPE_FP16)
    assert within_tolerance(base.double().numpy(), ref)[0]
    for _ in range(7):
        out, _ = run_gpu(q, kc, vc, bt, L, 1.0 / 16, 512, variant)
        assert torch.equal(out, base)


@pytest.mark.parametrize("variant", [SIMT, MMA])
def test_partition_bookkeeping(variant):
    """Workspace after a call: exactly NP_s partitions per (s, h) hold finite
    m_p and l_p >= 1; unused ones hold m = -inf and l = +0.0 bitwise; m_p, l_p
    and (multi-partition) o_p match the oracle's phase-1 states."""
    S, H, KH, D, BS, P = 5, 8, 2, 128, 16, 128
    lens = [1, 129, 640, 0, 300]
    q, kc, vc, bt, L = random_case(12, S=S, H=H, KH=KH, D=D, BS=BS, lens=lens, MB=40)
    out, ws = run_gpu(q, kc, vc, bt, L, 0.1, P, variant)
    (om, ol, oo, _, _), pmax = binding.workspace_layout(S, H, KH, D, 40, BS, P)
    w = ws.cpu()
    m = w[om:om + S * H * pmax * 4].view(torch.float32).view(S, H, pmax).double().numpy()
    l = w[ol:ol + S * H * pmax * 4].view(torch.float32).view(S, H, pmax).double().numpy()
    o = w[oo:oo + S * H * pmax * D * 4].view(torch.float32).view(S, H, pmax, D).double().numpy()
    rm, rl, ro = oracle.partitions(q, kc, vc, bt, L, 0.1, oracle.DTYPE_FP16, P, pmax)
    for s in range(S):
        np_s = -(-lens[s] // P)
        assert np.all(np.isneginf(m[s, :, np_s:]))
        assert np.all(l[s, :, np_s:] == 0.0) and not np.any(np.signbit(l[s, :, np_s:]))
        assert np.all(np.isfinite(m[s, :, :np_s])) and np.all(l[s, :, :np_s] >= 1.0)
        assert np.allclose(m[s, :, :np_s], rm[s, :, :np_s], rtol=1e-4, atol=1e-4)
        assert np.allclose(l[s, :, :np_s], rl[s, :, :np_s], rtol=2e-3, atol=0)
        if np_s > 1:
            ok, worst = within_tolerance(o[s, :, :np_s], ro[s, :, :np_s])
            assert ok, worst
    assert torch.all(out[3] == 0)


@pytest.mark.parametrize("variant", [SIMT, MMA])
def test_empty_and_garbage_past_end(variant):
    """seq_len 0 gives zeros; NaN in cache slots past each sequence's end and
    -1 in table entries past ceil(L/BS) change nothing and flag nothing."""
    S, H, KH, D, BS = 4, 8, 2, 128, 16
    lens = [0, 37, 5, 16]
    q, kc, vc, bt, L = random_case(13, S=S, H=H, KH=KH, D=D, BS=BS, lens=lens, MB=4)
    ref_out, _ = run_gpu(q, kc, vc, bt, L, 0.1, 512, variant)
    k_tok, v_tok = token_views(kc, vc)
    k2, v2 = k_tok.clone(), v_tok.clone()
    bt2 = bt.clone()
    used = set()
    for s in range(S):
        nb = -(-lens[s] // BS)
        for j in range(nb):
            b = int(bt[s, j])
            used.add(b)
            last = lens[s] - j * BS
            if last < BS:
                k2[b, last:] = float("nan")
                v2[b, last:] = float("nan")
        bt2[s, nb:] = -1
    for b in range(kc.shape[0]):
        if b not in used:
            k2[b] = float("nan")
            v2[b] = float("nan")
    kc2, vc2 = caches_from_tokens(k2, v2)
    out, _ = run_gpu(q, kc2, vc2, bt2, L, 0.1, 512, variant)
    assert torch.all(out[0] == 0)
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out, ref_out)
    ref = oracle.decode(q, kc, vc, bt, L, 0.1, oracle.DTYPE_FP16)
    assert within_tolerance(out.double().numpy(), ref)[0]


def test_bad_block_id_and_length_are_flagged():
    q, kc, vc, bt, lens = random_case(14, S=2, H=4, KH=4, D=64, BS=16, lens=[40, 20], MB=3)
    bad = bt.clone()
    bad[0, 1] = kc.shape[0]          # one past the pool
    run_gpu(q, kc, vc, bad, lens, 0.1, 512, expect_status=binding.PA_ERR_DEVICE_BOUNDS)
    long = lens.clone()
    long[1] = 3 * 16 + 1             # more tokens than the table row can hold
    run_gpu(q, kc, vc, bt, long, 0.1, 512, expect_status=binding.PA_ERR_DEVICE_BOUNDS)


@pytest.mark.parametrize("variant", [SIMT, MMA], ids=["simt", "mma"])
def test_batch_split_across_launches(variant):
    """More sequences than one launch takes (binding.MAX_ROWS_PER_LAUNCH): the
    batch is split into launches that share the workspace.  Every sequence
    matches the oracle, including multi-partition ones on both sides of each
    split and an empty last sequence."""
    g = torch.Generator().manual_seed(21)
    S = 2100
    lens = torch.randint(1, 700, (S,), generator=g).tolist()
    for k in range(binding.MAX_ROWS_PER_LAUNCH, S, binding.MAX_ROWS_PER_LAUNCH):
        lens[k - 1] = lens[k] = 1500
    lens[S - 1] = 0
    H, KH = (4, 4) if variant == SIMT else (8, 2)
    q, kc, vc, bt, L = random_case(22, S=S, H=H, KH=KH, D=64, BS=16, lens=lens, num_blocks=4096)
    check_parity(q, kc, vc, bt, L, 0.125, 256, variant, what=f"{S} sequences")


@pytest.mark.parametrize("S", [2000, 2100], ids=["rows-2000", "per-sequence-2100"])
def test_many_sequences_with_long_tables(S):
    """More than 16 partitions in the table: up to 2048 sequences the combine
    runs as persistent row groups (each sequence's warps per row from its own
    partition count, the row-group prefix over all sequences in shared
    memory), past that as a grid over sequences.  Both match the oracle."""
    g = torch.Generator().manual_seed(23 + S)
    lens = torch.randint(1, 300, (S,), generator=g).tolist()
    for k in range(0, S, 97):
        lens[k] = 1500  # 24 partitions of 64
    lens[S - 1] = 0
    q, kc, vc, bt, L = random_case(24, S=S, H=8, KH=2, D=64, BS=16, lens=lens, num_blocks=4096)
    check_parity(q, kc, vc, bt, L, 0.125, 64, MMA, what=f"{S} sequences, P = 64")


def test_more_than_1024_partitions():
    """600,000 tokens at P = 512 is 1172 partitions; all of them are combined."""
    L, BS, D = 600_000, 16, 64
    MB = L // BS
    g = torch.Generator().manual_seed(15)
    nb = 64
    q = torch.randn((1, 2, D), generator=g).half()
    kc = torch.randn((nb, 1, D // 8, BS, 8), generator=g).half()
    vc = torch.randn((nb, 1, D, BS), generator=g).half()
    bt = torch.randint(0, nb, (1, MB), generator=g, dtype=torch.int32)
    lens = torch.tensor([L], dtype=torch.int32)
    check_parity(q, kc, vc, bt, lens, 0.125, 512, what="1172 partitions")


def test_poisoned_workspace_two_level_combine():
    """The workspace's contents on entry do not matter.  It is filled with 0x7f
    bytes (3.4e38 as f32) before each of 20 calls on the long-context
    batch (one sequence of 131072 tokens = 256 partitions, combined in 16
    chunks of 16, eight heads per group): a partition or chunk state read
    before this call wrote it shows up as a wrong or non-finite output, or as
    a difference between calls (as does a ring stage refilled under reads
    still in flight, which corrupts single accumulator tiles)."""
    w = workloads.WORKLOADS["long_skew_bf16"]
    inp = workloads.make_inputs(w, device="cuda")
    need = binding.workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_size,
                                   w.max_blocks_per_seq, w.block_size, w.partition_size)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(20):
        ws.fill_(0x7F)
        out = torch.full_like(inp["query"], float("nan"))
        binding.pa_decode_v2(out, inp["query"], inp["key_cache"], inp["value_cache"], inp["block_tables"],
                             inp["seq_lens"], inp["scale"], partition_size=w.partition_size, workspace=ws)
        assert binding.device_status(ws) == binding.PA_OK
        assert torch.isfinite(out.float()).all()
        outs.append(out)
    for i, o in enumerate(outs[1:], 1):
        assert torch.equal(o, outs[0]), f"call {i} differs from call 0"
    seqs = [0, 1]   # 256 and 32 partitions: both combined in two levels
    sub = compact_sequences(inp, seqs)
    ref = oracle.decode(*sub, inp["scale"], workloads.DTYPE_CODES[w.dtype])
    ok, worst = within_tolerance(outs[0][torch.tensor(seqs, device="cuda")].cpu().double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    del inp, outs, ws
    torch.cuda.empty_cache()
