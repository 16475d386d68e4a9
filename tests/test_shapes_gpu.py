"""GPU parity of the tensor-core kernel family at the shapes beyond the
benchmark's (head sizes 80, 96, 112; 8- and 64-token blocks), through the C ABI,
against the fp64 oracle at the benchmark tolerance.  The page
"paged_attention_v2_triton.py -- Triton PagedAttention V2 for BI-V100" sizes its
key layout by x = 16 / sizeof(element) for any head size and block size; these
shapes use x = 8 like the others."""
import math

import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding
from pa_testutil import caches_from_tokens, random_case, token_views, within_tolerance
from test_lse_gpu import lse_close
from test_mq_gpu import mq_case, run_mq

pytestmark = pytest.mark.gpu

DT_CODE = {torch.float16: oracle.DTYPE_FP16, torch.bfloat16: oracle.DTYPE_BF16}
AUTO, SIMT, MMA = binding.PA_VARIANT_AUTO, binding.PA_VARIANT_SIMT, binding.PA_VARIANT_MMA


def run(q, kc, vc, bt, lens, scale, P, variant=AUTO, lse=False):
    dev = torch.device("cuda")
    qd, kd, vd, btd, ld = (t.to(dev) for t in (q, kc, vc, bt, lens))
    out = torch.full_like(qd, float("nan"))
    l = torch.full(q.shape[:2], float("nan"), device=dev) if lse else None
    ws = binding.pa_decode_v2(out, qd, kd, vd, btd.contiguous(), ld, scale, partition_size=P,
                              variant=variant, lse=l)
    st = binding.device_status(ws)
    assert st == binding.PA_OK, binding.status_string(st)
    return out.cpu(), (l.cpu() if lse else None)


NEW_D = [(dt, D, BS, G) for dt in (torch.float16, torch.bfloat16) for D in (80, 96, 112)
         for BS in (16, 32) for G in (1, 4, 8)]
NEW_BS = [(dt, D, BS, G) for dt in (torch.float16, torch.bfloat16) for D in (64, 80, 128, 256)
          for BS in (8, 64) for G in (1, 4)]


@pytest.mark.parametrize("dt,D,BS,G", NEW_D + NEW_BS,
                         ids=[f"{str(c[0])[6:]}-D{c[1]}-BS{c[2]}-G{c[3]}" for c in NEW_D + NEW_BS])
def test_parity_new_shapes(dt, D, BS, G):
    # Ragged ends inside a block, at a block edge, across partitions (P = 64)
    # and past 16 partitions (the two-level combine).
    P = 64
    lens = [1, BS - 1, BS + 1, 2 * P - 1, 3 * P + 5, 17 * P + 3]
    KH = 2
    q, kc, vc, bt, L = random_case(3000 + D + BS + G, S=len(lens), H=KH * G, KH=KH, D=D, BS=BS,
                                   lens=lens, dtype=dt)
    out, lse = run(q, kc, vc, bt, L, 1.0 / math.sqrt(D), P, lse=True)
    ref = oracle.decode(q, kc, vc, bt, L, 1.0 / math.sqrt(D), DT_CODE[dt])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), oracle.lse(q, kc, vc, bt, L, 1.0 / math.sqrt(D), DT_CODE[dt]))


SIMT_X = [(dt, D, BS, G, var) for dt in (torch.float16, torch.bfloat16)
          for D, BS in ((80, 16), (96, 32), (112, 64), (64, 64), (128, 64), (96, 64))
          for G in (1, 3) for var in (SIMT, MMA)]


@pytest.mark.parametrize("dt,D,BS,G,variant", SIMT_X,
                         ids=[f"{str(c[0])[6:]}-D{c[1]}-BS{c[2]}-G{c[3]}-{'simt' if c[4] == SIMT else 'mma'}"
                              for c in SIMT_X])
def test_parity_extra_shapes_both_families(dt, D, BS, G, variant):
    """Head sizes 80/96/112 and 64-token blocks on the CUDA-core family (head
    split in halves over lane pairs) and on the tensor cores."""
    P = 128
    lens = [1, BS - 1, BS + 1, 2 * P - 1, 17 * P + 3]
    q, kc, vc, bt, L = random_case(7000 + D + BS + G, S=len(lens), H=2 * G, KH=2, D=D, BS=BS, lens=lens,
                                   dtype=dt)
    out, _ = run(q, kc, vc, bt, L, 1.0 / math.sqrt(D), P, variant=variant)
    ref = oracle.decode(q, kc, vc, bt, L, 1.0 / math.sqrt(D), DT_CODE[dt])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"


@pytest.mark.parametrize("D,BS", [(80, 8), (112, 64), (256, 8), (64, 64)])
def test_garbage_past_end_new_shapes(D, BS):
    """NaN in every cache slot past each sequence's end (and in unused blocks)
    changes nothing: 8-token blocks read half a 16-token tile."""
    S, H, KH = 4, 8, 2
    lens = [3, BS, BS + 5, 200]
    q, kc, vc, bt, L = random_case(31 + D + BS, S=S, H=H, KH=KH, D=D, BS=BS, lens=lens)
    ref_out, _ = run(q, kc, vc, bt, L, 0.1, 64)
    k_tok, v_tok = token_views(kc, vc)
    k2, v2 = k_tok.clone(), v_tok.clone()
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
    for b in range(kc.shape[0]):
        if b not in used:
            k2[b] = float("nan")
            v2[b] = float("nan")
    kc2, vc2 = caches_from_tokens(k2, v2)
    out, _ = run(q, kc2, vc2, bt, L, 0.1, 64)
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out, ref_out)


@pytest.mark.parametrize("D,BS", [(96, 8), (80, 64), (112, 16)])
def test_multi_query_new_shapes(D, BS):
    q_len = 3
    lens = [q_len, 40, 129, 700]
    q, kc, vc, bt, L = mq_case(57 + D + BS, S=len(lens), q_len=q_len, H=8, KH=2, D=D, BS=BS, lens=lens,
                               dtype=torch.bfloat16)
    out, lse = run_mq(q, kc, vc, bt, L, 0.1, 64)
    ref, ref_lse = oracle.decode_mq(q, kc, vc, bt, L, 0.1, oracle.DTYPE_BF16)
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)


def test_deterministic_new_shapes():
    q, kc, vc, bt, L = random_case(71, S=6, H=16, KH=2, D=96, BS=8, lens=[5, 64, 300, 1100, 9, 2000])
    a, _ = run(q, kc, vc, bt, L, 0.1, 64)
    for _ in range(3):
        b, _ = run(q, kc, vc, bt, L, 0.1, 64)
        assert torch.equal(a, b)


WIDE = [(dt, D, BS, G) for dt in (torch.float16, torch.bfloat16) for D in (64, 128, 256)
        for BS in (16, 32) for G in (9, 16, 24)]


@pytest.mark.parametrize("dt,D,BS,G", WIDE, ids=[f"{str(c[0])[6:]}-D{c[1]}-BS{c[2]}-G{c[3]}" for c in WIDE])
def test_parity_wide_groups(dt, D, BS, G):
    """More than 8 query heads per kv head: units of 16 heads (the rows on the M
    side of the products; head size 256 keeps units of 8), partly filled when G
    is not a multiple of 16."""
    P = 64
    lens = [1, BS + 1, 2 * P - 1, 17 * P + 3]
    KH = 2
    q, kc, vc, bt, L = random_case(5000 + D + BS + G, S=len(lens), H=KH * G, KH=KH, D=D, BS=BS,
                                   lens=lens, dtype=dt)
    out, lse = run(q, kc, vc, bt, L, 1.0 / math.sqrt(D), P, lse=True)
    ref = oracle.decode(q, kc, vc, bt, L, 1.0 / math.sqrt(D), DT_CODE[dt])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), oracle.lse(q, kc, vc, bt, L, 1.0 / math.sqrt(D), DT_CODE[dt]))


@pytest.mark.parametrize("q_len,G", [(4, 4), (3, 4), (2, 8), (5, 4)])
def test_multi_query_wide_units(q_len, G):
    """q_len * G row heads per kv head above 8 share 16-row units."""
    lens = [q_len, 40, 129, 1500]
    q, kc, vc, bt, L = mq_case(91 + q_len + G, S=len(lens), q_len=q_len, H=2 * G, KH=2, D=128, BS=16,
                               lens=lens, dtype=torch.bfloat16)
    out, lse = run_mq(q, kc, vc, bt, L, 0.1, 64)
    ref, ref_lse = oracle.decode_mq(q, kc, vc, bt, L, 0.1, oracle.DTYPE_BF16)
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)


@pytest.mark.parametrize("D,BS", [(64, 16), (128, 32), (128, 16)])
def test_wide_units_ignore_garbage_past_the_end(D, BS):
    """NaN in every slot past each sequence's end and in unused blocks, under
    units of 16 query rows: the result is bitwise that of finite contents."""
    S, KH = 4, 2
    lens = [3, BS, BS + 5, 200]
    q, kc, vc, bt, L = random_case(131 + D + BS, S=S, H=16 * KH, KH=KH, D=D, BS=BS, lens=lens)
    ref_out, _ = run(q, kc, vc, bt, L, 0.1, 64)
    k_tok, v_tok = token_views(kc, vc)
    k2, v2 = k_tok.clone(), v_tok.clone()
    used = set()
    for s in range(S):
        for j in range(-(-lens[s] // BS)):
            b = int(bt[s, j])
            used.add(b)
            last = lens[s] - j * BS
            if last < BS:
                k2[b, last:] = float("nan")
                v2[b, last:] = float("nan")
    for b in range(kc.shape[0]):
        if b not in used:
            k2[b] = float("nan")
            v2[b] = float("nan")
    kc2, vc2 = caches_from_tokens(k2, v2)
    out, _ = run(q, kc2, vc2, bt, L, 0.1, 64)
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out, ref_out)


def test_wide_units_deterministic_across_grid_sizes():
    q, kc, vc, bt, L = random_case(97, S=4, H=32, KH=2, D=128, BS=16, lens=[5, 300, 2100, 64])
    dev = torch.device("cuda")
    outs = []
    for ctas in (0, 1, 13):
        out = torch.empty_like(q, device=dev)
        ws = binding.pa_decode_v2(out, q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), L.to(dev), 0.1,
                                  partition_size=64, max_ctas=ctas)
        assert binding.device_status(ws) == binding.PA_OK
        outs.append(out.cpu())
    assert all(torch.equal(outs[0], o) for o in outs[1:])
