"""GPU parity of decode with fp32 query, caches and output (key layout x = 4,
16 / sizeof(float) as the page "paged_attention_v2_triton.py -- Triton
PagedAttention V2 for BI-V100" sizes it), through the C ABI, against the fp64
oracle's decode_fp32.

Tolerance, from the arithmetic: every operand is an exact fp32 value, scores
are fp32 dot products of at most 256 terms, weights are fp32 exp2 of fp32
differences and the accumulators fp32, so each output is the weighted mean of
V with weights off by a few units of 2^-24 times |score|; bounded here by
|out - ref| <= 1e-5 + 1e-4 |ref| (two orders of magnitude under the 16-bit
tolerance), and the log-sum-exp by 1e-4 + 1e-5 |ref|."""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding
from pa_testutil import f32_caches_from_tokens, f32_random_case, token_views, within_tolerance
from test_lse_gpu import lse_close

pytestmark = pytest.mark.gpu

ATOL32, RTOL32 = 1e-5, 1e-4


def run(q, kc, vc, bt, lens, scale, P, variant=binding.PA_VARIANT_AUTO, lse=False, max_ctas=0):
    dev = torch.device("cuda")
    qd, kd, vd, btd, ld = (t.to(dev) for t in (q, kc, vc, bt, lens))
    out = torch.full_like(qd, float("nan"))
    l = torch.full(q.shape[:2], float("nan"), device=dev) if lse else None
    ws = binding.pa_decode_v2(out, qd, kd, vd, btd.contiguous(), ld, scale, partition_size=P,
                              variant=variant, lse=l, max_ctas=max_ctas)
    st = binding.device_status(ws)
    assert st == binding.PA_OK, binding.status_string(st)
    return out.cpu(), (l.cpu() if lse else None)


CASES = [(D, BS, G) for D in (64, 128, 256) for BS in (16, 32) for G in (1, 4)]


@pytest.mark.parametrize("D,BS,G", CASES, ids=[f"D{c[0]}-BS{c[1]}-G{c[2]}" for c in CASES])
def test_fp32_parity(D, BS, G):
    P = 64
    lens = [1, BS - 1, BS + 1, 2 * P - 1, 3 * P + 5, 17 * P + 3, 0]
    KH = 2
    q, kc, vc, bt, L = f32_random_case(4000 + D + BS + G, S=len(lens), H=KH * G, KH=KH, D=D, BS=BS, lens=lens)
    out, lse = run(q, kc, vc, bt, L, 1.0 / math.sqrt(D), P, lse=True)
    ref, ref_lse = oracle.decode_fp32(q, kc, vc, bt, L, 1.0 / math.sqrt(D))
    ok, worst = within_tolerance(out.double().numpy(), ref, ATOL32, RTOL32)
    assert ok, f"worst excess {worst:.3e}"
    assert torch.all(out[-1] == 0)
    lse_close(lse.numpy(), ref_lse)


def test_fp32_long_sequence_and_grid_sizes():
    """131 partitions (two-level combine), bitwise the same for every grid size."""
    q, kc, vc, bt, L = f32_random_case(4101, S=3, H=4, KH=4, D=128, BS=16, lens=[8400, 33, 2000])
    base, _ = run(q, kc, vc, bt, L, 0.088, 64)
    ref, _ = oracle.decode_fp32(q, kc, vc, bt, L, 0.088)
    assert within_tolerance(base.double().numpy(), ref, ATOL32, RTOL32)[0]
    for ctas in (1, 7, 152):
        out, _ = run(q, kc, vc, bt, L, 0.088, 64, max_ctas=ctas)
        assert torch.equal(out, base), ctas


def test_fp32_garbage_past_end():
    """NaN in cache slots past each sequence's end changes nothing."""
    BS = 16
    lens = [3, 16, 21, 200]
    q, kc, vc, bt, L = f32_random_case(4111, S=4, H=4, KH=2, D=64, BS=BS, lens=lens)
    a, _ = run(q, kc, vc, bt, L, 0.1, 64)
    k_tok, v_tok = token_views(kc, vc)
    k2, v2 = k_tok.clone(), v_tok.clone()
    for s in range(4):
        nb = -(-lens[s] // BS)
        last = lens[s] - (nb - 1) * BS
        b = int(bt[s, nb - 1])
        if last < BS:
            k2[b, last:] = float("nan")
            v2[b, last:] = float("nan")
    kc2, vc2 = f32_caches_from_tokens(k2, v2)
    b_, _ = run(q, kc2, vc2, bt, L, 0.1, 64)
    assert torch.isfinite(b_).all() and torch.equal(a, b_)


def test_fp32_host_io_matches_device_call():
    q, kc, vc, bt, L = f32_random_case(4121, S=5, H=8, KH=8, D=128, BS=32, lens=[40, 900, 1, 77, 513])
    a, _ = run(q, kc, vc, bt, L, 0.09, 512)
    dev = torch.device("cuda")
    need = binding.host_io_workspace_bytes(5, 8, 8, 128, bt.shape[1], 32, 512)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out_h = torch.empty_like(q).pin_memory()
    binding.pa_decode_v2_host_io(out_h, q.pin_memory(), kc.to(dev), vc.to(dev), bt.contiguous().pin_memory(),
                                 L.pin_memory(), 0.09, 512, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h, a)


def test_fp32_rejected_outside_its_family():
    q, kc, vc, bt, L = f32_random_case(4131, S=2, H=4, KH=2, D=128, BS=16, lens=[5, 9])
    dev = torch.device("cuda")
    out = torch.empty_like(q, device=dev)
    with pytest.raises(binding.PaError) as e:
        binding.pa_decode_v2(out, q.to(dev), kc.to(dev), vc.to(dev), bt.to(dev), L.to(dev), 0.1,
                             variant=binding.PA_VARIANT_MMA)
    assert e.value.status == binding.PA_ERR_UNSUPPORTED


# The CUDA-core family's further shapes with fp32 elements, 8-token blocks included.
XCASES = [(D, BS, G) for D, BS in ((80, 16), (96, 32), (112, 64), (64, 64), (128, 64), (80, 64),
                                    (64, 8), (80, 8), (96, 8), (112, 8), (128, 8), (256, 8)) for G in (1, 2)]


@pytest.mark.parametrize("D,BS,G", XCASES, ids=[f"D{c[0]}-BS{c[1]}-G{c[2]}" for c in XCASES])
def test_fp32_more_shapes(D, BS, G):
    P = 128
    lens = [1, BS - 1, BS + 1, 2 * P - 1, 3 * P + 5, 17 * P + 3, 0]
    KH = 2
    q, kc, vc, bt, L = f32_random_case(4200 + D + BS + G, S=len(lens), H=KH * G, KH=KH, D=D, BS=BS, lens=lens)
    out, lse = run(q, kc, vc, bt, L, 1.0 / math.sqrt(D), P, lse=True)
    ref, ref_lse = oracle.decode_fp32(q, kc, vc, bt, L, 1.0 / math.sqrt(D))
    ok, worst = within_tolerance(out.double().numpy(), ref, ATOL32, RTOL32)
    assert ok, f"worst excess {worst:.3e}"
    assert torch.all(out[-1] == 0)
    lse_close(lse.numpy(), ref_lse)


def run_mq32(q, kc, vc, bt, lens, scale, P):
    dev = torch.device("cuda")
    q, kc, vc, bt, lens = (t.to(dev) for t in (q, kc, vc, bt, lens))
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=dev)
    ws = binding.pa_decode_v2_mq(out, q, kc, vc, bt, lens, scale, partition_size=P, lse=lse)
    assert binding.device_status(ws) == binding.PA_OK
    return out.cpu(), lse.cpu()


MQ32_CASES = [(q_len, G, D, BS) for q_len, G in ((2, 1), (4, 2), (3, 4))
              for D, BS in ((128, 16), (64, 32), (96, 64), (112, 8), (256, 8))]


@pytest.mark.parametrize("q_len,G,D,BS", MQ32_CASES, ids=[f"q{c[0]}-G{c[1]}-D{c[2]}-BS{c[3]}" for c in MQ32_CASES])
def test_fp32_multi_query(q_len, G, D, BS):
    """Multi-query decode with fp32 elements (the CUDA-core family's causal
    instances): every row masked to its causal limit (L = q_len leaves row 0
    one token), partition edges inside the causal band, two-level combine."""
    KH, P = 2, 64
    lens = [q_len, q_len + 1, P, P + q_len - 1, P + 1, 700, 1500]
    S = len(lens)
    q, kc, vc, bt, L = f32_random_case(4300 + q_len + G + D + BS, S=S * q_len, H=KH * G, KH=KH, D=D, BS=BS,
                                       lens=lens * q_len)
    q = q.view(S, q_len, KH * G, D).contiguous()
    bt, L = bt[:S].contiguous(), L[:S].contiguous()
    out, lse = run_mq32(q, kc, vc, bt, L, 0.09, P)
    ref, ref_lse = oracle.decode_mq_fp32(q, kc, vc, bt, L, 0.09)
    ok, worst = within_tolerance(out.double().numpy(), ref, ATOL32, RTOL32)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)
