"""GPU parity of decode over an fp8 (E4M3) KV cache (pa_decode_v2_fp8): the
caches hold E4M3 codes (key layout x = 16), real keys and values are
k_scale * K and v_scale * V, queries and output fp16 / bf16.  Checked against
the fp64 oracle's restatement at the benchmark tolerance (every E4M3 value is
exact in fp16 and bf16, so the arithmetic is that of the 16-bit caches);
log-sum-exp at the tolerance derived in test_lse_gpu."""
import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding
from pa_testutil import fp8_random_case, within_tolerance
from test_lse_gpu import lse_close

pytestmark = pytest.mark.gpu

DT_CODE = {torch.float16: oracle.DTYPE_FP16, torch.bfloat16: oracle.DTYPE_BF16}


def run_fp8(q, kc, vc, bt, lens, scale, k_scale, v_scale, P):
    dev = torch.device("cuda")
    q, kc, vc, bt, lens = (t.to(dev) for t in (q, kc, vc, bt, lens))
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), device=dev)
    ws = binding.pa_decode_v2_fp8(out, q, kc, vc, bt, lens, scale, k_scale, v_scale, partition_size=P, lse=lse)
    assert binding.device_status(ws) == binding.PA_OK
    return out.cpu(), lse.cpu()


CASES = [  # (H, KH, D, BS, qdtype)
    (4, 4, 128, 16, torch.float16), (8, 2, 128, 16, torch.bfloat16), (16, 2, 128, 32, torch.float16),
    (8, 2, 64, 16, torch.float16), (8, 2, 64, 32, torch.bfloat16), (4, 2, 256, 16, torch.bfloat16),
    (8, 8, 256, 32, torch.float16), (12, 3, 128, 16, torch.bfloat16), (16, 4, 64, 32, torch.float16),
]


@pytest.mark.parametrize("H,KH,D,BS,qdtype", CASES,
                         ids=[f"h{c[0]}kh{c[1]}_d{c[2]}_bs{c[3]}_{'bf16' if c[4] == torch.bfloat16 else 'fp16'}"
                              for c in CASES])
def test_fp8kv_matches_oracle(H, KH, D, BS, qdtype):
    # one token, none, a partial block, block and partition edges, two-level (P = 64)
    lens = [1, 0, 5, BS, 64, 65, 700, 1500]
    q, kc, vc, bt, L = fp8_random_case(31 + D + BS + H, S=len(lens), H=H, KH=KH, D=D, BS=BS, lens=lens,
                                       qdtype=qdtype)
    out, lse = run_fp8(q, kc, vc, bt, L, 0.09, 0.75, 1.5, 64)
    ref, ref_lse = oracle.decode_fp8kv(q, kc, vc, bt, L, 0.09, 0.75, 1.5, DT_CODE[qdtype])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)


def test_fp8kv_scales_act_as_multipliers():
    """v_scale 2 doubles every output bitwise where the output is a normal fp16
    number (below 2^-14 the rounding to fp16 subnormals need not commute with
    the doubling: 2 round(x) and round(2 x) can differ by one subnormal step);
    k_scale 2 at scale s is scale 2 s."""
    q, kc, vc, bt, L = fp8_random_case(5, S=4, H=8, KH=2, D=128, BS=16, lens=[30, 513, 1, 2000])
    a, la = run_fp8(q, kc, vc, bt, L, 0.25, 1.0, 1.0, 512)
    b, lb = run_fp8(q, kc, vc, bt, L, 0.25, 1.0, 2.0, 512)
    normal = (2 * a).float().abs() >= 2.0 ** -14
    assert torch.equal(b[normal], (2 * a)[normal]) and torch.equal(la, lb)
    assert ((b.float() - 2 * a.float()).abs()[~normal] <= 2.0 ** -24).all()
    c, lc = run_fp8(q, kc, vc, bt, L, 0.25, 2.0, 1.0, 512)
    d, ld = run_fp8(q, kc, vc, bt, L, 0.5, 1.0, 1.0, 512)
    assert torch.equal(c, d) and torch.equal(lc, ld)


def test_fp8kv_nan_codes_past_the_end_are_ignored():
    """Cache slots past a sequence's end may hold any code, NaN included."""
    q, kc, vc, bt, L = fp8_random_case(6, S=2, H=8, KH=2, D=64, BS=16, lens=[20, 7])
    kc2, vc2 = kc.clone(), vc.clone()
    for s, n in ((0, 20), (1, 7)):
        b = int(bt[s, n // 16])
        kc2[b, :, :, n % 16:, :] = 0x7F
        vc2[b, :, :, n % 16:] = 0xFF
    a, _ = run_fp8(q, kc, vc, bt, L, 0.1, 1.0, 1.0, 512)
    b2, _ = run_fp8(q, kc2, vc2, bt, L, 0.1, 1.0, 1.0, 512)
    assert torch.isfinite(b2.float()).all() and torch.equal(a, b2)


# Head sizes 80/96/112 and blocks of 8 or 64 tokens over an fp8 cache: one,
# four (kv-head pairs; an odd kv-head count runs one kv head a unit) and eight
# query heads per kv head.
SHAPE_CASES = [  # (H, KH, D, BS, qdtype)
    (8, 8, 80, 16, torch.float16), (16, 4, 96, 32, torch.bfloat16), (8, 1, 112, 16, torch.float16),
    (12, 3, 112, 32, torch.bfloat16), (8, 2, 80, 32, torch.float16),
    (8, 2, 64, 8, torch.float16), (4, 4, 128, 8, torch.bfloat16), (16, 2, 256, 8, torch.float16),
    (8, 2, 80, 8, torch.bfloat16), (6, 3, 96, 8, torch.float16), (8, 2, 112, 8, torch.float16),
    (8, 2, 128, 64, torch.bfloat16), (4, 4, 256, 64, torch.float16), (8, 1, 80, 64, torch.float16),
    (16, 4, 64, 64, torch.bfloat16),
]


@pytest.mark.parametrize("H,KH,D,BS,qdtype", SHAPE_CASES,
                         ids=[f"h{c[0]}kh{c[1]}_d{c[2]}_bs{c[3]}_{'bf16' if c[4] == torch.bfloat16 else 'fp16'}"
                              for c in SHAPE_CASES])
def test_fp8kv_more_shapes_match_oracle(H, KH, D, BS, qdtype):
    # one token, none, a partial block, block and partition edges, two-level (P = 64)
    lens = [1, 0, 5, BS, BS + 3, 64, 65, 700, 1500]
    q, kc, vc, bt, L = fp8_random_case(47 + D + BS + H, S=len(lens), H=H, KH=KH, D=D, BS=BS, lens=lens,
                                       qdtype=qdtype)
    out, lse = run_fp8(q, kc, vc, bt, L, 0.09, 0.75, 1.5, 64)
    ref, ref_lse = oracle.decode_fp8kv(q, kc, vc, bt, L, 0.09, 0.75, 1.5, DT_CODE[qdtype])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)


@pytest.mark.parametrize("BS,H", [(8, 8), (8, 16), (64, 8), (64, 2)])
def test_fp8kv_nan_codes_past_the_end_other_blocks(BS, H):
    """NaN codes in every slot past each sequence's end, in 8- and 64-token
    blocks (8-token blocks pair up into one 16-token tile, a lone last block
    fills half of one): the result is bitwise that of finite codes there."""
    lens = [3, BS, BS + 5, 2 * BS + 1, 200]
    q, kc, vc, bt, L = fp8_random_case(66 + BS + H, S=len(lens), H=H, KH=2, D=128, BS=BS, lens=lens)
    kc2, vc2 = kc.clone(), vc.clone()
    for s, n in enumerate(lens):
        if n % BS:
            b = int(bt[s, n // BS])
            kc2[b, :, :, n % BS:, :] = 0x7F
            vc2[b, :, :, n % BS:] = 0xFF
    a, _ = run_fp8(q, kc, vc, bt, L, 0.1, 1.0, 1.0, 64)
    b2, _ = run_fp8(q, kc2, vc2, bt, L, 0.1, 1.0, 1.0, 64)
    assert torch.isfinite(b2.float()).all() and torch.equal(a, b2)


def run_mq_fp8(q, kc, vc, bt, lens, scale, k_scale, v_scale, P):
    dev = torch.device("cuda")
    q, kc, vc, bt, lens = (t.to(dev) for t in (q, kc, vc, bt, lens))
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=dev)
    ws = binding.pa_decode_v2_mq_fp8(out, q, kc, vc, bt, lens, scale, k_scale, v_scale, partition_size=P, lse=lse)
    assert binding.device_status(ws) == binding.PA_OK
    return out.cpu(), lse.cpu()


def mq_fp8_case(seed, S, q_len, H, KH, D, BS, lens, qdtype=torch.float16):
    q, kc, vc, bt, L = fp8_random_case(seed, S=S * q_len, H=H, KH=KH, D=D, BS=BS, lens=list(lens) * q_len,
                                       qdtype=qdtype)
    return q.view(S, q_len, H, D).contiguous(), kc, vc, bt[:S].contiguous(), L[:S].contiguous()


MQ_CASES = [  # (q_len, H, KH, D, BS, qdtype): q_len * H / KH rows per kv head
    (2, 4, 2, 128, 16, torch.float16), (4, 2, 2, 128, 32, torch.bfloat16), (3, 8, 2, 64, 16, torch.float16),
    (2, 8, 1, 256, 32, torch.bfloat16), (4, 4, 4, 96, 8, torch.float16), (2, 2, 1, 80, 64, torch.bfloat16),
    (8, 4, 2, 128, 16, torch.bfloat16), (2, 2, 2, 64, 16, torch.float16),
]


@pytest.mark.parametrize("q_len,H,KH,D,BS,qdtype", MQ_CASES,
                         ids=[f"q{c[0]}_h{c[1]}kh{c[2]}_d{c[3]}_bs{c[4]}_{'bf16' if c[5] == torch.bfloat16 else 'fp16'}"
                              for c in MQ_CASES])
def test_mq_fp8kv_matches_oracle(q_len, H, KH, D, BS, qdtype):
    """Multi-query decode over an fp8 cache: every query row masked to its
    causal limit (L = q_len leaves row 0 one token), partition and block edges
    inside the causal band, the two-level combine (P = 64)."""
    lens = [q_len, q_len + 1, 64, 64 + q_len - 1, 65, 700, 1500]
    q, kc, vc, bt, L = mq_fp8_case(8100 + q_len + H + D + BS, S=len(lens), q_len=q_len, H=H, KH=KH, D=D, BS=BS,
                                   lens=lens, qdtype=qdtype)
    out, lse = run_mq_fp8(q, kc, vc, bt, L, 0.09, 0.75, 1.5, 64)
    ref, ref_lse = oracle.decode_mq_fp8kv(q, kc, vc, bt, L, 0.09, 0.75, 1.5, DT_CODE[qdtype])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)


def test_mq_fp8kv_one_row_is_the_single_query_entry():
    """q_len = 1 through the multi-query entry is bitwise pa_decode_v2_fp8."""
    q, kc, vc, bt, L = fp8_random_case(91, S=5, H=8, KH=2, D=128, BS=16, lens=[1, 17, 300, 513, 2000])
    a, la = run_fp8(q, kc, vc, bt, L, 0.1, 0.5, 2.0, 512)
    b, lb = run_mq_fp8(q.unsqueeze(1).contiguous(), kc, vc, bt, L, 0.1, 0.5, 2.0, 512)
    assert torch.equal(a, b[:, 0]) and torch.equal(la, lb[:, 0])
