"""GPU parity of multi-query decode (pa_decode_v2_mq): q_len new tokens per
sequence, the i-th attending causally to positions 0 .. L - q_len + i, checked
against the fp64 oracle's direct causal restatement (output at the benchmark
tolerance, log-sum-exp at the tolerance derived in test_lse_gpu)."""
import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding
from pa_testutil import random_case, within_tolerance
from test_lse_gpu import lse_close

pytestmark = pytest.mark.gpu

DT_CODE = {torch.float16: oracle.DTYPE_FP16, torch.bfloat16: oracle.DTYPE_BF16}


def mq_case(seed, S, q_len, H, KH, D, BS, lens, dtype=torch.float16, num_blocks=None):
    q, kc, vc, bt, L = random_case(seed, S=S * q_len, H=H, KH=KH, D=D, BS=BS, lens=list(lens) * q_len,
                                   dtype=dtype, num_blocks=num_blocks)
    return q.view(S, q_len, H, D).contiguous(), kc, vc, bt[:S].contiguous(), L[:S].contiguous()


def run_mq(q, kc, vc, bt, lens, scale, P, expect=binding.PA_OK):
    dev = torch.device("cuda")
    q, kc, vc, bt, lens = (t.to(dev) for t in (q, kc, vc, bt, lens))
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=dev)
    ws = binding.pa_decode_v2_mq(out, q, kc, vc, bt, lens, scale, partition_size=P, lse=lse)
    assert binding.device_status(ws) == expect
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("q_len", [2, 4, 8])
@pytest.mark.parametrize("H,KH,D,BS", [(4, 4, 128, 16), (8, 2, 128, 16), (16, 2, 64, 32)],
                         ids=["simt", "mma_g4", "mma_g8_bs32"])
def test_mq_matches_oracle(H, KH, D, BS, q_len, dtype):
    # L = q_len: row 0 sees one token; partition (P = 64) and block boundaries
    # fall inside the causal band; 1500 tokens need the two-level combine.
    lens = [q_len, q_len + 1, 64, 64 + q_len - 1, 65, 700, 1500]
    q, kc, vc, bt, L = mq_case(5 + q_len + H, S=len(lens), q_len=q_len, H=H, KH=KH, D=D, BS=BS,
                               lens=lens, dtype=dtype)
    out, lse = run_mq(q, kc, vc, bt, L, 0.09, 64)
    ref, ref_lse = oracle.decode_mq(q, kc, vc, bt, L, 0.09, DT_CODE[dtype])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"q_len {q_len}: worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)


def test_mq_single_row_is_plain_decode():
    """q_len = 1 is the single-query path, bitwise (output and lse)."""
    q, kc, vc, bt, L = random_case(3, S=6, H=8, KH=2, D=128, BS=16, lens=[1, 17, 512, 513, 2000, 0])
    dev = torch.device("cuda")
    qd, kd, vd, btd, Ld = (t.to(dev) for t in (q, kc, vc, bt, L))
    out1 = torch.empty_like(qd)
    lse1 = torch.empty(qd.shape[:2], device=dev)
    binding.pa_decode_v2(out1, qd, kd, vd, btd, Ld, 0.1, partition_size=256, lse=lse1)
    out2 = torch.empty_like(qd).view(6, 1, 8, 128)
    lse2 = torch.empty((6, 1, 8), device=dev)
    ws = binding.pa_decode_v2_mq(out2, qd.view(6, 1, 8, 128), kd, vd, btd, Ld, 0.1, partition_size=256,
                                 lse=lse2)
    assert binding.device_status(ws) == binding.PA_OK
    assert torch.equal(out1, out2.view(6, 8, 128))
    assert torch.equal(lse1, lse2.view(6, 8))


def test_mq_length_below_q_len_is_flagged():
    q, kc, vc, bt, L = mq_case(9, S=2, q_len=4, H=4, KH=4, D=64, BS=16, lens=[10, 3])
    run_mq(q, kc, vc, bt, L, 0.1, 512, expect=binding.PA_ERR_DEVICE_BOUNDS)


def test_mq_rows_split_across_launches():
    """300 sequences x 4 rows = 1200 rows: split into launches of whole sequences."""
    g = torch.Generator().manual_seed(8)
    lens = (torch.randint(4, 600, (300,), generator=g)).tolist()
    q, kc, vc, bt, L = mq_case(10, S=300, q_len=4, H=8, KH=2, D=64, BS=16, lens=lens, num_blocks=4096)
    out, lse = run_mq(q, kc, vc, bt, L, 0.125, 128)
    ref, ref_lse = oracle.decode_mq(q, kc, vc, bt, L, 0.125, oracle.DTYPE_FP16)
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)
