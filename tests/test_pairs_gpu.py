"""GPU parity of the tensor-core units that take two kv heads at once (four
query heads per kv head: the unit's 8 columns hold both kv heads' query
heads, and one stage holds one block of each), through the C ABI, against the
fp64 oracle at the benchmark tolerance; with an odd number of kv heads the
same shapes run one kv head per unit.  The grouping is the one the page
"paged_attention_v2_triton.py -- Triton PagedAttention V2 for BI-V100" gives
its launcher (query head h reads kv head h // (H / KH))."""
import math

import pytest
import torch

import oracle
from pa_testutil import caches_from_tokens, random_case, token_views, within_tolerance
from test_lse_gpu import lse_close
from test_shapes_gpu import DT_CODE, run

pytestmark = pytest.mark.gpu

CASES = [(dt, D, BS, KH) for dt in (torch.float16, torch.bfloat16) for D in (64, 128)
         for BS in (8, 16, 32) for KH in (2, 3, 4)]


@pytest.mark.parametrize("dt,D,BS,KH", CASES,
                         ids=[f"{str(c[0])[6:]}-D{c[1]}-BS{c[2]}-KH{c[3]}" for c in CASES])
def test_kv_head_pairs_match_oracle(dt, D, BS, KH):
    # one token, a ragged block, block and partition edges, past 16 partitions
    P = 64
    lens = [1, BS - 1, BS + 1, 2 * P, 3 * P + 5, 17 * P + 3]
    q, kc, vc, bt, L = random_case(9100 + D + BS + KH, S=len(lens), H=4 * KH, KH=KH, D=D, BS=BS,
                                   lens=lens, dtype=dt)
    out, lse = run(q, kc, vc, bt, L, 1.0 / math.sqrt(D), P, lse=True)
    ref = oracle.decode(q, kc, vc, bt, L, 1.0 / math.sqrt(D), DT_CODE[dt])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), oracle.lse(q, kc, vc, bt, L, 1.0 / math.sqrt(D), DT_CODE[dt]))


@pytest.mark.parametrize("BS", [8, 16, 32])
def test_kv_head_pairs_ignore_garbage_past_the_end(BS):
    """NaN in every slot past each sequence's end, for both kv heads of a
    pair: the result is bitwise the same as with finite contents there."""
    S, KH, D = 4, 4, 128
    lens = [3, BS, BS + 5, 200]
    q, kc, vc, bt, L = random_case(77 + BS, S=S, H=4 * KH, KH=KH, D=D, BS=BS, lens=lens)
    ref_out, _ = run(q, kc, vc, bt, L, 0.1, 64)
    k_tok, v_tok = token_views(kc, vc)
    k2, v2 = k_tok.clone(), v_tok.clone()
    for s in range(S):
        for j in range(-(-lens[s] // BS)):
            last = lens[s] - j * BS
            if last < BS:
                b = int(bt[s, j])
                k2[b, last:] = float("nan")
                v2[b, last:] = float("nan")
    kc2, vc2 = caches_from_tokens(k2, v2)
    out, _ = run(q, kc2, vc2, bt, L, 0.1, 64)
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out, ref_out)


MQ_CASES = [(dt, q_len, G, KH, BS) for dt in (torch.float16, torch.bfloat16) for q_len, G in ((2, 2), (4, 1))
            for KH in (2, 3) for BS in (8, 16, 32)]


@pytest.mark.parametrize("dt,q_len,G,KH,BS", MQ_CASES,
                         ids=[f"{str(c[0])[6:]}-q{c[1]}-G{c[2]}-KH{c[3]}-BS{c[4]}" for c in MQ_CASES])
def test_kv_head_pairs_multi_query(dt, q_len, G, KH, BS):
    """Multi-query decode with four row heads per kv head (q_len x G = 4): the
    unit's 8 columns hold two kv heads' row heads, each masked to its causal
    limit (an odd kv-head count runs one kv head a unit)."""
    from test_mq_gpu import mq_case, run_mq
    lens = [q_len, q_len + 1, 64, 64 + q_len - 1, 65, 700, 1500]
    q, kc, vc, bt, L = mq_case(9300 + q_len + G + KH + BS, S=len(lens), q_len=q_len, H=G * KH, KH=KH, D=128,
                               BS=BS, lens=lens, dtype=dt)
    out, lse = run_mq(q, kc, vc, bt, L, 0.09, 64)
    ref, ref_lse = oracle.decode_mq(q, kc, vc, bt, L, 0.09, DT_CODE[dt])
    ok, worst = within_tolerance(out.double().numpy(), ref)
    assert ok, f"worst excess {worst:.3e}"
    lse_close(lse.numpy(), ref_lse)
