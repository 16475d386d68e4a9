"""GPU parity of the log-sum-exp output (pa_decode_v2_lse): the natural-log
log-sum-exp of each (sequence, head)'s scaled scores, checked against the fp64
oracle, and put to its use: two halves of a sequence decoded as separate
sequences merge, through their log-sum-exps, into the whole sequence's output.

Tolerance on lse: |got - ref| <= 1e-4 + 1e-5 |ref|.  The kernel's scores are
fp32 sums of exact 16-bit products (relative error ~1e-6 of sum |q_d k_d|,
well under 1e-5 absolute at these scales), its exp sums are fp32 over at most
131072 terms (relative error ~1e-5, so ~1e-5 absolute after the log), and the
maxima are exact; a log2/ln mix-up or a dropped maximum is off by far more."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding
from pa_testutil import random_case, within_tolerance

pytestmark = pytest.mark.gpu

DT_CODE = {torch.float16: oracle.DTYPE_FP16, torch.bfloat16: oracle.DTYPE_BF16}


def lse_close(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    empty = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), empty), "-inf exactly where a sequence has no tokens"
    g, r = got[~empty], ref[~empty]
    excess = np.abs(g - r) - (1e-4 + 1e-5 * np.abs(r))
    assert excess.size == 0 or excess.max() <= 0, f"lse worst excess {excess.max():.3e}"


def run(q, kc, vc, bt, lens, scale, P):
    dev = torch.device("cuda")
    q, kc, vc, bt, lens = (t.to(dev) for t in (q, kc, vc, bt, lens))
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[1]), float("nan"), device=dev)
    ws = binding.pa_decode_v2(out, q, kc, vc, bt, lens, scale, partition_size=P, lse=lse)
    assert binding.device_status(ws) == binding.PA_OK
    out2 = torch.full_like(q, float("nan"))
    ws = binding.pa_decode_v2(out2, q, kc, vc, bt, lens, scale, partition_size=P)
    assert binding.device_status(ws) == binding.PA_OK
    assert torch.equal(out, out2), "returning lse must not change the output"
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("H,KH,D,BS", [(4, 4, 128, 16), (8, 2, 128, 16), (16, 2, 64, 32), (4, 4, 256, 16)],
                         ids=["simt_d128", "mma_g4", "mma_g8_bs32", "simt_d256"])
def test_lse_matches_oracle(H, KH, D, BS, dtype):
    lens = [1, 0, 5, 64, 65, 700, 1500, 31]   # one, none, one partition, several, two-level (P = 64)
    q, kc, vc, bt, L = random_case(7 + H + D, S=len(lens), H=H, KH=KH, D=D, BS=BS, lens=lens, dtype=dtype)
    out, lse = run(q, kc, vc, bt, L, 0.09, 64)
    ref = oracle.lse(q, kc, vc, bt, L, 0.09, DT_CODE[dtype])
    lse_close(lse.numpy(), ref)
    ok, worst = within_tolerance(out.double().numpy(), oracle.decode(q, kc, vc, bt, L, 0.09, DT_CODE[dtype]))
    assert ok, f"output worst excess {worst:.3e}"


@pytest.mark.parametrize("H,KH", [(4, 4), (8, 2)], ids=["simt", "mma"])
def test_lse_merges_two_halves(H, KH):
    """A 2000-token sequence decoded whole, and its first 1024 and last 976 tokens
    decoded as two sequences of one batch: exp-weighting the halves by their
    lse gives the whole output, and their log-add-exp gives its lse."""
    D, BS, L, L1 = 128, 16, 2000, 1024
    q, kc, vc, bt, lens = random_case(77, S=1, H=H, KH=KH, D=D, BS=BS, lens=[L])
    nblk = -(-L // BS)
    halves_bt = torch.zeros((2, nblk), dtype=torch.int32)
    halves_bt[0, : L1 // BS] = bt[0, : L1 // BS]
    halves_bt[1, : nblk - L1 // BS] = bt[0, L1 // BS: nblk]
    q2 = torch.cat([q, q], dim=0)
    out_w, lse_w = run(q, kc, vc, bt, lens, 0.088, 512)
    out_h, lse_h = run(q2, kc, vc, halves_bt, torch.tensor([L1, L - L1], dtype=torch.int32), 0.088, 512)
    a, b = lse_h[0].double(), lse_h[1].double()
    big = torch.maximum(a, b)
    tot = big + torch.log(torch.exp(a - big) + torch.exp(b - big))
    merged = (torch.exp(a - tot)[:, None] * out_h[0].double() + torch.exp(b - tot)[:, None] * out_h[1].double())
    ref = oracle.decode(q, kc, vc, bt, lens, 0.088, oracle.DTYPE_FP16)
    ok, worst = within_tolerance(merged.numpy()[None], ref)
    assert ok, f"merged halves worst excess {worst:.3e}"
    lse_close(tot.numpy()[None], oracle.lse(q, kc, vc, bt, lens, 0.088, oracle.DTYPE_FP16))
    lse_close(lse_w.numpy(), oracle.lse(q, kc, vc, bt, lens, 0.088, oracle.DTYPE_FP16))
