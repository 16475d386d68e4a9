"""Repeated calls on the same inputs must agree bit for bit (the block-to-warp
grouping depends only on the unit, so any difference is a race: a stage read
while its next copy lands, a state handed over early).  One medium batch per
consumer variant -- fp8 codes (4-byte fragment loads), 16-row units, 8-token
blocks, fp32 on the CUDA cores -- each checked once against the oracle."""
import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding
from pa_testutil import f32_random_case, fp8_random_case, random_case, within_tolerance

pytestmark = pytest.mark.gpu

CALLS = 25
LENS = [4096, 17, 900, 2500, 1, 640, 3000, 77, 1800, 4000, 260, 1200]


def repeat(call):
    first = call().clone()
    for i in range(CALLS - 1):
        assert torch.equal(call(), first), f"call {i + 2} differs from the first"
    return first.cpu()


def device(*ts):
    return [t.to("cuda") for t in ts]


def test_repeat_fp8_gqa():
    q, kc, vc, bt, L = fp8_random_case(6001, S=len(LENS), H=16, KH=4, D=128, BS=16, lens=LENS,
                                       qdtype=torch.bfloat16)
    qd, kd, vd, btd, ld = device(q, kc, vc, bt, L)
    out = torch.empty_like(qd)
    ws = torch.empty(binding.workspace_bytes(len(LENS), 16, 4, 128, bt.shape[1], 16, 512),
                     dtype=torch.uint8, device="cuda")

    def call():
        binding.pa_decode_v2_fp8(out, qd, kd, vd, btd, ld, 0.09, 0.5, 1.5, workspace=ws)
        assert binding.device_status(ws) == binding.PA_OK
        return out

    got = repeat(call)
    ref, _ = oracle.decode_fp8kv(q, kc, vc, bt, L, 0.09, 0.5, 1.5, oracle.DTYPE_BF16)
    assert within_tolerance(got.double().numpy(), ref)[0]


@pytest.mark.parametrize("H,KH,BS,dt", [(32, 2, 16, torch.bfloat16), (16, 2, 8, torch.float16)],
                         ids=["16-row-units", "8-token-blocks"])
def test_repeat_tensor_core_variants(H, KH, BS, dt):
    q, kc, vc, bt, L = random_case(6002 + BS, S=len(LENS), H=H, KH=KH, D=128, BS=BS, lens=LENS, dtype=dt)
    qd, kd, vd, btd, ld = device(q, kc, vc, bt, L)
    out = torch.empty_like(qd)
    ws = torch.empty(binding.workspace_bytes(len(LENS), H, KH, 128, bt.shape[1], BS, 512),
                     dtype=torch.uint8, device="cuda")

    def call():
        binding.pa_decode_v2(out, qd, kd, vd, btd, ld, 0.09, workspace=ws)
        assert binding.device_status(ws) == binding.PA_OK
        return out

    got = repeat(call)
    ref = oracle.decode(q, kc, vc, bt, L, 0.09, oracle.DTYPE_FP16 if dt == torch.float16 else oracle.DTYPE_BF16)
    assert within_tolerance(got.double().numpy(), ref)[0]


def test_repeat_fp32():
    q, kc, vc, bt, L = f32_random_case(6003, S=len(LENS), H=8, KH=8, D=128, BS=16, lens=LENS)
    qd, kd, vd, btd, ld = device(q, kc, vc, bt, L)
    out = torch.empty_like(qd)
    ws = torch.empty(binding.workspace_bytes(len(LENS), 8, 8, 128, bt.shape[1], 16, 512),
                     dtype=torch.uint8, device="cuda")

    def call():
        binding.pa_decode_v2(out, qd, kd, vd, btd, ld, 0.09, workspace=ws)
        assert binding.device_status(ws) == binding.PA_OK
        return out

    got = repeat(call)
    ref, _ = oracle.decode_fp32(q, kc, vc, bt, L, 0.09)
    assert within_tolerance(got.double().numpy(), ref, 1e-5, 1e-4)[0]


def _split_lens(seed):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, 400, (1100,), generator=g).tolist()
    for k in range(binding.MAX_ROWS_PER_LAUNCH, len(lens), binding.MAX_ROWS_PER_LAUNCH):
        lens[k - 1] = lens[k] = 1300   # multi-partition on both sides of each split
    lens[-1] = 0
    return lens


def test_fp8_batch_split_across_launches():
    """More sequences than one launch takes, over an fp8 cache: split launches, one workspace."""
    lens = _split_lens(31)
    q, kc, vc, bt, L = fp8_random_case(6101, S=len(lens), H=8, KH=2, D=64, BS=16, lens=lens, num_blocks=2048)
    qd, kd, vd, btd, ld = device(q, kc, vc, bt, L)
    out = torch.full_like(qd, float("nan"))
    ws = binding.pa_decode_v2_fp8(out, qd, kd, vd, btd, ld, 0.125, 0.75, 1.25, partition_size=256)
    assert binding.device_status(ws) == binding.PA_OK
    ref, _ = oracle.decode_fp8kv(q, kc, vc, bt, L, 0.125, 0.75, 1.25, oracle.DTYPE_FP16)
    assert within_tolerance(out.cpu().double().numpy(), ref)[0]


def test_fp32_batch_split_across_launches():
    lens = _split_lens(32)
    q, kc, vc, bt, L = f32_random_case(6102, S=len(lens), H=4, KH=4, D=64, BS=16, lens=lens, num_blocks=2048)
    qd, kd, vd, btd, ld = device(q, kc, vc, bt, L)
    out = torch.full_like(qd, float("nan"))
    ws = binding.pa_decode_v2(out, qd, kd, vd, btd, ld, 0.125, partition_size=256)
    assert binding.device_status(ws) == binding.PA_OK
    ref, _ = oracle.decode_fp32(q, kc, vc, bt, L, 0.125)
    assert within_tolerance(out.cpu().double().numpy(), ref, 1e-5, 1e-4)[0]
