"""Failure detection on the GPU without a fault: every device-side wait of the
kernel is bounded.  A call whose bound is 1 ns gives up at its first wait,
records PA_ERR_TIMEOUT in the workspace error word (read by the host), lets
its in-flight copies land and exits; the context stays usable and the next
call is correct."""
import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding
from pa_testutil import random_case, within_tolerance

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", [binding.PA_VARIANT_SIMT, binding.PA_VARIANT_MMA])
def test_wait_bound_reports_timeout_and_context_survives(variant):
    q, kc, vc, bt, lens = random_case(31, S=16, H=8, KH=8 if variant == binding.PA_VARIANT_SIMT else 2,
                                      D=128, BS=16, lens=[4096] * 16)
    dev = torch.device("cuda")
    q, kc, vc, bt, lens = (t.to(dev) for t in (q, kc, vc, bt, lens))
    out = torch.empty_like(q)
    ws = binding.pa_decode_v2(out, q, kc, vc, bt, lens, 0.088, partition_size=512, variant=variant,
                              timeout_ns=1)
    assert binding.device_status(ws) == binding.PA_ERR_TIMEOUT
    ws = binding.pa_decode_v2(out, q, kc, vc, bt, lens, 0.088, partition_size=512, variant=variant,
                              workspace=ws)
    assert binding.device_status(ws) == binding.PA_OK
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), bt.cpu(), lens.cpu(), 0.088, oracle.DTYPE_FP16)
    assert within_tolerance(out.cpu().double().numpy(), ref)[0]
