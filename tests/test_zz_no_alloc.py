"""The entry point that allocates nothing (pa_decode_v2_static_scratch).

It exists for callers that cannot allocate device memory when they decode --
their memory is reserved up front by another allocator, or an allocation call
could stall a latency-critical loop, or their footprint is fixed at start-up --
so it takes its scratch from a fixed array inside the library.  Here it is
called through the C ABI twice in a row (with different batches, so the second
call meets the first call's leftovers in the shared array) and each output is
compared with the regular entry point's on the same inputs.  This file is
collected last, so a run that stops at its first failure has run every other
test before this one.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from decode_attention_paged_pa_gb300 import binding
from pa_testutil import random_case, within_tolerance

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024


def _entry():
    fn = binding.lib().pa_decode_v2_static_scratch
    vp, ci = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, ci, ci, ci, ci, ci, ci, ci, vp, ci, ci]
    fn.restype = ci
    return fn


def _call_static(fn, out, q, kc, vc, bt, lens, scale, P):
    S, H, D = q.shape
    NB, KH, _, BS, _ = kc.shape
    code = binding.PA_DTYPE_FP16 if q.dtype == torch.float16 else binding.PA_DTYPE_BF16
    return fn(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
              lens.data_ptr(), scale, S, H, KH, D, BS, P, code,
              torch.cuda.current_stream().cuda_stream, bt.shape[1], NB)


def test_static_scratch_matches_regular_entry_twice():
    fn = _entry()
    cases = [
        dict(seed=41, S=6, H=8, KH=2, D=128, BS=16, lens=[1, 700, 1500, 33, 512, 2049],
             dtype=torch.float16, P=256),
        dict(seed=42, S=4, H=16, KH=16, D=128, BS=32, lens=[4000, 3, 64, 900],
             dtype=torch.bfloat16, P=512),
    ]
    for c in cases:
        q, kc, vc, bt, lens = random_case(c["seed"], S=c["S"], H=c["H"], KH=c["KH"], D=c["D"],
                                          BS=c["BS"], lens=c["lens"], dtype=c["dtype"])
        dev = torch.device("cuda")
        q, kc, vc, bt, lens = (t.to(dev) for t in (q, kc, vc, bt, lens))
        scale = 1.0 / math.sqrt(c["D"])
        ref = torch.empty_like(q)
        binding.pa_decode_v2(ref, q, kc, vc, bt, lens, scale, partition_size=c["P"])
        out = torch.full_like(q, float("nan"))
        assert binding.workspace_bytes(c["S"], c["H"], c["KH"], c["D"], bt.shape[1], c["BS"],
                                       c["P"]) <= SCRATCH_BYTES
        st = _call_static(fn, out, q, kc, vc, bt, lens, scale, c["P"])
        assert st == binding.PA_OK, binding.status_string(st)
        torch.cuda.synchronize()
        ok, worst = within_tolerance(out.cpu().double().numpy(), ref.cpu().double().numpy())
        assert ok, f"worst excess {worst:.3e}"


def test_static_scratch_rejects_sizes_beyond_its_array():
    fn = _entry()
    # 64 sequences x 32 heads x 512 partitions x 128 dims of fp32 states: far over 32 MiB.
    S, H, D, BS, MB, P = 64, 32, 128, 16, 16384, 16
    assert binding.workspace_bytes(S, H, H, D, MB, BS, P) > SCRATCH_BYTES
    dev = torch.device("cuda")
    q = torch.zeros((S, H, D), dtype=torch.float16, device=dev)
    kc = torch.zeros((1, H, D // 8, BS, 8), dtype=torch.float16, device=dev)
    vc = torch.zeros((1, H, D, BS), dtype=torch.float16, device=dev)
    bt = torch.zeros((S, MB), dtype=torch.int32, device=dev)
    lens = torch.ones((S,), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    assert _call_static(fn, out, q, kc, vc, bt, lens, 0.1, P) == binding.PA_ERR_WORKSPACE
