"""The entry point that allocates nothing (pa_decode_v2_static_scratch).

It exists for callers that cannot allocate device memory when they decode --
their memory is reserved up front by another allocator, or an allocation call
could stall a latency-critical loop, or their footprint is fixed at start-up --
so it takes its scratch from a fixed array inside the library.  Here it is
called through the C ABI twice in a row (with different batches, so the second
call meets the first call's leftovers in the shared array) and each output is
compared with the regular entry point's on the same inputs: bit for bit,
since both run the same deterministic launch.  The device's default memory
pool (the one stream-ordered allocation draws from) must show no use at all
across the two calls.  This file is collected last, so a run that stops at
its first failure has run every other test before this one.
"""
import ctypes
import math

import pytest
import torch

from decode_attention_paged_pa_gb300 import binding
from pa_testutil import random_case

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


class DefaultPool:
    """Use of the current device's default memory pool, read through the driver
    (cuMemPoolGetAttribute; torch's caching allocator does not draw from it)."""

    USED_MEM_CURRENT, USED_MEM_HIGH = 7, 8   # CUmemPool_attribute

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int(0)
        assert self.cu.cuCtxGetDevice(ctypes.byref(dev)) == 0
        self.pool = ctypes.c_void_p(0)
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def get(self, attr):
        v = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset_high(self):
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, self.USED_MEM_HIGH, ctypes.byref(zero)) == 0


def test_static_scratch_matches_regular_entry_twice():
    fn = _entry()
    cases = [
        dict(seed=41, S=6, H=8, KH=2, D=128, BS=16, lens=[1, 700, 1500, 33, 512, 2049],
             dtype=torch.float16, P=256),
        dict(seed=42, S=4, H=16, KH=16, D=128, BS=32, lens=[4000, 3, 64, 900],
             dtype=torch.bfloat16, P=512),
    ]
    dev = torch.device("cuda")
    torch.cuda.synchronize()
    pool = DefaultPool()
    # The pool watch sees an allocation: the regular entry point without a
    # workspace draws one from this pool on its stream.
    q, kc, vc, bt, lens = (t.to(dev) for t in random_case(40, S=2, H=4, KH=4, D=64, BS=16, lens=[5, 70]))
    out = torch.empty_like(q)
    base = pool.get(DefaultPool.USED_MEM_CURRENT)
    pool.reset_high()
    lib = binding.lib()
    st = lib.pa_decode_v2(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                          lens.data_ptr(), 0.125, 2, 4, 4, 64, 16, 512, binding.PA_DTYPE_FP16,
                          torch.cuda.current_stream().cuda_stream, bt.shape[1], kc.shape[0], None, 0)
    assert st == binding.PA_OK
    torch.cuda.synchronize()
    assert pool.get(DefaultPool.USED_MEM_HIGH) > base, "the default-pool watch missed an allocation"

    prepared = []
    for c in cases:
        q, kc, vc, bt, lens = random_case(c["seed"], S=c["S"], H=c["H"], KH=c["KH"], D=c["D"],
                                          BS=c["BS"], lens=c["lens"], dtype=c["dtype"])
        q, kc, vc, bt, lens = (t.to(dev) for t in (q, kc, vc, bt, lens))
        scale = 1.0 / math.sqrt(c["D"])
        ref = torch.empty_like(q)
        binding.pa_decode_v2(ref, q, kc, vc, bt, lens, scale, partition_size=c["P"])
        assert binding.workspace_bytes(c["S"], c["H"], c["KH"], c["D"], bt.shape[1], c["BS"],
                                       c["P"]) <= SCRATCH_BYTES
        prepared.append((c, q, kc, vc, bt, lens, scale, ref, torch.full_like(q, float("nan"))))
    torch.cuda.synchronize()
    base = pool.get(DefaultPool.USED_MEM_CURRENT)   # whatever else holds pool memory stays as it is
    pool.reset_high()
    for c, q, kc, vc, bt, lens, scale, ref, out in prepared:   # two calls in a row
        st = _call_static(fn, out, q, kc, vc, bt, lens, scale, c["P"])
        assert st == binding.PA_OK, binding.status_string(st)
    torch.cuda.synchronize()
    assert pool.get(DefaultPool.USED_MEM_HIGH) <= base, "the static-scratch calls allocated device memory"
    for c, q, kc, vc, bt, lens, scale, ref, out in prepared:
        assert torch.equal(out, ref), f"static-scratch output differs from pa_decode_v2's ({c['dtype']})"


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
