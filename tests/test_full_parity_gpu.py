"""Full-size parity: every output element of every measured workload against
the fp64 oracle, through the C ABI.

The five benchmark configurations (tiny_fp16, mha_fp16, gqa_bf16,
long_skew_bf16, d256_fp16) are decoded whole in the launch the bench times
(AUTO, with the log-sum-exp returned) and in each kernel family forced (SIMT,
MMA); the whole [S, H, D] output is compared with ``oracle.decode`` at
|out - ref| <= 2e-3 + 1e-2 |ref| and the whole [S, H] log-sum-exp with
``oracle.lse`` at 1e-4 + 1e-5 |ref|.  The workloads of the further rows
(multi-query decode, the fp8 cache, fp32, head sizes 80 / 112 in 64- / 8-token
blocks) are compared whole with their own oracle functions.

Reference: the page "paged_attention_v2_triton.py -- Triton PagedAttention V2
for BI-V100", module docstring (the result the two phases reach) and
``_paged_attn_v2_reduce_kernel`` (the combine)."""
import gc

import pytest
import torch

import oracle
from decode_attention_paged_pa_gb300 import binding, workloads
from pa_testutil import within_tolerance
from test_lse_gpu import lse_close

pytestmark = pytest.mark.gpu

AUTO, SIMT, MMA = binding.PA_VARIANT_AUTO, binding.PA_VARIANT_SIMT, binding.PA_VARIANT_MMA
VNAME = {AUTO: "auto", SIMT: "simt", MMA: "mma"}
ATOL32, RTOL32 = 1e-5, 1e-4

_cache = {}


def inputs_and_reference(name):
    """The workload's device inputs and the oracle's answer over the whole batch
    (computed once per workload; the previous workload's tensors are freed)."""
    if name not in _cache:
        _cache.clear()
        gc.collect()
        torch.cuda.empty_cache()
        w = workloads.WORKLOADS[name]
        inp = workloads.make_inputs(w, device="cuda")
        args = (inp["query"], inp["key_cache"], inp["value_cache"], inp["block_tables"], inp["seq_lens"],
                inp["scale"])
        if w.kv_dtype == "e4m3":
            ref = oracle.decode_fp8kv(*args, w.k_scale, w.v_scale, workloads.DTYPE_CODES[w.dtype])
        elif w.dtype == "fp32":
            ref = oracle.decode_fp32(*args)
        elif w.q_len > 1:
            ref = oracle.decode_mq(*args, workloads.DTYPE_CODES[w.dtype])
        else:
            code = workloads.DTYPE_CODES[w.dtype]
            ref = (oracle.decode(*args, code), oracle.lse(*args, code))
        _cache[name] = (w, inp, ref)
    return _cache[name]


BASE = [(n, v) for n in workloads.WORKLOAD_ORDER for v in (AUTO, SIMT, MMA)]


@pytest.mark.parametrize("name,variant", BASE, ids=[f"{n}-{VNAME[v]}" for n, v in BASE])
def test_workload_full_parity(name, variant):
    w, inp, (ref, ref_lse) = inputs_and_reference(name)
    out = torch.full_like(inp["query"], float("nan"))
    lse = torch.full(inp["query"].shape[:2], float("nan"), device="cuda") if variant == AUTO else None
    ws = binding.pa_decode_v2(out, inp["query"], inp["key_cache"], inp["value_cache"], inp["block_tables"],
                              inp["seq_lens"], inp["scale"], partition_size=w.partition_size,
                              variant=variant, lse=lse)
    assert binding.device_status(ws) == binding.PA_OK
    ok, worst = within_tolerance(out.cpu().double().numpy(), ref)
    assert ok, f"{name} ({VNAME[variant]}): worst excess {worst:.3e} over {ref.size} elements"
    if lse is not None:
        lse_close(lse.cpu().numpy(), ref_lse)
    if name == workloads.WORKLOAD_ORDER[-1] and variant == MMA:
        _cache.clear()


def test_long_context_batch_in_reverse_order():
    """The long-context batch with its sequences in reverse order (the
    131072-token sequence last): units are scheduled longest sequence first
    whatever the batch order, and the reversed output is the forward one,
    row for row, bit for bit, and matches the oracle."""
    w, inp, (ref, ref_lse) = inputs_and_reference("long_skew_bf16")
    args = (inp["key_cache"], inp["value_cache"])
    fwd = torch.empty_like(inp["query"])
    ws = binding.pa_decode_v2(fwd, inp["query"], *args, inp["block_tables"], inp["seq_lens"], inp["scale"],
                              partition_size=w.partition_size)
    assert binding.device_status(ws) == binding.PA_OK
    rev = torch.arange(w.num_seqs - 1, -1, -1, device="cuda")
    out = torch.full_like(inp["query"], float("nan"))
    ws = binding.pa_decode_v2(out, inp["query"][rev].contiguous(), *args, inp["block_tables"][rev].contiguous(),
                              inp["seq_lens"][rev].contiguous(), inp["scale"], partition_size=w.partition_size)
    assert binding.device_status(ws) == binding.PA_OK
    assert torch.equal(out, fwd[rev])
    ok, worst = within_tolerance(out.cpu().double().numpy(), ref[rev.cpu().numpy()])
    assert ok, f"reversed long-context batch: worst excess {worst:.3e}"


NEXT = ["spec4_gqa_bf16", "spec4_mha_fp16", "gqa_fp8kv_bf16", "gqa_d112_bs8_bf16", "mha_d80_bs64_fp16",
        "mha_fp32"]


@pytest.mark.parametrize("name", NEXT)
def test_next_workload_full_parity(name):
    w, inp, ref = inputs_and_reference(name)
    q = inp["query"]
    out = torch.full_like(q, float("nan"))
    args = (inp["key_cache"], inp["value_cache"], inp["block_tables"], inp["seq_lens"], inp["scale"])
    ref_lse = None
    if w.kv_dtype == "e4m3":
        lse = torch.full(q.shape[:2], float("nan"), device="cuda")
        ws = binding.pa_decode_v2_fp8(out, q, *args, w.k_scale, w.v_scale, partition_size=w.partition_size,
                                      lse=lse)
        ref, ref_lse = ref
    elif w.q_len > 1:
        lse = torch.full(q.shape[:3], float("nan"), device="cuda")
        ws = binding.pa_decode_v2_mq(out, q, *args, partition_size=w.partition_size, lse=lse)
        ref, ref_lse = ref
    elif w.dtype == "fp32":
        lse = torch.full(q.shape[:2], float("nan"), device="cuda")
        ws = binding.pa_decode_v2(out, q, *args, partition_size=w.partition_size, lse=lse)
        ref, ref_lse = ref
    else:
        lse = None
        ws = binding.pa_decode_v2(out, q, *args, partition_size=w.partition_size)
        ref = ref[0]
    assert binding.device_status(ws) == binding.PA_OK
    atol, rtol = (ATOL32, RTOL32) if w.dtype == "fp32" else (2e-3, 1e-2)
    ok, worst = within_tolerance(out.cpu().double().numpy(), ref, atol, rtol)
    assert ok, f"{name}: worst excess {worst:.3e} over {ref.size} elements"
    if ref_lse is not None:
        lse_close(lse.cpu().numpy(), ref_lse)
    if name == NEXT[-1]:
        _cache.clear()
