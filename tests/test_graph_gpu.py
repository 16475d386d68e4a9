"""Calls captured into a CUDA graph and replayed: with a caller-owned
workspace a call is a fixed, stream-ordered chain of launches (the header
clear, phase 1, phase 2 as programmatic dependents), so it can be captured
once and replayed with new contents in its input buffers (query, block
table, lengths up to the table's capacity).  Each replay must give bitwise
the result of an eager call on the same inputs (the kernels are
deterministic)."""
import math

import pytest
import torch

from decode_attention_paged_pa_gb300 import binding
from pa_testutil import random_case

pytestmark = pytest.mark.gpu

CASES = [  # (dtype, H, KH, D, BS): CUDA-core MHA, tensor-core pairs, 16-row units
    (torch.float16, 8, 8, 128, 16), (torch.bfloat16, 16, 4, 128, 32), (torch.bfloat16, 32, 2, 64, 16),
]


@pytest.mark.parametrize("dt,H,KH,D,BS", CASES, ids=[f"{str(c[0])[6:]}-H{c[1]}-KH{c[2]}-D{c[3]}-BS{c[4]}"
                                                      for c in CASES])
def test_decode_replays_from_a_cuda_graph(dt, H, KH, D, BS):
    dev = torch.device("cuda")
    S, MB, P = 6, 64, 256
    lens_a = [1, 100, 700, 1024, 33, 513]
    lens_b = [1024, 5, 256, 257, 900, 64]
    q_a, kc, vc, bt, la = random_case(7100 + D + BS + H, S=S, H=H, KH=KH, D=D, BS=BS, lens=lens_a, dtype=dt, MB=MB)
    q_b, _, _, _, lb = random_case(7200 + D + BS + H, S=S, H=H, KH=KH, D=D, BS=BS, lens=lens_b, dtype=dt, MB=MB)
    kc, vc, bt = kc.to(dev), vc.to(dev), bt.to(dev)
    scale = 1.0 / math.sqrt(D)
    ws_bytes = binding.workspace_bytes(S, H, KH, D, MB, BS, P)

    def eager(q, lens):
        out = torch.empty_like(q)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        binding.pa_decode_v2(out, q, kc, vc, bt, lens, scale, partition_size=P, workspace=ws)
        assert binding.device_status(ws) == binding.PA_OK
        return out

    # Static buffers the graph reads and writes.
    q = q_a.to(dev).clone()
    lens = la.to(dev).clone()
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    graph = _capture(lambda: binding.pa_decode_v2(out, q, kc, vc, bt, lens, scale, partition_size=P,
                                                  workspace=ws))

    for q_new, l_new in ((q_a, la), (q_b, lb), (q_a, la)):
        q.copy_(q_new.to(dev))
        lens.copy_(l_new.to(dev))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert binding.device_status(ws) == binding.PA_OK
        ref = eager(q_new.to(dev), l_new.to(dev))
        assert torch.equal(out, ref)


def _capture(call):
    """call() once on a side stream (one-time set-up outside the capture), then
    captured into a CUDA graph, which is returned."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    return graph


def test_multi_query_and_fp8_calls_replay_from_a_cuda_graph():
    """The multi-query and fp8 entry points captured and replayed: bitwise the
    eager results on the same inputs."""
    from pa_testutil import fp8_random_case
    from test_mq_gpu import mq_case
    dev = torch.device("cuda")
    # multi-query, 16-row units (q_len 4 x 4 heads per kv head)
    S, q_len, H, KH, D, BS, P = 5, 4, 8, 2, 128, 16, 128
    lens = [q_len, 70, 300, 1000, 129]
    q0, kc, vc, bt, L0 = mq_case(7301, S=S, q_len=q_len, H=H, KH=KH, D=D, BS=BS, lens=lens, dtype=torch.bfloat16)
    q1, _, _, _, _ = mq_case(7302, S=S, q_len=q_len, H=H, KH=KH, D=D, BS=BS, lens=lens, dtype=torch.bfloat16)
    kc, vc, bt = kc.to(dev), vc.to(dev), bt.to(dev)
    ws_bytes = binding.workspace_bytes(S * q_len, H * q_len, KH, D, bt.shape[1], BS, P)
    q, lens_d = q0.to(dev).clone(), L0.to(dev).clone()
    out, ws = torch.empty_like(q), torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    call = lambda: binding.pa_decode_v2_mq(out, q, kc, vc, bt, lens_d, 0.1, partition_size=P, workspace=ws)
    graph = _capture(call)
    for qn in (q1, q0):
        q.copy_(qn.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        ref, ws2 = torch.empty_like(q), torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        binding.pa_decode_v2_mq(ref, qn.to(dev), kc, vc, bt, lens_d, 0.1, partition_size=P, workspace=ws2)
        assert binding.device_status(ws) == binding.PA_OK and torch.equal(out, ref)
    # fp8 cache, kv-head pairs
    S, H, KH, D, BS, P = 6, 16, 4, 128, 16, 256
    lens = [1, 40, 600, 1024, 257, 90]
    q0, kc, vc, bt, L0 = fp8_random_case(7401, S=S, H=H, KH=KH, D=D, BS=BS, lens=lens, qdtype=torch.bfloat16)
    q1, _, _, _, _ = fp8_random_case(7402, S=S, H=H, KH=KH, D=D, BS=BS, lens=lens, qdtype=torch.bfloat16)
    kc, vc, bt = kc.to(dev), vc.to(dev), bt.to(dev)
    ws_bytes = binding.workspace_bytes(S, H, KH, D, bt.shape[1], BS, P)
    q, lens_d = q0.to(dev).clone(), L0.to(dev).clone()
    out, ws = torch.empty_like(q), torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    call = lambda: binding.pa_decode_v2_fp8(out, q, kc, vc, bt, lens_d, 0.1, 0.5, 1.5, partition_size=P,
                                            workspace=ws)
    graph = _capture(call)
    for qn in (q1, q0):
        q.copy_(qn.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        ref, ws2 = torch.empty_like(q), torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        binding.pa_decode_v2_fp8(ref, qn.to(dev), kc, vc, bt, lens_d, 0.1, 0.5, 1.5, partition_size=P,
                                 workspace=ws2)
        assert binding.device_status(ws) == binding.PA_OK and torch.equal(out, ref)
