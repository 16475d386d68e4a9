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
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture (one-time set-up calls)
        binding.pa_decode_v2(out, q, kc, vc, bt, lens, scale, partition_size=P, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.pa_decode_v2(out, q, kc, vc, bt, lens, scale, partition_size=P, workspace=ws)

    for q_new, l_new in ((q_a, la), (q_b, lb), (q_a, la)):
        q.copy_(q_new.to(dev))
        lens.copy_(l_new.to(dev))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert binding.device_status(ws) == binding.PA_OK
        ref = eager(q_new.to(dev), l_new.to(dev))
        assert torch.equal(out, ref)
