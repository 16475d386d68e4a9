"""CPU tests of the seeded synthetic workloads and their byte accounting (the
numbers the bench divides by time).  No attention arithmetic is involved."""
import dataclasses

import torch

from decode_attention_paged_pa_gb300 import workloads

W = workloads.WORKLOADS


def _draw(w):
    gen = torch.Generator().manual_seed(w.seed)
    return workloads.draw_seq_lens(w, gen), workloads.draw_block_tables(w, gen)


def test_long_context_bytes_match_the_worked_figure():
    """The long-context batch (fixed lengths) moves exactly
    KV 671,059,968 + q/out 262,144 + tables 5121 * 4 + lens 32 = 671,342,628 B:
    163,833 tokens x 8 kv heads x 128 dims x 2 (K, V) x 2 bytes, q and out
    8 x 64 x 128 x 2 bytes each, one int32 per 32-token block in use."""
    w = W["long_skew_bf16"]
    lens = list(w.lens)
    assert sum(lens) == 163833
    assert sum(-(-L // 32) for L in lens) == 5121
    assert workloads.algorithmic_bytes(w, lens) == 671_342_628
    assert workloads.kv_tokens(lens) == 163833


def test_bytes_scale_with_the_element_size():
    lens = [100, 7, 513]
    base = dict(num_seqs=3, num_heads=8, num_kv_heads=2, head_size=64, block_size=16, lens=tuple(lens))
    b16 = workloads.algorithmic_bytes(workloads.custom(dtype="bf16", **base), lens)
    f32 = workloads.algorithmic_bytes(workloads.custom(dtype="fp32", **base), lens)
    fp8 = workloads.algorithmic_bytes(dataclasses.replace(workloads.custom(dtype="bf16", **base),
                                                          kv_dtype="e4m3"), lens)
    kv16 = sum(lens) * 2 * 64 * 2 * 2
    q16 = 2 * 3 * 8 * 64 * 2
    tables = 4 * sum(-(-L // 16) for L in lens) + 4 * 3
    assert b16 == kv16 + q16 + tables
    assert f32 == 2 * kv16 + 2 * q16 + tables
    assert fp8 == kv16 // 2 + q16 + tables
    mq = dataclasses.replace(workloads.custom(dtype="bf16", **base), q_len=4)
    assert workloads.algorithmic_bytes(mq, lens) == kv16 + 4 * q16 + tables


def test_benchmark_configurations_as_defined():
    tiny = W["tiny_fp16"]
    lens, bt = _draw(tiny)
    assert lens.min() >= 1 and lens.max() <= 300 and bt.shape == (4, 19)
    for row in bt:                                   # distinct block ids within a sequence
        assert len(set(row.tolist())) == 19 and int(row.max()) < 128
    mha = W["mha_fp16"]
    lens, bt = _draw(mha)
    assert lens.min() >= 512 and lens.max() <= 4096 and bt.shape == (64, 256)
    assert sorted(bt.flatten().tolist()) == list(range(64 * 256))   # a permutation of the pool
    gqa = W["gqa_bf16"]
    lens, _ = _draw(gqa)
    assert lens.min() >= 2048 and lens.max() <= 8192 and gqa.num_heads // gqa.num_kv_heads == 4
    d256 = W["d256_fp16"]
    lens, _ = _draw(d256)
    assert lens[:3].tolist() == [1, 2048, 17] and lens.max() <= 2048
    assert d256.k_std == 2.0 and d256.v_uniform and d256.scale == 1.0 / 16.0
    for i, name in enumerate(["tiny_fp16", "mha_fp16", "gqa_bf16", "long_skew_bf16", "d256_fp16"]):
        assert W[name].seed == 1000 + i


def test_inputs_are_seeded_and_laid_out_per_element_type():
    small = dict(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=32, block_size=16, lens=(5, 40))
    for dtype, x in (("fp16", 8), ("bf16", 8), ("fp32", 4)):
        w = workloads.custom(dtype=dtype, **small)
        a, b = workloads.make_inputs(w), workloads.make_inputs(w)
        assert a["key_cache"].shape[-1] == x and a["key_cache"].shape[2] == 32 // x
        assert a["query"].dtype == workloads.DTYPES[dtype]
        for k in ("query", "key_cache", "value_cache", "block_tables", "seq_lens"):
            assert torch.equal(a[k], b[k]), k
    w8 = dataclasses.replace(workloads.custom(dtype="bf16", **small), kv_dtype="e4m3")
    inp = workloads.make_inputs(w8)
    assert inp["key_cache"].dtype == torch.uint8 and inp["key_cache"].shape[-1] == 16
    assert inp["value_cache"].dtype == torch.uint8
    # No NaN codes (0x7f / 0xff): draws are clamped to the finite range first.
    codes = torch.cat([inp["key_cache"].flatten(), inp["value_cache"].flatten()])
    assert not bool(((codes & 0x7F) == 0x7F).any())
