"""CPU tests of the C ABI: the library loads, exports every symbol the header
declares, sizes its workspace as documented and rejects bad arguments before
it touches the GPU (no compute calls are made here)."""
import ctypes
import os
import re

import pytest

from decode_attention_paged_pa_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa_decode.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(binding.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = binding.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name


def _align(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("S,H,KH,D,MB,BS,P", [
    (4, 4, 4, 64, 19, 16, 512),
    (64, 32, 32, 128, 256, 16, 512),
    (8, 64, 8, 128, 4096, 32, 512),
    (3, 6, 2, 256, 7, 16, 32),
])
def test_workspace_bytes_and_layout(S, H, KH, D, MB, BS, P):
    pmax = -(-(MB * BS) // P)
    hdr = 256
    m = hdr
    l = _align(m + S * H * pmax * 4)
    o = _align(l + S * H * pmax * 4)
    total = _align(o + S * H * pmax * D * 4)
    assert binding.workspace_bytes(S, H, KH, D, MB, BS, P) == total
    offs, pm = binding.workspace_layout(S, H, KH, D, MB, BS, P)
    assert offs == (m, l, o, 0, total) and pm == pmax


def test_workspace_bytes_invalid_sizes_is_zero():
    assert binding.workspace_bytes(4, 6, 4, 64, 8, 16, 512) == 0   # H % KH != 0
    assert binding.workspace_bytes(4, 4, 4, 64, 0, 16, 512) == 0   # no blocks per sequence
    assert binding.workspace_bytes(-1, 4, 4, 64, 8, 16, 512) == 0


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced by these calls


def call(**kw):
    a = dict(out=FAKE, query=FAKE, key_cache=FAKE, value_cache=FAKE, block_tables=FAKE,
             seq_lens=FAKE, scale=0.125, num_seqs=2, num_heads=4, num_kv_heads=2, head_size=128,
             block_size=16, partition_size=512, dtype=0, stream=None, max_blocks_per_seq=4,
             num_blocks=8, workspace=FAKE, workspace_bytes=1 << 30)
    a.update(kw)
    return binding.lib().pa_decode_v2(
        a["out"], a["query"], a["key_cache"], a["value_cache"], a["block_tables"], a["seq_lens"],
        ctypes.c_float(a["scale"]), a["num_seqs"], a["num_heads"], a["num_kv_heads"], a["head_size"],
        a["block_size"], a["partition_size"], a["dtype"], a["stream"], a["max_blocks_per_seq"],
        a["num_blocks"], a["workspace"], a["workspace_bytes"])


@pytest.mark.parametrize("kw,status", [
    (dict(num_heads=6, num_kv_heads=4), binding.PA_ERR_INVALID_ARG),
    (dict(dtype=7), binding.PA_ERR_INVALID_ARG),
    (dict(head_size=72), binding.PA_ERR_UNSUPPORTED),
    (dict(head_size=100), binding.PA_ERR_UNSUPPORTED),
    (dict(block_size=4), binding.PA_ERR_UNSUPPORTED),
    (dict(block_size=24), binding.PA_ERR_UNSUPPORTED),
    (dict(block_size=64, partition_size=96), binding.PA_ERR_UNSUPPORTED),
    (dict(partition_size=100), binding.PA_ERR_UNSUPPORTED),
    (dict(partition_size=0), binding.PA_ERR_INVALID_ARG),
    (dict(out=None), binding.PA_ERR_INVALID_ARG),
    (dict(seq_lens=None), binding.PA_ERR_INVALID_ARG),
    (dict(query=FAKE + 8), binding.PA_ERR_INVALID_ARG),
    (dict(key_cache=FAKE + 2), binding.PA_ERR_INVALID_ARG),
    (dict(block_tables=FAKE + 2), binding.PA_ERR_INVALID_ARG),
    (dict(num_blocks=0), binding.PA_ERR_INVALID_ARG),
    (dict(max_blocks_per_seq=0), binding.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.PA_ERR_INVALID_ARG),
    (dict(workspace_bytes=1024), binding.PA_ERR_WORKSPACE),
    (dict(num_seqs=0), binding.PA_OK),
])
def test_rejects_bad_arguments_before_launch(kw, status):
    assert call(**kw) == status


def test_lse_entry_rejects_misaligned_lse():
    lib = binding.lib()
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125), 2, 4, 2, 128, 16, 512, 0, None, 4, 8,
            FAKE, 1 << 30)
    assert lib.pa_decode_v2_lse(FAKE, FAKE + 2, *args) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_decode_v2_lse(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125), 0, 4, 2,
                                128, 16, 512, 0, None, 4, 8, FAKE, 1 << 30) == binding.PA_OK


def test_mq_entry_rejects_bad_q_len():
    lib = binding.lib()
    for q_len in (0, -1, 1025):
        st = lib.pa_decode_v2_mq(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125), 2, q_len,
                                 4, 2, 128, 16, 512, 0, None, 4, 8, FAKE, 1 << 30)
        assert st == binding.PA_ERR_INVALID_ARG, q_len
    st = lib.pa_decode_v2_mq(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125), 2, 4,
                             4, 2, 128, 16, 512, 0, None, 4, 8, FAKE, 1024)
    assert st == binding.PA_ERR_WORKSPACE


def test_binding_launch_count_matches_kernel_limit():
    text = open(os.path.join(ROOT, "decode_attention_paged_pa_gb300", "csrc", "pa_kernel.cuh")).read()
    limit = int(re.search(r"#define PA_MAX_SEQS_PER_LAUNCH (\d+)", text).group(1))
    assert binding.MAX_ROWS_PER_LAUNCH == limit
    # the header clear and phase 1 per `limit` sequences, plus the phase-2 combine
    assert binding.launches_per_call(limit) == 3 and binding.launches_per_call(limit + 1) == 5
    assert binding.launches_per_call(300, 4) == 3   # multi-query rows share their sequence's launch
    # no phase 2 when no sequence can have two partitions
    assert binding.launches_per_call(300, 1, max_partitions=1) == 2


def test_fp8_entry_rejects_bad_scales():
    lib = binding.lib()
    for ks, vs in ((float("nan"), 1.0), (1.0, float("inf"))):
        st = lib.pa_decode_v2_fp8(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125),
                                  ctypes.c_float(ks), ctypes.c_float(vs), 2, 4, 2, 128, 16, 512, 0, None,
                                  4, 8, FAKE, 1 << 30)
        assert st == binding.PA_ERR_INVALID_ARG
        st = lib.pa_decode_v2_mq_fp8(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125),
                                     ctypes.c_float(ks), ctypes.c_float(vs), 2, 2, 4, 2, 128, 16, 512, 0, None,
                                     4, 8, FAKE, 1 << 30)
        assert st == binding.PA_ERR_INVALID_ARG
    for q_len in (0, 1025):
        st = lib.pa_decode_v2_mq_fp8(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125),
                                     ctypes.c_float(1.0), ctypes.c_float(1.0), 2, q_len, 4, 2, 128, 16, 512, 0,
                                     None, 4, 8, FAKE, 1 << 30)
        assert st == binding.PA_ERR_INVALID_ARG, q_len
    st = lib.pa_decode_v2_mq_fp8(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125),
                                 ctypes.c_float(1.0), ctypes.c_float(1.0), 2, 2, 4, 2, 128, 16, 512,
                                 binding.PA_DTYPE_FP32, None, 4, 8, FAKE, 1 << 30)
    assert st == binding.PA_ERR_UNSUPPORTED


def test_shapes_outside_a_family_are_rejected():
    """With 16-bit elements the tensor-core family takes every shape; the
    CUDA-core family head sizes 80/96/112 with 16/32/64-token blocks and
    64-token blocks at 64/128 next to its base shapes, never 8-token blocks
    (fp32 takes those: see the fp32 test); fp8 caches take every supported
    head size and block size, on tensor cores only."""
    lib = binding.lib()

    def ex(D, BS, variant):
        return lib.pa_decode_v2_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125), 0, 4, 2, D, BS,
                                   512, 0, None, 4, 8, FAKE, 1 << 30, variant, 0, 0)

    for D, BS in ((96, 16), (80, 32), (112, 64), (64, 64), (128, 64)):
        for variant in (binding.PA_VARIANT_SIMT, binding.PA_VARIANT_MMA, binding.PA_VARIANT_AUTO):
            assert ex(D, BS, variant) == binding.PA_OK, (D, BS, variant)
    for D, BS in ((128, 8), (80, 8), (256, 64)):
        assert ex(D, BS, binding.PA_VARIANT_SIMT) == binding.PA_ERR_UNSUPPORTED, (D, BS)
        assert ex(D, BS, binding.PA_VARIANT_MMA) == binding.PA_OK, (D, BS)
        assert ex(D, BS, binding.PA_VARIANT_AUTO) == binding.PA_OK, (D, BS)
    for D, BS in ((80, 16), (128, 8), (128, 64), (256, 8), (112, 64), (96, 32)):
        st = lib.pa_decode_v2_fp8(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125),
                                  ctypes.c_float(1.0), ctypes.c_float(1.0), 0, 4, 2, D, BS, 512, 0, None,
                                  4, 8, FAKE, 1 << 30)
        assert st == binding.PA_OK, (D, BS)
        st = lib.pa_decode_v2_mq_fp8(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125),
                                     ctypes.c_float(1.0), ctypes.c_float(1.0), 0, 2, 4, 2, D, BS, 512, 0, None,
                                     4, 8, FAKE, 1 << 30)
        assert st == binding.PA_OK, (D, BS)
    for D, BS in ((48, 16), (128, 24)):
        st = lib.pa_decode_v2_fp8(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125),
                                  ctypes.c_float(1.0), ctypes.c_float(1.0), 2, 4, 2, D, BS, 528, 0, None,
                                  4, 8, FAKE, 1 << 30)
        assert st == binding.PA_ERR_UNSUPPORTED, (D, BS)


def test_fp32_only_on_the_cuda_core_family():
    """fp32 (dtype 2) runs on the CUDA-core family, every shape (single- and
    multi-query, 8-token blocks included), never on tensor cores or over an fp8
    cache; 16-bit 8-token blocks stay off the CUDA-core family."""
    lib = binding.lib()

    def ex(D, BS, variant, dtype=binding.PA_DTYPE_FP32):
        return lib.pa_decode_v2_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125), 0, 4, 2, D, BS,
                                   512, dtype, None, 4, 8, FAKE, 1 << 30, variant, 0, 0)

    assert ex(128, 16, binding.PA_VARIANT_AUTO) == binding.PA_OK
    assert ex(128, 16, binding.PA_VARIANT_SIMT) == binding.PA_OK
    assert ex(128, 16, binding.PA_VARIANT_MMA) == binding.PA_ERR_UNSUPPORTED
    assert ex(96, 16, binding.PA_VARIANT_AUTO) == binding.PA_OK
    assert ex(112, 64, binding.PA_VARIANT_AUTO) == binding.PA_OK
    assert ex(128, 8, binding.PA_VARIANT_AUTO) == binding.PA_OK
    assert ex(80, 8, binding.PA_VARIANT_SIMT) == binding.PA_OK
    assert ex(128, 8, binding.PA_VARIANT_AUTO, dtype=binding.PA_DTYPE_FP16) == binding.PA_OK
    assert ex(128, 8, binding.PA_VARIANT_SIMT, dtype=binding.PA_DTYPE_FP16) == binding.PA_ERR_UNSUPPORTED
    assert ex(96, 16, binding.PA_VARIANT_MMA) == binding.PA_ERR_UNSUPPORTED
    assert ex(128, 16, binding.PA_VARIANT_AUTO, dtype=3) == binding.PA_ERR_INVALID_ARG
    for D, BS, want in ((128, 16, binding.PA_OK), (80, 64, binding.PA_OK), (112, 8, binding.PA_OK),
                        (128, 24, binding.PA_ERR_UNSUPPORTED)):
        st = lib.pa_decode_v2_mq(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125), 0, 4,
                                 4, 2, D, BS, 512, binding.PA_DTYPE_FP32, None, 4, 8, FAKE, 1 << 30)
        assert st == want, (D, BS)
    st = lib.pa_decode_v2_fp8(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.125),
                              ctypes.c_float(1.0), ctypes.c_float(1.0), 2, 4, 2, 128, 16, 512,
                              binding.PA_DTYPE_FP32, None, 4, 8, FAKE, 1 << 30)
    assert st == binding.PA_ERR_UNSUPPORTED


def test_host_io_staging_has_room_for_fp32():
    base = binding.workspace_bytes(3, 4, 2, 128, 8, 16, 512)
    need = binding.host_io_workspace_bytes(3, 4, 2, 128, 8, 16, 512)
    assert need >= base + 2 * 3 * 4 * 128 * 4 + 3 * 8 * 4 + 3 * 4


def test_status_strings():
    for code in range(7):
        s = binding.status_string(code)
        assert s and s != "unknown status"
    assert binding.status_string(99) == "unknown status"
