"""ctypes binding of ``libpa_decode.so`` (the C ABI in ``include/pa_decode.h``).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their data pointers and torch's current CUDA stream are handed to
the C entry points, and a non-zero status becomes a :class:`PaError`.  Every
step of the computation runs in the library's CUDA kernels; there is no other
code path.  If the library is missing it is built from ``csrc/`` with nvcc;
if that is impossible the call fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE_BOUNDS = 5
PA_ERR_TIMEOUT = 6

PA_DTYPE_FP16 = 0
PA_DTYPE_BF16 = 1
PA_DTYPE_FP32 = 2

PA_VARIANT_AUTO = 0
PA_VARIANT_SIMT = 1
PA_VARIANT_MMA = 2

_DTYPE_CODE = {torch.float16: PA_DTYPE_FP16, torch.bfloat16: PA_DTYPE_BF16}
# pa_decode_v2 and the host-I/O entry point also take fp32 (key layout x = 4).
_DTYPE_CODE_F32 = {**_DTYPE_CODE, torch.float32: PA_DTYPE_FP32}

# Every symbol the header declares.
EXPORTED_SYMBOLS = (
    "pa_decode_v2",
    "pa_decode_v2_ex",
    "pa_decode_v2_lse",
    "pa_decode_v2_mq",
    "pa_decode_v2_fp8",
    "pa_decode_v2_mq_fp8",
    "pa_decode_v2_workspace_bytes",
    "pa_decode_v2_workspace_layout",
    "pa_decode_v2_host_io",
    "pa_decode_v2_host_io_workspace_bytes",
    "pa_decode_v2_static_scratch",
    "pa_decode_v2_device_status",
    "pa_decode_v2_status_string",
)


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def _declare(lib):
    vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
    ci, cs, cf, cll = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_longlong
    lib.pa_decode_v2_workspace_bytes.argtypes = [ci] * 7
    lib.pa_decode_v2_workspace_bytes.restype = cs
    lib.pa_decode_v2_workspace_layout.argtypes = [ci] * 7 + [ctypes.POINTER(cs), ctypes.POINTER(ci)]
    lib.pa_decode_v2_workspace_layout.restype = ci
    base = [vp, vp, vp, vp, vp, vp, cf, ci, ci, ci, ci, ci, ci, ci, vp, ci, ci, vp, cs]
    lib.pa_decode_v2.argtypes = base
    lib.pa_decode_v2.restype = ci
    lib.pa_decode_v2_ex.argtypes = base + [ci, ci, cll]
    lib.pa_decode_v2_ex.restype = ci
    lib.pa_decode_v2_lse.argtypes = [vp, vp] + base[1:]   # out, lse, then pa_decode_v2's from query on
    lib.pa_decode_v2_lse.restype = ci
    lib.pa_decode_v2_mq.argtypes = [vp, vp] + base[1:8] + [ci] + base[8:]   # q_len after num_seqs
    lib.pa_decode_v2_mq.restype = ci
    # out, lse, query .. seq_lens, scale, k_scale, v_scale, then pa_decode_v2's from num_seqs on
    lib.pa_decode_v2_fp8.argtypes = [vp, vp] + base[1:7] + [cf, cf] + base[7:]
    lib.pa_decode_v2_fp8.restype = ci
    # pa_decode_v2_fp8's arguments with q_len after num_seqs
    lib.pa_decode_v2_mq_fp8.argtypes = [vp, vp] + base[1:7] + [cf, cf, ci, ci] + base[8:]
    lib.pa_decode_v2_mq_fp8.restype = ci
    lib.pa_decode_v2_host_io.argtypes = base
    lib.pa_decode_v2_host_io.restype = ci
    lib.pa_decode_v2_host_io_workspace_bytes.argtypes = [ci] * 7
    lib.pa_decode_v2_host_io_workspace_bytes.restype = cs
    lib.pa_decode_v2_device_status.argtypes = [vp, vp, ctypes.POINTER(ci)]
    lib.pa_decode_v2_device_status.restype = ci
    lib.pa_decode_v2_status_string.argtypes = [ci]
    lib.pa_decode_v2_status_string.restype = ctypes.c_char_p
    return lib


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (built on first use if absent)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not _build.up_to_date():
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing and could not be built")
            _lib = _declare(ctypes.CDLL(path))
        return _lib


def status_string(status: int) -> str:
    return lib().pa_decode_v2_status_string(int(status)).decode()


def workspace_bytes(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, block_size,
                    partition_size) -> int:
    return int(lib().pa_decode_v2_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_size,
                                                  max_blocks_per_seq, block_size, partition_size))


def workspace_layout(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, block_size,
                     partition_size):
    """Byte offsets (max_logits, exp_sums, tmp_output, header, total) and Pmax."""
    offs = (ctypes.c_size_t * 5)()
    pmax = ctypes.c_int(0)
    st = lib().pa_decode_v2_workspace_layout(num_seqs, num_heads, num_kv_heads, head_size,
                                             max_blocks_per_seq, block_size, partition_size, offs,
                                             ctypes.byref(pmax))
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_workspace_layout")
    return tuple(int(v) for v in offs), int(pmax.value)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, like: torch.Tensor | None = None) -> int | None:
    """The CUDA stream handle to launch on: ``stream`` (a torch stream or a raw
    handle), else PyTorch's current stream on ``like``'s device (looked up
    through the raw-stream accessor where PyTorch has one: the public
    ``torch.cuda.current_stream()`` costs about 3 us a call)."""
    if stream is None:
        if _raw_stream is not None and like is not None:
            return _raw_stream(like.get_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_tensor(name, t, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")


def pa_decode_v2(out, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                 partition_size: int = 512, workspace: torch.Tensor | None = None, stream=None,
                 variant: int = PA_VARIANT_AUTO, max_ctas: int = 0, timeout_ns: int = 0,
                 lse: torch.Tensor | None = None):
    """Paged decode attention into ``out`` (see include/pa_decode.h).

    Shapes: query/out [S, H, D]; key_cache [NB, KH, D/x, BS, x] with
    x = 16 / element size (8 for fp16/bf16, 4 for fp32); value_cache
    [NB, KH, D, BS]; block_tables [S, MB] int32; seq_lens [S] int32.
    ``workspace`` (uint8, >= workspace_bytes(...)) is allocated if omitted.
    ``lse`` (float32 [S, H], optional) receives each (sequence, head)'s
    log-sum-exp of the scaled scores (``pa_decode_v2_lse``; the kernel family
    is then chosen automatically).
    Returns the workspace used."""
    _check_tensor("query", query, ndim=3)
    dt = query.dtype
    if dt not in _DTYPE_CODE_F32:
        raise TypeError("query must be float16, bfloat16 or float32")
    _check_tensor("out", out, dt, 3)
    _check_tensor("key_cache", key_cache, dt, 5)
    _check_tensor("value_cache", value_cache, dt, 4)
    _check_tensor("block_tables", block_tables, torch.int32, 2)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    S, H, D = query.shape
    NB, KH, DX, BS, X = key_cache.shape
    if tuple(out.shape) != (S, H, D) or X != 16 // query.element_size() or DX * X != D:
        raise ValueError("inconsistent query / out / key_cache shapes")
    if tuple(value_cache.shape) != (NB, KH, D, BS):
        raise ValueError("value_cache must be [num_blocks, KH, D, BS]")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens must have num_seqs rows")
    MB = block_tables.shape[1]
    if workspace is None:  # (a caller's workspace is checked by the library: PA_ERR_WORKSPACE)
        workspace = torch.empty(max(workspace_bytes(S, H, KH, D, MB, BS, partition_size), 256), dtype=torch.uint8,
                                device=query.device)
    _check_tensor("workspace", workspace, torch.uint8)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, 2)
        if tuple(lse.shape) != (S, H):
            raise ValueError("lse must be [num_seqs, num_heads]")
        if variant != PA_VARIANT_AUTO or max_ctas or timeout_ns:
            raise ValueError("lse is returned with the automatic kernel choice and defaults only")
        st = lib().pa_decode_v2_lse(
            _ptr(out), _ptr(lse), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
            _ptr(seq_lens), float(scale), S, H, KH, D, BS, int(partition_size), _DTYPE_CODE_F32[dt],
            _stream_handle(stream, query), MB, NB, _ptr(workspace), workspace.numel())
        if st != PA_OK:
            raise PaError(st, "pa_decode_v2_lse")
        return workspace
    st = lib().pa_decode_v2_ex(
        _ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        _ptr(seq_lens), float(scale), S, H, KH, D, BS, int(partition_size), _DTYPE_CODE_F32[dt],
        _stream_handle(stream, query), MB, NB, _ptr(workspace), workspace.numel(), int(variant),
        int(max_ctas), int(timeout_ns))
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2")
    return workspace


def pa_decode_v2_mq(out, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                    partition_size: int = 512, workspace: torch.Tensor | None = None, stream=None,
                    lse: torch.Tensor | None = None):
    """Multi-query decode into ``out`` (see include/pa_decode.h): query/out
    [S, q_len, H, D] (fp16, bf16 or fp32, key layout as for
    :func:`pa_decode_v2`); each query row i of sequence s attends to positions
    0 .. seq_lens[s] - q_len + i.  ``lse`` (float32 [S, q_len, H]) is optional.
    Returns the workspace used."""
    _check_tensor("query", query, ndim=4)
    dt = query.dtype
    if dt not in _DTYPE_CODE_F32:
        raise TypeError("query must be float16, bfloat16 or float32")
    _check_tensor("out", out, dt, 4)
    _check_tensor("key_cache", key_cache, dt, 5)
    _check_tensor("value_cache", value_cache, dt, 4)
    _check_tensor("block_tables", block_tables, torch.int32, 2)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    S, QL, H, D = query.shape
    NB, KH, DX, BS, X = key_cache.shape
    if tuple(out.shape) != (S, QL, H, D) or X != 16 // query.element_size() or DX * X != D:
        raise ValueError("inconsistent query / out / key_cache shapes")
    if tuple(value_cache.shape) != (NB, KH, D, BS):
        raise ValueError("value_cache must be [num_blocks, KH, D, BS]")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens must have num_seqs rows")
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, 3)
        if tuple(lse.shape) != (S, QL, H):
            raise ValueError("lse must be [num_seqs, q_len, num_heads]")
    MB = block_tables.shape[1]
    if workspace is None:  # (a caller's workspace is checked by the library: PA_ERR_WORKSPACE)
        workspace = torch.empty(max(workspace_bytes(S * QL, H, KH, D, MB, BS, partition_size), 256), dtype=torch.uint8,
                                device=query.device)
    _check_tensor("workspace", workspace, torch.uint8)
    st = lib().pa_decode_v2_mq(
        _ptr(out), _ptr(lse), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        _ptr(seq_lens), float(scale), S, QL, H, KH, D, BS, int(partition_size), _DTYPE_CODE_F32[dt],
        _stream_handle(stream, query), MB, NB, _ptr(workspace), workspace.numel())
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_mq")
    return workspace


# Sequences one phase-1 kernel launch takes (the kernel's order and prefix
# arrays); a call launches phase 1 once per this many sequences, whatever q_len.
MAX_ROWS_PER_LAUNCH = 512


def launches_per_call(num_seqs: int, q_len: int = 1, max_partitions: int = 2) -> int:
    """Kernel launches one call makes (for launch counts in measurements):
    the header clear and phase 1 once per MAX_ROWS_PER_LAUNCH sequences, and
    the phase-2 combine once if a sequence can have more than one partition
    (``max_partitions`` = ceil(max_blocks_per_seq * block_size / partition_size))."""
    return 2 * max(1, -(-num_seqs // MAX_ROWS_PER_LAUNCH)) + (1 if max_partitions > 1 else 0)


def pa_decode_v2_fp8(out, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                     k_scale: float = 1.0, v_scale: float = 1.0, partition_size: int = 512,
                     workspace: torch.Tensor | None = None, stream=None, lse: torch.Tensor | None = None):
    """Decode over an fp8 (E4M3) KV cache (see include/pa_decode.h): query/out
    [S, H, D] fp16 or bf16; key_cache uint8 [NB, KH, D/16, BS, 16] and
    value_cache uint8 [NB, KH, D, BS] hold E4M3 codes; real keys / values are
    k_scale * K and v_scale * V.  ``lse`` (float32 [S, H]) is optional.
    Returns the workspace used."""
    _check_tensor("query", query, ndim=3)
    dt = query.dtype
    if dt not in _DTYPE_CODE:
        raise TypeError("query must be float16 or bfloat16")
    _check_tensor("out", out, dt, 3)
    _check_tensor("key_cache", key_cache, torch.uint8, 5)
    _check_tensor("value_cache", value_cache, torch.uint8, 4)
    _check_tensor("block_tables", block_tables, torch.int32, 2)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    S, H, D = query.shape
    NB, KH, DX, BS, X = key_cache.shape
    if tuple(out.shape) != (S, H, D) or X != 16 or DX * X != D:
        raise ValueError("inconsistent query / out / key_cache shapes (fp8 key_cache is [NB, KH, D/16, BS, 16])")
    if tuple(value_cache.shape) != (NB, KH, D, BS):
        raise ValueError("value_cache must be [num_blocks, KH, D, BS]")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens must have num_seqs rows")
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, 2)
        if tuple(lse.shape) != (S, H):
            raise ValueError("lse must be [num_seqs, num_heads]")
    MB = block_tables.shape[1]
    if workspace is None:  # (a caller's workspace is checked by the library: PA_ERR_WORKSPACE)
        workspace = torch.empty(max(workspace_bytes(S, H, KH, D, MB, BS, partition_size), 256), dtype=torch.uint8,
                                device=query.device)
    _check_tensor("workspace", workspace, torch.uint8)
    st = lib().pa_decode_v2_fp8(
        _ptr(out), _ptr(lse), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        _ptr(seq_lens), float(scale), float(k_scale), float(v_scale), S, H, KH, D, BS,
        int(partition_size), _DTYPE_CODE[dt], _stream_handle(stream, query), MB, NB, _ptr(workspace),
        workspace.numel())
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_fp8")
    return workspace


def pa_decode_v2_mq_fp8(out, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                        k_scale: float = 1.0, v_scale: float = 1.0, partition_size: int = 512,
                        workspace: torch.Tensor | None = None, stream=None, lse: torch.Tensor | None = None):
    """Multi-query decode over an fp8 (E4M3) KV cache (see include/pa_decode.h):
    query/out [S, q_len, H, D] fp16 or bf16, each query row i of sequence s
    attending to positions 0 .. seq_lens[s] - q_len + i; the caches hold E4M3
    codes as for :func:`pa_decode_v2_fp8`.  ``lse`` (float32 [S, q_len, H]) is
    optional.  Returns the workspace used."""
    _check_tensor("query", query, ndim=4)
    dt = query.dtype
    if dt not in _DTYPE_CODE:
        raise TypeError("query must be float16 or bfloat16")
    _check_tensor("out", out, dt, 4)
    _check_tensor("key_cache", key_cache, torch.uint8, 5)
    _check_tensor("value_cache", value_cache, torch.uint8, 4)
    _check_tensor("block_tables", block_tables, torch.int32, 2)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    S, QL, H, D = query.shape
    NB, KH, DX, BS, X = key_cache.shape
    if tuple(out.shape) != (S, QL, H, D) or X != 16 or DX * X != D:
        raise ValueError("inconsistent query / out / key_cache shapes (fp8 key_cache is [NB, KH, D/16, BS, 16])")
    if tuple(value_cache.shape) != (NB, KH, D, BS):
        raise ValueError("value_cache must be [num_blocks, KH, D, BS]")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens must have num_seqs rows")
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, 3)
        if tuple(lse.shape) != (S, QL, H):
            raise ValueError("lse must be [num_seqs, q_len, num_heads]")
    MB = block_tables.shape[1]
    if workspace is None:  # (a caller's workspace is checked by the library: PA_ERR_WORKSPACE)
        workspace = torch.empty(max(workspace_bytes(S * QL, H, KH, D, MB, BS, partition_size), 256), dtype=torch.uint8,
                                device=query.device)
    _check_tensor("workspace", workspace, torch.uint8)
    st = lib().pa_decode_v2_mq_fp8(
        _ptr(out), _ptr(lse), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        _ptr(seq_lens), float(scale), float(k_scale), float(v_scale), S, QL, H, KH, D, BS,
        int(partition_size), _DTYPE_CODE[dt], _stream_handle(stream, query), MB, NB, _ptr(workspace),
        workspace.numel())
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_mq_fp8")
    return workspace


def host_io_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq,
                            block_size, partition_size) -> int:
    return int(lib().pa_decode_v2_host_io_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_size,
                                                          max_blocks_per_seq, block_size,
                                                          partition_size))


def pa_decode_v2_host_io(out_host, query_host, key_cache, value_cache, block_tables_host,
                         seq_lens_host, scale: float, partition_size: int, workspace: torch.Tensor,
                         stream=None):
    """Decode with per-step inputs and output in host memory (pinned CPU
    tensors) and the caches on the device; enqueued on ``stream``, not
    synchronised."""
    for name, t in (("out_host", out_host), ("query_host", query_host),
                    ("block_tables_host", block_tables_host), ("seq_lens_host", seq_lens_host)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    _check_tensor("key_cache", key_cache, query_host.dtype, 5)
    _check_tensor("value_cache", value_cache, query_host.dtype, 4)
    _check_tensor("workspace", workspace, torch.uint8)
    if query_host.dtype not in _DTYPE_CODE_F32 or out_host.dtype != query_host.dtype:
        raise TypeError("query_host / out_host must be float16, bfloat16 or float32")
    if block_tables_host.dtype != torch.int32 or seq_lens_host.dtype != torch.int32:
        raise TypeError("block_tables_host / seq_lens_host must be int32")
    S, H, D = query_host.shape
    NB, KH, _, BS, _ = key_cache.shape
    MB = block_tables_host.shape[1]
    st = lib().pa_decode_v2_host_io(
        _ptr(out_host), _ptr(query_host), _ptr(key_cache), _ptr(value_cache),
        _ptr(block_tables_host), _ptr(seq_lens_host), float(scale), S, H, KH, D, BS,
        int(partition_size), _DTYPE_CODE_F32[query_host.dtype], _stream_handle(stream, key_cache), MB, NB,
        _ptr(workspace), workspace.numel())
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_host_io")


def device_status(workspace: torch.Tensor, stream=None) -> int:
    """Device-side error word of the last call on ``workspace`` (synchronises the stream)."""
    v = ctypes.c_int(0)
    st = lib().pa_decode_v2_device_status(_ptr(workspace), _stream_handle(stream, workspace), ctypes.byref(v))
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_device_status")
    return int(v.value)
