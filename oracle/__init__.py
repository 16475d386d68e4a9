"""fp64 CPU oracle for single-query paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
CUDA library never links, loads or calls it, and this package imports nothing
from the CUDA library: the two sides share only the seeded input generators.

What it computes follows the page "paged_attention_v2_triton.py -- Triton
PagedAttention V2 for BI-V100" (phase-1 kernel ``_paged_attn_v2_partition_kernel``
for the paged gather and scores, the module docstring and
``_paged_attn_v2_reduce_kernel`` for the combine), written as its plain
definition in ``pa_oracle.c``:

* :func:`decode`      -- softmax(scale * q . K^T) . V over all tokens, fp64,
                         no partitioning (the result the two-phase method
                         reaches);
* :func:`partitions`  -- per-partition (m_p, l_p, o_p), the phase-1 outputs,
                         with the unused-partition sentinels (-inf, 0);
* :func:`combine`     -- the phase-2 log-sum-exp combine of those states;
* :func:`lse`         -- log-sum-exp of each (sequence, head)'s scaled scores,
                         the value the forward kernel of the page
                         "flash_attention.metal -- Flash Attention Metal Shaders"
                         stores beside its output (max plus log of the sum);
* :func:`combine_lse` -- the same from phase-1 states (M + log total);
* :func:`decode_mq`   -- multi-query decode: q_len new tokens per sequence, the
                         i-th at position L - q_len + i attending causally to
                         positions 0 .. L - q_len + i (output and log-sum-exp);
* :func:`decode_fp8kv` -- decode over an E4M3 (fp8) KV cache with per-tensor
                         k_scale / v_scale (key layout x = 16), and
  :func:`e4m3_decode`   the code -> value map it uses;
* :func:`decode_mq_fp8kv` -- multi-query decode (the causal rows of
                         :func:`decode_mq`) over an E4M3 cache (the keys and
                         values of :func:`decode_fp8kv`);
* :func:`decode_fp32` -- decode with fp32 query and caches (key layout x = 4);
* :func:`decode_mq_fp32` -- multi-query decode (the causal rows of
                         :func:`decode_mq`) with fp32 query and caches.

Inputs are the raw 16-bit patterns of fp16 / bf16 tensors (numpy ``uint16``)
in the page's layouts; the fp32 ``scale`` is widened to double exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpa_oracle.so")

DTYPE_FP16 = 0
DTYPE_BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile ``pa_oracle.c`` (or ``src``) with gcc + OpenMP into a shared library."""
    src = src or _SRC
    out = out or _LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    up = ctypes.POINTER(ctypes.c_uint16)
    ip = ctypes.POINTER(ctypes.c_int32)
    c_int, c_double = ctypes.c_int, ctypes.c_double
    lib.pa_oracle_decode.argtypes = [dp, up, up, up, ip, ip, c_double] + [c_int] * 8
    lib.pa_oracle_decode.restype = c_int
    lib.pa_oracle_partitions.argtypes = [dp, dp, dp, up, up, up, ip, ip, c_double] + [c_int] * 10
    lib.pa_oracle_partitions.restype = c_int
    lib.pa_oracle_combine.argtypes = [dp, dp, dp, dp, ip] + [c_int] * 5
    lib.pa_oracle_combine.restype = c_int
    lib.pa_oracle_lse.argtypes = [dp, up, up, ip, ip, c_double] + [c_int] * 8
    lib.pa_oracle_lse.restype = c_int
    lib.pa_oracle_combine_lse.argtypes = [dp, dp, dp, ip] + [c_int] * 4
    lib.pa_oracle_combine_lse.restype = c_int
    lib.pa_oracle_decode_mq.argtypes = [dp, dp, up, up, up, ip, ip, c_double] + [c_int] * 9
    lib.pa_oracle_decode_mq.restype = c_int
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.pa_oracle_e4m3_decode.argtypes = [dp, u8p, c_int]
    lib.pa_oracle_e4m3_decode.restype = c_int
    lib.pa_oracle_decode_fp8kv.argtypes = [dp, dp, up, u8p, u8p, ip, ip, c_double, c_double, c_double] + [c_int] * 8
    lib.pa_oracle_decode_fp8kv.restype = c_int
    lib.pa_oracle_decode_mq_fp8kv.argtypes = ([dp, dp, up, u8p, u8p, ip, ip, c_double, c_double, c_double]
                                              + [c_int] * 9)
    lib.pa_oracle_decode_mq_fp8kv.restype = c_int
    fp = ctypes.POINTER(ctypes.c_float)
    lib.pa_oracle_decode_fp32.argtypes = [dp, dp, fp, fp, fp, ip, ip, c_double] + [c_int] * 7
    lib.pa_oracle_decode_fp32.restype = c_int
    lib.pa_oracle_decode_mq_fp32.argtypes = [dp, dp, fp, fp, fp, ip, ip, c_double] + [c_int] * 8
    lib.pa_oracle_decode_mq_fp32.restype = c_int
    lib.pa_oracle_max_threads.argtypes = []
    lib.pa_oracle_max_threads.restype = c_int
    return lib


def load_library(path: str) -> ctypes.CDLL:
    """Load an oracle shared library built from ``pa_oracle.c`` (or a variant of it)."""
    return _declare(ctypes.CDLL(path))


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def max_threads() -> int:
    return int(lib().pa_oracle_max_threads())


def _u16(a) -> np.ndarray:
    """Raw 16-bit pattern of an fp16 / bf16 array (numpy or torch) as contiguous uint16."""
    if hasattr(a, "detach"):  # torch tensor: reinterpret the bits on the CPU
        import torch

        a = a.detach().cpu().contiguous()
        if a.dtype in (torch.float16, torch.bfloat16):
            a = a.view(torch.int16)
        a = a.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected 16-bit float data, got {a.dtype}")
    return a


def _u8(a) -> np.ndarray:
    """Raw bytes of an fp8 / uint8 array (numpy or torch) as contiguous uint8."""
    if hasattr(a, "detach"):
        import torch

        a = a.detach().cpu().contiguous()
        if a.dtype != torch.uint8:
            a = a.view(torch.uint8)
        a = a.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"expected 8-bit codes, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _shapes(query, key_cache, value_cache, block_tables):
    S, H, D = query.shape
    nb, KH, dx, BS, x = key_cache.shape
    if x != 8 or dx * x != D:
        raise ValueError("key_cache must be [num_blocks, KH, D/8, BS, 8]")
    if tuple(value_cache.shape) != (nb, KH, D, BS):
        raise ValueError("value_cache must be [num_blocks, KH, D, BS]")
    MB = block_tables.shape[1]
    return S, H, KH, D, BS, MB


def _f32(a) -> np.ndarray:
    """An fp32 array (numpy or torch) as contiguous float32."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"expected float32 data, got {a.dtype}")
    return a


class Oracle:
    """The oracle's entry points bound to one compiled copy of ``pa_oracle.c``."""

    def __init__(self, library: ctypes.CDLL):
        self.lib = library

    def decode(self, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
               dtype: int, nthreads: int = 0) -> np.ndarray:
        """fp64 softmax(scale * q . K^T) . V over each sequence's tokens; returns [S, H, D] float64."""
        q, kc, vc = _u16(query), _u16(key_cache), _u16(value_cache)
        bt, lens = _i32(block_tables), _i32(seq_lens)
        S, H, KH, D, BS, MB = _shapes(q, kc, vc, bt)
        out = np.zeros((S, H, D), dtype=np.float64)
        rc = self.lib.pa_oracle_decode(
            _ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16), _ptr(kc, ctypes.c_uint16),
            _ptr(vc, ctypes.c_uint16), _ptr(bt, ctypes.c_int32), _ptr(lens, ctypes.c_int32),
            float(np.float32(scale)), S, H, KH, D, BS, MB, dtype, nthreads)
        if rc != 0:
            raise ValueError("oracle decode rejected its arguments")
        return out

    def partitions(self, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                   dtype: int, partition_size: int, max_partitions: int | None = None,
                   nthreads: int = 0):
        """Phase-1 states: (m [S,H,Pmax], l [S,H,Pmax], o [S,H,Pmax,D]) in float64."""
        q, kc, vc = _u16(query), _u16(key_cache), _u16(value_cache)
        bt, lens = _i32(block_tables), _i32(seq_lens)
        S, H, KH, D, BS, MB = _shapes(q, kc, vc, bt)
        P = int(partition_size)
        if max_partitions is None:
            max_partitions = -(-(MB * BS) // P)
        Pm = int(max_partitions)
        m = np.zeros((S, H, Pm), dtype=np.float64)
        l = np.zeros((S, H, Pm), dtype=np.float64)
        o = np.zeros((S, H, Pm, D), dtype=np.float64)
        rc = self.lib.pa_oracle_partitions(
            _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double), _ptr(o, ctypes.c_double),
            _ptr(q, ctypes.c_uint16), _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16),
            _ptr(bt, ctypes.c_int32), _ptr(lens, ctypes.c_int32), float(np.float32(scale)),
            S, H, KH, D, BS, MB, P, Pm, dtype, nthreads)
        if rc != 0:
            raise ValueError("oracle partitions rejected its arguments")
        return m, l, o

    def combine(self, m, l, o, seq_lens, partition_size: int) -> np.ndarray:
        """Phase-2 combine of phase-1 states; returns [S, H, D] float64."""
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        o = np.ascontiguousarray(o, dtype=np.float64)
        lens = _i32(seq_lens)
        S, H, Pm, D = o.shape
        out = np.zeros((S, H, D), dtype=np.float64)
        rc = self.lib.pa_oracle_combine(
            _ptr(out, ctypes.c_double), _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double),
            _ptr(o, ctypes.c_double), _ptr(lens, ctypes.c_int32), S, H, D, int(partition_size), Pm)
        if rc != 0:
            raise ValueError("oracle combine rejected its arguments")
        return out


    def lse(self, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
            dtype: int, nthreads: int = 0) -> np.ndarray:
        """fp64 log-sum-exp of scale * q . K^T over each sequence's tokens; [S, H] (-inf if empty)."""
        q, kc, vc = _u16(query), _u16(key_cache), _u16(value_cache)
        bt, lens = _i32(block_tables), _i32(seq_lens)
        S, H, KH, D, BS, MB = _shapes(q, kc, vc, bt)
        out = np.zeros((S, H), dtype=np.float64)
        rc = self.lib.pa_oracle_lse(
            _ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16), _ptr(kc, ctypes.c_uint16),
            _ptr(bt, ctypes.c_int32), _ptr(lens, ctypes.c_int32), float(np.float32(scale)),
            S, H, KH, D, BS, MB, dtype, nthreads)
        if rc != 0:
            raise ValueError("oracle lse rejected its arguments")
        return out

    def combine_lse(self, m, l, seq_lens, partition_size: int) -> np.ndarray:
        """Log-sum-exp from phase-1 states (M + log total); [S, H] float64."""
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        lens = _i32(seq_lens)
        S, H, Pm = m.shape
        out = np.zeros((S, H), dtype=np.float64)
        rc = self.lib.pa_oracle_combine_lse(
            _ptr(out, ctypes.c_double), _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double),
            _ptr(lens, ctypes.c_int32), S, H, int(partition_size), Pm)
        if rc != 0:
            raise ValueError("oracle combine_lse rejected its arguments")
        return out


    def decode_mq(self, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                  dtype: int, nthreads: int = 0):
        """Multi-query decode; query is [S, q_len, H, D].  Returns (out [S, q_len, H, D],
        lse [S, q_len, H]) in float64."""
        q, kc, vc = _u16(query), _u16(key_cache), _u16(value_cache)
        bt, lens = _i32(block_tables), _i32(seq_lens)
        S, q_len, H, D = q.shape
        _, KH, _, BS, _ = kc.shape
        _shapes(q.reshape(S * q_len, H, D), kc, vc, np.zeros((S * q_len, bt.shape[1]), np.int32))
        MB = bt.shape[1]
        out = np.zeros((S, q_len, H, D), dtype=np.float64)
        lse = np.zeros((S, q_len, H), dtype=np.float64)
        rc = self.lib.pa_oracle_decode_mq(
            _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), _ptr(q, ctypes.c_uint16),
            _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16), _ptr(bt, ctypes.c_int32),
            _ptr(lens, ctypes.c_int32), float(np.float32(scale)), S, q_len, H, KH, D, BS, MB, dtype,
            nthreads)
        if rc != 0:
            raise ValueError("oracle decode_mq rejected its arguments")
        return out, lse


    def e4m3_decode(self, codes) -> np.ndarray:
        """Values of E4M3 codes (uint8 array-like) as float64."""
        c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
        out = np.zeros(c.shape, dtype=np.float64)
        rc = self.lib.pa_oracle_e4m3_decode(_ptr(out, ctypes.c_double), _ptr(c, ctypes.c_uint8), c.size)
        if rc != 0:
            raise ValueError("oracle e4m3_decode rejected its arguments")
        return out

    def decode_fp8kv(self, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                     k_scale: float, v_scale: float, qdtype: int, nthreads: int = 0):
        """Decode over E4M3 caches (uint8 codes: key_cache [NB, KH, D/16, BS, 16], value_cache
        [NB, KH, D, BS]); returns (out [S, H, D], lse [S, H]) in float64."""
        q = _u16(query)
        kc, vc = _u8(key_cache), _u8(value_cache)
        bt, lens = _i32(block_tables), _i32(seq_lens)
        S, H, D = q.shape
        nb, KH, dx, BS, x = kc.shape
        if x != 16 or dx * x != D or tuple(vc.shape) != (nb, KH, D, BS):
            raise ValueError("fp8 caches must be [NB, KH, D/16, BS, 16] and [NB, KH, D, BS]")
        MB = bt.shape[1]
        out = np.zeros((S, H, D), dtype=np.float64)
        lse = np.zeros((S, H), dtype=np.float64)
        rc = self.lib.pa_oracle_decode_fp8kv(
            _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), _ptr(q, ctypes.c_uint16),
            _ptr(kc, ctypes.c_uint8), _ptr(vc, ctypes.c_uint8), _ptr(bt, ctypes.c_int32),
            _ptr(lens, ctypes.c_int32), float(np.float32(scale)), float(np.float32(k_scale)),
            float(np.float32(v_scale)), S, H, KH, D, BS, MB, qdtype, nthreads)
        if rc != 0:
            raise ValueError("oracle decode_fp8kv rejected its arguments")
        return out, lse


    def decode_mq_fp8kv(self, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                        k_scale: float, v_scale: float, qdtype: int, nthreads: int = 0):
        """Multi-query decode (query [S, q_len, H, D]) over E4M3 caches laid out as for
        decode_fp8kv; returns (out [S, q_len, H, D], lse [S, q_len, H]) in float64."""
        q = _u16(query)
        kc, vc = _u8(key_cache), _u8(value_cache)
        bt, lens = _i32(block_tables), _i32(seq_lens)
        S, q_len, H, D = q.shape
        nb, KH, dx, BS, x = kc.shape
        if x != 16 or dx * x != D or tuple(vc.shape) != (nb, KH, D, BS):
            raise ValueError("fp8 caches must be [NB, KH, D/16, BS, 16] and [NB, KH, D, BS]")
        if bt.shape[0] != S or lens.shape[0] != S:
            raise ValueError("block_tables and seq_lens need one row per sequence")
        MB = bt.shape[1]
        out = np.zeros((S, q_len, H, D), dtype=np.float64)
        lse = np.zeros((S, q_len, H), dtype=np.float64)
        rc = self.lib.pa_oracle_decode_mq_fp8kv(
            _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), _ptr(q, ctypes.c_uint16),
            _ptr(kc, ctypes.c_uint8), _ptr(vc, ctypes.c_uint8), _ptr(bt, ctypes.c_int32),
            _ptr(lens, ctypes.c_int32), float(np.float32(scale)), float(np.float32(k_scale)),
            float(np.float32(v_scale)), S, q_len, H, KH, D, BS, MB, qdtype, nthreads)
        if rc != 0:
            raise ValueError("oracle decode_mq_fp8kv rejected its arguments")
        return out, lse

    def decode_fp32(self, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                        nthreads: int = 0):
        """Decode with fp32 query and caches (key_cache [NB, KH, D/4, BS, 4], value_cache
        [NB, KH, D, BS]); returns (out [S, H, D], lse [S, H]) in float64."""
        q, kc, vc = _f32(query), _f32(key_cache), _f32(value_cache)
        bt, lens = _i32(block_tables), _i32(seq_lens)
        S, H, D = q.shape
        nb, KH, dx, BS, x = kc.shape
        if x != 4 or dx * x != D or tuple(vc.shape) != (nb, KH, D, BS):
            raise ValueError("fp32 caches must be [NB, KH, D/4, BS, 4] and [NB, KH, D, BS]")
        MB = bt.shape[1]
        out = np.zeros((S, H, D), dtype=np.float64)
        lse = np.zeros((S, H), dtype=np.float64)
        rc = self.lib.pa_oracle_decode_fp32(
            _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), _ptr(q, ctypes.c_float),
            _ptr(kc, ctypes.c_float), _ptr(vc, ctypes.c_float), _ptr(bt, ctypes.c_int32),
            _ptr(lens, ctypes.c_int32), float(np.float32(scale)), S, H, KH, D, BS, MB, nthreads)
        if rc != 0:
            raise ValueError("oracle decode_fp32 rejected its arguments")
        return out, lse

    def decode_mq_fp32(self, query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                       nthreads: int = 0):
        """Multi-query decode (query [S, q_len, H, D]) with fp32 query and caches laid
        out as for decode_fp32; returns (out [S, q_len, H, D], lse [S, q_len, H]) in float64."""
        q, kc, vc = _f32(query), _f32(key_cache), _f32(value_cache)
        bt, lens = _i32(block_tables), _i32(seq_lens)
        S, q_len, H, D = q.shape
        nb, KH, dx, BS, x = kc.shape
        if x != 4 or dx * x != D or tuple(vc.shape) != (nb, KH, D, BS):
            raise ValueError("fp32 caches must be [NB, KH, D/4, BS, 4] and [NB, KH, D, BS]")
        if bt.shape[0] != S or lens.shape[0] != S:
            raise ValueError("block_tables and seq_lens need one row per sequence")
        MB = bt.shape[1]
        out = np.zeros((S, q_len, H, D), dtype=np.float64)
        lse = np.zeros((S, q_len, H), dtype=np.float64)
        rc = self.lib.pa_oracle_decode_mq_fp32(
            _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), _ptr(q, ctypes.c_float),
            _ptr(kc, ctypes.c_float), _ptr(vc, ctypes.c_float), _ptr(bt, ctypes.c_int32),
            _ptr(lens, ctypes.c_int32), float(np.float32(scale)), S, q_len, H, KH, D, BS, MB, nthreads)
        if rc != 0:
            raise ValueError("oracle decode_mq_fp32 rejected its arguments")
        return out, lse

_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(lib())
    return _default


def decode(*args, **kwargs) -> np.ndarray:
    return default().decode(*args, **kwargs)


def partitions(*args, **kwargs):
    return default().partitions(*args, **kwargs)


def combine(*args, **kwargs) -> np.ndarray:
    return default().combine(*args, **kwargs)


def lse(*args, **kwargs) -> np.ndarray:
    return default().lse(*args, **kwargs)


def combine_lse(*args, **kwargs) -> np.ndarray:
    return default().combine_lse(*args, **kwargs)


def decode_mq(*args, **kwargs):
    return default().decode_mq(*args, **kwargs)


def e4m3_decode(*args, **kwargs) -> np.ndarray:
    return default().e4m3_decode(*args, **kwargs)


def decode_fp8kv(*args, **kwargs):
    return default().decode_fp8kv(*args, **kwargs)


def decode_mq_fp8kv(*args, **kwargs):
    return default().decode_mq_fp8kv(*args, **kwargs)


def decode_fp32(*args, **kwargs):
    return default().decode_fp32(*args, **kwargs)


def decode_mq_fp32(*args, **kwargs):
    return default().decode_mq_fp32(*args, **kwargs)
