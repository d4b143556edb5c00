"""fp64 CPU oracle for paged KV-cache attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library (``paged_kv_cache_27_gb300``) and never imports it.

Contents:
  * ``oracle.c`` (built into ``liboracle.so`` by :func:`build`): decode over a
    paged cache, full causal attention, varlen prefill, append scatter, and
    the split-softmax partial/merge pair, all in fp64; :func:`decode_multi`
    (several new tokens per sequence) composes the decode; the fp8 e4m3
    codec, the per-row quantizer and the decode over an fp8 cache.
  * :mod:`oracle.page_pool`: the block pool and per-request block table of
    the PagedAttention article, restated.
  * :mod:`oracle.paging`: slot arithmetic, cache filling and the serving-mix
    protocol driven on :class:`oracle.page_pool.PagePool`.
  * :mod:`oracle.geometry`: the KV-cache byte-count formula.

Parity status of each function is recorded in its docstring; every function
here is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (strict IEEE fp64: no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_half_to_double.restype = D
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_array_to_double.restype = None
            lib.oracle_half_array_to_double.argtypes = [P, P, ctypes.c_int64]
            lib.oracle_decode.restype = I
            lib.oracle_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I, D, P, I]
            lib.oracle_causal_attention.restype = I
            lib.oracle_causal_attention.argtypes = [P, P, P, I, I, D, P]
            lib.oracle_prefill.restype = I
            lib.oracle_prefill.argtypes = [P, P, P, P, I, I, I, I, D, I, P, I]
            lib.oracle_append.restype = I
            lib.oracle_append.argtypes = [P, P, P, P, P, I, I, I, I, I]
            lib.oracle_partial.restype = None
            lib.oracle_partial.argtypes = [P, P, P, I, I, I, D, P, P, P]
            lib.oracle_merge.restype = None
            lib.oracle_merge.argtypes = [P, P, P, I, I, P]
            lib.oracle_e4m3_to_double.restype = D
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_quantize_fp8.restype = None
            lib.oracle_quantize_fp8.argtypes = [P, ctypes.c_int64, I, P, P]
            lib.oracle_decode_fp8.restype = I
            lib.oracle_decode_fp8.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I, I, D, P, I]
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits: np.ndarray) -> np.ndarray:
    """Exact binary16 -> fp64 widening from the bit patterns (uint16 array)."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_half_array_to_double(_ptr(bits), _ptr(out), bits.size)
    return out


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float16, a.dtype
    return a.view(np.uint16)


def decode(q, k_cache, v_cache, block_table, context_lens, scale, nthreads=None):
    """Decode over one layer of a paged cache, fp64.

    q [B][Hq][D] f16; k_cache/v_cache [NB][Hkv][bs][D] f16; block_table int32
    [B][max_blocks]; context_lens int32 [B] (including the appended token).
    Returns out [B][Hq][D] float64.  Raises on an out-of-range index.
    """
    q = _bits(q)
    kc, vc = _bits(k_cache), _bits(v_cache)
    NB, Hkv, bs, D = kc.shape
    B, Hq, Dq = q.shape
    assert Dq == D and vc.shape == kc.shape
    table = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = _load().oracle_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(table), table.shape[1], _ptr(ctx), B,
                               Hq, Hkv, D, bs, NB, float(scale), _ptr(out),
                               nthreads or default_threads())
    if rc != 0:
        raise IndexError("oracle_decode: context length or block id out of range")
    return out


def decode_multi(q, k_cache, v_cache, block_table, context_lens, scale, nthreads=None):
    """Multi-token decode, fp64: q [B][T][Hq][D] holds each sequence's T newest tokens (in the cache already,
    context_lens including them); token t sits at position ctx - T + t and attends to positions 0 .. ctx - T + t
    (verifying T drafted tokens in one pass over them: speculative-decoding paragraph of "Tornar a inferência
    barata", neuralialabs.com).  Each token is the plain decode over its own prefix of the context.
    Returns out [B][T][Hq][D] float64.  Pinned against full causal attention on gathered sequences."""
    q = np.asarray(q)
    B, T = q.shape[:2]
    ctx = np.asarray(context_lens, dtype=np.int32)
    if np.any(ctx < T):
        raise IndexError("decode_multi: a context is shorter than the new tokens")
    out = np.empty(q.shape, dtype=np.float64)
    for t in range(T):
        out[:, t] = decode(np.ascontiguousarray(q[:, t]), k_cache, v_cache, block_table, ctx - T + 1 + t, scale,
                           nthreads)
    return out


# ---- fp8 e4m3 cache (an extension; the pages fix no quantized KV format) ------------------------------
def e4m3_to_float64(codes) -> np.ndarray:
    """Value of every e4m3 code (1 sign, 4 exponent bits bias 7, 3 fraction bits; 0x7F / 0xFF are NaN)."""
    codes = np.asarray(codes, dtype=np.uint8)
    lib = _load()
    table = np.array([lib.oracle_e4m3_to_double(c) for c in range(256)], dtype=np.float64)
    return table[codes]


def e4m3_from_float32(x) -> np.ndarray:
    """Nearest e4m3 code of each binary32 value, ties to even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float32)
    lib = _load()
    return np.array([lib.oracle_e4m3_from_float(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def quantize_fp8(x):
    """Rows of D fp16 values (last axis) -> (codes uint8 like x, scales float32 x.shape[:-1]): scale = absmax /
    448 in binary32 (1 for an all-zero row), code = e4m3(x / scale) with the quotient in binary32."""
    x = _bits(np.asarray(x))
    D = x.shape[-1]
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.float32)
    _load().oracle_quantize_fp8(_ptr(x), rows, D, _ptr(codes), _ptr(scales))
    return codes, scales


def decode_fp8(q, k_codes, v_codes, k_scales, v_scales, block_table, context_lens, scale, nthreads=None):
    """Decode over an fp8 cache: codes [NB][Hkv][bs][D] uint8, scales [NB][Hkv][bs] float32; every cached value
    is code value x scale (exact in fp64); otherwise :func:`decode`.  Returns out [B][Hq][D] float64."""
    q = _bits(q)
    kq, vq = _c(k_codes, np.uint8), _c(v_codes, np.uint8)
    ks, vs = _c(k_scales, np.float32), _c(v_scales, np.float32)
    NB, Hkv, bs, D = kq.shape
    B, Hq, Dq = q.shape
    assert Dq == D and vq.shape == kq.shape and ks.shape == (NB, Hkv, bs) and vs.shape == ks.shape
    table = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = _load().oracle_decode_fp8(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ks), _ptr(vs), _ptr(table), table.shape[1],
                                   _ptr(ctx), B, Hq, Hkv, D, bs, NB, float(scale), _ptr(out),
                                   nthreads or default_threads())
    if rc != 0:
        raise IndexError("oracle_decode_fp8: context length or block id out of range")
    return out


def causal_attention(Q, K, V, scale):
    """Full n x n causal attention on one contiguous sequence (fp64 arrays [n][D])."""
    Q, K, V = (_c(x, np.float64) for x in (Q, K, V))
    n, D = Q.shape
    O = np.empty((n, D), dtype=np.float64)
    if _load().oracle_causal_attention(_ptr(Q), _ptr(K), _ptr(V), n, D, float(scale), _ptr(O)) != 0:
        raise MemoryError("oracle_causal_attention")
    return O


def prefill(q, k, v, cu_seqlens, scale, causal=True, nthreads=None):
    """Varlen packed prefill: q [T][Hq][D], k/v [T][Hkv][D] f16 -> out [T][Hq][D] fp64."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    cu = _c(cu_seqlens, np.int32)
    out = np.empty((T, Hq, D), dtype=np.float64)
    rc = _load().oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, Hq, Hkv, D,
                                float(scale), int(bool(causal)), _ptr(out),
                                nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_prefill: bad cu_seqlens")
    return out


def append(k_cache, v_cache, k_new, v_new, slot_mapping):
    """Scatter rows of k_new/v_new ([n][Hkv][D] f16) into one layer's cache in place."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    kc, vc = k_cache.view(np.uint16), v_cache.view(np.uint16)
    NB, Hkv, bs, D = kc.shape
    kn, vn = _bits(k_new), _bits(v_new)
    slots = _c(slot_mapping, np.int64)
    rc = _load().oracle_append(_ptr(kc), _ptr(vc), _ptr(kn), _ptr(vn), _ptr(slots), len(slots), Hkv, D,
                               bs, NB)
    if rc != 0:
        raise IndexError("oracle_append: slot out of range")


def partial(q, K, V, j0, j1, scale):
    """Partial softmax over rows [j0, j1): returns (m, l, acc[D]), fp64."""
    q, K, V = (_c(x, np.float64) for x in (q, K, V))
    D = q.shape[0]
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(D)
    _load().oracle_partial(_ptr(q), _ptr(K), _ptr(V), int(j0), int(j1), D, float(scale), _ptr(m), _ptr(l),
                           _ptr(acc))
    return float(m[0]), float(l[0]), acc


def merge(ms, ls, accs):
    """Merge split partials (m_s, l_s, acc_s) into the normalised output."""
    ms, ls, accs = _c(ms, np.float64), _c(ls, np.float64), _c(accs, np.float64)
    n, D = accs.shape
    out = np.zeros(D)
    _load().oracle_merge(_ptr(ms), _ptr(ls), _ptr(accs), n, D, _ptr(out))
    return out
