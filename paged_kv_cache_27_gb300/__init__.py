"""Paged KV-cache attention for GB300 (sm_103a): Python binding of ``libkvc.so``.

Every function here marshals arguments (tensor pointers, sizes, the current
CUDA stream) and calls the C ABI of the same name declared in
``include/kvc.h``; all arithmetic runs in the library's CUDA kernels or its
native host code.  There is no fallback: if the library has not been built
(``paged_kv_cache_27_gb300.build()``), importing this package raises.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch  # loads the CUDA runtime that libkvc.so links against

from ._build import LIB as _LIB_PATH
from ._build import build

__all__ = [
    "KvcError", "KvcConfig", "KVC_F16", "KVC_F32", "build", "lib_path",
    "kvc_version", "kvc_set_checked_mode", "kvc_device_error_flags", "kv_cache_pool_bytes",
    "kv_cache_create", "kv_cache_destroy", "kv_cache_layer", "kv_block_alloc", "kv_block_share",
    "kv_block_release", "kv_block_refcount", "kv_block_num_free", "kv_cache_utilisation",
    "kv_block_cow", "kv_copy_blocks", "kv_slot_mapping", "kv_step_prepare", "kv_append",
    "paged_decode_plan", "paged_decode_workspace_init", "paged_decode_attention",
    "paged_decode_append_attention", "kvc_set_launch_overlap", "kvc_set_cascade_min_saved_blocks", "kvc_set_multi_tc", "kvc_copy_async", "KVC_COPY_AHEAD", "PreparedCall",
    "kvc_trace_read",
    "paged_decode_attention_static_workspace", "paged_decode_cascade_plan", "paged_decode_cascade_attention", "kv_cascade_groups",
    "paged_decode_multi_plan", "paged_decode_multi_attention", "kv_append_fp8", "paged_decode_attention_fp8",
    "kv_fp8_record_bytes",
    "prefill_attention", "prefill_attention_ex", "fp8_v_position", "DEVERR",
]

KVC_F16, KVC_F32 = 0, 1
KVC_PREFILL_P_F16, KVC_PREFILL_P_SPLIT = 0, 1
STATUS = {0: "KVC_OK", 1: "KVC_ERR_INVALID", 2: "KVC_ERR_OOM", 3: "KVC_ERR_CAPACITY", 4: "KVC_ERR_CUDA",
          5: "KVC_ERR_UNSUPPORTED"}
DEVERR = {"BLOCK_ID": 0x1, "CONTEXT": 0x2, "SLOT": 0x4, "TIMEOUT": 0x8, "SEQLENS": 0x10}


class KvcError(RuntimeError):
    def __init__(self, status: int, func: str, msg: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{func}: {self.name}: {msg}")


class _Config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int), ("num_blocks", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int)]


@dataclass
class KvcConfig:
    num_layers: int
    num_blocks: int
    num_kv_heads: int
    head_dim: int
    block_size: int = 16
    dtype: int = KVC_F16

    def _c(self) -> _Config:
        return _Config(self.num_layers, self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim,
                       self.dtype)

    @property
    def pool_shape(self):
        return (self.num_layers, self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)


def lib_path() -> str:
    return _LIB_PATH


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libkvc.so is not built ({_LIB_PATH}); run paged_kv_cache_27_gb300.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, I32, I64, SZ, D = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                             ctypes.c_double)
    PI32, PI64, PSZ, PI = (ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64),
                           ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_int))
    sig = {
        "kvc_last_error_string": (ctypes.c_char_p, []),
        "kvc_version": (I, []),
        "kvc_set_checked_mode": (I, [I]),
        "kvc_device_error_flags": (I, [ctypes.POINTER(ctypes.c_uint32), I]),
        "kv_cache_pool_bytes": (I, [ctypes.POINTER(_Config), PSZ]),
        "kv_cache_create": (I, [ctypes.POINTER(_Config), P, P, ctypes.POINTER(P)]),
        "kv_cache_destroy": (I, [P]),
        "kv_cache_layer": (I, [P, I, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "kv_block_alloc": (I, [P, PI32]),
        "kv_block_share": (I, [P, I32]),
        "kv_block_release": (I, [P, I32]),
        "kv_block_refcount": (I, [P, I32, PI32]),
        "kv_block_num_free": (I, [P, PI32]),
        "kv_cache_utilisation": (I, [P, ctypes.POINTER(D)]),
        "kv_block_cow": (I, [P, I32, PI32, P]),
        "kv_copy_blocks": (I, [P, P, P, I, P]),
        "kv_slot_mapping": (I, [P, I, I, P, P, I, P]),
        "kv_step_prepare": (I, [P, P, I, P, P, I, P, P, P, PI]),
        "kv_append": (I, [P, I, P, P, P, I, P]),
        "paged_decode_plan": (I, [I, I, I, I, I, I, I, PI, PI, PSZ]),
        "paged_decode_workspace_init": (I, [P, SZ, P]),
        "paged_decode_attention": (I, [P, P, P, I, P, I, P, I, I, I, I, I, I, ctypes.c_float, P, I, P, SZ, I, P]),
        "paged_decode_append_attention": (I, [P, P, P, P, P, I, P, I, P, I, I, I, I, I, I, ctypes.c_float, P,
                                              I, P, SZ, I, P]),
        "kvc_set_launch_overlap": (I, [I]),
        "kvc_set_cascade_min_saved_blocks": (I, [I]),
        "kvc_set_multi_tc": (I, [I]),
        "kvc_copy_async": (I, [P, P, SZ, ctypes.c_uint, P]),
        "paged_decode_attention_static_workspace": (I, [P, P, P, I, P, I, P, I, I, I, I, I, I, ctypes.c_float, P, I,
                                                        I, P]),
        "kvc_trace_read": (I, [P, I, PI, I]),
        "paged_decode_cascade_plan": (I, [I, I, I, I, I, I, I, I, PSZ]),
        "kv_cascade_groups": (I, [P, I, I, P, I, I, P, PI, P, PI]),
        "paged_decode_multi_plan": (I, [I, I, I, I, I, I, I, PSZ]),
        "kv_fp8_record_bytes": (I, [I, PSZ]),
        "kv_append_fp8": (I, [P, P, P, I, P, I, I, I, I, P]),
        "paged_decode_attention_fp8": (I, [P, P, I, P, I, P, I, I, I, I, I, I, ctypes.c_float, P, I, P, SZ, I, P]),
        "paged_decode_multi_attention": (I, [P, P, P, I, P, I, P, I, I, I, I, I, I, I, ctypes.c_float, P, I, P, SZ,
                                             P]),
        "paged_decode_cascade_attention": (I, [P, P, P, I, P, I, P, P, P, I, I, I, I, I, I, I, I, ctypes.c_float, P,
                                               I, P, SZ, P]),
        "prefill_attention": (I, [P, P, P, P, I, I, I, I, I, I, ctypes.c_float, I, P, I, P]),
        "prefill_attention_ex": (I, [P, P, P, P, I, I, I, I, I, I, ctypes.c_float, I, I, P, I, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(status: int, func: str):
    if status != 0:
        raise KvcError(status, func, _lib.kvc_last_error_string().decode(errors="replace"))


# the current stream of a device as a raw handle, without building a torch.cuda.Stream object (a few µs per call)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, *tensors) -> Optional[int]:
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    for t in tensors:
        if isinstance(t, torch.Tensor) and t.is_cuda:
            if _raw_stream is not None:
                return _raw_stream(t.get_device())
            return torch.cuda.current_stream(t.device).cuda_stream
    return None


def _dptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    # the common case in one expression (dtypes are singletons); the checks below only name the failure
    if isinstance(t, torch.Tensor) and t.is_cuda and (dtype is None or t.dtype is dtype) and t.is_contiguous():
        return t.data_ptr()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    raise ValueError(f"{name} must be contiguous")


class PreparedCall:
    """One library call whose arguments were checked and converted once (the `prepare=True` form of a launching
    call): calling it launches that call again, on `stream` or else the current stream of the call's device.  It
    keeps its tensors alive; their contents may change between launches, their storage must stay where it is.
    Saves the per-call checks and conversions (~5 µs of host time per decode call)."""
    __slots__ = ("_fn", "_args", "_name", "_device", "_keep")

    def __init__(self, fn, args, name, device, keep):
        self._fn, self._name, self._device, self._keep = fn, name, device, keep
        self._args = tuple(a if a is None else at(a) for a, at in zip(args, fn.argtypes))

    def __call__(self, stream=None) -> None:
        if stream is not None:
            st = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        elif _raw_stream is not None:
            st = _raw_stream(self._device)
        else:
            st = torch.cuda.current_stream(self._device).cuda_stream
        _check(self._fn(*self._args, st), self._name)


def _launch(fn, args, name, stream, prepare, keep):
    """Launch fn(*args, stream), or return it as a PreparedCall; keep[0] is a CUDA tensor of the call."""
    if prepare:
        return PreparedCall(fn, args, name, keep[0].get_device(), keep)
    _check(fn(*args, _stream(stream, keep[0])), name)
    return None


def _host(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _np_ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ---------------------------------------------------------------- diagnostics
def kvc_version() -> int:
    return _lib.kvc_version()


def kvc_set_checked_mode(on: bool) -> None:
    _check(_lib.kvc_set_checked_mode(int(bool(on))), "kvc_set_checked_mode")


def kvc_set_cascade_min_saved_blocks(blocks: int) -> None:
    """Cascade calls saving fewer than `blocks` block reads per KV head ((B - n_groups) * max_shared_blocks) run the
    plain decode (0: always the cascade kernels)."""
    _check(_lib.kvc_set_cascade_min_saved_blocks(int(blocks)), "kvc_set_cascade_min_saved_blocks")


def kvc_set_multi_tc(on: bool) -> None:
    """Multi-token calls at head dim 64 with up to 64 query rows on the tensor-core kernel (off: the mma.sync kernel)."""
    _check(_lib.kvc_set_multi_tc(int(bool(on))), "kvc_set_multi_tc")


def kvc_set_launch_overlap(on: bool) -> None:
    """Launch decode kernels as programmatic dependents of the previous kernel (see include/kvc.h)."""
    _check(_lib.kvc_set_launch_overlap(int(bool(on))), "kvc_set_launch_overlap")


KVC_COPY_AHEAD = 1


def _stage_ptr(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda or t.device.type == "cpu"):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def kvc_copy_async(dst: torch.Tensor, src: torch.Tensor, ahead: bool = False, stream=None, prepare: bool = False):
    """Copy src's bytes into dst with the library's staging kernel (see include/kvc.h for the two orderings).

    Each of dst and src is a CUDA tensor or a pinned CPU tensor; both hold the same number of bytes, a multiple
    of 16, at 16-byte aligned addresses.  prepare=True returns a PreparedCall instead of launching."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src must hold the same number of bytes")
    args = (_stage_ptr(dst, "dst"), _stage_ptr(src, "src"), nbytes, KVC_COPY_AHEAD if ahead else 0)
    if prepare:
        cuda = dst if dst.is_cuda else src
        return PreparedCall(_lib.kvc_copy_async, args, "kvc_copy_async",
                            cuda.get_device() if cuda.is_cuda else torch.cuda.current_device(), (dst, src))
    _check(_lib.kvc_copy_async(*args, _stream(stream, dst, src)), "kvc_copy_async")


TRACE_DTYPE = np.dtype([("t", "<u8", (8,)), ("seq", "<u4"), ("smid", "<u4"), ("x", "<u4"), ("yz", "<u4")])


def kvc_trace_read(capacity: int = 1 << 16, clear: bool = True) -> np.ndarray:
    """Decode-kernel timeline records (library built with -DKVC_TRACE=1)."""
    buf = np.zeros(capacity, dtype=TRACE_DTYPE)
    n = ctypes.c_int(0)
    _check(_lib.kvc_trace_read(_np_ptr(buf), capacity, ctypes.byref(n), int(bool(clear))), "kvc_trace_read")
    return buf[:n.value]


def kvc_device_error_flags(clear: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _check(_lib.kvc_device_error_flags(ctypes.byref(v), int(bool(clear))), "kvc_device_error_flags")
    return v.value


# ------------------------------------------------------------ cache / pool
def kv_cache_pool_bytes(cfg: KvcConfig) -> int:
    n = ctypes.c_size_t(0)
    c = cfg._c()
    _check(_lib.kv_cache_pool_bytes(ctypes.byref(c), ctypes.byref(n)), "kv_cache_pool_bytes")
    return n.value


def kv_cache_create(cfg: KvcConfig, k_pool: Optional[torch.Tensor] = None,
                    v_pool: Optional[torch.Tensor] = None) -> int:
    """Handle over caller-owned pools (fp16 [L][NB][Hkv][bs][D]); None, None = host-only pool."""
    if (k_pool is None) != (v_pool is None):
        raise ValueError("k_pool and v_pool: both or neither")
    if k_pool is not None:
        need = kv_cache_pool_bytes(cfg)
        for t, nm in ((k_pool, "k_pool"), (v_pool, "v_pool")):
            if t.numel() * t.element_size() < need:
                raise ValueError(f"{nm} holds {t.numel() * t.element_size()} bytes, needs {need}")
    h = ctypes.c_void_p()
    c = cfg._c()
    _check(_lib.kv_cache_create(ctypes.byref(c), _dptr(k_pool, torch.float16, "k_pool"),
                                _dptr(v_pool, torch.float16, "v_pool"), ctypes.byref(h)), "kv_cache_create")
    return h.value


def kv_cache_destroy(h: int) -> None:
    _check(_lib.kv_cache_destroy(h), "kv_cache_destroy")


def kv_cache_layer(h: int, layer: int):
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(_lib.kv_cache_layer(h, layer, ctypes.byref(k), ctypes.byref(v)), "kv_cache_layer")
    return k.value, v.value


def kv_block_alloc(h: int) -> int:
    b = ctypes.c_int32()
    _check(_lib.kv_block_alloc(h, ctypes.byref(b)), "kv_block_alloc")
    return b.value


def kv_block_share(h: int, block: int) -> None:
    _check(_lib.kv_block_share(h, int(block)), "kv_block_share")


def kv_block_release(h: int, block: int) -> None:
    _check(_lib.kv_block_release(h, int(block)), "kv_block_release")


def kv_block_refcount(h: int, block: int) -> int:
    r = ctypes.c_int32()
    _check(_lib.kv_block_refcount(h, int(block), ctypes.byref(r)), "kv_block_refcount")
    return r.value


def kv_block_num_free(h: int) -> int:
    r = ctypes.c_int32()
    _check(_lib.kv_block_num_free(h, ctypes.byref(r)), "kv_block_num_free")
    return r.value


def kv_cache_utilisation(h: int) -> float:
    r = ctypes.c_double()
    _check(_lib.kv_cache_utilisation(h, ctypes.byref(r)), "kv_cache_utilisation")
    return r.value


def kv_block_cow(h: int, block: int, stream=None) -> int:
    r = ctypes.c_int32()
    _check(_lib.kv_block_cow(h, int(block), ctypes.byref(r), _stream(stream)), "kv_block_cow")
    return r.value


def kv_copy_blocks(h: int, src: Sequence[int], dst: Sequence[int], stream=None) -> None:
    s, d = _host(src, np.int32), _host(dst, np.int32)
    if s.shape != d.shape:
        raise ValueError("src and dst differ in length")
    _check(_lib.kv_copy_blocks(h, _np_ptr(s), _np_ptr(d), len(s), _stream(stream)), "kv_copy_blocks")


# ------------------------------------------------------------ slots (host)
def kv_slot_mapping(block_table: np.ndarray, first_pos, count, block_size: int = 16) -> np.ndarray:
    table = _host(block_table, np.int32)
    fp, cn = _host(first_pos, np.int32), _host(count, np.int32)
    B, mb = table.shape
    out = np.empty(int(cn.astype(np.int64).sum()), dtype=np.int64)
    _check(_lib.kv_slot_mapping(_np_ptr(table), mb, B, _np_ptr(fp), _np_ptr(cn), block_size, _np_ptr(out)),
           "kv_slot_mapping")
    return out


def kv_step_prepare(h: int, block_table: np.ndarray, num_blocks: np.ndarray, positions):
    """One decode step's allocation / copy-on-write; block_table and num_blocks are updated in place.

    Returns (slot_mapping int64 [B], copy pairs int32 [n][2])."""
    if block_table.dtype != np.int32 or not block_table.flags.c_contiguous:
        raise TypeError("block_table must be a C-contiguous int32 array")
    if num_blocks.dtype != np.int32 or not num_blocks.flags.c_contiguous:
        raise TypeError("num_blocks must be a C-contiguous int32 array")
    pos = _host(positions, np.int32)
    B, mb = block_table.shape
    slots = np.empty(B, dtype=np.int64)
    src = np.empty(max(B, 1), dtype=np.int32)
    dst = np.empty(max(B, 1), dtype=np.int32)
    n = ctypes.c_int(0)
    _check(_lib.kv_step_prepare(h, _np_ptr(block_table), mb, _np_ptr(num_blocks), _np_ptr(pos), B, _np_ptr(slots),
                                _np_ptr(src), _np_ptr(dst), ctypes.byref(n)), "kv_step_prepare")
    return slots, np.stack([src[:n.value], dst[:n.value]], axis=1)


# ------------------------------------------------------------ device ops
def kv_append(h: int, layer: int, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
              stream=None, prepare: bool = False):
    """Scatter rows of k_new/v_new ([n][Hkv][D] fp16) to slot_mapping (int64 [n]) of one layer.

    prepare=True returns a PreparedCall instead of launching."""
    n = k_new.shape[0]
    if v_new.shape != k_new.shape or slot_mapping.numel() != n:
        raise ValueError("k_new, v_new and slot_mapping must agree in n")
    args = (h, layer, _dptr(k_new, torch.float16, "k_new"), _dptr(v_new, torch.float16, "v_new"),
            _dptr(slot_mapping, torch.int64, "slot_mapping"), n)
    return _launch(_lib.kv_append, args, "kv_append", stream, prepare, (k_new, v_new, slot_mapping))


def paged_decode_plan(B: int, Hq: int, Hkv: int, head_dim: int, max_context_len: int, blocks_per_split: int = 0,
                      block_size: int = 16):
    ns, bps, ws = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    _check(_lib.paged_decode_plan(B, Hq, Hkv, head_dim, block_size, max_context_len, blocks_per_split,
                                  ctypes.byref(ns), ctypes.byref(bps), ctypes.byref(ws)), "paged_decode_plan")
    return ns.value, bps.value, ws.value


def paged_decode_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    _check(_lib.paged_decode_workspace_init(_dptr(workspace, None, "workspace"),
                                            workspace.numel() * workspace.element_size(),
                                            _stream(stream, workspace)), "paged_decode_workspace_init")


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                           context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                           workspace: Optional[torch.Tensor], max_context_len: int, blocks_per_split: int = 0,
                           stream=None, prepare: bool = False):
    """out = softmax(q K^T * scale) V per sequence over its paged context.

    q [B][Hq][D] fp16; k_cache/v_cache [NB][Hkv][bs][D] fp16 (one layer); block_table int32 [B][max_blocks];
    context_lens int32 [B]; out [B][Hq][D] fp16 or fp32; workspace: paged_decode_plan(...) bytes (uint8/any).
    prepare=True returns a PreparedCall instead of launching.
    """
    B, Hq, D = q.shape
    NB, Hkv, bs, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shapes do not match q")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_table.dim() != 2 or block_table.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_table / context_lens do not match B")
    if out.dtype == torch.float16:
        od = KVC_F16
    elif out.dtype == torch.float32:
        od = KVC_F32
    else:
        raise TypeError("out must be float16 or float32")
    ws_ptr = _dptr(workspace, None, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (_dptr(q, torch.float16, "q"), _dptr(k_cache, torch.float16, "k_cache"),
            _dptr(v_cache, torch.float16, "v_cache"), NB, _dptr(block_table, torch.int32, "block_table"),
            block_table.shape[1], _dptr(context_lens, torch.int32, "context_lens"), B, Hq, Hkv, D, bs,
            int(max_context_len), float(scale), _dptr(out, None, "out"), od, ws_ptr, ws_bytes,
            int(blocks_per_split))
    return _launch(_lib.paged_decode_attention, args, "paged_decode_attention", stream, prepare,
                   (q, k_cache, v_cache, block_table, context_lens, out, workspace))


def kv_cascade_groups(block_table: np.ndarray, context_lens, max_group: int = 8, block_size: int = 16):
    """Groups for paged_decode_cascade_attention from a host block table [B][max_blocks] and context lengths:
    returns (group_start int32 [n_groups + 1], shared_blocks int32 [B], max_shared)."""
    table = _host(block_table, np.int32)
    if table.ndim != 2:
        raise ValueError("block_table must be [B][max_blocks]")
    B, mb = table.shape
    ctx = _host(context_lens, np.int32)
    gs = np.zeros(B + 1, dtype=np.int32)
    sh = np.zeros(max(B, 1), dtype=np.int32)
    ng, mx = ctypes.c_int(), ctypes.c_int()
    _check(_lib.kv_cascade_groups(_np_ptr(table), B, mb, _np_ptr(ctx), block_size, max_group, _np_ptr(gs),
                                  ctypes.byref(ng), _np_ptr(sh), ctypes.byref(mx)), "kv_cascade_groups")
    return gs[:ng.value + 1].copy(), sh[:B].copy(), mx.value


def paged_decode_cascade_plan(B: int, Hq: int, Hkv: int, head_dim: int, max_context_len: int, n_groups: int,
                              max_shared_blocks: int, block_size: int = 16) -> int:
    """Workspace bytes of paged_decode_cascade_attention for these sizes."""
    ws = ctypes.c_size_t()
    _check(_lib.paged_decode_cascade_plan(B, Hq, Hkv, head_dim, block_size, max_context_len, n_groups,
                                          max_shared_blocks, ctypes.byref(ws)), "paged_decode_cascade_plan")
    return ws.value


def paged_decode_cascade_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                   block_table: torch.Tensor, context_lens: torch.Tensor, group_start: torch.Tensor,
                                   shared_blocks: torch.Tensor, max_shared_blocks: int, scale: float,
                                   out: torch.Tensor, workspace: torch.Tensor, max_context_len: int,
                                   stream=None) -> None:
    """paged_decode_attention's result, with each group's shared leading blocks read once for the group.

    group_start int32 [n_groups + 1] (groups of consecutive sequences, at most 8 each); shared_blocks int32 [B]
    (leading blocks every member of the sequence's group has in common); workspace: paged_decode_cascade_plan bytes.
    """
    B, Hq, D = q.shape
    NB, Hkv, bs, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shapes do not match q")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_table.dim() != 2 or block_table.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_table / context_lens do not match B")
    if shared_blocks.numel() != B or group_start.numel() < 2:
        raise ValueError("shared_blocks must have B entries and group_start at least 2")
    if out.dtype == torch.float16:
        od = KVC_F16
    elif out.dtype == torch.float32:
        od = KVC_F32
    else:
        raise TypeError("out must be float16 or float32")
    _check(_lib.paged_decode_cascade_attention(
        _dptr(q, torch.float16, "q"), _dptr(k_cache, torch.float16, "k_cache"),
        _dptr(v_cache, torch.float16, "v_cache"), NB, _dptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _dptr(context_lens, torch.int32, "context_lens"),
        _dptr(group_start, torch.int32, "group_start"), _dptr(shared_blocks, torch.int32, "shared_blocks"),
        group_start.numel() - 1, int(max_shared_blocks), B, Hq, Hkv, D, bs, int(max_context_len), float(scale),
        _dptr(out, None, "out"), od, _dptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream, q)), "paged_decode_cascade_attention")


def paged_decode_multi_plan(B: int, Hq: int, Hkv: int, head_dim: int, max_context_len: int, q_len: int,
                            block_size: int = 16) -> int:
    """Workspace bytes of paged_decode_multi_attention for these sizes."""
    ws = ctypes.c_size_t()
    _check(_lib.paged_decode_multi_plan(B, Hq, Hkv, head_dim, block_size, max_context_len, q_len, ctypes.byref(ws)),
           "paged_decode_multi_plan")
    return ws.value


def paged_decode_multi_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 block_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                 out: torch.Tensor, workspace: torch.Tensor, max_context_len: int,
                                 stream=None) -> None:
    """q [B][q_len][Hq][D] fp16: the q_len newest tokens of every sequence (already in the cache), causal among
    themselves; out like q (fp16 or fp32); workspace: paged_decode_multi_plan bytes."""
    B, T, Hq, D = q.shape
    NB, Hkv, bs, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shapes do not match q")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_table.dim() != 2 or block_table.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_table / context_lens do not match B")
    if out.dtype == torch.float16:
        od = KVC_F16
    elif out.dtype == torch.float32:
        od = KVC_F32
    else:
        raise TypeError("out must be float16 or float32")
    _check(_lib.paged_decode_multi_attention(
        _dptr(q, torch.float16, "q"), _dptr(k_cache, torch.float16, "k_cache"),
        _dptr(v_cache, torch.float16, "v_cache"), NB, _dptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _dptr(context_lens, torch.int32, "context_lens"), T, B, Hq, Hkv, D, bs,
        int(max_context_len), float(scale), _dptr(out, None, "out"), od, _dptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream, q)), "paged_decode_multi_attention")


def fp8_v_position(tau: int) -> int:
    """Byte position of token tau (0..15) of a block within each 16-byte dim row of an fp8 record's V codes."""
    return 4 * ((tau & 7) >> 1) + 2 * (tau >> 3) + (tau & 1)


def kv_fp8_record_bytes(head_dim: int) -> int:
    """Bytes of one fp8 cache record (one per (block, KV head)): 32 * head_dim + 128."""
    n = ctypes.c_size_t()
    _check(_lib.kv_fp8_record_bytes(int(head_dim), ctypes.byref(n)), "kv_fp8_record_bytes")
    return n.value


def kv_append_fp8(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor, kv_fp8: torch.Tensor,
                  stream=None) -> None:
    """Quantize k_new / v_new (fp16 [n][Hkv][D]) into an fp8 cache layer kv_fp8, uint8 [NB][Hkv][record] (one
    record of kv_fp8_record_bytes(D) per (block, KV head): K codes, K scales, V codes, V scales; value = e4m3
    code value * scale); slot_mapping int64 [n]."""
    n, Hkv, D = k_new.shape
    NB, Hkv2, rec = kv_fp8.shape
    if Hkv2 != Hkv or rec != kv_fp8_record_bytes(D) or v_new.shape != k_new.shape or slot_mapping.numel() != n:
        raise ValueError("fp8 cache shapes do not match")
    _check(_lib.kv_append_fp8(
        _dptr(k_new, torch.float16, "k_new"), _dptr(v_new, torch.float16, "v_new"),
        _dptr(slot_mapping, torch.int64, "slot_mapping"), n, _dptr(kv_fp8, torch.uint8, "kv_fp8"), NB, Hkv, D, 16,
        _stream(stream, k_new)), "kv_append_fp8")


def paged_decode_attention_fp8(q: torch.Tensor, kv_fp8: torch.Tensor, block_table: torch.Tensor,
                               context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                               workspace: Optional[torch.Tensor], max_context_len: int, blocks_per_split: int = 0,
                               stream=None) -> None:
    """paged_decode_attention over an fp8 cache layer (kv_fp8 uint8 [NB][Hkv][record] as kv_append_fp8 writes it)."""
    B, Hq, D = q.shape
    NB, Hkv, rec = kv_fp8.shape
    if rec != kv_fp8_record_bytes(D):
        raise ValueError("fp8 cache records do not match q's head dim")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_table.dim() != 2 or block_table.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_table / context_lens do not match B")
    od = {torch.float16: KVC_F16, torch.float32: KVC_F32}.get(out.dtype)
    if od is None:
        raise TypeError("out must be float16 or float32")
    ws_ptr = _dptr(workspace, None, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.paged_decode_attention_fp8(
        _dptr(q, torch.float16, "q"), _dptr(kv_fp8, torch.uint8, "kv_fp8"), NB,
        _dptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dptr(context_lens, torch.int32, "context_lens"), B, Hq, Hkv, D, 16, int(max_context_len), float(scale),
        _dptr(out, None, "out"), od, ws_ptr, ws_bytes, int(blocks_per_split), _stream(stream, q)),
        "paged_decode_attention_fp8")


def paged_decode_append_attention(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                                  v_cache: torch.Tensor, block_table: torch.Tensor, context_lens: torch.Tensor,
                                  scale: float, out: torch.Tensor, workspace: Optional[torch.Tensor],
                                  max_context_len: int, blocks_per_split: int = 0, stream=None,
                                  prepare: bool = False):
    """Append k_new/v_new ([B][Hkv][D] fp16) at position ctx-1 of every sequence, then attend (one kernel).

    prepare=True returns a PreparedCall instead of launching."""
    B, Hq, D = q.shape
    NB, Hkv, bs, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("shape mismatch")
    if k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B][Hkv][D]")
    if block_table.dim() != 2 or block_table.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_table / context_lens do not match B")
    od = KVC_F16 if out.dtype == torch.float16 else KVC_F32 if out.dtype == torch.float32 else None
    if od is None:
        raise TypeError("out must be float16 or float32")
    ws_ptr = _dptr(workspace, None, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (_dptr(q, torch.float16, "q"), _dptr(k_new, torch.float16, "k_new"), _dptr(v_new, torch.float16, "v_new"),
            _dptr(k_cache, torch.float16, "k_cache"), _dptr(v_cache, torch.float16, "v_cache"), NB,
            _dptr(block_table, torch.int32, "block_table"), block_table.shape[1],
            _dptr(context_lens, torch.int32, "context_lens"), B, Hq, Hkv, D, bs, int(max_context_len), float(scale),
            _dptr(out, None, "out"), od, ws_ptr, ws_bytes, int(blocks_per_split))
    return _launch(_lib.paged_decode_append_attention, args, "paged_decode_append_attention", stream, prepare,
                   (q, k_new, v_new, k_cache, v_cache, block_table, context_lens, out, workspace))


def paged_decode_attention_static_workspace(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                            block_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                            out: torch.Tensor, max_context_len: int, blocks_per_split: int = 0,
                                            stream=None) -> None:
    """paged_decode_attention without a workspace argument: split scratch comes from the library's fixed
    16 MiB device array, so the call allocates nothing (for callers that must not allocate device memory).

    The first call on a device looks up that array's address; make it before any stream capture. Calls that
    overlap on the GPU share the array and race on it."""
    B, Hq, D = q.shape
    NB, Hkv, bs, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("shape mismatch")
    if block_table.dim() != 2 or block_table.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_table / context_lens do not match B")
    od = KVC_F16 if out.dtype == torch.float16 else KVC_F32 if out.dtype == torch.float32 else None
    if od is None:
        raise TypeError("out must be float16 or float32")
    _check(_lib.paged_decode_attention_static_workspace(
        _dptr(q, torch.float16, "q"), _dptr(k_cache, torch.float16, "k_cache"),
        _dptr(v_cache, torch.float16, "v_cache"), NB, _dptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _dptr(context_lens, torch.int32, "context_lens"), B, Hq, Hkv, D, bs,
        int(max_context_len), float(scale), _dptr(out, None, "out"), od, int(blocks_per_split), _stream(stream, q)),
        "paged_decode_attention_static_workspace")


def paged_decode_attention_raw(q_ptr: int, k_ptr: int, v_ptr: int, num_blocks: int, table_ptr: int, max_blocks: int,
                               ctx_ptr: int, B: int, Hq: int, Hkv: int, D: int, max_context_len: int, scale: float,
                               out_ptr: int, out_dtype: int, ws_ptr: int, ws_bytes: int, blocks_per_split: int,
                               stream: int) -> None:
    """Same call with raw device pointers (e.g. a layer slice from kv_cache_layer)."""
    _check(_lib.paged_decode_attention(q_ptr, k_ptr, v_ptr, num_blocks, table_ptr, max_blocks, ctx_ptr, B, Hq, Hkv,
                                       D, 16, max_context_len, float(scale), out_ptr, out_dtype, ws_ptr, ws_bytes,
                                       blocks_per_split, stream), "paged_decode_attention")


def prefill_attention_ex(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                         max_seqlen: int, scale: float, causal: bool, p_precision: int, out: torch.Tensor,
                         stream=None) -> None:
    """Packed varlen prefill with a choice of P precision (KVC_PREFILL_P_F16 or KVC_PREFILL_P_SPLIT):
    q [T][Hq][D], k/v [T][Hkv][D] fp16, cu_seqlens int32 [nseq+1] -> out [T][Hq][D]."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, D) or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("shape mismatch")
    od = KVC_F16 if out.dtype == torch.float16 else KVC_F32 if out.dtype == torch.float32 else None
    if od is None:
        raise TypeError("out must be float16 or float32")
    _check(_lib.prefill_attention_ex(_dptr(q, torch.float16, "q"), _dptr(k, torch.float16, "k"),
                                     _dptr(v, torch.float16, "v"), _dptr(cu_seqlens, torch.int32, "cu_seqlens"),
                                     cu_seqlens.numel() - 1, T, int(max_seqlen), Hq, Hkv, D, float(scale),
                                     int(bool(causal)), int(p_precision), _dptr(out, None, "out"), od,
                                     _stream(stream, q)),
           "prefill_attention_ex")


def prefill_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor, max_seqlen: int,
                      scale: float, causal: bool, out: torch.Tensor, stream=None, precise: bool = False) -> None:
    """Packed varlen prefill: q [T][Hq][D], k/v [T][Hkv][D] fp16, cu_seqlens int32 [nseq+1] -> out [T][Hq][D].

    precise=False rounds the softmax weights P to fp16 (KVC_PREFILL_P_F16); precise=True multiplies V by
    P's fp16 high part and residual (KVC_PREFILL_P_SPLIT)."""
    prefill_attention_ex(q, k, v, cu_seqlens, max_seqlen, scale, causal,
                         KVC_PREFILL_P_SPLIT if precise else KVC_PREFILL_P_F16, out, stream)
