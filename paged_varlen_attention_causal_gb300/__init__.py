"""GB300 (sm_103a) paged varlen causal GQA attention with the Inkling relative bias.

Thin Python binding over the C ABI in ``include/ink_attn.h`` (libinkattn.so):
argument checking and marshalling only; every step of the computation runs in
the library's CUDA kernels.  PyTorch provides device memory and the stream.
The binding raises if the library is not built: there is no fallback path.

    out = ink_rel_attn_varlen(q, key_cache, value_cache, block_table=...,
                              cache_seqlens=..., cu_seqlens_q=..., max_seqlen_q=...,
                              softmax_scale=..., causal=True, window_left=-1,
                              window_right=-1, rel_extent=E, rel_logits=...)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

__all__ = [
    "LibraryNotBuilt", "InkError", "Dims", "build", "load", "ink_rel_attn_varlen", "workspace_size",
    "num_splits", "read_device_errors", "version", "DEVERR", "set_timing_events", "launch_count",
    "reshape_and_cache", "ink_rel_attn_varlen_fp8kv", "reshape_and_cache_fp8", "stage_bytes",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libinkattn.so")

DEVERR = {
    "PAGE_ID": 0x01, "CU_SEQLENS": 0x02, "SEQLEN_Q": 0x04, "SEQLEN_K": 0x08, "EMPTY_ROWS": 0x10,
    "TIMEOUT": 0x100, "SMEM": 0x200, "STAGE": 0x400,
}
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "workspace too small",
           4: "CUDA error"}


class LibraryNotBuilt(RuntimeError):
    pass


class InkError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_tokens", "batch", "num_heads", "num_kv_heads", "head_dim", "num_blocks", "block_size",
        "max_blocks_per_seq")]


_lock = threading.Lock()
_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libinkattn.so in-tree (nvcc, sm_103a)."""
    from ._build import build as _b

    return _b(force=force, verbose=verbose)


def load(path: Optional[str] = None):
    """Load the C-ABI library (raises LibraryNotBuilt when it is missing)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise LibraryNotBuilt(f"{p} is missing: run paged_varlen_attention_causal_gb300.build() first")
        lib = ctypes.CDLL(p)
        i32, sz, vp = ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p
        dp = ctypes.POINTER(Dims)
        lib.ink_rel_attn_workspace_size.restype = sz
        lib.ink_rel_attn_workspace_size.argtypes = [dp, i32, i32]
        lib.ink_rel_attn_stage_bytes.restype = sz
        lib.ink_rel_attn_stage_bytes.argtypes = [dp, ctypes.c_int64]
        lib.ink_rel_attn_num_splits.restype = i32
        lib.ink_rel_attn_num_splits.argtypes = [dp, i32, i32, i32, i32]
        lib.ink_rel_attn_varlen.restype = ctypes.c_int
        lib.ink_rel_attn_varlen.argtypes = [
            dp, vp, vp, vp, vp, vp, vp, i32, ctypes.c_float, ctypes.c_int, i32, i32, i32, vp, i32,
            vp, vp, vp, sz, vp]
        lib.ink_rel_attn_varlen_fp8kv.restype = ctypes.c_int
        lib.ink_rel_attn_varlen_fp8kv.argtypes = [
            dp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp, vp, i32, ctypes.c_float, ctypes.c_int, i32,
            i32, i32, vp, i32, vp, vp, vp, sz, vp]
        lib.ink_status_string.restype = ctypes.c_char_p
        lib.ink_status_string.argtypes = [ctypes.c_int]
        lib.ink_rel_attn_read_device_errors.restype = ctypes.c_int
        lib.ink_rel_attn_read_device_errors.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.ink_attn_version.restype = i32
        lib.ink_set_timing_events.restype = None
        lib.ink_set_timing_events.argtypes = [ctypes.c_int, vp, vp]
        lib.ink_launch_count.restype = ctypes.c_uint64
        lib.ink_reshape_and_cache.restype = ctypes.c_int
        lib.ink_reshape_and_cache.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp]
        lib.ink_reshape_and_cache_fp8.restype = ctypes.c_int
        lib.ink_reshape_and_cache_fp8.argtypes = [dp, vp, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp]
        if path is None:
            _lib = lib
        return lib


def version() -> int:
    return int(load().ink_attn_version())


KERNELS = {"prepass": 1, "decode": 2, "prefill": 3, "combine": 4, "append": 5, "stage": 6}


def set_timing_events(kernel: str, start=None, stop=None) -> None:
    """Record torch.cuda.Event `start`/`stop` around the named kernel's launches (None clears)."""
    load().ink_set_timing_events(KERNELS[kernel], None if start is None else start.cuda_event,
                                 None if stop is None else stop.cuda_event)


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load().ink_launch_count())


def _dims(q, key_cache, block_table) -> Dims:
    T, H, D = q.shape
    NB, BS, Hkv, D2 = key_cache.shape
    if D2 != D:
        raise ValueError("q and the caches differ in head_dim")
    B, W = block_table.shape
    return Dims(T, B, H, Hkv, D, NB, BS, W)


def workspace_size(dims: Dims, max_seqlen_q: int, num_splits: int = 0) -> int:
    n = load().ink_rel_attn_workspace_size(ctypes.byref(dims), int(max_seqlen_q), int(num_splits))
    if n == 0:
        raise InkError(1, "ink_rel_attn_workspace_size")
    return int(n)


def stage_bytes(dims: Dims, prefill_kv_tokens: int) -> int:
    """Extra workspace bytes that stage the K/V of prefill-shaped requests holding `prefill_kv_tokens` cache
    keys in total (ink_rel_attn_stage_bytes)."""
    return int(load().ink_rel_attn_stage_bytes(ctypes.byref(dims), int(prefill_kv_tokens)))


def num_splits(dims: Dims, max_seqlen_q: int, max_kv_len: int, window_left: int = -1,
               window_right: int = -1) -> int:
    return int(load().ink_rel_attn_num_splits(ctypes.byref(dims), int(max_seqlen_q), int(max_kv_len),
                                              int(window_left), int(window_right)))


_ws_cache: dict = {}


def _workspace(device: torch.device, nbytes: int, stream) -> torch.Tensor:
    """Per (device, stream) workspace, grown on demand (calls on one stream are ordered)."""
    key = (device.index, int(stream.cuda_stream))
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _check(t: torch.Tensor, name: str, dtype, dim: int, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, got shape {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _prepare(q, key_cache, value_cache, cache_dtype, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
             rel_extent, rel_logits, num_splits, out, lse, return_lse, workspace, stream, stage_kv_tokens=0):
    """Checks and marshals the arguments both attention entry points share."""
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _check(q, "q", torch.bfloat16, 3, dev)
    _check(key_cache, "key_cache", cache_dtype, 4, dev)
    _check(value_cache, "value_cache", cache_dtype, 4, dev)
    if value_cache.shape != key_cache.shape:
        raise ValueError("value_cache and key_cache shapes differ")
    _check(block_table, "block_table", torch.int32, 2, dev)
    _check(cache_seqlens, "cache_seqlens", torch.int32, 1, dev)
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, dev)
    dims = _dims(q, key_cache, block_table)
    if cache_seqlens.shape[0] != dims.batch or cu_seqlens_q.shape[0] != dims.batch + 1:
        raise ValueError("cache_seqlens / cu_seqlens_q do not match block_table's batch")
    rel_ptr = None
    if rel_extent > 0:
        if rel_logits is None:
            raise ValueError("rel_extent > 0 needs rel_logits")
        _check(rel_logits, "rel_logits", torch.float32, 3, dev)
        if tuple(rel_logits.shape) != (dims.num_tokens, dims.num_heads, rel_extent):
            raise ValueError("rel_logits must be (num_tokens, num_heads, rel_extent)")
        rel_ptr = rel_logits.data_ptr()
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if lse is None and return_lse:
        lse = torch.empty((dims.num_tokens, dims.num_heads), dtype=torch.float32, device=dev)
    if lse is not None:
        _check(lse, "lse", torch.float32, 2, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    need = workspace_size(dims, max_seqlen_q, num_splits)
    if stage_kv_tokens:
        need += stage_bytes(dims, stage_kv_tokens)
    if workspace is None:
        workspace = _workspace(dev, need, stream)
    return dims, rel_ptr, out, lse, workspace, stream


def ink_rel_attn_varlen(q, key_cache, value_cache, *, block_table, cache_seqlens, cu_seqlens_q,
                        max_seqlen_q: int, softmax_scale: float, causal: bool = True,
                        window_left: int = -1, window_right: int = -1, rel_extent: int = 0,
                        rel_logits=None, num_splits: int = 0, out=None, lse=None,
                        return_lse: bool = False, workspace=None, stream=None, stage_kv_tokens: int = 0):
    """Paged varlen attention with the Inkling relative bias (see include/ink_attn.h).

    Keyword arguments follow ``inkling_fa4_rel_attention`` (fa4_rel_attention.py
    as quoted by the nxmr.cn article, its wrapper signature), with the window
    passed as two integers (-1 = unbounded).  ``stage_kv_tokens`` (the cache
    keys of the prefill-shaped requests, summed) sizes the workspace so that
    their K/V is staged contiguously (ink_rel_attn_stage_bytes); results do not
    depend on it.  Returns ``out`` (and ``lse`` when ``return_lse``).
    """
    lib = load()
    dims, rel_ptr, out, lse, workspace, stream = _prepare(
        q, key_cache, value_cache, torch.bfloat16, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
        rel_extent, rel_logits, num_splits, out, lse, return_lse, workspace, stream, stage_kv_tokens)
    rc = lib.ink_rel_attn_varlen(
        ctypes.byref(dims), q.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(),
        block_table.data_ptr(), cache_seqlens.data_ptr(), cu_seqlens_q.data_ptr(), int(max_seqlen_q),
        float(softmax_scale), int(bool(causal)), int(window_left), int(window_right), int(rel_extent),
        rel_ptr, int(num_splits), out.data_ptr(), None if lse is None else lse.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), int(stream.cuda_stream))
    if rc != 0:
        raise InkError(rc, "ink_rel_attn_varlen")
    return (out, lse) if return_lse else out


def ink_rel_attn_varlen_fp8kv(q, key_cache, value_cache, *, k_scale: float, v_scale: float, block_table,
                              cache_seqlens, cu_seqlens_q, max_seqlen_q: int, softmax_scale: float,
                              causal: bool = True, window_left: int = -1, window_right: int = -1,
                              rel_extent: int = 0, rel_logits=None, num_splits: int = 0, out=None, lse=None,
                              return_lse: bool = False, workspace=None, stream=None, stage_kv_tokens: int = 0):
    """``ink_rel_attn_varlen`` over an FP8 KV cache (see include/ink_attn.h).

    key_cache / value_cache: E4M3 bytes as uint8 (or float8_e4m3fn) tensors of shape
    (num_blocks, block_size, Hkv, 128); the values attended over are k_scale * E4M3 and v_scale * E4M3.
    Prefill-shaped requests are read from the K/V staging area: ``stage_kv_tokens`` (their cache keys,
    summed) sizes it.
    """
    lib = load()
    if key_cache.dtype == torch.float8_e4m3fn:
        key_cache = key_cache.view(torch.uint8)
    if value_cache.dtype == torch.float8_e4m3fn:
        value_cache = value_cache.view(torch.uint8)
    dims, rel_ptr, out, lse, workspace, stream = _prepare(
        q, key_cache, value_cache, torch.uint8, block_table, cache_seqlens, cu_seqlens_q, max_seqlen_q,
        rel_extent, rel_logits, num_splits, out, lse, return_lse, workspace, stream, stage_kv_tokens)
    rc = lib.ink_rel_attn_varlen_fp8kv(
        ctypes.byref(dims), q.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(), float(k_scale),
        float(v_scale), block_table.data_ptr(), cache_seqlens.data_ptr(), cu_seqlens_q.data_ptr(),
        int(max_seqlen_q), float(softmax_scale), int(bool(causal)), int(window_left), int(window_right),
        int(rel_extent), rel_ptr, int(num_splits), out.data_ptr(), None if lse is None else lse.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), int(stream.cuda_stream))
    if rc != 0:
        raise InkError(rc, "ink_rel_attn_varlen_fp8kv")
    return (out, lse) if return_lse else out


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, *, flags=None, stream=None) -> None:
    """Write this step's keys and values into the paged cache at ``slot_mapping`` (see include/ink_attn.h).

    key/value: bf16 (T, Hkv, D) with D = 64, 128 or 256; caches: bf16 (num_blocks, block_size, Hkv, D), written in place;
    slot_mapping: int64 (T,), negative = padding; flags: optional int32 (1,) device tensor that receives
    DEVERR["PAGE_ID"] for slots past the cache.
    """
    lib = load()
    dev = key.device
    if dev.type != "cuda":
        raise ValueError("key must be a CUDA tensor")
    _check(key, "key", torch.bfloat16, 3, dev)
    _check(value, "value", torch.bfloat16, 3, dev)
    _check(key_cache, "key_cache", torch.bfloat16, 4, dev)
    _check(value_cache, "value_cache", torch.bfloat16, 4, dev)
    _check(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    if value.shape != key.shape or value_cache.shape != key_cache.shape:
        raise ValueError("key/value or key_cache/value_cache shapes differ")
    T, Hkv, D = key.shape
    NB, BS, Hkv2, D2 = key_cache.shape
    if (Hkv, D) != (Hkv2, D2) or slot_mapping.shape[0] != T:
        raise ValueError("key, key_cache and slot_mapping shapes do not match")
    if flags is not None:
        _check(flags, "flags", torch.int32, 1, dev)
    dims = Dims(T, 1, Hkv, Hkv, D, NB, BS, 1)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = lib.ink_reshape_and_cache(ctypes.byref(dims), key.data_ptr(), value.data_ptr(), key_cache.data_ptr(),
                                   value_cache.data_ptr(), slot_mapping.data_ptr(),
                                   None if flags is None else flags.data_ptr(), int(stream.cuda_stream))
    if rc != 0:
        raise InkError(rc, "ink_reshape_and_cache")


def reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, *, k_scale: float, v_scale: float,
                          flags=None, stream=None) -> None:
    """``reshape_and_cache`` into an FP8 (E4M3) cache: each element stored as E4M3(x / scale) (see
    include/ink_attn.h).  key/value: bf16 (T, Hkv, 128); caches: uint8 or float8_e4m3fn
    (num_blocks, block_size, Hkv, 128), written in place; slot_mapping: int64 (T,)."""
    lib = load()
    dev = key.device
    if dev.type != "cuda":
        raise ValueError("key must be a CUDA tensor")
    if key_cache.dtype == torch.float8_e4m3fn:
        key_cache = key_cache.view(torch.uint8)
    if value_cache.dtype == torch.float8_e4m3fn:
        value_cache = value_cache.view(torch.uint8)
    _check(key, "key", torch.bfloat16, 3, dev)
    _check(value, "value", torch.bfloat16, 3, dev)
    _check(key_cache, "key_cache", torch.uint8, 4, dev)
    _check(value_cache, "value_cache", torch.uint8, 4, dev)
    _check(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    if value.shape != key.shape or value_cache.shape != key_cache.shape:
        raise ValueError("key/value or key_cache/value_cache shapes differ")
    T, Hkv, D = key.shape
    NB, BS, Hkv2, D2 = key_cache.shape
    if (Hkv, D) != (Hkv2, D2) or slot_mapping.shape[0] != T:
        raise ValueError("key, key_cache and slot_mapping shapes do not match")
    if flags is not None:
        _check(flags, "flags", torch.int32, 1, dev)
    dims = Dims(T, 1, Hkv, Hkv, D, NB, BS, 1)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = lib.ink_reshape_and_cache_fp8(ctypes.byref(dims), key.data_ptr(), value.data_ptr(), key_cache.data_ptr(),
                                       value_cache.data_ptr(), slot_mapping.data_ptr(), float(k_scale),
                                       float(v_scale), None if flags is None else flags.data_ptr(),
                                       int(stream.cuda_stream))
    if rc != 0:
        raise InkError(rc, "ink_reshape_and_cache_fp8")


def read_device_errors(workspace: Optional[torch.Tensor] = None, stream=None, device=None) -> int:
    """Error word (DEVERR bits) of the last call that used `workspace`; synchronises the stream."""
    lib = load()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        workspace = _ws_cache.get((dev.index, int(stream.cuda_stream)))
        if workspace is None:
            return 0
    flags = ctypes.c_uint32(0)
    rc = lib.ink_rel_attn_read_device_errors(workspace.data_ptr(), int(stream.cuda_stream), ctypes.byref(flags))
    if rc != 0:
        raise InkError(rc, "ink_rel_attn_read_device_errors")
    return int(flags.value)
