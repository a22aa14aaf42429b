"""fp64 CPU oracle for paged varlen causal GQA attention with the Inkling
relative bias.

TEST INFRASTRUCTURE ONLY.  The product package never imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (``bench.py``) use it.  It shares no code with the CUDA path: the
attention itself is the plain C file ``ink_oracle.c`` (fp64, OpenMP over
rows), the scheduling helpers are in ``helpers.py``.

Parity status of each function is stated in its docstring; the pins live in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .helpers import (  # noqa: F401  (re-exported)
    bucket_max_seqlen_q,
    cu_seqlens_from_lengths,
    page_index_csr,
    page_num_splits,
    slot_mapping,
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ink_oracle.c")
_LIB = os.path.join(_HERE, "libinkoracle.so")
# Tests that plant mistakes in the oracle build mutant copies and point here.
_LIB_OVERRIDE = os.environ.get("INK_ORACLE_LIB")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ink_oracle.c into a shared library next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_LIB_OVERRIDE or build())
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.ink_oracle_attn.restype = ctypes.c_int
            lib.ink_oracle_attn.argtypes = [
                i32, i32, i32, i32, i32, i32, i32, i32,
                vp, vp, vp, vp, vp, vp,
                f64, ctypes.c_int, i32, i32, i32, vp,
                vp, i64, i64, vp, vp,
            ]
            lib.ink_oracle_attn_fp8kv.restype = ctypes.c_int
            lib.ink_oracle_attn_fp8kv.argtypes = [
                i32, i32, i32, i32, i32, i32, i32, i32,
                vp, vp, vp, f64, f64, vp, vp, vp,
                f64, ctypes.c_int, i32, i32, i32, vp,
                vp, i64, i64, vp, vp,
            ]
            lib.ink_oracle_e4m3_decode.restype = None
            lib.ink_oracle_e4m3_decode.argtypes = [vp, i64, vp]
            lib.ink_oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP thread count the oracle runs with."""
    return int(_load().ink_oracle_threads())


class OracleError(RuntimeError):
    pass


_ERRORS = {1: "invalid argument", 2: "page id out of range", 3: "bad cu_seqlens_q", 4: "out of memory"}


def _as_u16(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 bit patterns."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch

        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(np.asarray(x))
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns, got {a.dtype}")
    return a


def _as(x, dtype) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=dtype))


def _as_u8(x) -> np.ndarray:
    """uint8 tensor / array (E4M3 bytes) -> contiguous uint8 array."""
    if hasattr(x, "detach"):
        import torch

        x = x.detach().cpu().contiguous()
        if x.dtype != torch.uint8:
            x = x.view(torch.uint8)
        x = x.numpy()
    a = np.ascontiguousarray(np.asarray(x))
    if a.dtype != np.uint8:
        raise TypeError(f"expected E4M3 bytes as uint8, got {a.dtype}")
    return a


def e4m3_to_float64(codes) -> np.ndarray:
    """Values of OCP FP8 E4M3 bytes (NaN for the two NaN codes), decoded by the oracle's C routine."""
    a = _as_u8(codes)
    out = np.empty(a.shape, dtype=np.float64)
    _load().ink_oracle_e4m3_decode(a.ctypes.data_as(ctypes.c_void_p), int(a.size),
                                   out.ctypes.data_as(ctypes.c_void_p))
    return out


def attention(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, *,
              softmax_scale: float, causal: bool = True, window_left: int = -1,
              window_right: int = -1, rel_extent: int = 0, rel_logits=None,
              rows=None, chunk_keys: int = 0):
    """Exact (fp64) paged varlen attention with the Inkling relative bias.

    Follows the score definition of ``score_mod_rel_bias`` (nxmr.cn article
    on fa4_rel_attention.py) and the wrapper arguments of
    ``inkling_fa4_rel_attention`` (its layer 3 "参数签名").

    q: (T, H, D) bf16; key_cache/value_cache: (NB, BS, Hkv, D) bf16;
    block_table: (B, MAXBLK) int32; cache_seqlens: (B,); cu_seqlens_q: (B+1,).
    rows: optional flat indices t*H + h to evaluate (default: all rows).
    chunk_keys > 0 selects the split-and-merge variant (PagedAttention V2
    page, Phase 2).  Returns (out (n_rows, D) float64, lse (n_rows,) float64);
    with rows=None, out is shaped (T, H, D) and lse (T, H).
    """
    lib = _load()
    qa = _as_u16(q)
    ka = _as_u16(key_cache)
    va = _as_u16(value_cache)
    T, H, D = qa.shape
    NB, BS, Hkv, D2 = ka.shape
    if D2 != D or va.shape != ka.shape:
        raise ValueError("cache shapes do not match q")
    bt = _as(block_table, np.int32)
    if bt.ndim != 2:
        raise ValueError("block_table must be 2-D")
    B, MAXBLK = bt.shape
    sk = _as(cache_seqlens, np.int32)
    cu = _as(cu_seqlens_q, np.int32)
    if sk.shape != (B,) or cu.shape != (B + 1,):
        raise ValueError("cache_seqlens / cu_seqlens_q shapes do not match block_table")
    rel = None
    if rel_extent > 0:
        rel = _as(rel_logits, np.float32)
        if rel.shape != (T, H, rel_extent):
            raise ValueError("rel_logits must be (T, H, rel_extent)")
    if rows is None:
        rows_a = None
        n_rows = T * H
    else:
        rows_a = _as(rows, np.int64).reshape(-1)
        n_rows = rows_a.size
    out = np.empty((max(n_rows, 0), D), dtype=np.float64)
    lse = np.empty((max(n_rows, 0),), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = lib.ink_oracle_attn(
        T, B, H, Hkv, D, NB, BS, MAXBLK,
        ptr(qa), ptr(ka), ptr(va), ptr(bt), ptr(sk), ptr(cu),
        float(softmax_scale), int(bool(causal)), int(window_left), int(window_right),
        int(rel_extent), ptr(rel),
        ptr(rows_a), int(n_rows), int(chunk_keys), ptr(out), ptr(lse),
    )
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))
    if rows is None:
        return out.reshape(T, H, D), lse.reshape(T, H)
    return out, lse


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping):
    """KV append: the new tokens' keys and values into copies of the paged caches.

    vLLM V1 attention page, metadata builder step 2 and appendix O: token t
    is stored at slot s = slot_mapping[t], i.e. in page s // block_size at
    offset s % block_size, all KV heads at once; a negative slot is padding
    and stores nothing.  Written out one token at a time.  Returns the new
    (key_cache, value_cache) as numpy arrays of the input dtype's bits; the
    inputs are not modified.  Pinned in ``tests/test_oracle_pins.py`` (every
    stored token reads back through the slot's page and offset, nothing else
    changes, padding changes nothing).
    """
    k = _as_u16(key)
    v = _as_u16(value)
    kc = _as_u16(key_cache).copy()
    vc = _as_u16(value_cache).copy()
    slots = np.asarray(slot_mapping.cpu() if hasattr(slot_mapping, "cpu") else slot_mapping, dtype=np.int64)
    bs = kc.shape[1]
    for t in range(k.shape[0]):
        s = int(slots[t])
        if s < 0:
            continue
        kc[s // bs, s % bs] = k[t]
        vc[s // bs, s % bs] = v[t]
    return kc, vc


def e4m3_encode(y) -> np.ndarray:
    """fp32 values -> OCP FP8 E4M3 bytes: the nearest finite E4M3 value, ties to the even code (the code whose
    last mantissa bit is 0), magnitudes above the largest finite value 448 saturated to it, NaN -> 0x7F.
    The sign is kept, zero included (-0.0 -> 0x80).

    Written as a plain search over the 127 non-negative finite codes and their values (decoded by the
    oracle's own E4M3 decoder), not as bit arithmetic.  Pinned in ``tests/test_oracle_pins.py`` (an
    independent E4M3 cast on a dense sweep, round trips, ties, saturation)."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    codes = np.arange(0x7F, dtype=np.uint8)                  # 0x00 .. 0x7E: every finite magnitude
    vals = e4m3_to_float64(codes)                              # ascending
    mag = np.minimum(np.abs(y), vals[-1])                      # saturate
    hi = np.clip(np.searchsorted(vals, mag, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo, d_hi = mag - vals[lo], vals[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    out = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    out = out | np.where(np.signbit(y), np.uint8(0x80), np.uint8(0))
    out[np.isnan(y)] = 0x7F
    return out


def reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, k_scale: float, v_scale: float):
    """KV append into an FP8 (E4M3) cache: like ``reshape_and_cache``, with each stored element quantized as
    E4M3(fp32(x) / fp32(scale)), k_scale for keys and v_scale for values.  The division is one IEEE fp32
    division, then ``e4m3_encode``.  This is the quantize-on-store of the vLLM V1 attention page's
    TurboQuant backend (section 12.1), inverse to the K = k_scale * E4M3 read of ``attention_fp8kv``.
    Returns the new (key_cache, value_cache) as uint8 arrays; the inputs are not modified."""
    import torch

    k32 = _as_u16(key).astype(np.uint32) << 16
    v32 = _as_u16(value).astype(np.uint32) << 16
    with np.errstate(over="ignore"):  # a quotient beyond fp32 is inf, which the encoder saturates
        kq = e4m3_encode(k32.view(np.float32) / np.float32(k_scale))
        vq = e4m3_encode(v32.view(np.float32) / np.float32(v_scale))
    kc = _as_u8(key_cache).copy()
    vc = _as_u8(value_cache).copy()
    slots = np.asarray(slot_mapping.cpu() if isinstance(slot_mapping, torch.Tensor) else slot_mapping,
                       dtype=np.int64)
    bs = kc.shape[1]
    for t in range(kq.shape[0]):
        s = int(slots[t])
        if s < 0:
            continue
        kc[s // bs, s % bs] = kq[t]
        vc[s // bs, s % bs] = vq[t]
    return kc, vc


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (round half to even), returned as float64.

    Written from the bf16 format definition (8 exponent bits, 7 stored
    mantissa bits): the value is first rounded to fp32 precision range and
    then to 8 significant bits with ties to even on the fp32 bit pattern.
    """
    f32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = f32.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(f32)
    out = rounded.astype(np.uint32).view(np.float32).astype(np.float64)
    out[nan] = np.nan
    return out


def attention_fp8kv(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, *,
                    k_scale: float, v_scale: float, softmax_scale: float, causal: bool = True,
                    window_left: int = -1, window_right: int = -1, rel_extent: int = 0, rel_logits=None,
                    rows=None, chunk_keys: int = 0):
    """``attention`` over an FP8 KV cache: key_cache / value_cache are (NB, BS, Hkv, D) E4M3 bytes and
    K = k_scale * E4M3(byte), V = v_scale * E4M3(byte).

    The scales enter as the PagedAttention V2 page's paged_attention_v2_pytorch applies k_scale and
    v_scale to the gathered K and V rows; the cache format is OCP FP8 E4M3, the FP8 KV cache of the
    vLLM V1 attention page's TurboQuant backend (section 12.1), dequantized when the cache is read.
    Pinned in ``tests/test_oracle_pins.py``: the decoder against every one of the 256 codes of an
    independent E4M3 implementation, and the attention against ``attention`` on bf16 caches holding
    the same values.
    """
    lib = _load()
    qa = _as_u16(q)
    ka = _as_u8(key_cache)
    va = _as_u8(value_cache)
    T, H, D = qa.shape
    NB, BS, Hkv, D2 = ka.shape
    if D2 != D or va.shape != ka.shape:
        raise ValueError("cache shapes do not match q")
    bt = _as(block_table, np.int32)
    B, MAXBLK = bt.shape
    sk = _as(cache_seqlens, np.int32)
    cu = _as(cu_seqlens_q, np.int32)
    if sk.shape != (B,) or cu.shape != (B + 1,):
        raise ValueError("cache_seqlens / cu_seqlens_q shapes do not match block_table")
    rel = None
    if rel_extent > 0:
        rel = _as(rel_logits, np.float32)
        if rel.shape != (T, H, rel_extent):
            raise ValueError("rel_logits must be (T, H, rel_extent)")
    if rows is None:
        rows_a, n_rows = None, T * H
    else:
        rows_a = _as(rows, np.int64).reshape(-1)
        n_rows = rows_a.size
    out = np.empty((max(n_rows, 0), D), dtype=np.float64)
    lse = np.empty((max(n_rows, 0),), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = lib.ink_oracle_attn_fp8kv(
        T, B, H, Hkv, D, NB, BS, MAXBLK,
        ptr(qa), ptr(ka), ptr(va), float(k_scale), float(v_scale), ptr(bt), ptr(sk), ptr(cu),
        float(softmax_scale), int(bool(causal)), int(window_left), int(window_right),
        int(rel_extent), ptr(rel),
        ptr(rows_a), int(n_rows), int(chunk_keys), ptr(out), ptr(lse),
    )
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))
    if rows is None:
        return out.reshape(T, H, D), lse.reshape(T, H)
    return out, lse
