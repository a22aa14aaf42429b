"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol include/ink_attn.h declares, and rejects bad arguments on the host
before anything is launched."""
import ctypes
import os
import re

import pytest

import paged_varlen_attention_causal_gb300 as ink

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ink_attn.h")


@pytest.fixture(scope="module")
def lib():
    ink.build()
    return ink.load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"INK_API\s+[\w\s\*]+?\b(ink_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    assert {"ink_rel_attn_varlen", "ink_rel_attn_workspace_size", "ink_rel_attn_num_splits",
            "ink_status_string", "ink_rel_attn_read_device_errors", "ink_attn_version"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(lib):
    for code, text in [(0, b"ok"), (1, b"invalid argument"), (2, b"unsupported configuration"),
                       (3, b"workspace too small"), (4, b"CUDA error")]:
        assert lib.ink_status_string(code) == text
    assert ink.version() >= 100


def _dims(**kw):
    d = dict(num_tokens=130, batch=3, num_heads=8, num_kv_heads=2, head_dim=128, num_blocks=64,
             block_size=16, max_blocks_per_seq=20)
    d.update(kw)
    return ink.Dims(**d)


def test_workspace_size_is_positive_and_grows_with_splits(lib):
    d = _dims()
    a = ink.workspace_size(d, 128, 1)
    b = ink.workspace_size(d, 128, 8)
    assert 256 <= a < b
    assert lib.ink_rel_attn_workspace_size(ctypes.byref(_dims(head_dim=0)), 128, 1) == 0
    assert lib.ink_rel_attn_workspace_size(ctypes.byref(_dims(num_heads=6, num_kv_heads=4)), 128, 1) == 0
    assert lib.ink_rel_attn_workspace_size(ctypes.byref(_dims()), 0, 1) == 0


def _call(lib, dims, **over):
    P = 4096  # a fake, 256-byte aligned address: these calls must fail before any use of it
    args = dict(q=P, k=P, v=P, bt=P, sk=P, cu=P, msq=128, scale=0.088, causal=1, wl=-1, wr=-1, E=0,
                rel=None, splits=0, out=P, lse=None, ws=P, wsb=1 << 40, stream=None)
    args.update(over)
    return lib.ink_rel_attn_varlen(ctypes.byref(dims), args["q"], args["k"], args["v"], args["bt"],
                                   args["sk"], args["cu"], args["msq"], args["scale"], args["causal"],
                                   args["wl"], args["wr"], args["E"], args["rel"], args["splits"],
                                   args["out"], args["lse"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(out=None), 1), (dict(ws=None), 1),
    (dict(msq=0), 1), (dict(wl=-2), 1), (dict(wr=-5), 1), (dict(E=-1), 1), (dict(E=8, rel=None), 1),
    (dict(splits=-1), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("nan")), 1),
    (dict(q=4096 + 8), 1), (dict(out=4096 + 2), 1), (dict(ws=4096 + 16), 1), (dict(bt=4096 + 2), 1),
])
def test_host_validation(lib, over, status):
    assert _call(lib, _dims(), **over) == status


@pytest.mark.parametrize("dims_over,status", [
    (dict(head_dim=96), 2), (dict(head_dim=32), 2), (dict(head_dim=512), 2), (dict(block_size=8), 2),
    (dict(block_size=24), 2),
    (dict(num_heads=6, num_kv_heads=4), 1), (dict(batch=0), 1), (dict(num_tokens=-1), 1),
])
def test_unsupported_or_invalid_dims(lib, dims_over, status):
    assert _call(lib, _dims(**dims_over)) == status


def test_empty_batch_is_a_no_op(lib):
    assert _call(lib, _dims(num_tokens=0)) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ink.LibraryNotBuilt):
        ink.load(str(tmp_path / "missing.so"))


def test_append_host_validation(lib):
    """ink_reshape_and_cache rejects bad arguments before touching the GPU."""
    import ctypes

    f = lib.ink_reshape_and_cache
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ink.Dims)] + [ctypes.c_void_p] * 7
    good = 0x10000
    dims = ink.Dims(8, 1, 4, 4, 128, 16, 16, 1)
    assert f(ctypes.byref(dims), None, good, good, good, good, None, None) == 1          # null key
    assert f(ctypes.byref(dims), good, good, good, good, good + 4, None, None) == 1      # misaligned slots
    assert f(ctypes.byref(dims), good + 8, good, good, good, good, None, None) == 1      # misaligned key
    bad = ink.Dims(8, 1, 4, 4, 96, 16, 16, 1)
    assert f(ctypes.byref(bad), good, good, good, good, good, None, None) == 2           # head_dim 96
    empty = ink.Dims(0, 1, 4, 4, 128, 16, 16, 1)
    assert f(ctypes.byref(empty), good, good, good, good, good, None, None) == 0         # nothing to do


def test_fp8_entry_host_validation(lib):
    """ink_rel_attn_varlen_fp8kv rejects bad scales, pointers and shapes before touching the GPU."""
    import ctypes

    f = lib.ink_rel_attn_varlen_fp8kv
    f.restype = ctypes.c_int
    vp, i32, fl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    f.argtypes = [ctypes.POINTER(ink.Dims), vp, vp, vp, fl, fl, vp, vp, vp, i32, fl, ctypes.c_int, i32, i32, i32,
                  vp, i32, vp, vp, vp, ctypes.c_size_t, vp]
    good = 0x10000
    dims = ink.Dims(4, 2, 8, 2, 128, 16, 16, 4)

    def call(ks=0.5, vs=0.5, q=good, d=dims, scale=0.1):
        return f(ctypes.byref(d), q, good, good, ks, vs, good, good, good, 2, scale, 1, -1, -1, 0, None, 0,
                 good, None, good, 1 << 20, None)

    for ks, vs in [(0.0, 1.0), (1.0, 0.0), (-2.0, 1.0), (float("nan"), 1.0), (1.0, float("inf")),
                   (2.0 ** -127, 1.0), (1.0, 2.0 ** 127), (1e-40, 1.0)]:   # outside [2^-126, 2^126]
        assert call(ks, vs) == 1
    assert call(q=None) == 1                                   # null q
    assert call(q=good + 2) == 1                               # misaligned q
    assert call(scale=0.0) == 1                                # softmax_scale must be > 0
    assert call(d=ink.Dims(4, 2, 8, 2, 64, 16, 16, 4)) == 2    # head_dim 64
    assert call(d=ink.Dims(0, 2, 8, 2, 128, 16, 16, 4)) == 0   # nothing to do


def test_fp8_append_host_validation(lib):
    """ink_reshape_and_cache_fp8 rejects bad scales, pointers and shapes before touching the GPU."""
    import ctypes

    f = lib.ink_reshape_and_cache_fp8
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(ink.Dims), vp, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp]
    good = 0x10000
    dims = ink.Dims(8, 1, 4, 4, 128, 16, 16, 1)
    for ks, vs in [(0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf")), (2.0 ** -127, 1.0),
                   (1.0, 2.0 ** 127), (1e-40, 1.0)]:   # the reciprocal of a scale below 2^-126 overflows
        assert f(ctypes.byref(dims), good, good, good, good, good, ks, vs, None, None) == 1
    assert f(ctypes.byref(dims), None, good, good, good, good, 1.0, 1.0, None, None) == 1       # null key
    assert f(ctypes.byref(dims), good, good, good + 8, good, good, 1.0, 1.0, None, None) == 1   # misaligned cache
    bad = ink.Dims(8, 1, 4, 4, 256, 16, 16, 1)
    assert f(ctypes.byref(bad), good, good, good, good, good, 1.0, 1.0, None, None) == 2        # head_dim 256
    empty = ink.Dims(0, 1, 4, 4, 128, 16, 16, 1)
    assert f(ctypes.byref(empty), good, good, good, good, good, 1.0, 1.0, None, None) == 0     # nothing to do


def test_head_sizes_64_and_256(lib):
    """D = 64 and 256 are served (decode items by the decode kernel, prefill tiles by the head-size-generic
    kernel): workspace sizes follow D, nothing is staged, and an FP8 cache is refused at those sizes."""
    sizes = {D: ink.workspace_size(_dims(head_dim=D), 128, 8) for D in (64, 128, 256)}
    assert 0 < sizes[64] < sizes[256]
    assert ink.stage_bytes(_dims(head_dim=64), 1000) == 0 and ink.stage_bytes(_dims(head_dim=256), 1000) == 0
    assert ink.stage_bytes(_dims(head_dim=128), 1000) > 0
    f = lib.ink_rel_attn_varlen_fp8kv
    vp, fl, i32 = ctypes.c_void_p, ctypes.c_float, ctypes.c_int32
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ink.Dims), vp, vp, vp, fl, fl, vp, vp, vp, i32, fl, ctypes.c_int, i32, i32, i32,
                  vp, i32, vp, vp, vp, ctypes.c_size_t, vp]
    P = 4096
    d = _dims(head_dim=64)
    assert f(ctypes.byref(d), P, P, P, 1.0, 1.0, P, P, P, 128, 0.088, 1, -1, -1, 0, None, 0, P, None, P, 1 << 40,
             None) == 2
