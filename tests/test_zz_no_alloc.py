"""The allocation-free entry point, ink_rel_attn_varlen_static.

It serves callers that cannot allocate device memory: programs running inside a
host that owns all device memory itself (a serving engine that has reserved HBM
for its paged KV-cache pool, or a plugin interface that passes an operator its
tensors but no workspace and no allocator).  The test calls it through the C
ABI, twice in a row on the library's one fixed scratch area, and requires each
result to equal the workspace-taking entry point's bit for bit (both run the
same kernels on the same inputs).

The file name makes pytest collect it last, so that a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import paged_varlen_attention_causal_gb300 as ink
from workloads import build_case, workload

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 << 20   # INK_STATIC_SCRATCH_BYTES in include/ink_attn.h
INK_ERR_WORKSPACE = 3


def _static_fn():
    ink.build()
    fn = ink.load().ink_rel_attn_varlen_static
    i32, vp = ctypes.c_int32, ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ink.Dims), vp, vp, vp, vp, vp, vp, i32, ctypes.c_float, ctypes.c_int, i32, i32,
                   i32, vp, i32, vp, vp, vp]
    return fn


def _dims(case, T=None):
    return ink.Dims(case.T if T is None else T, case.B, case.H, case.Hkv, case.D, case.num_blocks, case.BS,
                    case.block_table.shape[1])


def _call_static(case, out, lse, num_splits):
    dims = _dims(case)
    rel = case.rel_logits.data_ptr() if case.E > 0 else None
    return _static_fn()(ctypes.byref(dims), case.q.data_ptr(), case.key_cache.data_ptr(),
                        case.value_cache.data_ptr(), case.block_table.data_ptr(), case.cache_seqlens.data_ptr(),
                        case.cu_seqlens_q.data_ptr(), case.max_seqlen_q, case.softmax_scale, int(case.causal),
                        case.window_left, case.window_right, case.E, rel, num_splits, out.data_ptr(),
                        lse.data_ptr(), int(torch.cuda.current_stream().cuda_stream))


def _case(name):
    if name == "mixed":
        return build_case("mixed", [1, 300, 1, 40], [2000, 900, 70, 40], H=16, Hkv=4, E=128, seed=17,
                          device="cuda")
    return workload(name, device="cuda")


@pytest.mark.parametrize("name,splits", [("tiny_mix", 0), ("tiny_mix", 4), ("mixed", 0), ("mixed", 1)])
def test_static_entry_point_matches_workspace_entry_point(name, splits):
    case = _case(name)
    assert ink.workspace_size(_dims(case), case.max_seqlen_q, splits) <= STATIC_SCRATCH_BYTES
    ref_out, ref_lse = ink.ink_rel_attn_varlen(
        case.q, case.key_cache, case.value_cache, block_table=case.block_table, cache_seqlens=case.cache_seqlens,
        cu_seqlens_q=case.cu_seqlens_q, max_seqlen_q=case.max_seqlen_q, softmax_scale=case.softmax_scale,
        causal=case.causal, window_left=case.window_left, window_right=case.window_right, rel_extent=case.E,
        rel_logits=case.rel_logits, num_splits=splits, return_lse=True)
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row on the same scratch area, which keeps the previous call's contents
        out = torch.full_like(case.q, float("nan"))
        lse = torch.full((case.T, case.H), float("nan"), device="cuda")
        assert _call_static(case, out, lse, splits) == 0
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the results are identical bit for bit
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)


def test_static_entry_point_refuses_work_beyond_its_scratch():
    case = workload("tiny_mix", device="cuda")
    big = 1 << 20
    dims = _dims(case, T=big)
    assert ink.workspace_size(dims, big, 64) > STATIC_SCRATCH_BYTES
    out = torch.empty_like(case.q)
    lse = torch.empty(case.T, case.H, device="cuda")
    rc = _static_fn()(ctypes.byref(dims), case.q.data_ptr(), case.key_cache.data_ptr(), case.value_cache.data_ptr(),
                      case.block_table.data_ptr(), case.cache_seqlens.data_ptr(), case.cu_seqlens_q.data_ptr(), big,
                      case.softmax_scale, 1, -1, -1, case.E, case.rel_logits.data_ptr(), 64, out.data_ptr(),
                      lse.data_ptr(), int(torch.cuda.current_stream().cuda_stream))
    assert rc == INK_ERR_WORKSPACE
