"""K/V staging for the prefill (workspace beyond the minimum; ink_rel_attn_stage_bytes).

A staged prefill-shaped request reads its K and V tiles from a contiguous copy
of its pages instead of the paged cache.  Only where the kernel reads from
changes, not the arithmetic, so a staged call must equal the unstaged call bit
for bit, and both must match the fp64 oracle.  Partial staging (room for some
requests only), bad page ids and split and window shapes are covered too.
"""
import pytest
import torch

import oracle
import paged_varlen_attention_causal_gb300 as ink
from test_gpu_parity import check, oracle_run, sampled_rows
from workloads import build_case, random_case, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ink.build()
    ink.load()
    oracle.build()


def _dims(case):
    return ink.Dims(case.T, case.B, case.H, case.Hkv, 128, case.num_blocks, case.BS, case.block_table.shape[1])


def _prefill_keys(case):
    G = case.H // case.Hkv
    return sum(lk for lq, lk in zip(case.q_lens, case.kv_lens) if lq * G > 16)


def _run(case, ws_bytes, **kw):
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    args = dict(block_table=case.block_table, cache_seqlens=case.cache_seqlens, cu_seqlens_q=case.cu_seqlens_q,
                max_seqlen_q=case.max_seqlen_q, softmax_scale=case.softmax_scale, causal=case.causal,
                window_left=case.window_left, window_right=case.window_right, rel_extent=case.E,
                rel_logits=case.rel_logits, return_lse=True, workspace=ws)
    args.update(kw)
    out, lse = ink.ink_rel_attn_varlen(case.q, case.key_cache, case.value_cache, **args)
    torch.cuda.synchronize()
    return out, lse, ink.read_device_errors(ws)


def _both(case, what, splits=0):
    base = ink.workspace_size(_dims(case), case.max_seqlen_q, splits)
    full = base + ink.stage_bytes(_dims(case), _prefill_keys(case))
    out0, lse0, e0 = _run(case, base, num_splits=splits)
    out1, lse1, e1 = _run(case, full, num_splits=splits)
    assert torch.equal(out0, out1), f"{what}: staged out differs from paged"
    assert torch.equal(lse0, lse1), f"{what}: staged lse differs from paged"
    assert e0 == e1
    ref_out, ref_lse = oracle_run(case)
    check(out1, lse1, ref_out, ref_lse, what=what)
    return e1


@pytest.mark.parametrize("splits", [1, 4, 0])
def test_tiny_mix_staged(splits):
    _both(workload("tiny_mix", device="cuda"), f"tiny_mix splits={splits}", splits)


@pytest.mark.parametrize("seed", range(16))
def test_random_staged(seed):
    case = random_case(300 + seed, D=128, BS=[16, 32][seed % 2], device="cuda", max_q=90, max_kv_extra=700)
    _both(case, f"random{300 + seed}")


@pytest.mark.parametrize("seed", range(6))
def test_random_staged_split(seed):
    case = random_case(400 + seed, D=128, BS=16, device="cuda", max_q=60, max_kv_extra=900)
    _both(case, f"random{400 + seed} splits 3", splits=3)


@pytest.mark.parametrize("H,Hkv", [(8, 8), (32, 8), (8, 1), (64, 2), (12, 4), (128, 1), (6, 2)])
def test_head_layouts_staged(H, Hkv):
    case = build_case(f"stage-{H}-{Hkv}", [150, 1, 37], [150, 900, 500], H=H, Hkv=Hkv, E=96, seed=H + Hkv,
                      device="cuda")
    _both(case, f"H{H} Hkv{Hkv}")


@pytest.mark.parametrize("window", [(64, 0), (200, 17), (5, -1)])
@pytest.mark.parametrize("causal", [True, False])
def test_windows_staged(window, causal):
    case = build_case("stage-win", [140, 1, 33], [400, 800, 33], H=16, Hkv=4, E=64, seed=7, device="cuda",
                      causal=causal, window=window)
    _both(case, f"window {window} causal={causal}")


def test_partial_staging():
    """Room for the first prefill request only: it is staged, the others read the paged cache."""
    case = build_case("stage-part", [200, 1, 130, 64], [900, 300, 1300, 64], H=32, Hkv=8, E=256, seed=21,
                      device="cuda")
    base = ink.workspace_size(_dims(case), case.max_seqlen_q, 0)
    per_key = case.Hkv * 128 * 2 * 2  # K and V of every KV head
    out0, lse0, _ = _run(case, base)
    # the prefill-shaped requests take 1024, 1408 and 128 staged keys, in that order
    for keys in (1024, 1152, 2560, 10 ** 5):
        out1, lse1, _ = _run(case, base + keys * per_key)
        assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    ref_out, ref_lse = oracle_run(case)
    check(out0, lse0, ref_out, ref_lse, what="partial staging")


def test_bad_page_staged():
    """A bad block_table entry of a staged request is flagged and reads as zeros, as on the paged path."""
    case = build_case("stage-bad", [100, 80], [300, 200], H=16, Hkv=4, E=32, seed=5, device="cuda")
    case.block_table[1, 3] = case.num_blocks + 7
    base = ink.workspace_size(_dims(case), case.max_seqlen_q, 0)
    full = base + ink.stage_bytes(_dims(case), 500)
    out0, lse0, e0 = _run(case, base)
    out1, lse1, e1 = _run(case, full)
    assert e0 & ink.DEVERR["PAGE_ID"] and e1 & ink.DEVERR["PAGE_ID"]
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


@pytest.mark.slow
def test_chunked_prefill_staged_sampled():
    """The full-size chunked prefill, staged: equal to the paged result, and sampled rows against the oracle."""
    case = workload("chunked_prefill", device="cuda")
    base = ink.workspace_size(_dims(case), case.max_seqlen_q, 0)
    full = base + ink.stage_bytes(_dims(case), _prefill_keys(case))
    out0, lse0, _ = _run(case, base)
    out1, lse1, _ = _run(case, full)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    rows = sampled_rows(case, 96, 11)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    check(out1, lse1, ref_out, ref_lse, rows=rows, what="chunked prefill staged")
