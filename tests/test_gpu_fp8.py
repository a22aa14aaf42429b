"""Attention over an FP8 (E4M3) KV cache on the GPU against the fp64 oracle.

The cache bytes come from the seeded generator (bf16 workload values divided
by a per-tensor scale and rounded to E4M3); the oracle decodes the same bytes
exactly, so the only differences are the kernels' fp32 accumulation and their
fp16 (decode) or bf16 (prefill) q and probabilities.  Prefill-shaped requests
read a staged bf16 copy of their pages.  Tolerances are those of the bf16 path.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_causal_gb300 as ink
from test_gpu_parity import check, sampled_rows
from workloads import build_case, fp8_kv, workload

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 0.0625, 0.05


@pytest.fixture(scope="module", autouse=True)
def _built():
    ink.build()
    ink.load()
    oracle.build()


def run_fp8(case, k8, v8, ks=K_SCALE, vs=V_SCALE, **kw):
    args = dict(block_table=case.block_table, cache_seqlens=case.cache_seqlens, cu_seqlens_q=case.cu_seqlens_q,
                max_seqlen_q=case.max_seqlen_q, softmax_scale=case.softmax_scale, causal=case.causal,
                window_left=case.window_left, window_right=case.window_right, rel_extent=case.E,
                rel_logits=case.rel_logits, return_lse=True)
    args.update(kw)
    out, lse = ink.ink_rel_attn_varlen_fp8kv(case.q, k8, v8, k_scale=ks, v_scale=vs, **args)
    torch.cuda.synchronize()
    return out, lse


def oracle_fp8(case, k8, v8, ks=K_SCALE, vs=V_SCALE, rows=None):
    c = case.to("cpu")
    return oracle.attention_fp8kv(c.q, k8.cpu(), v8.cpu(), c.block_table, c.cache_seqlens, c.cu_seqlens_q,
                                  k_scale=ks, v_scale=vs, rows=rows, **c.oracle_kwargs())


def prefill_keys(case):
    """Cache keys of the prefill-shaped requests: what the call stages (converted to bf16)."""
    G = case.H // case.Hkv
    return sum(lk for lq, lk in zip(case.q_lens, case.kv_lens) if lq * G > 16)


def parity_fp8(case, what, ks=K_SCALE, vs=V_SCALE, **kw):
    k8, v8 = fp8_kv(case, ks, vs)
    kw.setdefault("stage_kv_tokens", prefill_keys(case))
    out, lse = run_fp8(case, k8, v8, ks, vs, **kw)
    ref_out, ref_lse = oracle_fp8(case, k8, v8, ks, vs)
    return check(out, lse, ref_out, ref_lse, what=what)


@pytest.mark.parametrize("H,Hkv", [(32, 8), (8, 1), (16, 2), (32, 4), (64, 8), (8, 8)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fp8_decode_matches_oracle(H, Hkv, splits):
    G = H // Hkv
    lq = max(1, 16 // G)  # the most tokens per request a decode-shaped call allows
    q_lens = [1, lq, 1, min(2, lq)]
    kv_lens = [37, 700, 2049, 16]
    case = build_case(f"fp8-{H}-{Hkv}", q_lens, kv_lens, H=H, Hkv=Hkv, E=300, seed=H + Hkv, device="cuda")
    parity_fp8(case, f"fp8 H={H} Hkv={Hkv} splits={splits}", num_splits=splits)
    assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0


@pytest.mark.parametrize("window,causal", [((-1, -1), False), ((100, 0), True), ((64, 64), False), ((0, 0), True)])
def test_fp8_windows(window, causal):
    case = build_case(f"fp8-w{window}", [1, 2, 1], [1000, 301, 5], H=16, Hkv=4, E=64, seed=21, device="cuda",
                      window=window, causal=causal)
    parity_fp8(case, f"fp8 window={window} causal={causal}")


@pytest.mark.parametrize("ks,vs", [(1.0, 1.0), (0.013, 2.5), (3.0, 0.004)])
def test_fp8_scales(ks, vs):
    case = build_case("fp8-scales", [1, 1, 4], [513, 90, 2000], H=32, Hkv=8, E=128, seed=23, device="cuda")
    parity_fp8(case, f"fp8 k_scale={ks} v_scale={vs}", ks=ks, vs=vs)


def test_fp8_nan_bytes_past_the_cache_length_are_never_used():
    """Every byte of the last page beyond Lk is an E4M3 NaN; rows must stay finite and match the oracle."""
    case = build_case("fp8-tail", [1, 1], [35, 70], H=16, Hkv=2, E=8, seed=25, device="cuda")
    k8, v8 = fp8_kv(case, K_SCALE, V_SCALE)
    for b, lk in enumerate(case.kv_lens):
        last = int(case.block_table[b, (lk - 1) // case.BS])
        off = lk % case.BS
        if off:
            k8[last, off:] = 0x7F
            v8[last, off:] = 0xFF
    out, lse = run_fp8(case, k8, v8)
    ref_out, ref_lse = oracle_fp8(case, k8, v8)
    check(out, lse, ref_out, ref_lse, what="fp8 NaN tail")


def test_fp8_bad_page_reads_as_zero_and_is_flagged():
    case = build_case("fp8-badpage", [1, 1], [100, 50], H=8, Hkv=2, E=0, seed=27, device="cuda")
    k8, v8 = fp8_kv(case, K_SCALE, V_SCALE)
    case.block_table[0, 2] = case.num_blocks + 5
    run_fp8(case, k8, v8)
    assert ink.read_device_errors() & ink.DEVERR["PAGE_ID"]


def _dims(case):
    return ink.Dims(case.T, case.B, case.H, case.Hkv, 128, case.num_blocks, case.BS, case.block_table.shape[1])


def test_fp8_prefill_needs_staging_room_and_valid_scales():
    """Prefill-shaped requests over an E4M3 cache are read through the staging copy: a workspace with no
    room for it is refused; scales outside [2^-126, 2^126] are refused."""
    case = build_case("fp8-pf", [1, 64], [100, 64], H=16, Hkv=4, E=0, seed=29, device="cuda")
    k8, v8 = fp8_kv(case, K_SCALE, V_SCALE)
    base = ink.workspace_size(_dims(case), case.max_seqlen_q, 0)
    with pytest.raises(ink.InkError) as e:
        run_fp8(case, k8, v8, workspace=torch.empty(base, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 3  # workspace too small: nowhere to stage the prefill request
    for ks, vs in [(0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf")), (2.0 ** -127, 1.0),
                   (1.0, 2.0 ** 127)]:
        with pytest.raises(ink.InkError) as e:
            run_fp8(case, k8, v8, ks, vs, stage_kv_tokens=64)
        assert e.value.status == 1


@pytest.mark.parametrize("H,Hkv", [(32, 8), (8, 1), (16, 2), (64, 8), (8, 8), (12, 4)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fp8_prefill_and_mixed_match_oracle(H, Hkv, splits):
    """Prefill-shaped requests (read from the staged bf16 copy) next to decodes (read from the E4M3 pages)."""
    case = build_case(f"fp8-pf-{H}-{Hkv}", [1, 130, 1, 37, 300], [700, 130, 33, 900, 300], H=H, Hkv=Hkv, E=96,
                      seed=H * 3 + Hkv, device="cuda")
    parity_fp8(case, f"fp8 prefill H={H} Hkv={Hkv} splits={splits}", num_splits=splits)
    assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0


def test_fp8_tiny_mix():
    case = workload("tiny_mix", device="cuda")
    for splits in (1, 4):
        parity_fp8(case, f"fp8 tiny_mix splits={splits}", num_splits=splits)


@pytest.mark.parametrize("window,causal", [((64, 0), True), ((100, 30), False), ((-1, -1), False)])
def test_fp8_prefill_windows(window, causal):
    case = build_case(f"fp8-pfw{window}", [140, 1, 33], [400, 800, 33], H=16, Hkv=4, E=64, seed=7, device="cuda",
                      window=window, causal=causal)
    parity_fp8(case, f"fp8 prefill window={window} causal={causal}")


@pytest.mark.parametrize("ks,vs", [(1.0, 1.0), (0.013, 2.5), (3.0, 0.004)])
def test_fp8_prefill_scales(ks, vs):
    case = build_case("fp8-pf-scales", [200, 1], [513, 90], H=32, Hkv=8, E=128, seed=23, device="cuda")
    parity_fp8(case, f"fp8 prefill k_scale={ks} v_scale={vs}", ks=ks, vs=vs)


def test_fp8_prefill_without_room_is_skipped_and_flagged():
    """Room for the first prefill request only: the second is skipped (its rows keep their contents) and
    flagged; the decode and the first prefill request match the oracle."""
    case = build_case("fp8-part", [100, 1, 120], [300, 500, 1000], H=16, Hkv=4, E=32, seed=37, device="cuda")
    k8, v8 = fp8_kv(case, K_SCALE, V_SCALE)
    base = ink.workspace_size(_dims(case), case.max_seqlen_q, 0)
    ws = torch.empty(base + 384 * case.Hkv * 128 * 2 * 2, dtype=torch.uint8, device="cuda")  # 384 staged keys
    out = torch.full_like(case.q, 7.0)
    out, lse = run_fp8(case, k8, v8, workspace=ws, out=out)
    assert ink.read_device_errors(ws) & ink.DEVERR["STAGE"]
    cu = case.cu_seqlens_q.tolist()
    assert torch.all(out[cu[2]:cu[3]] == 7.0)  # skipped: left as it was
    rows = np.arange(0, cu[2] * case.H, dtype=np.int64)
    ref_out, ref_lse = oracle_fp8(case, k8, v8, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what="fp8 partial staging")


@pytest.mark.slow
def test_fp8_chunked_prefill_full_size():
    """The chunked prefill (4 x Lq 2048 on prior 0 .. 14336 keys, H 32, Hkv 8, E 4096) over an E4M3 cache,
    staged; sampled rows against the oracle."""
    case = workload("chunked_prefill", device="cuda")
    k8, v8 = fp8_kv(case, K_SCALE, V_SCALE)
    case.key_cache = case.value_cache = None
    torch.cuda.empty_cache()
    out, lse = run_fp8(case, k8, v8, stage_kv_tokens=prefill_keys(case))
    assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    rows = sampled_rows(case, 128, 13)
    ref_out, ref_lse = oracle_fp8(case, k8, v8, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what="fp8 chunked_prefill")
    del k8, v8, out, lse
    torch.cuda.empty_cache()


def test_fp8_batch_of_decodes_reads_half_the_bytes():
    """A batch of single-token decodes over lengths from 1 to 4096 against the oracle; the E4M3 cache is
    half the bf16 cache's bytes."""
    case = build_case("fp8-vs-bf16", [1] * 6, [3000, 17, 999, 4096, 1, 250], H=32, Hkv=8, E=512, seed=31,
                      device="cuda")
    parity_fp8(case, "fp8 batch")
    k8, v8 = fp8_kv(case, K_SCALE, V_SCALE)
    assert k8.numel() * k8.element_size() * 2 == case.key_cache.numel() * case.key_cache.element_size()


@pytest.mark.slow
def test_fp8_decode_batch_full_size():
    """The 64-request decode batch (Lk up to 32768, H 32, Hkv 8, E 1024) on an FP8 cache, sampled rows."""
    case = workload("decode_batch", device="cuda")
    k8, v8 = fp8_kv(case, K_SCALE, V_SCALE)
    out, lse = run_fp8(case, k8, v8)
    assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    rows = sampled_rows(case, 192, 11)
    ref_out, ref_lse = oracle_fp8(case, k8, v8, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what="fp8 decode_batch")
    del case, k8, v8, out, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("bs", [32, 64, 128])
def test_fp8_block_sizes(bs):
    """Pages of 32 to 128 keys: the kernel reads them as 16-key groups at the right offsets."""
    case = build_case(f"fp8-bs{bs}", [1, 2, 1, 1], [700, 129, 33, 4000], H=32, Hkv=8, E=200, BS=bs, seed=41 + bs,
                      device="cuda")
    parity_fp8(case, f"fp8 block_size={bs}")
    parity_fp8(case, f"fp8 block_size={bs} splits=5", num_splits=5)


@pytest.mark.slow
def test_fp8_long_decode_full_size():
    """One decode over 1,048,576 keys (H 64, Hkv 8, E 8192) on an E4M3 cache: the transposed path with 8 rows
    and the split-KV merge over many splits; the rows of the first and last KV heads against the oracle."""
    case = workload("long_decode", device="cuda")
    k8, v8 = fp8_kv(case, K_SCALE, V_SCALE)
    case.key_cache = case.value_cache = None
    torch.cuda.empty_cache()
    out, lse = run_fp8(case, k8, v8)
    assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    rows = np.concatenate([np.arange(8), np.arange(case.H - 8, case.H)]).astype(np.int64)
    ref_out, ref_lse = oracle_fp8(case, k8, v8, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what="fp8 long_decode")
    del k8, v8, out, lse
    torch.cuda.empty_cache()
