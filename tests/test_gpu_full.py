"""The five workloads at full size on the GPU, in the launch configuration the
benchmark times (K/V staging room for the prefill-shaped requests), checked
against the fp64 oracle on stratified rows (the oracle computes each chosen row
exactly), plus the split-count sweep of the long batch-1 decode.

Stratified rows: for every prefill work item (request, q tile, KV head) its
first, middle and last token with the first and last query head of the KV
head's group -- the item's first and last packed rows among them; every head of
every decode-shaped token; every token whose causal diagonal or window edge
falls on a 128-key tile boundary (either side); and seeded random rows.  The
chunked prefill is also run with a forced split count, so that split boundaries
cut through every q tile's key range.
"""
import numpy as np
import pytest
import torch

import paged_varlen_attention_causal_gb300 as ink
from test_gpu_parity import check, errors_of_last_call, gpu_run, oracle_run
from workloads import workload

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def prefill_keys(case):
    G = case.H // case.Hkv
    return sum(lk for lq, lk in zip(case.q_lens, case.kv_lens) if lq * G > 16)


def stratified_rows(case, extra=1024, seed=7):
    H, G = case.H, case.H // case.Hkv
    tpt = 128 // G  # tokens of a 128-row prefill tile
    cu = case.cu_seqlens_q.tolist()
    g = np.random.default_rng(seed)
    rows = set()
    for b in range(case.B):
        lq, lk, t0 = case.q_lens[b], case.kv_lens[b], cu[b]
        if lq == 0:
            continue
        if lq * G <= 16:  # decode-shaped: every head of every token
            rows.update(range(t0 * H, (t0 + lq) * H))
            continue
        for qt in range((lq + tpt - 1) // tpt):
            i0, i1 = qt * tpt, min(lq, qt * tpt + tpt) - 1
            for i in {i0, (i0 + i1) // 2, i1}:
                for kvh in range(case.Hkv):
                    rows.add((t0 + i) * H + kvh * G)
                    rows.add((t0 + i) * H + kvh * G + G - 1)
        for i in range(lq):
            qa = i + lk - lq
            lo = qa - case.window_left if case.window_left >= 0 else -1
            if qa % 128 in (0, 127) or (lo >= 0 and lo % 128 in (0, 127)):
                rows.add((t0 + i) * H + int(g.integers(0, H)))
    rows.update(g.integers(0, case.T * H, size=extra).tolist())
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", ["decode_batch", "chunked_prefill", "long_decode", "continuous_batch"])
def test_workload_full_size(name):
    case = workload(name, device="cuda")
    out, lse = gpu_run(case, stage_kv_tokens=prefill_keys(case))
    assert errors_of_last_call() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    assert torch.isfinite(out.float()).all()
    rows = stratified_rows(case)
    assert rows.size >= min(4096, case.T * case.H)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what=name)
    del case, out, lse
    torch.cuda.empty_cache()


def test_chunked_prefill_forced_splits():
    """Three splits per q tile: every row's key range is cut at two split boundaries and merged."""
    case = workload("chunked_prefill", device="cuda")
    out, lse = gpu_run(case, num_splits=3, stage_kv_tokens=prefill_keys(case))
    assert errors_of_last_call() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    rows = stratified_rows(case, extra=256, seed=9)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what="chunked_prefill splits=3")
    del case, out, lse
    torch.cuda.empty_cache()


def test_long_decode_split_sweep():
    case = workload("long_decode", device="cuda")
    rows = np.arange(case.H, dtype=np.int64)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    for s in (16, 32, 64, 128):
        out, lse = gpu_run(case, num_splits=s)
        check(out, lse, ref_out, ref_lse, rows=rows, what=f"long_decode splits={s}")
    del case
    torch.cuda.empty_cache()
