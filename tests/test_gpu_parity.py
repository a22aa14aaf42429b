"""CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Tolerances follow the target the pages' tutorial uses for bf16 attention
(max |out - ref| < 2e-2) and a 1e-3 relative bound on the fp32 log-sum-exp
(relative to max(1, |lse|), so that rows with lse near 0 get 1e-3 absolute);
rows without a visible key must give -inf exactly and out = 0.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_causal_gb300 as ink
from workloads import build_case, random_case, workload

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_RTOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    ink.build()
    ink.load()
    oracle.build()


def gpu_run(case, **kw):
    args = dict(block_table=case.block_table, cache_seqlens=case.cache_seqlens, cu_seqlens_q=case.cu_seqlens_q,
                max_seqlen_q=case.max_seqlen_q, softmax_scale=case.softmax_scale, causal=case.causal,
                window_left=case.window_left, window_right=case.window_right, rel_extent=case.E,
                rel_logits=case.rel_logits, return_lse=True)
    args.update(kw)
    out, lse = ink.ink_rel_attn_varlen(case.q, case.key_cache, case.value_cache, **args)
    torch.cuda.synchronize()
    return out, lse


def oracle_run(case, rows=None):
    c = case.to("cpu")
    return oracle.attention(c.q, c.key_cache, c.value_cache, c.block_table, c.cache_seqlens, c.cu_seqlens_q,
                            rows=rows, **c.oracle_kwargs())


def check(out, lse, ref_out, ref_lse, rows=None, what=""):
    o = out.float().cpu().double().numpy().reshape(-1, out.shape[-1])
    l = lse.cpu().double().numpy().reshape(-1)
    ro = ref_out.reshape(-1, o.shape[-1])
    rl = ref_lse.reshape(-1)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.all(np.isfinite(o)), f"{what}: non-finite outputs"
    err = np.max(np.abs(o - ro)) if o.size else 0.0
    assert err <= OUT_TOL, f"{what}: max |out - ref| = {err}"
    inf_ref = ~np.isfinite(rl)
    assert np.array_equal(inf_ref, ~np.isfinite(l)), f"{what}: -inf rows differ"
    assert np.all(l[inf_ref] == -np.inf)
    assert np.all(o[inf_ref] == 0.0)
    if (~inf_ref).any():
        rel = np.abs(l[~inf_ref] - rl[~inf_ref]) / np.maximum(1.0, np.abs(rl[~inf_ref]))
        assert rel.max() <= LSE_RTOL, f"{what}: lse rel err {rel.max()}"
    return err


def parity(case, what="", **kw):
    out, lse = gpu_run(case, **kw)
    ref_out, ref_lse = oracle_run(case)
    return check(out, lse, ref_out, ref_lse, what=what)


def errors_of_last_call():
    return ink.read_device_errors()


# --- the tiny mixed batch: decode 47, decode 312, prefill 128/128 --------------------

@pytest.mark.parametrize("splits", [1, 4, 0])
def test_tiny_mix(splits):
    case = workload("tiny_mix", device="cuda")
    parity(case, f"tiny_mix splits={splits}", num_splits=splits)
    assert errors_of_last_call() & ~ink.DEVERR["EMPTY_ROWS"] == 0


# --- small random cases across shapes -------------------------------------------------

@pytest.mark.parametrize("seed", range(40))
def test_random_small(seed):
    case = random_case(seed, D=128, BS=[16, 32][seed % 2], device="cuda", max_q=70, max_kv_extra=300)
    parity(case, f"random{seed}")


@pytest.mark.parametrize("seed", range(12))
def test_random_small_split(seed):
    case = random_case(100 + seed, D=128, BS=16, device="cuda", max_q=40, max_kv_extra=400)
    parity(case, f"random{100 + seed} splits 3", num_splits=3)


# G = H / Hkv covers every prefill packing: warp-strided (G divides 32) and plain, and every number of
# tokens per bias box the host picks (8: G 1-4, 6, 8, 16; 4: G 5, 7, 12, 32; 2: G 64; 1: G 128).
@pytest.mark.parametrize("H,Hkv", [(8, 8), (16, 8), (8, 1), (16, 1), (32, 1), (64, 2), (12, 4), (48, 16),
                                   (128, 1), (6, 2), (10, 2), (12, 2), (14, 2), (24, 2), (64, 1)])
@pytest.mark.parametrize("kind", ["decode", "prefill", "mixed"])
def test_head_layouts(H, Hkv, kind):
    if kind == "decode":
        q_lens, kv_lens = [1, 1, 1], [17, 300, 1029]
    elif kind == "prefill":
        q_lens, kv_lens = [150, 37], [150, 500]
    else:
        q_lens, kv_lens = [1, 200, 2, 3], [77, 260, 40, 9]
    case = build_case(f"{kind}-{H}-{Hkv}", q_lens, kv_lens, H=H, Hkv=Hkv, E=96, seed=H * 100 + Hkv,
                      device="cuda")
    parity(case, f"H{H} Hkv{Hkv} {kind}")


@pytest.mark.parametrize("E", [0, 1, 5, 64, 130, 1000])
def test_bias_extents(E):
    case = build_case(f"E{E}", [1, 64, 300], [900, 64, 700], H=16, Hkv=4, E=E, seed=E + 7, device="cuda")
    parity(case, f"E={E}")


@pytest.mark.parametrize("window", [(0, 0), (5, -1), (127, 0), (300, 0), (-1, 0), (64, 64), (4095, 0)])
@pytest.mark.parametrize("causal", [True, False])
def test_windows(window, causal):
    case = build_case(f"w{window}", [1, 3, 260], [1000, 40, 900], H=8, Hkv=2, E=200, seed=11, device="cuda",
                      window=window, causal=causal)
    parity(case, f"window={window} causal={causal}")


@pytest.mark.parametrize("lq", [2, 3, 4, 5, 16, 17])
def test_multi_token_decode(lq):
    case = build_case(f"spec{lq}", [lq, lq], [lq + 100, lq + 2000], H=16, Hkv=4, E=128, seed=lq,
                      device="cuda")
    parity(case, f"lq={lq}")


@pytest.mark.parametrize("E,window", [(256, (-1, -1)), (0, (-1, -1)), (64, (700, 0)), (4096, (-1, -1))])
def test_multi_item_prefill(E, window):
    """Several work items per CTA and interior tiles that need neither bias nor masks."""
    case = build_case(f"multi{E}", [3000, 1, 700], [9000, 5000, 700], H=8, Hkv=2, E=E, seed=31, device="cuda",
                      window=window)
    out, lse = gpu_run(case)
    assert errors_of_last_call() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    rows = sampled_rows(case, 600, 3)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what=f"multi-item E={E} window={window}")


@pytest.mark.parametrize("splits", [0, 1])
def test_partial_warp_rescale(splits):
    """Only some rows of a warp move their running maximum late in the key range.

    A +20 bias on the four nearest distances of the odd heads makes the rows of
    those heads (every other lane of each softmax warp) raise their maximum by far
    more than the rescale threshold on the diagonal tile, while the even heads keep
    theirs; the warp must rescale its O rows together.
    """
    case = build_case("late_max", [1536], [1536], H=16, Hkv=2, E=64, seed=41, device="cuda")
    case.rel_logits[:, 1::2, :4] += 20.0
    out, lse = gpu_run(case, num_splits=splits)
    assert errors_of_last_call() == 0
    rows = sampled_rows(case, 600, 5)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what=f"late maximum, splits={splits}")


# --- edge cases -------------------------------------------------------------------------

def test_empty_requests_and_empty_rows():
    # request 1 has no query tokens; request 2 has fewer keys than queries (causal: early rows see nothing)
    case = build_case("edge", [5, 0, 20, 1], [50, 30, 8, 1], H=8, Hkv=2, E=16, seed=3, device="cuda")
    parity(case, "edge")
    assert errors_of_last_call() & ink.DEVERR["EMPTY_ROWS"]


def test_zero_length_kv():
    case = build_case("nokv", [1, 4], [0, 4], H=8, Hkv=2, E=4, seed=5, device="cuda", causal=False)
    parity(case, "zero-length kv")


def test_large_block_size():
    case = build_case("bs64", [1, 100], [3000, 500], H=16, Hkv=4, E=64, BS=64, seed=9, device="cuda")
    parity(case, "block_size 64")


def test_stacked_cache_and_shared_pages():
    case = build_case("stack", [1, 50], [300, 90], H=8, Hkv=2, E=32, seed=21, device="cuda")
    stacked = torch.stack([case.key_cache, case.value_cache])
    case.key_cache, case.value_cache = stacked[0], stacked[1]
    case.block_table[1, :3] = case.block_table[0, :3]  # request 1 shares request 0's first pages
    parity(case, "stacked")


def test_lse_optional_and_out_preallocated():
    case = workload("tiny_mix", device="cuda")
    out = torch.full_like(case.q, float("nan"))
    res = ink.ink_rel_attn_varlen(case.q, case.key_cache, case.value_cache, block_table=case.block_table,
                                  cache_seqlens=case.cache_seqlens, cu_seqlens_q=case.cu_seqlens_q,
                                  max_seqlen_q=case.max_seqlen_q, softmax_scale=case.softmax_scale,
                                  rel_extent=case.E, rel_logits=case.rel_logits, out=out)
    torch.cuda.synchronize()
    assert res.data_ptr() == out.data_ptr()
    ref_out, ref_lse = oracle_run(case)
    o = out.float().cpu().double().numpy()
    assert np.max(np.abs(o - ref_out)) <= OUT_TOL


# --- invariants on the GPU ----------------------------------------------------------------

def test_split_sweep_agrees():
    case = build_case("sweep", [1, 1, 300], [5000, 20000, 2000], H=32, Hkv=8, E=1024, seed=77, device="cuda")
    ref_out, ref_lse = oracle_run(case)
    for s in (1, 2, 3, 7, 16, 64, 0):
        out, lse = gpu_run(case, num_splits=s)
        check(out, lse, ref_out, ref_lse, what=f"splits={s}")


def test_max_seqlen_q_bucketing_is_bit_identical():
    case = build_case("bucket", [1, 45, 130], [100, 400, 130], H=16, Hkv=4, E=64, seed=5, device="cuda")
    out1, lse1 = gpu_run(case, max_seqlen_q=130)
    out2, lse2 = gpu_run(case, max_seqlen_q=oracle.bucket_max_seqlen_q(130))
    out3, lse3 = gpu_run(case, max_seqlen_q=4096)
    assert torch.equal(out1, out2) and torch.equal(out1, out3)
    assert torch.equal(lse1, lse2) and torch.equal(lse1, lse3)


def test_page_permutation_invariance():
    case = build_case("perm", [1, 70], [3000, 600], H=16, Hkv=4, E=200, seed=8, device="cuda")
    out1, lse1 = gpu_run(case)
    g = torch.Generator().manual_seed(1)
    perm = torch.randperm(case.num_blocks, generator=g).cuda()
    kc = torch.empty_like(case.key_cache)
    vc = torch.empty_like(case.value_cache)
    kc[perm] = case.key_cache
    vc[perm] = case.value_cache
    bt = case.block_table.clone()
    valid = bt >= 0
    bt[valid] = perm[bt[valid].long()].to(torch.int32)
    out2, lse2 = ink.ink_rel_attn_varlen(case.q, kc, vc, block_table=bt, cache_seqlens=case.cache_seqlens,
                                         cu_seqlens_q=case.cu_seqlens_q, max_seqlen_q=case.max_seqlen_q,
                                         softmax_scale=case.softmax_scale, rel_extent=case.E,
                                         rel_logits=case.rel_logits, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_request_order_invariance():
    case = build_case("order", [1, 90, 1, 33], [700, 300, 50, 2000], H=16, Hkv=4, E=128, seed=12, device="cuda")
    out, lse = gpu_run(case)
    cu = case.cu_seqlens_q.tolist()
    order = [3, 1, 0, 2]
    q = torch.cat([case.q[cu[b]:cu[b + 1]] for b in order])
    rel = torch.cat([case.rel_logits[cu[b]:cu[b + 1]] for b in order])
    cu2 = torch.tensor(oracle.cu_seqlens_from_lengths([case.q_lens[b] for b in order]), dtype=torch.int32,
                       device="cuda")
    idx = torch.tensor(order, device="cuda")
    out2, lse2 = ink.ink_rel_attn_varlen(q, case.key_cache, case.value_cache, block_table=case.block_table[idx],
                                         cache_seqlens=case.cache_seqlens[idx], cu_seqlens_q=cu2,
                                         max_seqlen_q=case.max_seqlen_q, softmax_scale=case.softmax_scale,
                                         rel_extent=case.E, rel_logits=rel, return_lse=True)
    torch.cuda.synchronize()
    want = torch.cat([out[cu[b]:cu[b + 1]] for b in order])
    assert torch.equal(out2, want)


# --- device-side data errors ---------------------------------------------------------

def test_bad_page_id_is_flagged():
    case = build_case("badpage", [1, 20], [100, 60], H=8, Hkv=2, E=8, seed=4, device="cuda")
    case.block_table[0, 2] = case.num_blocks + 5
    gpu_run(case)
    assert errors_of_last_call() & ink.DEVERR["PAGE_ID"]
    case.block_table[0, 2] = -1
    gpu_run(case)
    assert errors_of_last_call() & ink.DEVERR["PAGE_ID"]


def test_bad_cu_and_lengths_are_flagged():
    case = build_case("badcu", [2, 3], [10, 10], H=8, Hkv=2, E=8, seed=4, device="cuda")
    case.cu_seqlens_q[1] = 7  # beyond cu[2]
    gpu_run(case)
    assert errors_of_last_call() & ink.DEVERR["CU_SEQLENS"]
    case = build_case("badk", [2, 3], [10, 10], H=8, Hkv=2, E=8, seed=4, device="cuda")
    case.cache_seqlens[0] = 10_000
    gpu_run(case)
    assert errors_of_last_call() & ink.DEVERR["SEQLEN_K"]
    case = build_case("badq", [2, 30], [10, 40], H=8, Hkv=2, E=8, seed=4, device="cuda", max_seqlen_q=8)
    gpu_run(case)
    assert errors_of_last_call() & ink.DEVERR["SEQLEN_Q"]


@pytest.mark.parametrize("splits", [1, 4])
def test_overlapping_requests_beyond_the_tile_budget_run_nothing(splits):
    """cu = [0, 100, 0, 100, 120]: requests 0 and 2 are valid but cover the same 100 tokens, so the
    valid requests need 9 q tiles of 32 tokens where T = 120 allows 8 (ceil(T / 32) + B): flagged,
    and every output row is left as it was."""
    case = build_case("overlap", [100, 0, 0, 20], [300, 10, 400, 50], H=8, Hkv=2, E=16, seed=6,
                      device="cuda", max_seqlen_q=100)
    case.cu_seqlens_q.copy_(torch.tensor([0, 100, 0, 100, 120], dtype=torch.int32))
    out = torch.full_like(case.q, 3.0)
    lse = torch.full((case.T, case.H), 7.0, dtype=torch.float32, device="cuda")
    gpu_run(case, num_splits=splits, out=out, lse=lse)
    assert errors_of_last_call() & ink.DEVERR["CU_SEQLENS"]
    assert bool((out == 3.0).all()) and bool((lse == 7.0).all())


def sampled_rows(case, n, seed):
    g = np.random.default_rng(seed)
    T, H = case.T, case.H
    rows = set(g.integers(0, T * H, size=n).tolist())
    # always include the first/last row of every request
    cu = case.cu_seqlens_q.tolist()
    for b in range(case.B):
        if cu[b + 1] > cu[b]:
            rows.add(cu[b] * H)
            rows.add((cu[b + 1] - 1) * H + H - 1)
    return np.array(sorted(rows), dtype=np.int64)
