"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: a
printed example, an independent dense formulation (tests/dense_ref.py), a
library routine on a special case, a closed form, or an invariant.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from dense_ref import dense_attention
from workloads import build_case, random_case, workload_lengths

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _run(case, **over):
    kw = case.oracle_kwargs()
    kw.update(over)
    return oracle.attention(case.q, case.key_cache, case.value_cache, case.block_table,
                            case.cache_seqlens, case.cu_seqlens_q, **kw)


def _dense(case, **over):
    kw = case.oracle_kwargs()
    kw.update(over)
    return dense_attention(case.q, case.key_cache, case.value_cache, case.block_table,
                           case.cache_seqlens, case.cu_seqlens_q, **kw)


def _close(a, b, tol):
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape
    fa, fb = np.isfinite(a), np.isfinite(b)
    assert np.array_equal(fa, fb), "finite / -inf pattern differs"
    assert np.array_equal(a[~fa], b[~fb])
    if fa.any():
        err = np.max(np.abs(a[fa] - b[fb]))
        assert err <= tol, f"max abs diff {err}"


# --- printed examples ---------------------------------------------------------

def test_page_index_csr_printed_examples():
    g = _golden("page_index_csr.json")
    for c in g["cases"]:
        indptr, indices, last = oracle.page_index_csr(c["block_table"], c["seq_lens"], g["block_size"],
                                                      count=c["count"])
        assert indptr == c["indptr"]
        assert indices == c["indices"]
        assert last == c["last_page_len"]


def test_cu_seqlens_printed_examples():
    for c in _golden("cu_seqlens.json")["cases"]:
        assert oracle.cu_seqlens_from_lengths(c["lengths"]) == c["cu_seqlens"]


def test_bucket_max_seqlen_q():
    g = _golden("bucket_max_seqlen_q.json")
    for n, want in g["printed"] + g["from_the_formula"]:
        assert oracle.bucket_max_seqlen_q(n) == want


def test_page_num_splits_reading_at_workloads():
    for c in _golden("page_num_splits_workloads.json")["cases"]:
        kw = {k: c[k] for k in ("is_local", "batch_size", "max_query_len", "num_heads", "num_kv_heads",
                                "max_kv_len")}
        if "capability_major" in c:
            kw["capability_major"] = c["capability_major"]
        assert oracle.page_num_splits(**kw) == c["splits"], c["workload"]


def test_workload_shapes_match_heuristic_inputs():
    # the golden shapes above are the workloads' own maxima
    _, kv = workload_lengths("decode_batch")
    assert max(kv) <= 32768 and min(kv) >= 1024
    q, kv = workload_lengths("chunked_prefill")
    assert max(q) == 2048 and max(kv) == 16384


def test_slot_mapping_brute_force():
    g = torch.Generator().manual_seed(3)
    bs = 4
    block_table = torch.randperm(40, generator=g)[:30].view(3, 10).tolist()
    seq_lens = [13, 1, 29]
    query_lens = [5, 1, 29]
    got = oracle.slot_mapping(block_table, seq_lens, query_lens, bs)
    want = []
    for row, n, ql in zip(block_table, seq_lens, query_lens):
        dense = [p * bs + o for p in row for o in range(bs)]  # logical position -> slot
        want += dense[n - ql:n]
    assert got == want


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_reshape_and_cache_reads_back_through_the_block_table(bs):
    """The append stores every new token where attention later finds it, and nothing else.

    Read back through the definition (request i's logical position p lives in page
    block_table[i][p // bs] at offset p % bs), not through the slot arithmetic.
    """
    g = torch.Generator().manual_seed(11 + bs)
    H = 3
    seq_lens, query_lens = [13, 1, 29, 7], [5, 1, 29, 0]
    pages = [(n + bs - 1) // bs for n in seq_lens]
    pool = sum(pages) + 5
    perm = torch.randperm(pool, generator=g).tolist()
    block_table, o = [], 0
    for n in pages:
        block_table.append(perm[o:o + n] + [-1] * (max(pages) - n))
        o += n
    slots = oracle.slot_mapping(block_table, seq_lens, query_lens, bs)
    T = len(slots)
    # two padding tokens (slot -1) in the middle of the step
    slots = slots[:3] + [-1, -1] + slots[3:]
    T += 2
    key = torch.randn(T, H, 128, generator=g).to(torch.bfloat16)
    value = torch.randn(T, H, 128, generator=g).to(torch.bfloat16)
    kc0 = torch.randn(pool, bs, H, 128, generator=g).to(torch.bfloat16)
    vc0 = torch.randn(pool, bs, H, 128, generator=g).to(torch.bfloat16)
    kc, vc = oracle.reshape_and_cache(key, value, kc0, vc0, slots)
    ku, vu = key.view(torch.int16).numpy().view(np.uint16), value.view(torch.int16).numpy().view(np.uint16)
    k0, v0 = kc0.view(torch.int16).numpy().view(np.uint16), vc0.view(torch.int16).numpy().view(np.uint16)
    written = np.zeros((pool, bs), dtype=bool)
    t = 0
    for i, (n, ql) in enumerate(zip(seq_lens, query_lens)):
        for j in range(ql):
            if t == 3:
                t += 2  # the padding tokens
            p = n - ql + j
            page, off = block_table[i][p // bs], p % bs
            assert np.array_equal(kc[page, off], ku[t]) and np.array_equal(vc[page, off], vu[t])
            written[page, off] = True
            t += 1
    assert written.sum() == T - 2
    assert np.array_equal(kc[~written], k0[~written]) and np.array_equal(vc[~written], v0[~written])


# --- attention core against the independent dense formulation ---------------

@pytest.mark.parametrize("seed", range(240))
def test_oracle_matches_dense_bruteforce(seed):
    case = random_case(seed, D=[8, 16, 32][seed % 3])
    out, lse = _run(case)
    dout, dlse = _dense(case)
    _close(out, dout, 1e-12)
    _close(lse, dlse, 1e-12)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("seed", range(8))
def test_oracle_matches_dense_wide_head_dims(seed, D):
    """The head sizes a paged backend serves (64, 128, 256) against the dense formulation."""
    case = random_case(500 + seed + 31 * D, D=D)
    out, lse = _run(case)
    dout, dlse = _dense(case)
    _close(out, dout, 1e-12)
    _close(lse, dlse, 1e-12)


@pytest.mark.parametrize("seed", range(16))
def test_zero_bias_is_sdpa_with_explicit_mask(seed):
    """rel_logits == 0 reduces to plain causal GQA attention (fp64 SDPA), at head sizes 32, 64 and 256."""
    case = random_case(900 + seed, D=[32, 64, 256][seed % 3], E=16)
    case.rel_logits = torch.zeros_like(case.rel_logits)
    out, lse = _run(case)
    out0, _ = _run(case, rel_extent=0, rel_logits=None)
    _close(out, out0, 0.0)
    G = case.H // case.Hkv
    for b in range(case.B):
        t0, t1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        Lq, Lk = t1 - t0, case.kv_lens[b]
        if Lq == 0:
            continue
        npg = -(-Lk // case.BS)
        pages = case.block_table[b, :npg].long()
        K = case.key_cache[pages].reshape(-1, case.Hkv, case.D)[:Lk].double()
        V = case.value_cache[pages].reshape(-1, case.Hkv, case.D)[:Lk].double()
        K = K.repeat_interleave(G, dim=1).permute(1, 0, 2)
        V = V.repeat_interleave(G, dim=1).permute(1, 0, 2)
        Q = case.q[t0:t1].double().permute(1, 0, 2)
        i = torch.arange(Lq)[:, None] + (Lk - Lq)
        j = torch.arange(Lk)[None, :]
        mask = torch.ones(Lq, Lk, dtype=torch.bool)
        if case.causal:
            mask &= j <= i
        if case.window_left >= 0:
            mask &= j >= i - case.window_left
        if case.window_right >= 0:
            mask &= j <= i + case.window_right
        rows = mask.any(dim=1)
        if not rows.any():
            assert np.all(out[t0:t1] == 0)
            continue
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[:, rows], K, V, attn_mask=mask[rows], scale=case.softmax_scale)
        got = torch.from_numpy(out[t0:t1][rows.numpy()]).permute(1, 0, 2)
        assert torch.max(torch.abs(got - ref)) < 1e-12
        assert np.all(out[t0:t1][~rows.numpy()] == 0)


# --- closed forms -------------------------------------------------------------

@pytest.mark.parametrize("D", [16, 64, 256])
def test_single_key_decode_closed_form(D):
    """Lk = 1: the output is the single V row and lse the single score."""
    case = build_case("one", [1, 1], [1, 1], H=4, Hkv=2, D=D, BS=4, E=3, seed=7)
    out, lse = _run(case)
    for b in range(2):
        t = b
        page = int(case.block_table[b, 0])
        for h in range(4):
            g = h // 2
            v = case.value_cache[page, 0, g].double().numpy()
            k = case.key_cache[page, 0, g].double().numpy()
            qv = case.q[t, h].double().numpy()
            s = case.softmax_scale * float(np.dot(qv, k)) + float(case.rel_logits[t, h, 0])
            assert np.array_equal(out[t, h], v)
            assert abs(lse[t, h] - s) <= 1e-12 * max(1.0, abs(s))


def test_zero_query_is_mean_of_visible_values():
    case = build_case("zq", [3, 1], [9, 20], H=2, Hkv=1, D=8, BS=4, E=0, seed=9, window=(5, -1))
    case.q = torch.zeros_like(case.q)
    out, lse = _run(case)
    for b, (t0, Lq, Lk) in enumerate([(0, 3, 9), (3, 1, 20)]):
        npg = -(-Lk // 4)
        V = case.value_cache[case.block_table[b, :npg].long()].reshape(-1, 1, 8)[:Lk, 0].double().numpy()
        for i in range(Lq):
            qa = i + Lk - Lq
            lo = max(0, qa - 5)
            vis = V[lo:qa + 1]
            for h in range(2):
                assert np.max(np.abs(out[t0 + i, h] - vis.mean(axis=0))) < 1e-14
                assert abs(lse[t0 + i, h] - math.log(len(vis))) < 1e-14


# --- bias algebra ---------------------------------------------------------------

def test_constant_bias_shifts_lse_only():
    case = random_case(77, D=16, E=64, max_kv_extra=40, max_q=20, causal=True, window=(-1, -1))
    assert case.E >= max(case.kv_lens)
    out0, lse0 = _run(case, rel_extent=0, rel_logits=None)
    c = 0.625
    case.rel_logits = torch.full_like(case.rel_logits, c)
    out, lse = _run(case)
    # every visible key has 0 <= rd <= q_abs < Lk <= E, so the bias is c everywhere
    _close(out, out0, 1e-13)
    fin = np.isfinite(lse0)
    assert fin.any()
    assert np.max(np.abs(lse[fin] - (lse0[fin] + c))) < 1e-12


def test_extent_one_biases_only_the_diagonal():
    """E = 1 equals a wider table that is zero except at rd = 0."""
    case = build_case("diag", [4, 1, 7], [6, 5, 7], H=2, Hkv=1, D=8, BS=2, E=1, seed=11)
    out, lse = _run(case)
    wide = torch.zeros(case.T, case.H, 9)
    wide[:, :, 0] = case.rel_logits[:, :, 0]
    out9, lse9 = _run(case, rel_extent=9, rel_logits=wide)
    _close(out, out9, 0.0)
    _close(lse, lse9, 0.0)
    z_out, _ = _run(case, rel_extent=0, rel_logits=None)
    assert not np.allclose(out, z_out)


def test_unread_bias_entries_have_no_effect():
    """Entries at rd > q_abs (no such key) or beyond a left window are never read."""
    case = build_case("nan", [3, 1, 6], [3, 9, 14], H=4, Hkv=2, D=16, BS=4, E=12, seed=13,
                      window=(4, -1))
    ref_out, ref_lse = _run(case)
    rel = case.rel_logits.clone()
    for b in range(case.B):
        t0 = int(case.cu_seqlens_q[b])
        Lq, Lk = case.q_lens[b], case.kv_lens[b]
        for i in range(Lq):
            qa = i + Lk - Lq
            rel[t0 + i, :, min(case.E, qa + 1):] = float("nan")   # rd > q_abs
            rel[t0 + i, :, min(case.E, 5):] = float("nan")        # rd > window_left
    case.rel_logits = rel
    out, lse = _run(case)
    assert np.all(np.isfinite(out))
    _close(out, ref_out, 0.0)
    _close(lse, ref_lse, 0.0)


# --- split-and-merge and invariances ------------------------------------------------

@pytest.mark.parametrize("seed", range(30))
def test_split_merge_equals_unsplit(seed):
    case = random_case(2000 + seed, D=16)
    out, lse = _run(case)
    for chunk in (1, 3, 16, 64):
        so, sl = _run(case, chunk_keys=chunk)
        _close(so, out, 1e-12)
        _close(sl, lse, 1e-12)


def test_unnormalised_partials_with_page_weights_would_be_wrong():
    """Reading of the PagedAttention V2 Phase-2 weights exp(m_c - gmax) * l_c:
    they are right for partition outputs normalised by l_c, and count l_c
    twice for the unnormalised sum the page's partition step stores."""
    rng = np.random.default_rng(5)
    s = rng.normal(size=40) * 2
    v = rng.normal(size=(40, 3))
    p = np.exp(s - s.max())
    exact = (p[:, None] * v).sum(0) / p.sum()
    chunks = [slice(0, 7), slice(7, 25), slice(25, 40)]
    m = np.array([s[c].max() for c in chunks])
    l = np.array([np.exp(s[c] - s[c].max()).sum() for c in chunks])
    acc = np.array([(np.exp(s[c] - s[c].max())[:, None] * v[c]).sum(0) for c in chunks])
    w = np.exp(m - m.max()) * l
    normalised = (w[:, None] * (acc / l[:, None])).sum(0) / w.sum()
    unnormalised = (w[:, None] * acc).sum(0) / w.sum()
    assert np.allclose(normalised, exact, atol=1e-14)
    assert not np.allclose(unnormalised, exact, atol=1e-3)


def test_page_permutation_is_bit_identical():
    case = random_case(31, D=32, BS=4, B=3, max_q=12, max_kv_extra=60, E=5)
    out, lse = _run(case)
    g = torch.Generator().manual_seed(99)
    NB = case.num_blocks
    perm = torch.randperm(NB, generator=g)          # new physical slot of old page p is perm[p]
    kc = torch.empty_like(case.key_cache)
    vc = torch.empty_like(case.value_cache)
    kc[perm] = case.key_cache
    vc[perm] = case.value_cache
    bt = case.block_table.clone()
    valid = bt >= 0
    bt[valid] = perm[bt[valid].long()].to(torch.int32)
    case.key_cache, case.value_cache, case.block_table = kc, vc, bt
    out2, lse2 = _run(case)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_block_size_one_equals_block_size_sixteen():
    case16 = random_case(41, D=16, BS=16, B=2, E=7)
    out16, lse16 = _run(case16)
    # re-page the same logical K/V with one token per page
    K, V, rows = [], [], []
    off = 0
    for b in range(case16.B):
        Lk = case16.kv_lens[b]
        npg = -(-Lk // 16)
        pages = case16.block_table[b, :npg].long()
        K.append(case16.key_cache[pages].reshape(-1, case16.Hkv, case16.D)[:Lk])
        V.append(case16.value_cache[pages].reshape(-1, case16.Hkv, case16.D)[:Lk])
        rows.append(list(range(off, off + Lk)))
        off += Lk
    kc = torch.cat(K).unsqueeze(1)
    vc = torch.cat(V).unsqueeze(1)
    width = max(len(r) for r in rows)
    bt = torch.full((case16.B, width), -1, dtype=torch.int32)
    for b, r in enumerate(rows):
        bt[b, :len(r)] = torch.tensor(r, dtype=torch.int32)
    out1, lse1 = oracle.attention(case16.q, kc, vc, bt, case16.cache_seqlens, case16.cu_seqlens_q,
                                  **case16.oracle_kwargs())
    assert np.array_equal(out1, out16) and np.array_equal(lse1, lse16)


def test_request_permutation_and_one_at_a_time():
    case = random_case(51, D=16, B=4, E=9, max_q=10)
    out, lse = _run(case)
    cu = case.cu_seqlens_q.tolist()
    for b in range(case.B):
        t0, t1 = cu[b], cu[b + 1]
        sub = build_case("one", [case.q_lens[b]], [case.kv_lens[b]], H=case.H, Hkv=case.Hkv, D=case.D,
                         BS=case.BS, E=0, seed=0)
        sub.q = case.q[t0:t1]
        sub.key_cache, sub.value_cache = case.key_cache, case.value_cache
        sub.block_table = case.block_table[b:b + 1]
        sub.cache_seqlens = case.cache_seqlens[b:b + 1]
        sub.E = case.E
        sub.rel_logits = case.rel_logits[t0:t1]
        sub.causal, sub.window_left, sub.window_right = case.causal, case.window_left, case.window_right
        o1, l1 = _run(sub)
        assert np.array_equal(o1, out[t0:t1]) and np.array_equal(l1, lse[t0:t1])
    # reverse the request order
    order = list(reversed(range(case.B)))
    q = torch.cat([case.q[cu[b]:cu[b + 1]] for b in order])
    rel = torch.cat([case.rel_logits[cu[b]:cu[b + 1]] for b in order])
    cu2 = oracle.cu_seqlens_from_lengths([case.q_lens[b] for b in order])
    o2, l2 = oracle.attention(q, case.key_cache, case.value_cache, case.block_table[order],
                              case.cache_seqlens[order], torch.tensor(cu2, dtype=torch.int32),
                              **{**case.oracle_kwargs(), "rel_logits": rel})
    want = np.concatenate([out[cu[b]:cu[b + 1]] for b in order])
    assert np.array_equal(o2, want)


def test_sampled_rows_equal_full_rows():
    case = random_case(61, D=16, B=3, E=9)
    out, lse = _run(case)
    rows = np.array([0, 5, case.T * case.H - 1, 3], dtype=np.int64)
    rows = rows[rows < case.T * case.H]
    o, l = _run(case, rows=rows)
    flat_o = out.reshape(-1, case.D)
    flat_l = lse.reshape(-1)
    assert np.array_equal(o, flat_o[rows]) and np.array_equal(l, flat_l[rows])


# --- error behaviour ---------------------------------------------------------------

def test_bad_page_id_is_reported():
    case = build_case("bad", [2], [20], H=2, Hkv=1, D=8, BS=4, E=0, seed=1)
    case.block_table[0, 2] = case.num_blocks + 3
    with pytest.raises(oracle.OracleError):
        _run(case)


def test_non_monotone_cu_is_reported():
    case = build_case("cu", [2, 3], [4, 5], H=2, Hkv=1, D=8, BS=4, E=0, seed=1)
    case.cu_seqlens_q = torch.tensor([0, 4, 5], dtype=torch.int32)  # request 0 claims 4 tokens
    case.cu_seqlens_q[1] = 6
    with pytest.raises(oracle.OracleError):
        _run(case)


# --- FP8 (E4M3) KV cache ------------------------------------------------------

def test_fp8_decoder_matches_an_independent_e4m3_for_every_code():
    """All 256 codes against torch's float8_e4m3fn (an independent implementation of the OCP format),
    plus the format's landmarks: 1, -1, the largest finite value 448, the smallest subnormal 2^-9, the
    smallest normal 2^-6, +-0, and NaN for S.1111.111."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    mine = oracle.e4m3_to_float64(codes)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.flatnonzero(nan).tolist() == [0x7F, 0xFF]
    assert np.array_equal(mine[~nan], ref[~nan])
    got = oracle.e4m3_to_float64(np.array([0x38, 0xB8, 0x7E, 0x01, 0x08, 0x00, 0x80], dtype=np.uint8))
    assert got.tolist() == [1.0, -1.0, 448.0, 2.0 ** -9, 2.0 ** -6, 0.0, -0.0]
    assert math.copysign(1.0, got[-1]) == -1.0


def _fp8_case(seed, **over):
    case = random_case(seed, D=32, **over)
    g = torch.Generator().manual_seed(7000 + seed)
    shape = case.key_cache.shape
    k8 = (torch.randn(shape, generator=g) * 6).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (torch.randn(shape, generator=g) * 6).to(torch.float8_e4m3fn).view(torch.uint8)
    return case, k8, v8


def _fp8_run(case, k8, v8, ks, vs, **over):
    kw = case.oracle_kwargs()
    kw.update(over)
    return oracle.attention_fp8kv(case.q, k8, v8, case.block_table, case.cache_seqlens, case.cu_seqlens_q,
                                  k_scale=ks, v_scale=vs, **kw)


@pytest.mark.parametrize("seed", range(24))
def test_fp8_cache_equals_bf16_cache_of_the_same_values(seed):
    """With power-of-two scales every k_scale * E4M3 value is exact in bf16, so the FP8-cache attention
    must equal the (dense-pinned) bf16-cache attention on those values, to the last bit of fp64."""
    case, k8, v8 = _fp8_case(seed)
    ks, vs = 2.0 ** -3, 2.0 ** 2
    kb = torch.from_numpy(oracle.e4m3_to_float64(k8) * ks).to(torch.bfloat16)
    vb = torch.from_numpy(oracle.e4m3_to_float64(v8) * vs).to(torch.bfloat16)
    assert np.array_equal(kb.double().numpy(), oracle.e4m3_to_float64(k8) * ks)  # exact in bf16
    out, lse = _fp8_run(case, k8, v8, ks, vs)
    bout, blse = oracle.attention(case.q, kb, vb, case.block_table, case.cache_seqlens, case.cu_seqlens_q,
                                  **case.oracle_kwargs())
    _close(out, bout, 0.0)
    _close(lse, blse, 0.0)


@pytest.mark.parametrize("seed", range(8))
def test_fp8_scales_are_a_logit_scale_and_an_output_scale(seed):
    """K = k_scale * E4M3 multiplies every q.k by k_scale (the same as softmax_scale * k_scale with unit
    scales); V = v_scale * E4M3 multiplies the output by v_scale and leaves the log-sum-exp alone."""
    case, k8, v8 = _fp8_case(100 + seed)
    ks, vs = 0.37, 1.9
    out, lse = _fp8_run(case, k8, v8, ks, vs)
    uout, ulse = _fp8_run(case, k8, v8, 1.0, 1.0, softmax_scale=case.softmax_scale * ks)
    _close(out, vs * uout, 1e-12)
    _close(lse, ulse, 1e-12)


def test_e4m3_encoder_matches_an_independent_cast_in_range():
    """Every finite E4M3 value, every midpoint between neighbours (and a hair either side of it) and random
    fp32 values in [-448, 448] against torch's float8_e4m3fn cast (round to nearest even)."""
    vals = oracle.e4m3_to_float64(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2
    pts = np.concatenate([vals, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                          np.nextafter(mids.astype(np.float32), np.float32(1e9))])
    g = np.random.default_rng(5)
    rnd = np.concatenate([g.uniform(-448, 448, 20000), g.standard_normal(20000) * 2.0 ** g.integers(-12, 8, 20000)])
    y = np.concatenate([pts, -pts, rnd]).astype(np.float32)
    y = y[np.abs(y) <= 448]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(y), ref)


def test_e4m3_encoder_round_trip_ties_saturation():
    codes = np.concatenate([np.arange(0x7F), np.arange(0x80, 0xFF)]).astype(np.uint8)
    vals = oracle.e4m3_to_float64(codes).astype(np.float32)
    back = oracle.e4m3_encode(vals)
    assert np.array_equal(back[vals != 0], codes[vals != 0])     # every finite value encodes to its own code
    tie = lambda a, b: np.float32((oracle.e4m3_to_float64(np.array([a], np.uint8))[0] +
                                   oracle.e4m3_to_float64(np.array([b], np.uint8))[0]) / 2)
    # halfway cases go to the code with an even last mantissa bit
    for a, b in [(0x38, 0x39), (0x39, 0x3A), (0x00, 0x01), (0x07, 0x08), (0x7D, 0x7E)]:
        want = a if a % 2 == 0 else b
        assert oracle.e4m3_encode(np.array([tie(a, b)]))[0] == want
        assert oracle.e4m3_encode(np.array([-tie(a, b)]))[0] == want | 0x80
    big = np.array([448.0, 449.0, 464.0, 1e6, np.inf, -500.0, -np.inf], dtype=np.float32)
    assert oracle.e4m3_encode(big).tolist() == [0x7E] * 5 + [0xFE] * 2
    assert oracle.e4m3_encode(np.array([np.nan, 0.0, -0.0], np.float32)).tolist() == [0x7F, 0x00, 0x80]


@pytest.mark.parametrize("bs", [1, 16])
def test_reshape_and_cache_fp8_reads_back_quantized(bs):
    """Each stored byte, read back through the block table, is the E4M3 code of the fp32 quotient
    x / scale (the encoder above); nothing else in the cache changes; padding stores nothing."""
    g = torch.Generator().manual_seed(17 + bs)
    kv_lens, q_lens = [40, 7], [5, 7]
    pages = [(k + bs - 1) // bs for k in kv_lens]
    perm = torch.randperm(sum(pages) + 3, generator=g).tolist()
    table = [perm[:pages[0]], perm[pages[0]:pages[0] + pages[1]]]
    slots = oracle.slot_mapping(table, kv_lens, q_lens, bs) + [-1]
    T = len(slots)
    key = (torch.randn(T, 2, 128, generator=g) * 40).to(torch.bfloat16)    # some beyond 448 * k_scale
    value = (torch.randn(T, 2, 128, generator=g) * 0.01).to(torch.bfloat16)
    kc = torch.randint(0, 255, (len(perm), bs, 2, 128), generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 255, (len(perm), bs, 2, 128), generator=g, dtype=torch.uint8)
    ks, vs = 0.07, 0.0003
    nk, nv = oracle.reshape_and_cache_fp8(key, value, kc, vc, torch.tensor(slots), ks, vs)
    touched = np.zeros(kc.shape[:2], dtype=bool)
    t = 0
    for b, (lq, lk) in enumerate(zip(q_lens, kv_lens)):
        for j in range(lk - lq, lk):
            page, off = table[b][j // bs], j % bs
            kf = key[t].float().numpy() / np.float32(ks)
            vf = value[t].float().numpy() / np.float32(vs)
            assert np.array_equal(nk[page, off], oracle.e4m3_encode(kf))
            assert np.array_equal(nv[page, off], oracle.e4m3_encode(vf))
            touched[page, off] = True
            t += 1
    assert np.array_equal(nk[~touched], kc.numpy()[~touched])
    assert np.array_equal(nv[~touched], vc.numpy()[~touched])
    assert (nk[touched] == 0x7E).any() or (nk[touched] == 0xFE).any()       # saturation was exercised


def test_round_to_bf16_matches_torch():
    x = np.random.default_rng(0).normal(size=10000) * 10.0 ** np.random.default_rng(1).integers(-6, 6, 10000)
    want = torch.from_numpy(x).float().to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_to_bf16(x), want)
