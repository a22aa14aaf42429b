"""KV append (ink_reshape_and_cache) on the GPU against the oracle, bit for bit.

The append is a byte copy, so every cache byte must equal the oracle's, at
every block size and KV head count, with padding tokens and with a slot past
the cache (flagged and skipped).  The last test appends a step's new tokens
and then runs attention over the updated cache, as a serving step does.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_causal_gb300 as ink
from workloads import build_case, fp8_kv, workload

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_RTOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    ink.build()
    ink.load()
    oracle.build()


def _step(q_lens, kv_lens, bs, Hkv, seed, pad_at=()):
    """Random cache and block table, and this step's new tokens with their slots."""
    g = torch.Generator().manual_seed(seed)
    pages = [(k + bs - 1) // bs for k in kv_lens]
    pool = sum(pages) + 7
    perm = torch.randperm(pool, generator=g).tolist()
    table, o = [], 0
    for n in pages:
        table.append(perm[o:o + n])
        o += n
    slots = oracle.slot_mapping(table, kv_lens, q_lens, bs)
    for at in sorted(pad_at):
        slots.insert(min(at, len(slots)), -1)
    T = len(slots)
    key = torch.randn(T, Hkv, 128, generator=g).to(torch.bfloat16)
    value = torch.randn(T, Hkv, 128, generator=g).to(torch.bfloat16)
    kc = torch.randn(pool, bs, Hkv, 128, generator=g).to(torch.bfloat16)
    vc = torch.randn(pool, bs, Hkv, 128, generator=g).to(torch.bfloat16)
    return key, value, kc, vc, torch.tensor(slots, dtype=torch.int64)


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("bs,Hkv", [(16, 8), (1, 4), (32, 1), (16, 2), (64, 8)])
def test_append_matches_oracle(bs, Hkv):
    key, value, kc, vc, slots = _step([1, 200, 3, 77], [900, 200, 40, 300], bs, Hkv, seed=bs * 10 + Hkv,
                                      pad_at=(0, 50, 151))
    want_k, want_v = oracle.reshape_and_cache(key, value, kc, vc, slots)
    dk, dv = kc.cuda(), vc.cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ink.reshape_and_cache(key.cuda(), value.cuda(), dk, dv, slots.cuda(), flags=flags)
    torch.cuda.synchronize()
    assert flags.item() == 0
    assert np.array_equal(_bits(dk), want_k) and np.array_equal(_bits(dv), want_v)


def test_append_flags_and_skips_a_slot_past_the_cache():
    key, value, kc, vc, slots = _step([40], [40], 16, 4, seed=5)
    slots[7] = kc.shape[0] * kc.shape[1] + 3  # past the pool
    ok = slots.clone()
    ok[7] = -1
    want_k, want_v = oracle.reshape_and_cache(key, value, kc, vc, ok)
    dk, dv = kc.cuda(), vc.cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ink.reshape_and_cache(key.cuda(), value.cuda(), dk, dv, slots.cuda(), flags=flags)
    torch.cuda.synchronize()
    assert flags.item() & ink.DEVERR["PAGE_ID"]
    assert np.array_equal(_bits(dk), want_k) and np.array_equal(_bits(dv), want_v)


def test_append_at_the_chunked_prefill_size():
    """8192 new tokens, 8 KV heads, 16-key pages (the chunked prefill's step)."""
    c = workload("chunked_prefill", device="cpu", E=0)  # the bias is not needed here
    table = c.block_table.tolist()
    slots = torch.tensor(oracle.slot_mapping(table, c.kv_lens, c.q_lens, c.BS), dtype=torch.int64)
    g = torch.Generator().manual_seed(77)
    key = torch.randn(c.T, c.Hkv, 128, generator=g).to(torch.bfloat16)
    value = torch.randn(c.T, c.Hkv, 128, generator=g).to(torch.bfloat16)
    want_k, want_v = oracle.reshape_and_cache(key, value, c.key_cache, c.value_cache, slots)
    dk, dv = c.key_cache.cuda(), c.value_cache.cuda()
    ink.reshape_and_cache(key.cuda(), value.cuda(), dk, dv, slots.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_bits(dk), want_k) and np.array_equal(_bits(dv), want_v)


def test_append_then_attend():
    """A serving step: write the new tokens' K/V, then attend over the updated cache."""
    case = build_case("append-step", [1, 64, 3], [500, 64, 130], H=16, Hkv=4, E=96, seed=9)
    table = case.block_table.tolist()
    slots = torch.tensor(oracle.slot_mapping(table, case.kv_lens, case.q_lens, case.BS), dtype=torch.int64)
    g = torch.Generator().manual_seed(10)
    key = torch.randn(case.T, case.Hkv, 128, generator=g).to(torch.bfloat16)
    value = torch.randn(case.T, case.Hkv, 128, generator=g).to(torch.bfloat16)
    want_k, want_v = oracle.reshape_and_cache(key, value, case.key_cache, case.value_cache, slots)
    ref_out, ref_lse = oracle.attention(case.q, torch.from_numpy(want_k.view(np.int16)).view(torch.bfloat16),
                                        torch.from_numpy(want_v.view(np.int16)).view(torch.bfloat16),
                                        case.block_table, case.cache_seqlens, case.cu_seqlens_q,
                                        **case.oracle_kwargs())
    d = case.to("cuda")
    ink.reshape_and_cache(key.cuda(), value.cuda(), d.key_cache, d.value_cache, slots.cuda())
    out, lse = ink.ink_rel_attn_varlen(d.q, d.key_cache, d.value_cache, block_table=d.block_table,
                                       cache_seqlens=d.cache_seqlens, cu_seqlens_q=d.cu_seqlens_q,
                                       max_seqlen_q=d.max_seqlen_q, softmax_scale=d.softmax_scale,
                                       causal=d.causal, rel_extent=d.E, rel_logits=d.rel_logits, return_lse=True)
    torch.cuda.synchronize()
    o = out.float().cpu().double().numpy().reshape(ref_out.shape)
    assert np.max(np.abs(o - ref_out)) <= OUT_TOL
    l = lse.cpu().double().numpy().reshape(ref_lse.shape)
    rel = np.abs(l - ref_lse) / np.maximum(1.0, np.abs(ref_lse))
    assert rel.max() <= LSE_RTOL


# --- FP8 (E4M3) cache: quantize on store --------------------------------------

def _fp8_step(q_lens, kv_lens, bs, Hkv, seed, pad_at=()):
    """A step of new bf16 tokens over random E4M3 caches; keys span the whole E4M3 range at k_scale 0.05
    (some saturate), values are small (some E4M3 subnormals), and a few are exact zeros of either sign."""
    key, value, _, _, slots = _step(q_lens, kv_lens, bs, Hkv, seed, pad_at)
    g = torch.Generator().manual_seed(seed + 1000)
    key = (key.float() * 12).to(torch.bfloat16)
    value = (value.float() * 0.002).to(torch.bfloat16)
    key.view(-1)[::97] = 0.0
    value.view(-1)[::89] = -0.0
    pool = int(slots.max().item()) // bs + 8
    kc = torch.randint(0, 255, (pool, bs, Hkv, 128), generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 255, (pool, bs, Hkv, 128), generator=g, dtype=torch.uint8)
    return key, value, kc, vc, slots


@pytest.mark.parametrize("bs,Hkv,ks,vs", [(16, 8, 0.05, 1e-4), (1, 4, 1.0, 1.0), (32, 1, 0.3, 7e-5),
                                          (16, 2, 0.05, 0.0017)])
def test_append_fp8_matches_oracle_bit_for_bit(bs, Hkv, ks, vs):
    key, value, kc, vc, slots = _fp8_step([1, 200, 3, 77], [900, 200, 40, 300], bs, Hkv, seed=bs * 7 + Hkv,
                                          pad_at=(0, 50, 151))
    want_k, want_v = oracle.reshape_and_cache_fp8(key, value, kc, vc, slots, ks, vs)
    dk, dv = kc.cuda(), vc.cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ink.reshape_and_cache_fp8(key.cuda(), value.cuda(), dk, dv, slots.cuda(), k_scale=ks, v_scale=vs, flags=flags)
    torch.cuda.synchronize()
    assert flags.item() == 0
    assert np.array_equal(dk.cpu().numpy(), want_k) and np.array_equal(dv.cpu().numpy(), want_v)
    if ks == 0.05:
        assert (want_k == 0x7E).any() and (want_k == 0xFE).any()   # saturated on both sides


def test_append_fp8_flags_a_slot_past_the_cache():
    key, value, kc, vc, slots = _fp8_step([40], [40], 16, 4, seed=6)
    slots[3] = kc.shape[0] * kc.shape[1]
    ok = slots.clone()
    ok[3] = -1
    want_k, want_v = oracle.reshape_and_cache_fp8(key, value, kc, vc, ok, 0.5, 0.25)
    dk, dv = kc.cuda(), vc.cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ink.reshape_and_cache_fp8(key.cuda(), value.cuda(), dk, dv, slots.cuda(), k_scale=0.5, v_scale=0.25,
                              flags=flags)
    torch.cuda.synchronize()
    assert flags.item() & ink.DEVERR["PAGE_ID"]
    assert np.array_equal(dk.cpu().numpy(), want_k) and np.array_equal(dv.cpu().numpy(), want_v)


def test_append_fp8_then_attend():
    """A serving step over an E4M3 cache: quantize the new tokens into it, then decode over it."""
    case = build_case("append-fp8", [1, 1, 2], [500, 64, 130], H=32, Hkv=8, E=96, seed=19)
    ks, vs = 0.06, 0.05
    k8, v8 = fp8_kv(case, ks, vs)
    slots = torch.tensor(oracle.slot_mapping(case.block_table.tolist(), case.kv_lens, case.q_lens, case.BS),
                         dtype=torch.int64)
    g = torch.Generator().manual_seed(20)
    key = torch.randn(case.T, case.Hkv, 128, generator=g).to(torch.bfloat16)
    value = torch.randn(case.T, case.Hkv, 128, generator=g).to(torch.bfloat16)
    want_k, want_v = oracle.reshape_and_cache_fp8(key, value, k8, v8, slots, ks, vs)
    ref_out, ref_lse = oracle.attention_fp8kv(case.q, want_k, want_v, case.block_table, case.cache_seqlens,
                                              case.cu_seqlens_q, k_scale=ks, v_scale=vs, **case.oracle_kwargs())
    d = case.to("cuda")
    dk, dv = k8.cuda(), v8.cuda()
    ink.reshape_and_cache_fp8(key.cuda(), value.cuda(), dk, dv, slots.cuda(), k_scale=ks, v_scale=vs)
    out, lse = ink.ink_rel_attn_varlen_fp8kv(d.q, dk, dv, k_scale=ks, v_scale=vs, block_table=d.block_table,
                                             cache_seqlens=d.cache_seqlens, cu_seqlens_q=d.cu_seqlens_q,
                                             max_seqlen_q=d.max_seqlen_q, softmax_scale=d.softmax_scale,
                                             rel_extent=d.E, rel_logits=d.rel_logits, return_lse=True)
    torch.cuda.synchronize()
    assert np.array_equal(dk.cpu().numpy(), want_k)
    o = out.float().cpu().double().numpy().reshape(ref_out.shape)
    assert np.max(np.abs(o - ref_out)) <= OUT_TOL
    l = lse.cpu().double().numpy().reshape(ref_lse.shape)
    assert (np.abs(l - ref_lse) / np.maximum(1.0, np.abs(ref_lse))).max() <= LSE_RTOL


@pytest.mark.parametrize("scale", [0.05, 1.0, 3.7e-3, 123.0, 2.0 ** -10, 0.3, 2.0 ** -126, 2.0 ** 126])
def test_append_fp8_every_bf16_value(scale):
    """Every bf16 bit pattern except the NaNs (zeros, subnormals, normals, infinities, both signs) quantized
    with one scale: the stored codes equal the oracle's, which divides in IEEE fp32 and rounds with ties to
    even.  Checks the kernel's quotient and conversion on the whole input range, not a sample, down to the
    extreme scales the entry point accepts (2^-126: zeros stay zero, everything else saturates)."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch.bfloat16)
    nan = torch.isnan(vals.float())
    vals = torch.where(nan, torch.zeros_like(vals), vals)        # NaN codes are not compared
    key = vals.reshape(512, 1, 128).contiguous()
    value = (-vals).reshape(512, 1, 128).contiguous()
    slots = torch.arange(512, dtype=torch.int64)
    kc = torch.zeros(32, 16, 1, 128, dtype=torch.uint8)
    vc = torch.zeros_like(kc)
    want_k, want_v = oracle.reshape_and_cache_fp8(key, value, kc, vc, slots, scale, scale)
    dk, dv = kc.cuda(), vc.cuda()
    ink.reshape_and_cache_fp8(key.cuda(), value.cuda(), dk, dv, slots.cuda(), k_scale=scale, v_scale=scale)
    torch.cuda.synchronize()
    got_k, got_v = dk.cpu().numpy(), dv.cpu().numpy()
    diff = np.flatnonzero(got_k.reshape(-1) != want_k.reshape(-1))
    assert diff.size == 0, f"{diff.size} codes differ, first at bf16 {int(bits[diff[0]]) & 0xffff:#06x}"
    assert np.array_equal(got_v, want_v)
