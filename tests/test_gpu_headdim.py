"""Head sizes 64 and 256 on the GPU against the fp64 oracle.

The vLLM V1 attention page lists 64, 128 and 256 among the head sizes a paged
backend serves; the PagedAttention V2 page's GQA example has H 24, Hkv 4 (G 6)
at head size 256.  Same tolerances as head size 128.  Decode-shaped requests run
in the decode kernel templated on D (the head-size-generic kernel where a warp's
share of the head would be narrower than 16, or two bf16 pages do not fit its
ring: D 64 with one KV head, D 256 with eight), prefill-shaped ones in the
head-size-generic kernel, with splits merged by the split-KV combine at the same
head size.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_causal_gb300 as ink
from test_gpu_parity import check, errors_of_last_call, gpu_run, oracle_run, sampled_rows
from workloads import build_case, random_case, workload_lengths

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ink.build()
    ink.load()
    oracle.build()


def parity(case, what, **kw):
    out, lse = gpu_run(case, **kw)
    assert errors_of_last_call() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    ref_out, ref_lse = oracle_run(case)
    return check(out, lse, ref_out, ref_lse, what=what)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("splits", [1, 4, 0])
def test_tiny_mix(D, splits):
    case = build_case(f"tiny-d{D}", [1, 1, 128], [47, 312, 128], H=8, Hkv=2, D=D, E=64, seed=1000,
                      pool_pages=64, device="cuda")
    parity(case, f"tiny mix D={D} splits={splits}", num_splits=splits)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("seed", range(10))
def test_random(D, seed):
    case = random_case(700 + seed, D=D, BS=[16, 32][seed % 2], device="cuda", max_q=90, max_kv_extra=500)
    parity(case, f"random{700 + seed} D={D}")


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("seed", range(4))
def test_random_split(D, seed):
    case = random_case(750 + seed, D=D, BS=16, device="cuda", max_q=50, max_kv_extra=900)
    parity(case, f"random{750 + seed} D={D} splits 3", num_splits=3)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("H,Hkv", [(24, 4), (8, 8), (32, 8), (16, 1), (128, 1), (6, 2)])
def test_head_layouts(D, H, Hkv):
    case = build_case(f"hl-{D}-{H}-{Hkv}", [1, 150, 3, 40], [900, 150, 300, 700], H=H, Hkv=Hkv, D=D, E=96,
                      seed=H * 7 + Hkv + D, device="cuda")
    parity(case, f"D={D} H={H} Hkv={Hkv}")


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("window,causal", [((64, 0), True), ((100, 30), False), ((-1, -1), False), ((4095, 0), True)])
def test_windows(D, window, causal):
    case = build_case(f"w-{D}", [140, 1, 33], [400, 800, 33], H=16, Hkv=4, D=D, E=64, seed=7, device="cuda",
                      window=window, causal=causal)
    parity(case, f"D={D} window={window} causal={causal}")


@pytest.mark.parametrize("D", [64, 256])
def test_bad_page_reads_zeros_and_is_flagged(D):
    case = build_case(f"bad-{D}", [100, 1], [300, 200], H=16, Hkv=4, D=D, E=32, seed=5, device="cuda")
    good_out, good_lse = gpu_run(case)
    case.block_table[1, 3] = case.num_blocks + 7
    out, lse = gpu_run(case)
    assert errors_of_last_call() & ink.DEVERR["PAGE_ID"]
    cu = case.cu_seqlens_q.tolist()
    assert torch.equal(out[:cu[1]], good_out[:cu[1]])  # the other request is untouched


@pytest.mark.parametrize("D", [64, 256])
def test_append_then_attend(D):
    """ink_reshape_and_cache at head size D is bit-exact against the oracle's append."""
    g = torch.Generator().manual_seed(D)
    T, Hkv, pool, bs = 300, 4, 40, 16
    key = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    value = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    kc = torch.randn(pool, bs, Hkv, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(pool, bs, Hkv, D, generator=g).to(torch.bfloat16)
    slots = torch.randperm(pool * bs, generator=g)[:T].to(torch.int64)
    slots[5] = -1
    want_k, want_v = oracle.reshape_and_cache(key, value, kc, vc, slots)
    dk, dv = kc.cuda(), vc.cuda()
    ink.reshape_and_cache(key.cuda(), value.cuda(), dk, dv, slots.cuda())
    torch.cuda.synchronize()
    bits = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits(dk), want_k) and np.array_equal(bits(dv), want_v)


def test_fp8_cache_is_refused_at_other_head_sizes():
    case = build_case("fp8-d64", [1, 1], [40, 70], H=8, Hkv=2, D=64, E=0, seed=3, device="cuda")
    k8 = case.key_cache.view(torch.uint8)[..., :64].contiguous()
    with pytest.raises(ink.InkError) as e:
        ink.ink_rel_attn_varlen_fp8kv(case.q, k8, k8, k_scale=1.0, v_scale=1.0, block_table=case.block_table,
                                      cache_seqlens=case.cache_seqlens, cu_seqlens_q=case.cu_seqlens_q,
                                      max_seqlen_q=case.max_seqlen_q, softmax_scale=case.softmax_scale)
    assert e.value.status == 2


@pytest.mark.slow
@pytest.mark.parametrize("D,H,Hkv", [(64, 32, 8), (256, 24, 4)])
def test_chunked_prefill_shape_sampled(D, H, Hkv):
    """The chunked prefill's request shape (4 x Lq 2048 on prior KV 0 / 2048 / 6144 / 14336, E 4096) at head
    size D; sampled rows (every request's first and last row among them) against the oracle."""
    q_lens, kv_lens = workload_lengths("chunked_prefill")
    case = build_case(f"cp-d{D}", q_lens, kv_lens, H=H, Hkv=Hkv, D=D, E=4096, bias_std=0.5, seed=1002 + D,
                      device="cuda")
    out, lse = gpu_run(case)
    assert errors_of_last_call() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    rows = sampled_rows(case, 512, 3)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what=f"chunked prefill D={D}")
    del case, out, lse
    torch.cuda.empty_cache()
