"""The decode kernel's launch variants on the GPU against the fp64 oracle.

The host picks, per call, how many CTAs share an SM (two when half of the SM's
shared memory still holds a three-stage ring: E4M3 pages, or bf16 pages of at
most 4 KV heads; one otherwise) and, at two an SM, whether the 16-row path is
compiled in (left out when max_seqlen_q * G <= 8, so that no decode item can
need it).  Each case below lands in one of those variants; all must agree with
the oracle at the bf16 path's tolerances, splits and windows included.
"""
import pytest
import torch

import paged_varlen_attention_causal_gb300 as ink
from test_gpu_fp8 import parity_fp8
from test_gpu_parity import check, gpu_run, oracle_run
from workloads import build_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import oracle

    ink.build()
    ink.load()
    oracle.build()


def decode_case(H, Hkv, lq, seed, window=(-1, -1)):
    """Decode-shaped requests of up to `lq` tokens (lq * G <= 16), a mix of lengths."""
    q_lens = [1, lq, 1, lq, 1, min(2, lq)]
    kv_lens = [5, 333, 1500, 4100, 17, 900]
    return build_case(f"dv-{H}-{Hkv}-{lq}", q_lens, kv_lens, H=H, Hkv=Hkv, E=400, seed=seed, device="cuda",
                      window=window, causal=True)


# (H, Hkv): bf16 pages of 8 KV heads always keep one CTA an SM; fewer heads, and E4M3 pages, take two where
# the token bound leaves room for three stages in half an SM
HEADS = [(32, 8), (16, 4), (32, 4), (8, 2), (16, 1)]


def lq_cases(H, Hkv):
    """Token bounds that land in different variants: the stage's bias room grows with max_seqlen_q, so one
    token a request is the bound at which 8 KV heads of E4M3 (or 4 of bf16) still fit three stages in half an
    SM; max_seqlen_q * G <= 8 leaves the 16-row path out; up to 16 packed rows needs the full kernel."""
    G = H // Hkv
    small = max(1, 8 // G)
    large = max(1, 16 // G)
    return sorted({1, small, large})


@pytest.mark.parametrize("H,Hkv", HEADS)
@pytest.mark.parametrize("splits", [0, 3])
def test_bf16_decode_variants(H, Hkv, splits):
    for lq in lq_cases(H, Hkv):
        case = decode_case(H, Hkv, lq, seed=31 * H + Hkv + lq)
        out, lse = gpu_run(case, num_splits=splits)
        assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0
        ref_out, ref_lse = oracle_run(case)
        check(out, lse, ref_out, ref_lse, what=f"bf16 H={H} Hkv={Hkv} lq={lq} splits={splits}")


@pytest.mark.parametrize("H,Hkv", HEADS)
@pytest.mark.parametrize("splits", [0, 3])
def test_fp8_decode_variants(H, Hkv, splits):
    for lq in lq_cases(H, Hkv):
        case = decode_case(H, Hkv, lq, seed=37 * H + Hkv + lq)
        parity_fp8(case, f"fp8 H={H} Hkv={Hkv} lq={lq} splits={splits}", num_splits=splits)
        assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_variants_with_window(fp8):
    case = decode_case(16, 4, 2, seed=5, window=(300, 0))
    if fp8:
        parity_fp8(case, "fp8 window")
    else:
        out, lse = gpu_run(case)
        ref_out, ref_lse = oracle_run(case)
        check(out, lse, ref_out, ref_lse, what="bf16 window")
    assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0


# --- decode-only calls of at most 32 requests: each decode CTA finds its first item from the inputs and streams
# it while the prepass runs, waiting on the prepass only after that item

def test_small_call_bad_page_in_a_first_item_is_flagged():
    """A bad page id met while the first item streams (before the producer's wait on the prepass) is reported
    after that wait, so the prepass's error word does not hide it; the other requests are untouched."""
    case = decode_case(16, 4, 1, seed=91)
    good_out, good_lse = gpu_run(case, num_splits=1)
    assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    case.block_table[1, 0] = case.num_blocks + 3  # request 1's first page: item 1's first group
    out, lse = gpu_run(case, num_splits=1)
    assert ink.read_device_errors() & ink.DEVERR["PAGE_ID"]
    cu = case.cu_seqlens_q.tolist()
    keep = torch.ones(case.T, dtype=torch.bool)
    keep[cu[1]:cu[2]] = False
    assert torch.equal(out[keep.cuda()], good_out[keep.cuda()])


def test_small_call_request_beyond_max_seqlen_q_is_flagged_and_others_exact():
    """Request 1 has 3 tokens against max_seqlen_q 2 (so the call is decode-only: 2 x G <= 16): it is flagged
    and gets no items, by the prepass and by the decode CTAs' own first-item rule alike; the others match the
    oracle."""
    case = build_case("dv-msq", [1, 3, 1, 2], [700, 500, 90, 3000], H=16, Hkv=4, E=200, seed=17, device="cuda",
                      max_seqlen_q=2)
    out, lse = gpu_run(case)
    assert ink.read_device_errors() & ink.DEVERR["SEQLEN_Q"]
    cu = case.cu_seqlens_q.tolist()
    rows = [t * case.H + h for t in list(range(cu[0], cu[1])) + list(range(cu[2], cu[4])) for h in range(case.H)]
    ref_out, ref_lse = oracle_run(case, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what="requests within max_seqlen_q")


@pytest.mark.parametrize("fp8", [False, True])
def test_small_call_with_more_items_than_ctas(fp8):
    """Three long decodes cut into more splits than there are CTAs: each CTA streams its first item before the
    prepass is done and takes the rest from the prepass's queue."""
    case = build_case("dv-many", [1, 1, 1], [60000, 45000, 70000], H=32, Hkv=8, E=1024, seed=23, device="cuda")
    if fp8:
        parity_fp8(case, "fp8 many items", num_splits=400)
    else:
        out, lse = gpu_run(case, num_splits=400)
        ref_rows = list(range(case.T * case.H))
        ref_out, ref_lse = oracle_run(case, rows=ref_rows)
        check(out, lse, ref_out, ref_lse, rows=ref_rows, what="bf16 many items")
    assert ink.read_device_errors() & ~ink.DEVERR["EMPTY_ROWS"] == 0
