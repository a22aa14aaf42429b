"""The decode kernel's launch variants on the GPU against the fp64 oracle.

The host picks, per call, how many CTAs share an SM (two when half of the SM's
shared memory still holds a three-stage ring: E4M3 pages, or bf16 pages of at
most 4 KV heads; one otherwise) and, at two an SM, whether the 16-row path is
compiled in (left out when max_seqlen_q * G <= 8, so that no decode item can
need it).  Each case below lands in one of those variants; all must agree with
the oracle at the bf16 path's tolerances, splits and windows included.
"""
import pytest

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
