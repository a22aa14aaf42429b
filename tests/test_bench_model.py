"""Host logic of bench.py: the algorithmic work counted per step must match
the visibility definition (checked against dense masks on small shapes)."""
import numpy as np
import pytest

import bench
from workloads import WORKLOAD_ORDER, workload_lengths


class _Shape:
    def __init__(self, q_lens, kv_lens, H, Hkv, E=0, causal=True, window=(-1, -1)):
        self.q_lens, self.kv_lens, self.H, self.Hkv, self.E = q_lens, kv_lens, H, Hkv, E
        self.causal = causal
        self.window_left, self.window_right = window


def _dense_pairs(lq, lk, causal, wl, wr):
    i = np.arange(lq)[:, None] + lk - lq
    j = np.arange(lk)[None, :]
    m = np.ones((lq, lk), bool)
    if causal:
        m &= j <= i
    if wl >= 0:
        m &= j >= i - wl
    if wr >= 0:
        m &= j <= i + wr
    return m


@pytest.mark.parametrize("seed", range(20))
def test_work_model_matches_dense_masks(seed):
    g = np.random.default_rng(seed)
    B = int(g.integers(1, 5))
    Hkv = int(g.choice([1, 2, 4]))
    G = int(g.choice([1, 4, 8]))
    q_lens = [int(g.choice([1, 2, int(g.integers(3, 60))])) for _ in range(B)]
    kv_lens = [q + int(g.integers(0, 90)) for q in q_lens]
    causal = bool(g.integers(0, 2))
    window = (int(g.choice([-1, 0, 7, 30])), int(g.choice([-1, 0, 5])))
    s = _Shape(q_lens, kv_lens, Hkv * G, Hkv, causal=causal, window=window)
    kv, flops, pairs = bench.work_of(s)
    want_kv = want_pairs = 0
    for lq, lk in zip(q_lens, kv_lens):
        m = _dense_pairs(lq, lk, causal, *window)
        if lq * G <= 16:
            want_kv += int(m.any(axis=0).sum()) * Hkv * 128 * 2 * 2
        else:
            want_pairs += int(m.sum())
    assert pairs == want_pairs
    assert flops == 4 * 128 * s.H * want_pairs
    # decode bytes: the model counts the union range [lo(first row), hi(last row)]
    assert kv >= want_kv


def test_workload_totals():
    shapes = {
        "decode_batch": dict(H=32, Hkv=8, E=1024),
        "chunked_prefill": dict(H=32, Hkv=8, E=4096),
        "long_decode": dict(H=64, Hkv=8, E=8192),
    }
    for name, kw in shapes.items():
        q, k = workload_lengths(name)
        kv, flops, pairs = bench.work_of(_Shape(q, k, **kw))
        if name == "chunked_prefill":
            assert pairs == 54_530_048          # sum over requests of visible causal pairs
            assert abs(flops / 1e12 - 0.8934) < 1e-4
        if name == "long_decode":
            assert kv == (1 << 20) * 8 * 128 * 2 * 2


class _FakeNvml:
    max_sm = 2070.0

    def __init__(self):
        self.calls = 0

    def sample(self):
        self.calls += 1
        return (1965.0 if self.calls % 2 else 2070.0), (["sw_power_cap"] if self.calls == 3 else [])


def test_clock_sampler_summarises_polled_samples():
    import time

    cs = bench.ClockSampler(0)
    cs.nvml = _FakeNvml()
    with cs:
        time.sleep(0.05)
    s = cs.summary()
    assert s["samples"] >= 3 and s["source"] == "nvml"
    assert s["sm_max_mhz"] == 2070.0 and s["sm_mhz"] in (1965.0, 2017.5, 2070.0)
    assert s["reasons"] == ["sw_power_cap"]


def test_cpu_baseline_splits_its_budget_between_decode_and_prefill():
    """The tiny mixed batch has decode-shaped and prefill-shaped requests: the oracle runs whole decode
    requests for half the budget and stratified prefill rows for the other half, and the line reports
    both rates and the step time they imply."""
    from workloads import workload

    r = bench.cpu_baseline("tiny_mix", 0.5)
    assert r["kind"] == "oracle" and r["cores"] >= 1 and r["seconds"] >= 0.5
    assert r["unit"].startswith("ms per step")
    assert r["decode_gbs"] > 0 and r["prefill_tflops"] > 0
    assert "whole decode requests" in r["sample"] and "stratified prefill rows" in r["sample"]
    kv, flops, _ = bench.work_of(workload("tiny_mix"))
    implied = (kv / (r["decode_gbs"] * 1e9) + flops / (r["prefill_tflops"] * 1e12)) * 1e3
    assert abs(implied - r["value"]) <= 0.01 * r["value"]

