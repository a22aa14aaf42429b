"""One attention call (and a whole serving step) captured in a CUDA graph and replayed on new batches.

Everything the launches depend on is known on the host from the shapes and
bounds (T, B, H, Hkv, page pool, max_seqlen_q, num_splits, window, E): the
per-request work lists are built on the device by the prepass kernel.  So a
graph captured once serves every batch with the same shapes and bounds, even
when the mix of decode and prefill requests changes between replays.  Each
replay here is checked against the oracle on that replay's batch.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_causal_gb300 as ink
from workloads import build_case

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_RTOL = 1e-3

# Batches of one shape (B 4, T 120): decode-heavy, prefill-only, mixed, and one with empty requests.
BATCHES = [
    ([1, 1, 1, 117], [300, 40, 1000, 500]),
    ([40, 30, 20, 30], [40, 600, 20, 900]),
    ([1, 1, 117, 1], [1, 2000, 117, 60]),
    ([0, 120, 0, 0], [5, 1500, 0, 0]),
]
POOL = 160          # pages: enough for the largest batch above
WIDTH = 128         # block_table columns (2000 keys / 16)
MAX_Q = 120


@pytest.fixture(scope="module", autouse=True)
def _built():
    ink.build()
    ink.load()
    oracle.build()


def _case(i, *, H, Hkv, E, window, seed):
    q_lens, kv_lens = BATCHES[i]
    return build_case(f"graph-{i}", q_lens, kv_lens, H=H, Hkv=Hkv, E=E, window=window, seed=seed + i,
                      pool_pages=POOL, max_blocks_per_seq=WIDTH, max_seqlen_q=MAX_Q)


def _compare(out, lse, case, what):
    ref_out, ref_lse = oracle.attention(case.q, case.key_cache, case.value_cache, case.block_table,
                                        case.cache_seqlens, case.cu_seqlens_q, **case.oracle_kwargs())
    o = out.float().cpu().double().numpy().reshape(ref_out.shape)
    l = lse.cpu().double().numpy().reshape(ref_lse.shape)
    assert np.all(np.isfinite(o)), what
    err = np.max(np.abs(o - ref_out))
    assert err <= OUT_TOL, f"{what}: max |out - ref| = {err}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(l)), f"{what}: -inf rows differ"
    if fin.any():
        rel = np.abs(l[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))
        assert rel.max() <= LSE_RTOL, f"{what}: lse rel err {rel.max()}"


class _Static:
    """Device buffers a captured graph reads and writes; each batch is copied in before a replay."""

    def __init__(self, case):
        d = case.to("cuda")
        self.q, self.kc, self.vc = d.q.clone(), d.key_cache.clone(), d.value_cache.clone()
        self.bt, self.seqk, self.cu = d.block_table.clone(), d.cache_seqlens.clone(), d.cu_seqlens_q.clone()
        self.rel = None if d.rel_logits is None else d.rel_logits.clone()
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(case.T, case.H, dtype=torch.float32, device="cuda")

    def load(self, case):
        self.q.copy_(case.q)
        self.kc.copy_(case.key_cache)
        self.vc.copy_(case.value_cache)
        self.bt.copy_(case.block_table)
        self.seqk.copy_(case.cache_seqlens)
        self.cu.copy_(case.cu_seqlens_q)
        if self.rel is not None:
            self.rel.copy_(case.rel_logits)


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("H,Hkv,E,window,splits", [
    (16, 4, 64, (-1, -1), 0),
    (16, 4, 64, (-1, -1), 1),
    (32, 4, 200, (300, 0), 4),
    (8, 8, 0, (-1, -1), 0),
])
def test_one_graph_serves_every_batch_of_its_shape(H, Hkv, E, window, splits):
    cases = [_case(i, H=H, Hkv=Hkv, E=E, window=window, seed=700 + H + E) for i in range(len(BATCHES))]
    st = _Static(cases[0])
    c0 = cases[0]
    ws = torch.empty(ink.workspace_size(ink.Dims(c0.T, c0.B, H, Hkv, 128, POOL, 16, WIDTH), MAX_Q, splits),
                     dtype=torch.uint8, device="cuda")

    def run():
        ink.ink_rel_attn_varlen(st.q, st.kc, st.vc, block_table=st.bt, cache_seqlens=st.seqk,
                                cu_seqlens_q=st.cu, max_seqlen_q=MAX_Q, softmax_scale=c0.softmax_scale,
                                causal=True, window_left=window[0], window_right=window[1], rel_extent=E,
                                rel_logits=st.rel, num_splits=splits, out=st.out, lse=st.lse, workspace=ws)

    g = _capture(run)
    launches = ink.launch_count()
    for i in [1, 2, 3, 0, 2]:
        st.out.fill_(float("nan"))
        st.load(cases[i].to("cuda"))
        g.replay()
        torch.cuda.synchronize()
        _compare(st.out, st.lse, cases[i], f"replay of batch {i}")
        errs = ink.read_device_errors(ws)
        assert errs & ~ink.DEVERR["EMPTY_ROWS"] == 0, f"batch {i}: device errors {errs:#x}"
    # replays launch the captured kernels without calling the library again
    assert ink.launch_count() == launches


def test_error_word_is_rebuilt_on_every_replay():
    """A replay on a bad batch flags it; the next replay on a good batch clears the flag."""
    case = _case(1, H=16, Hkv=4, E=32, window=(-1, -1), seed=90)
    st = _Static(case)
    ws = torch.empty(ink.workspace_size(ink.Dims(case.T, case.B, 16, 4, 128, POOL, 16, WIDTH), MAX_Q, 0),
                     dtype=torch.uint8, device="cuda")

    def run():
        ink.ink_rel_attn_varlen(st.q, st.kc, st.vc, block_table=st.bt, cache_seqlens=st.seqk,
                                cu_seqlens_q=st.cu, max_seqlen_q=MAX_Q, softmax_scale=case.softmax_scale,
                                rel_extent=32, rel_logits=st.rel, out=st.out, lse=st.lse, workspace=ws)

    g = _capture(run)
    good = case.to("cuda")
    bad_cu = good.cu_seqlens_q.clone()
    bad_cu[2] = bad_cu[1] - 1                      # cu_seqlens_q decreasing: the request is skipped
    st.load(good)
    st.cu.copy_(bad_cu)
    g.replay()
    assert ink.read_device_errors(ws) & ink.DEVERR["CU_SEQLENS"]
    st.load(good)
    g.replay()
    assert ink.read_device_errors(ws) & ~ink.DEVERR["EMPTY_ROWS"] == 0
    _compare(st.out, st.lse, case, "good replay after a bad one")


def test_graph_of_a_whole_serving_step():
    """KV append and attention captured together; each replay appends its own new tokens."""
    cases = [_case(i, H=16, Hkv=4, E=48, window=(-1, -1), seed=40) for i in range(3)]
    c0 = cases[0]
    st = _Static(c0)
    T = c0.T
    key = torch.empty(T, 4, 128, dtype=torch.bfloat16, device="cuda")
    value = torch.empty_like(key)
    slots = torch.empty(T, dtype=torch.int64, device="cuda")
    ws = torch.empty(ink.workspace_size(ink.Dims(T, c0.B, 16, 4, 128, POOL, 16, WIDTH), MAX_Q, 0),
                     dtype=torch.uint8, device="cuda")

    def step():
        ink.reshape_and_cache(key, value, st.kc, st.vc, slots)
        ink.ink_rel_attn_varlen(st.q, st.kc, st.vc, block_table=st.bt, cache_seqlens=st.seqk,
                                cu_seqlens_q=st.cu, max_seqlen_q=MAX_Q, softmax_scale=c0.softmax_scale,
                                rel_extent=48, rel_logits=st.rel, out=st.out, lse=st.lse, workspace=ws)

    slots.fill_(-1)                                # the warm-up and capture runs append nothing
    g = _capture(step)
    for i, case in enumerate(cases):
        gen = torch.Generator().manual_seed(500 + i)
        new_k = torch.randn(T, 4, 128, generator=gen).to(torch.bfloat16)
        new_v = torch.randn(T, 4, 128, generator=gen).to(torch.bfloat16)
        sm = torch.tensor(oracle.slot_mapping(case.block_table.tolist(), case.kv_lens, case.q_lens, case.BS),
                          dtype=torch.int64)
        want_k, want_v = oracle.reshape_and_cache(new_k, new_v, case.key_cache, case.value_cache, sm)
        st.load(case.to("cuda"))
        key.copy_(new_k)
        value.copy_(new_v)
        slots.copy_(sm)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(st.kc.cpu().view(torch.int16).numpy().view(np.uint16), want_k)
        assert np.array_equal(st.vc.cpu().view(torch.int16).numpy().view(np.uint16), want_v)
        after = case.to("cpu")
        after.key_cache = torch.from_numpy(want_k.view(np.int16)).view(torch.bfloat16)
        after.value_cache = torch.from_numpy(want_v.view(np.int16)).view(torch.bfloat16)
        _compare(st.out, st.lse, after, f"step {i}")


def test_graph_of_an_fp8_serving_step():
    """E4M3 cache: quantizing KV append and decode-shaped attention captured together, replayed on batches
    with different mixes of 1- to 4-token requests (T = 8, G = 4)."""
    from workloads import fp8_kv

    batches = [([1, 1, 2, 4], [300, 17, 900, 64]), ([2, 2, 2, 2], [40, 40, 2000, 5]),
               ([4, 4, 0, 0], [1000, 4, 0, 0]), ([1, 3, 4, 0], [1, 700, 33, 0])]
    ks, vs = 0.07, 0.05
    cases = [build_case(f"fp8-graph-{i}", q, k, H=16, Hkv=4, E=40, seed=60 + i, pool_pages=POOL,
                        max_blocks_per_seq=WIDTH, max_seqlen_q=4) for i, (q, k) in enumerate(batches)]
    c0 = cases[0]
    T = c0.T
    q = c0.q.cuda().clone()
    bt, seqk, cu = c0.block_table.cuda().clone(), c0.cache_seqlens.cuda().clone(), c0.cu_seqlens_q.cuda().clone()
    rel = c0.rel_logits.cuda().clone()
    k8, v8 = (x.cuda() for x in fp8_kv(c0, ks, vs))
    key = torch.empty(T, 4, 128, dtype=torch.bfloat16, device="cuda")
    value = torch.empty_like(key)
    slots = torch.full((T,), -1, dtype=torch.int64, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(T, 16, dtype=torch.float32, device="cuda")
    ws = torch.empty(ink.workspace_size(ink.Dims(T, c0.B, 16, 4, 128, POOL, 16, WIDTH), 4, 0), dtype=torch.uint8,
                     device="cuda")

    def step():
        ink.reshape_and_cache_fp8(key, value, k8, v8, slots, k_scale=ks, v_scale=vs)
        ink.ink_rel_attn_varlen_fp8kv(q, k8, v8, k_scale=ks, v_scale=vs, block_table=bt, cache_seqlens=seqk,
                                      cu_seqlens_q=cu, max_seqlen_q=4, softmax_scale=c0.softmax_scale,
                                      rel_extent=40, rel_logits=rel, out=out, lse=lse, workspace=ws)

    g = _capture(step)
    for i, case in enumerate(cases):
        gen = torch.Generator().manual_seed(900 + i)
        new_k = torch.randn(T, 4, 128, generator=gen).to(torch.bfloat16)
        new_v = torch.randn(T, 4, 128, generator=gen).to(torch.bfloat16)
        sm = torch.tensor(oracle.slot_mapping(case.block_table.tolist(), case.kv_lens, case.q_lens, case.BS),
                          dtype=torch.int64)
        c8k, c8v = fp8_kv(case, ks, vs)
        want_k, want_v = oracle.reshape_and_cache_fp8(new_k, new_v, c8k, c8v, sm, ks, vs)
        ref_out, ref_lse = oracle.attention_fp8kv(case.q, want_k, want_v, case.block_table, case.cache_seqlens,
                                                  case.cu_seqlens_q, k_scale=ks, v_scale=vs,
                                                  **case.oracle_kwargs())
        q.copy_(case.q)
        bt.copy_(case.block_table)
        seqk.copy_(case.cache_seqlens)
        cu.copy_(case.cu_seqlens_q)
        rel.copy_(case.rel_logits)
        k8.copy_(c8k)
        v8.copy_(c8v)
        key.copy_(new_k)
        value.copy_(new_v)
        slots.copy_(sm)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(k8.cpu().numpy(), want_k) and np.array_equal(v8.cpu().numpy(), want_v)
        o = out.float().cpu().double().numpy().reshape(ref_out.shape)
        assert np.max(np.abs(o - ref_out)) <= OUT_TOL, f"step {i}"
        fin = np.isfinite(ref_lse)
        l = lse.cpu().double().numpy().reshape(ref_lse.shape)
        assert np.array_equal(fin, np.isfinite(l))
        assert (np.abs(l[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))).max() <= LSE_RTOL
