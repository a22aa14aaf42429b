"""Seeded synthetic inputs for paged varlen attention.

This module is the one piece shared by the oracle tests, the CUDA parity
tests and the benchmark.  It holds none of the method's arithmetic: it draws
lengths, a random physical page assignment and normally distributed tensors,
and lays them out in the shapes the pages use (q (T, H, D); K/V caches
(num_blocks, block_size, Hkv, D); block_table (B, max_blocks_per_seq) padded
with -1; cache_seqlens including this step's query tokens; cu_seqlens_q with
a leading 0; rel_logits (T, H, rel_extent)).

Recipe (same for every workload):
  * lengths are drawn on the CPU from torch.Generator(seed);
  * the page pool holds sum(ceil(Lk/bs)) pages plus `spare_frac` unreferenced
    pages (or a fixed pool size); one torch.randperm(pool) is cut into
    consecutive runs, one run per request;
  * q/K/V are N(0, 1) fp32 draws rounded to bf16 (round to nearest even,
    torch's conversion); rel_logits is N(0, bias_std) fp32;
  * large tensors are drawn in chunks from a generator on `device`
    (seed + 1), so a case drawn on the GPU differs from the CPU draw with the
    same seed; within one run both sides always see the same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

CHUNK = 1 << 26  # elements per random draw


@dataclass
class Case:
    name: str
    H: int
    Hkv: int
    D: int
    BS: int
    E: int
    causal: bool
    window_left: int
    window_right: int
    softmax_scale: float
    q_lens: list
    kv_lens: list
    q: torch.Tensor
    key_cache: torch.Tensor
    value_cache: torch.Tensor
    block_table: torch.Tensor
    cache_seqlens: torch.Tensor
    cu_seqlens_q: torch.Tensor
    rel_logits: Optional[torch.Tensor]
    max_seqlen_q: int
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def B(self) -> int:
        return len(self.q_lens)

    @property
    def num_blocks(self) -> int:
        return int(self.key_cache.shape[0])

    def to(self, device) -> "Case":
        """Copy of the case with every tensor on `device`."""
        mv = lambda t: None if t is None else t.to(device)
        return Case(self.name, self.H, self.Hkv, self.D, self.BS, self.E, self.causal,
                    self.window_left, self.window_right, self.softmax_scale,
                    list(self.q_lens), list(self.kv_lens), mv(self.q), mv(self.key_cache),
                    mv(self.value_cache), mv(self.block_table), mv(self.cache_seqlens),
                    mv(self.cu_seqlens_q), mv(self.rel_logits), self.max_seqlen_q, dict(self.meta))

    def oracle_kwargs(self) -> dict:
        return dict(softmax_scale=self.softmax_scale, causal=self.causal,
                    window_left=self.window_left, window_right=self.window_right,
                    rel_extent=self.E, rel_logits=self.rel_logits)


def _normal(shape, gen, device, std=1.0, dtype=torch.float32) -> torch.Tensor:
    n = math.prod(shape)
    out = torch.empty(n, dtype=dtype, device=device)
    for s in range(0, n, CHUNK):
        e = min(n, s + CHUNK)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[s:e] = x.to(dtype)
    return out.view(*shape)


def build_case(name: str, q_lens: Sequence[int], kv_lens: Sequence[int], *, H: int, Hkv: int,
               D: int = 128, BS: int = 16, E: int = 0, bias_std: float = 1.0, causal: bool = True,
               window=(-1, -1), seed: int = 0, pool_pages: Optional[int] = None,
               spare_frac: float = 0.05, max_blocks_per_seq: Optional[int] = None,
               softmax_scale: Optional[float] = None, device="cpu", pad_value: int = -1,
               max_seqlen_q: Optional[int] = None) -> Case:
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    if len(q_lens) != len(kv_lens):
        raise ValueError("q_lens and kv_lens differ in length")
    B = len(q_lens)
    T = sum(q_lens)
    cpu = torch.Generator().manual_seed(seed)
    pages_per = [(k + BS - 1) // BS for k in kv_lens]
    used = sum(pages_per)
    if pool_pages is None:
        pool_pages = used + int(math.ceil(spare_frac * used))
    if pool_pages < used:
        raise ValueError("page pool smaller than the pages the requests need")
    width = max([1] + pages_per) if max_blocks_per_seq is None else int(max_blocks_per_seq)
    perm = torch.randperm(pool_pages, generator=cpu).to(torch.int32)
    bt = torch.full((B, width), pad_value, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[off:off + n]
        off += n
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    seqk = torch.tensor(kv_lens, dtype=torch.int32)

    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed + 1)
    q = _normal((T, H, D), gen, dev, dtype=torch.bfloat16)
    kc = _normal((pool_pages, BS, Hkv, D), gen, dev, dtype=torch.bfloat16)
    vc = _normal((pool_pages, BS, Hkv, D), gen, dev, dtype=torch.bfloat16)
    rel = _normal((T, H, E), gen, dev, std=bias_std) if E > 0 else None
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    msq = max([1] + q_lens) if max_seqlen_q is None else int(max_seqlen_q)
    return Case(name, H, Hkv, D, BS, E, causal, int(window[0]), int(window[1]), scale,
                q_lens, kv_lens, q, kc, vc, bt.to(dev), seqk.to(dev), cu.to(dev), rel, msq,
                {"seed": seed, "pool_pages": pool_pages, "used_pages": used})


# --- the five workloads -----------------------------------------------------

WORKLOADS = {
    "tiny_mix": "3 requests (decode Lk 47, decode Lk 312, prefill 128/128), H 8, Hkv 2, E 64, 64-page pool",
    "decode_batch": "64 decodes, Lk ~ U{1024..32768}, H 32, Hkv 8, E 1024",
    "chunked_prefill": "4 x Lq 2048 on prior KV 0/2048/6144/14336, H 32, Hkv 8, E 4096, bias N(0, 0.5)",
    "long_decode": "1 decode, Lk 1,048,576, H 64, Hkv 8, E 8192",
    "continuous_batch": "128 decodes (Lk log-uniform 64..65536) + 8 prefills (Lq = Lk ~ U{128..4096}), "
                        "H 32, Hkv 4, window (4095, 0), E 2048",
}
WORKLOAD_ORDER = list(WORKLOADS)

# Reduced variants for profiler captures (a few GB on the device, still larger than L2).
PROFILE_WORKLOADS = {
    "decode_batch_quarter": "first 16 requests of decode_batch (same lengths, pool and head shapes)",
    "chunked_prefill_quarter": "one request of chunked_prefill: Lq 2048 on prior KV 6144, H 32, Hkv 8, E 4096",
}


# Head sizes 64 and 256 (the other sizes a paged backend serves): the decode batch's and the chunked
# prefill's request lengths, at D = 64 with H 32, Hkv 8 and at D = 256 with H 24, Hkv 4 (G 6, the
# PagedAttention V2 page's GQA example); seeds 1101 .. 1104.
HEADDIM_WORKLOADS = {
    "decode_batch_d64": "decode_batch lengths (64 decodes, Lk ~ U{1024..32768}), H 32, Hkv 8, D 64, E 1024",
    "chunked_prefill_d64": "chunked_prefill lengths (4 x Lq 2048 on 0/2048/6144/14336), H 32, Hkv 8, D 64, E 4096",
    "decode_batch_d256": "decode_batch lengths (64 decodes, Lk ~ U{1024..32768}), H 24, Hkv 4, D 256, E 1024",
    "chunked_prefill_d256": "chunked_prefill lengths (4 x Lq 2048 on 0/2048/6144/14336), H 24, Hkv 4, D 256, E 4096",
}


def workload_lengths(name: str):
    """(q_lens, kv_lens) of a named workload, drawn from seed 1000 + index."""
    idx = WORKLOAD_ORDER.index(name)
    g = torch.Generator().manual_seed(1000 + idx)
    if name == "tiny_mix":
        return [1, 1, 128], [47, 312, 128]
    if name == "decode_batch":
        kv = torch.randint(1024, 32768 + 1, (64,), generator=g).tolist()
        return [1] * 64, kv
    if name == "chunked_prefill":
        prior = [0, 2048, 6144, 14336]
        return [2048] * 4, [p + 2048 for p in prior]
    if name == "long_decode":
        return [1], [1 << 20]
    if name == "continuous_batch":
        u = torch.rand(128, generator=g, dtype=torch.float64)
        dec = torch.floor(torch.exp(math.log(64) + u * (math.log(65536) - math.log(64)))).long()
        dec = dec.clamp(64, 65536).tolist()
        pre = torch.randint(128, 4096 + 1, (8,), generator=g).tolist()
        return [1] * 128 + pre, dec + pre
    raise KeyError(name)


def workload(name: str, device="cpu", **overrides) -> Case:
    """Build a named workload with its recipe (seed 1000 + index)."""
    if name == "decode_batch_quarter":
        q, k = workload_lengths("decode_batch")
        return build_case(name, q[:16], k[:16], H=32, Hkv=8, E=1024, seed=1001, device=device, **overrides)
    if name == "chunked_prefill_quarter":
        return build_case(name, [2048], [8192], H=32, Hkv=8, E=4096, bias_std=0.5, seed=1002, device=device,
                          **overrides)
    if name in HEADDIM_WORKLOADS:
        base, d = name.rsplit("_d", 1)
        D = int(d)
        q, k = workload_lengths(base)
        heads = dict(H=32, Hkv=8) if D == 64 else dict(H=24, Hkv=4)
        extra = dict(E=1024) if base == "decode_batch" else dict(E=4096, bias_std=0.5)
        seed = 1100 + list(HEADDIM_WORKLOADS).index(name) + 1
        return build_case(name, q, k, D=D, seed=seed, device=device, **heads, **extra, **overrides)
    idx = WORKLOAD_ORDER.index(name)
    q_lens, kv_lens = workload_lengths(name)
    kw = dict(seed=1000 + idx, device=device)
    if name == "tiny_mix":
        kw.update(H=8, Hkv=2, E=64, pool_pages=64)
    elif name == "decode_batch":
        kw.update(H=32, Hkv=8, E=1024)
    elif name == "chunked_prefill":
        kw.update(H=32, Hkv=8, E=4096, bias_std=0.5)
    elif name == "long_decode":
        kw.update(H=64, Hkv=8, E=8192)
    elif name == "continuous_batch":
        kw.update(H=32, Hkv=4, E=2048, window=(4095, 0))
    kw.update(overrides)
    return build_case(name, q_lens, kv_lens, **kw)


def random_case(seed: int, *, B: Optional[int] = None, device="cpu", D: int = 128, BS: Optional[int] = None,
                max_q: int = 40, max_kv_extra: int = 80, **over) -> Case:
    """Small random case (mixed decode / prefill, random window and bias)."""
    g = torch.Generator().manual_seed(10_000 + seed)
    ri = lambda lo, hi: int(torch.randint(lo, hi + 1, (1,), generator=g))
    B = ri(1, 4) if B is None else B
    Hkv = [1, 2, 4][ri(0, 2)]
    G = [1, 2, 4, 8][ri(0, 3)]
    BS = [1, 4, 16][ri(0, 2)] if BS is None else BS
    q_lens, kv_lens = [], []
    for _ in range(B):
        lq = 1 if ri(0, 1) == 0 else ri(0, max_q)
        lk = lq + ri(0, max_kv_extra)
        q_lens.append(lq)
        kv_lens.append(lk)
    E = [0, 1, 5, 64][ri(0, 3)]
    wl = [-1, -1, 0, 3, 17][ri(0, 4)]
    wr = [-1, -1, 0, 2][ri(0, 3)]
    causal = ri(0, 3) != 0
    kw = dict(H=Hkv * G, Hkv=Hkv, D=D, BS=BS, E=E, causal=causal, window=(wl, wr), seed=seed,
              device=device)
    kw.update(over)
    return build_case(f"random{seed}", q_lens, kv_lens, **kw)


def fp8_kv(case: Case, k_scale: float, v_scale: float):
    """E4M3 bytes for an FP8 KV cache holding about the case's bf16 K and V: each element divided by its
    tensor's scale and rounded to E4M3 (torch's float8_e4m3fn cast; values clamped to the format's 448).
    Returns (key_cache, value_cache) as uint8 tensors of the case's cache shape on its device."""
    def q8(x, s):
        return (x.float() / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return q8(case.key_cache, k_scale), q8(case.value_cache, v_scale)
