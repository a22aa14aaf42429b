"""Scheduling and indexing helpers of the oracle, restated from the pages.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Each function says
which passage it follows and what pins it.
"""
from __future__ import annotations

from typing import Sequence


def bucket_max_seqlen_q(max_seqlen_q: int) -> int:
    """Round the scheduling bound on query length up to a power of two.

    ``bucket_max_seqlen_q`` in fa4_rel_attention.py (nxmr.cn article, layer 1
    of its walk-through): one shifted left by the
    bit length of max(0, n - 1).  The article's example maps 45000 to 65536.
    Pinned by that example and by the closed form at 0, 1 and powers of two.
    """
    return 1 << max(0, int(max_seqlen_q) - 1).bit_length()


def page_num_splits(*, is_local: bool, batch_size: int, max_query_len: int, num_heads: int,
                    num_kv_heads: int, max_kv_len: int, capability_major: int = 10) -> int:
    """Split-KV count of ``inkling_fa4_num_splits`` as the article prints it.

    nxmr.cn article, layer 1 steps 1-5.  The page
    lost its comparison operators; the reading taken is the one that keeps
    the cap monotone in the number of KV heads per rank:
      major 9 -> 1; local attention -> 1;
      q_tiles = ceil(max_query_len * G / 256), base = batch * Hkv * q_tiles;
      target = 256 (one q tile, batch 1), 128 (one q tile), else 64;
      cap = 128, and for one q tile at batch 1:
        16 if Hkv >= 8, elif Hkv >= 4 or max_kv <= 8192: 32,
        elif max_kv <= 65536: 64, else 128;
      result = max(1, min(target // base, cap, ceil(max_kv / 128))).
    This is the page's Hopper/Blackwell-FA4 heuristic, kept as a pinned
    reference function; the library's own split choice is derived for the
    GB300 SM count.  Pinned by the five workload shapes (3, 1, 1, 16, 1).
    """
    if capability_major == 9:
        return 1
    if is_local:
        return 1
    q_rows = max_query_len * (num_heads // num_kv_heads)
    q_tiles = (q_rows + 255) // 256
    base_ctas = batch_size * num_kv_heads * q_tiles
    if q_tiles == 1 and batch_size == 1:
        target_ctas = 256
    elif q_tiles == 1:
        target_ctas = 128
    else:
        target_ctas = 64
    max_splits = 128
    if q_tiles == 1 and batch_size == 1:
        if num_kv_heads >= 8:
            max_splits = 16
        elif num_kv_heads >= 4 or max_kv_len <= 8192:
            max_splits = 32
        elif max_kv_len <= 65536:
            max_splits = 64
        else:
            max_splits = 128
    return max(1, min(target_ctas // base_ctas, max_splits, (max_kv_len + 127) // 128))


def cu_seqlens_from_lengths(lengths: Sequence[int]) -> list[int]:
    """Exclusive prefix sum with a leading zero: request i owns tokens
    [cu[i], cu[i+1]).  Mini-vllm tutorial step 15 (varlen section) and the
    vLLM FlashAttention metadata builder on the vLLM V1 attention page.
    Pinned by the printed examples [47,312,128] -> [0,47,359,487] and
    [10,20,5] -> [0,10,30,35].
    """
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out


def page_index_csr(block_table: Sequence[Sequence[int]], seq_lens: Sequence[int],
                   block_size: int, *, count: str = "valid"):
    """FlashInfer-style CSR page index (indptr, indices, last_page_len).

    vLLM V1 attention page, FlashInfer metadata section and appendix U.1.
    ``count="valid"`` takes every non-negative entry of a row (the page's
    first example, whose third request lists 3 pages); ``count="ceil"`` takes
    the first ceil(seq_len / block_size) entries (appendix U.1's corrected
    table).  last_page_len = seq_len mod block_size, or block_size when that
    is zero.  Pinned by both printed examples.
    """
    indptr = [0]
    indices: list[int] = []
    last = []
    for row, n in zip(block_table, seq_lens):
        if count == "valid":
            pages = [int(p) for p in row if int(p) >= 0]
        elif count == "ceil":
            pages = [int(p) for p in row[: (int(n) + block_size - 1) // block_size]]
        else:
            raise ValueError(count)
        indices.extend(pages)
        indptr.append(len(indices))
        r = int(n) % block_size
        last.append(r if r != 0 else block_size)
    return indptr, indices, last


def slot_mapping(block_table: Sequence[Sequence[int]], seq_lens: Sequence[int],
                 query_lens: Sequence[int], block_size: int) -> list[int]:
    """Cache slot of every new token: the KV write that precedes attention.

    vLLM V1 attention page, metadata builder step 2: for request i with
    start = seq_len - query_len, token j goes to
    block_table[i][(start + j) // bs] * bs + (start + j) % bs.
    Pinned by brute force against a dense logical->physical map in the tests.
    """
    out = []
    for row, n, ql in zip(block_table, seq_lens, query_lens):
        start = int(n) - int(ql)
        for j in range(int(ql)):
            pos = start + j
            out.append(int(row[pos // block_size]) * block_size + pos % block_size)
    return out
