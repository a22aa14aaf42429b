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
    """Split-KV cap of the article's ``inkling_fa4_num_splits``, restated from its prose.

    nxmr.cn article, layer 1, the five steps that explain the function:
      1. Hopper (capability 9) and local (windowed) attention take no split.
      2. A KV head serves a group of max_query_len * (Hq / Hkv) query rows,
         cut into tiles of 256 rows; one split of the whole batch launches
         batch * Hkv * tiles CTAs.
      3. The CTA count wanted: a lone one-tile request (long decode) 256, a
         batch of one-tile requests 128, multi-tile prefill 64.
      4. A hard cap, tuned only for the lone one-tile request (below); 128
         otherwise.
      5. The wanted CTAs over the CTAs of one split, limited by the cap and by
         one split per 128 keys, and at least 1.
    The page lost its comparison operators (reading R6): the caps of step 4
    are taken as the first rule that holds in the order the article lists
    them, with the comparisons that keep the cap monotone (more KV heads per
    rank, fewer splits).  This is the page's heuristic, kept as a pinned
    reference function; the library's own split choice is derived for the
    GB300 SM count.  Pinned by the five workload shapes (3, 1, 1, 16, 1).
    """
    if capability_major == 9 or is_local:  # step 1
        return 1
    rows_per_group = max_query_len * (num_heads // num_kv_heads)  # step 2
    tiles = -(-rows_per_group // 256)
    ctas_per_split = batch_size * num_kv_heads * tiles
    lone_decode = tiles == 1 and batch_size == 1
    if lone_decode:  # step 3
        ctas_wanted = 256
    else:
        ctas_wanted = 128 if tiles == 1 else 64
    cap = 128  # step 4
    if lone_decode:
        rules = (
            (num_kv_heads >= 8, 16),
            (num_kv_heads >= 4 or max_kv_len <= 8192, 32),
            (max_kv_len <= 65536, 64),
            (True, 128),
        )
        cap = next(c for holds, c in rules if holds)
    per_key_limit = -(-max_kv_len // 128)  # step 5
    return max(1, min(ctas_wanted // ctas_per_split, cap, per_key_limit))


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
