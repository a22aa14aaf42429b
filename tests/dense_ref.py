"""Second, independent formulation of the attention for tiny inputs (NumPy, fp64).

Where the C oracle walks keys one by one through the page table, this module
first materialises each request's logical K/V by gathering whole pages, then
builds the full (H, Lq, Lk) score matrix, a boolean visibility matrix and a
bias matrix, and takes a log-sum-exp over keys.  It shares nothing with the
oracle but the definition it restates (score_mod_rel_bias and the wrapper of
fa4_rel_attention.py, nxmr.cn article) and is used only to pin the oracle.
"""
from __future__ import annotations

import numpy as np
import torch


def _f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def _i64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().to(torch.int64).numpy()
    return np.asarray(t, dtype=np.int64)


def dense_attention(q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q, *,
                    softmax_scale, causal=True, window_left=-1, window_right=-1, rel_extent=0,
                    rel_logits=None):
    """Returns (out (T, H, D), lse (T, H)) as float64 arrays."""
    Q = _f64(q)
    Kc = _f64(key_cache)
    Vc = _f64(value_cache)
    bt = _i64(block_table)
    seqk = _i64(cache_seqlens)
    cu = _i64(cu_seqlens_q)
    R = _f64(rel_logits) if rel_extent > 0 else None
    T, H, D = Q.shape
    _, BS, Hkv, _ = Kc.shape
    G = H // Hkv
    out = np.zeros((T, H, D))
    lse = np.full((T, H), -np.inf)
    for b in range(len(seqk)):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        Lq, Lk = t1 - t0, int(seqk[b])
        if Lq == 0:
            continue
        npg = -(-Lk // BS)
        pages = bt[b, :npg]
        K = Kc[pages].reshape(npg * BS, Hkv, D)[:Lk]          # logical keys
        V = Vc[pages].reshape(npg * BS, Hkv, D)[:Lk]
        K = np.repeat(K, G, axis=1)                           # (Lk, H, D)
        V = np.repeat(V, G, axis=1)
        qb = Q[t0:t1]                                         # (Lq, H, D)
        S = np.einsum("ihd,jhd->hij", qb, K) * softmax_scale  # (H, Lq, Lk)
        qpos = np.arange(Lq)[:, None] + (Lk - Lq)             # bottom-right alignment
        kpos = np.arange(Lk)[None, :]
        vis = np.ones((Lq, Lk), dtype=bool)
        if causal:
            vis &= kpos <= qpos
        if window_left >= 0:
            vis &= kpos >= qpos - window_left
        if window_right >= 0:
            vis &= kpos <= qpos + window_right
        if R is not None:
            rd = qpos - kpos                                  # (Lq, Lk)
            inside = (rd >= 0) & (rd < rel_extent)
            rdc = np.clip(rd, 0, rel_extent - 1)
            Rb = R[t0:t1]                                     # (Lq, H, E)
            bias = np.take_along_axis(Rb, np.broadcast_to(rdc[:, None, :], (Lq, H, Lk)), axis=2)
            bias = np.where(inside[:, None, :], bias, 0.0)    # (Lq, H, Lk)
            S = S + bias.transpose(1, 0, 2)
        S = np.where(vis[None], S, -np.inf)
        m = S.max(axis=2, keepdims=True)
        any_vis = vis.any(axis=1)                             # (Lq,)
        m_safe = np.where(np.isfinite(m), m, 0.0)
        P = np.exp(S - m_safe)
        l = P.sum(axis=2)                                     # (H, Lq)
        O = np.einsum("hij,jhd->ihd", P, V)                   # (Lq, H, D)
        with np.errstate(divide="ignore", invalid="ignore"):
            O = O / l.T[:, :, None]
            L = (m[:, :, 0] + np.log(l)).T                    # (Lq, H)
        O[~any_vis] = 0.0
        L[~any_vis] = -np.inf
        out[t0:t1] = O
        lse[t0:t1] = L
    return out, lse
