"""fp64 decoding attention over a paged KV cache (oracle, test infrastructure).

Decoding ("FlexAttention: A Programming Model for Generating Optimized
Attention Kernels", summary page, §3.4 Modification Conversion for
Inference): the query rows are the newest tokens of each sequence, at
absolute position offset + q_idx, and the mask and score_mod are evaluated
there (mask(b, h, q_idx + offset, kv_idx); an ALiBi score_mod adds
slope_h * (kv_idx - (q_idx + offset)); the tanh softcap does not depend on
positions).  Here offset = k_len - q_len:
the new tokens' keys are already in the cache.  The interval endpoints of
a decode row are given at its absolute position (``DecodeWorkload.mask_func``),
so the visible keys are [0, F0) U [F1, F2) U ... over the logical keys
0..k_len-1, exactly as for a training row ("Flex Attention Mask Plan
Design", §2).

Paging (same page, §3.4 Paged Attention Integration): logical key j of
sequence b is stored at physical page page_table[b][j // page_size], row
j % page_size.  The oracle gathers the logical K and V of each sequence
through that definition and then computes Eq. 1 with ``attention_dense``:
paging relocates keys, it does not change which are visible.
"""
from __future__ import annotations

import numpy as np
import torch

from . import attention as A
from . import mask as M


def gather_logical(cache: torch.Tensor, table_row: np.ndarray, k_len: int, page_size: int) -> np.ndarray:
    """Logical rows [k_len, H, d] (fp64) of one sequence from a paged cache [pages, page_size, H, d]."""
    j = np.arange(int(k_len), dtype=np.int64)
    pages = np.asarray(table_row, np.int64)[j // page_size]
    rows = cache[torch.from_numpy(pages), torch.from_numpy(j % page_size)]
    return A.as_f64(rows)


def _rows(w, b: int, h: int, k: np.ndarray, v: np.ndarray):
    """O [q_len, d], LSE [q_len] of sequence b, Q head h, from its logical
    K/V [k_len, Hk, d].  Mask head: 0 for a mask shared by the heads, else h."""
    k_len = int(w.k_lens[b])
    hk = h // (w.Hq // w.Hk)
    hm = 0 if w.mask_func.shape[0] == 1 else h
    rows = np.arange(b * w.q_len, (b + 1) * w.q_len)
    q = A.as_f64(w.q[torch.from_numpy(rows), h])
    vis = M.interval_visible(w.mask_func[hm][:, rows], k_len)
    # absolute positions: the score_mod converted for inference sees q_idx + offset
    q_abs = (k_len - w.q_len) + np.arange(w.q_len)
    slope = None if w.alibi_slopes is None else float(w.alibi_slopes[h])
    return A.attention_dense(q, k[:, hk], v[:, hk], vis, q_abs, w.scale, softcap=w.softcap, slope=slope)


def decode_rows(w, b: int, h: int):
    """O [q_len, d] and LSE [q_len] (fp64) of the query rows of sequence b, Q head h."""
    k_len = int(w.k_lens[b])
    k = gather_logical(w.k_cache, w.page_table[b], k_len, w.page_size)
    v = gather_logical(w.v_cache, w.page_table[b], k_len, w.page_size)
    return _rows(w, b, h, k, v)


def decode_sequence(w, b: int, heads=None):
    """{h: (O [q_len, d], LSE [q_len])} of sequence b for the given Q heads (all by default)."""
    k_len = int(w.k_lens[b])
    k = gather_logical(w.k_cache, w.page_table[b], k_len, w.page_size)
    v = gather_logical(w.v_cache, w.page_table[b], k_len, w.page_size)
    return {h: _rows(w, b, h, k, v) for h in (range(w.Hq) if heads is None else heads)}


def decode_full(w):
    """O [B*q_len, Hq, d] and LSE [Hq, B*q_len] (fp64) of every query row."""
    o = np.zeros((w.B * w.q_len, w.Hq, w.d))
    lse = np.full((w.Hq, w.B * w.q_len), -np.inf)
    for b in range(w.B):
        for h, (ob, lb) in decode_sequence(w, b).items():
            o[b * w.q_len:(b + 1) * w.q_len, h] = ob
            lse[h, b * w.q_len:(b + 1) * w.q_len] = lb
    return o, lse
