"""Mask semantics, written out as dense boolean matrices (oracle, test infrastructure).

Interval masks ("Flex Attention Mask Plan Design", §2 Public Mask
Representation): row q of ``mask_func[hm, :, q]`` holds nfunc (odd) endpoints
F0..F(n-1); the visible keys of that row are

    [0, F0) U [F1, F2) U [F3, F4) U ...

with sample-local key positions and the requirement
0 <= F0 <= F1 <= ... <= F(n-1) <= k_len of the row's sample (§2, §3.3).
Equal neighbours give an empty interval.

Block masks ("Decoupling Logical Masks from GPU Execution for Dynamic
Block-Sparse Attention", §2, definition of E(M)): a logical mask M over block
pairs of geometry (B_Q, B_KV) makes token pair (q, k) visible exactly when
M[q // B_Q, k // B_KV] is active, restricted to q < q_len and k < k_len.
"""
from __future__ import annotations

import numpy as np


class MaskError(ValueError):
    """Raised for endpoints or sequence prefixes that violate §2 / §3.2."""


def validate_endpoints(F: np.ndarray, k_len) -> None:
    """Check 0 <= F0 <= ... <= F(n-1) <= k_len for every row.

    ``F`` is ``[nfunc, rows]``; ``k_len`` is a scalar or per-row array.
    """
    F = np.asarray(F, dtype=np.int64)
    if F.shape[0] % 2 != 1:
        raise MaskError("nfunc must be odd")
    if np.any(F < 0):
        raise MaskError("negative endpoint")
    if F.shape[0] > 1 and np.any(np.diff(F, axis=0) < 0):
        raise MaskError("endpoints not ordered")
    if np.any(F[-1] > np.asarray(k_len)):
        raise MaskError("endpoint beyond sample k_len")


def validate_seqlens(cu_q, cu_k, total_q, total_k, max_q, max_k) -> None:
    """Prefix checks of "Flex Attention Mask Plan Design" §3.2."""
    cu_q = np.asarray(cu_q, np.int64)
    cu_k = np.asarray(cu_k, np.int64)
    if cu_q.shape != cu_k.shape or cu_q.ndim != 1 or cu_q.size < 2:
        raise MaskError("cu_seqlens shapes")
    if cu_q[0] != 0 or cu_k[0] != 0:
        raise MaskError("cu_seqlens must start at 0")
    if cu_q[-1] != total_q or cu_k[-1] != total_k:
        raise MaskError("cu_seqlens must end at the token totals")
    dq, dk = np.diff(cu_q), np.diff(cu_k)
    if np.any(dq < 0) or np.any(dk < 0):
        raise MaskError("cu_seqlens not monotone")
    if np.any(dq > max_q) or np.any(dk > max_k):
        raise MaskError("sample longer than max_seqlen")


def interval_visible(F: np.ndarray, k_len: int) -> np.ndarray:
    """Dense visibility of rows with endpoints ``F[nfunc, rows]``: bool [rows, k_len]."""
    F = np.asarray(F, dtype=np.int64)
    k = np.arange(k_len, dtype=np.int64)[None, :]
    vis = k < F[0][:, None]
    for i in range(1, F.shape[0], 2):
        vis |= (k >= F[i][:, None]) & (k < F[i + 1][:, None])
    return vis


def interval_visible_rows(w, hm: int, b: int, q_local: np.ndarray) -> np.ndarray:
    """Visibility of selected sample-local rows of sample b, mask head hm."""
    q_off, q_len, k_off, k_len = w.sample_bounds()[b]
    F = w.mask_func[hm][:, q_off + np.asarray(q_local)]
    return interval_visible(F, k_len)


def block_visible_rows(block_mask: np.ndarray, BQ: int, BKV: int, hm: int,
                       q_local: np.ndarray, k_len: int) -> np.ndarray:
    """E(M) rows: vis[r, k] = M[hm, q_r // BQ, k // BKV] for k < k_len."""
    qb = np.asarray(q_local, np.int64) // BQ
    kb = np.arange(k_len, dtype=np.int64) // BKV
    return block_mask[hm][np.ix_(qb, kb)].astype(bool)


def visible_rows(w, hm: int, b: int, q_local) -> np.ndarray:
    """Dense bool [len(q_local), k_len] for workload ``w`` (either mask kind)."""
    q_local = np.asarray(q_local, np.int64)
    _, q_len, _, k_len = w.sample_bounds()[b]
    if w.mask_kind == "intervals":
        return interval_visible_rows(w, hm, b, q_local)
    return block_visible_rows(w.block_mask, w.block_q, w.block_kv, hm, q_local, k_len)
