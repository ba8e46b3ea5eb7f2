"""fp64 masked attention with score_mods (oracle, test infrastructure).

FlexAttention Eq. 1 ("FlexAttention: A Programming Model for Generating
Optimized Attention Kernels", §3, summary page):

    O = softmax(mod(Q K^T / sqrt(d))) V,

where ``mod`` is pointwise.  Masking sets a score to -inf; the score_mods of
this library are a tanh softcap, cap * tanh(s / cap), followed by an ALiBi
bias slope_h * (k - q) (positions sample-local, head h of the Q heads).

The log-sum-exp of the row is LSE = ln sum_{visible k} exp(mod(s)).  A row
without any visible key has O = 0 and LSE = -inf ("Flex Attention Mask Plan
Design", §6.1).  Masked pairs contribute exactly zero, so the sums run over
the visible pairs only.

Inputs are the bf16 tensors both sides consume, upcast exactly to fp64.
"""
from __future__ import annotations

import numpy as np
import torch

from . import mask as M


def as_f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def attention_dense(q: np.ndarray, k: np.ndarray, v: np.ndarray, vis: np.ndarray,
                    q_pos: np.ndarray, scale: float, softcap: float = 0.0,
                    slope=None):
    """One (sample, head): q [n, d], k/v [m, d], vis bool [n, m], q_pos [n] local positions.

    Returns (O [n, d] float64, LSE [n] float64).
    """
    s = (q @ k.T) * scale
    if softcap and softcap > 0.0:
        s = softcap * np.tanh(s / softcap)
    if slope is not None:
        kpos = np.arange(k.shape[0], dtype=np.float64)
        s = s + float(slope) * (kpos[None, :] - np.asarray(q_pos, np.float64)[:, None])
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, initial=-np.inf)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    p = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 on masked pairs
    l = p.sum(axis=1)
    lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    o = (p @ v) / np.where(has, l, 1.0)[:, None]
    o[~has] = 0.0
    return o, lse


def head_slice(w, b: int, h: int):
    """fp64 (q [q_len, d], k [k_len, d], v [k_len, d]) of sample b, Q head h."""
    q_off, q_len, k_off, k_len = w.sample_bounds()[b]
    hk = h // (w.Hq // w.Hk)
    if w.layout == 0:
        q = w.q[b, :, h, :]
        k = w.k[b, :, hk, :]
        v = w.v[b, :, hk, :]
    else:
        q = w.q[q_off:q_off + q_len, h, :]
        k = w.k[k_off:k_off + k_len, hk, :]
        v = w.v[k_off:k_off + k_len, hk, :]
    return as_f64(q), as_f64(k), as_f64(v)


def attention_rows(w, b: int, h: int, q_local=None):
    """Oracle O/LSE for sample b, Q head h, at sample-local rows ``q_local`` (all if None)."""
    q, k, v = head_slice(w, b, h)
    if q_local is None:
        q_local = np.arange(q.shape[0])
    q_local = np.asarray(q_local, np.int64)
    hm = 0 if w.Hmask == 1 else h
    vis = M.visible_rows(w, hm, b, q_local)
    slope = None if w.alibi_slopes is None else float(w.alibi_slopes[h])
    return attention_dense(q[q_local], k, v, vis, q_local, w.scale, w.softcap, slope)


def attention_full(w):
    """Oracle over every row (small workloads only): O like w.q in float64, LSE [Hq, total_q]."""
    o = np.zeros(tuple(w.q.shape), np.float64)
    lse = np.full((w.Hq, w.total_q), -np.inf)
    for b, (q_off, q_len, k_off, k_len) in enumerate(w.sample_bounds()):
        for h in range(w.Hq):
            ob, lb = attention_rows(w, b, h)
            if w.layout == 0:
                o[b, :, h, :] = ob
            else:
                o[q_off:q_off + q_len, h, :] = ob
            lse[h, q_off:q_off + q_len] = lb
    return o, lse
