"""Backward views of a MaskPlan and fp64 attention gradients (oracle, test
infrastructure).

"Flex Attention Mask Plan Design":

* §4.4 / §4.7 K2Q view: for every K plan row (mask head, sample, K tile)
  two independent ascending CSR lists of the sample-local Q tiles whose tile
  pair is partial, respectively full.  It is the sparse transpose of the
  Q2K classification (§9 invariant 7: both views describe the same block
  relation); here the backward consumer uses the forward's tile geometry, so
  the classes are those of the same tiles.  K plan rows are compacted per
  sample like the Q rows (§4.2: ceil(k_len / T_KV) rows per sample, prefix
  ``cu_k_rows``).
* The K2Q payload follows the K-major consumer's accumulator ownership (one
  TMEM lane = one key): k2q_payload[e, c, w] bit l = element (query row
  32w + l, key column c) of the tile is visible; out-of-sample bits are 0.
* dq_write_order / dq_write_order_full (§4.7), parallel to the K2Q partial
  and full lists: the rank of the entry's K tile among all non-empty K
  tiles of its Q tile in ascending K order, i.e. a legal order of the dQ
  contributions of that Q tile.  (The page fixes only that the ranks define
  a legal accumulation order; ascending K order is the plainest one.)
* §4.5 header with backward fields: {fwd Q rows, fwd partial nnz, fwd full
  nnz, bwd Q rows, bwd K rows, bwd partial nnz, bwd full nnz, error}.  The
  dQ consumer reads the forward Q2K view (same geometry), so bwd Q rows is
  the forward row count.

Gradients: FlexAttention Eq. 1 differentiated by hand.  With S = scale Q K^T,
Z = mod(S) (tanh softcap then ALiBi), P = softmax over the visible keys and
O = P V:  dV = P^T dO,  dP = dO V^T,  dZ = P * (dP - rowsum(dO * O)),
dS = dZ * (1 - tanh^2(S / cap)) (1 without softcap),  dQ = scale dS K,
dK = scale dS^T Q.  Masked pairs have P = 0 and contribute nothing; a row
without visible keys has zero gradient.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import mask as M
from .attention import as_f64, head_slice


@dataclasses.dataclass
class BackwardView:
    T_Q: int
    T_KV: int
    Hmask: int
    k_rows: int                     # valid K plan rows over all samples
    cu_k_rows: np.ndarray           # int64 [B+1]
    krow_batch: np.ndarray          # int64 [k_rows]
    krow_nblock: np.ndarray         # int64 [k_rows]: sample-local K tile of the row
    partial_offset: np.ndarray      # int64 [Hmask*k_rows + 1]
    full_offset: np.ndarray         # int64 [Hmask*k_rows + 1]
    partial_idx: np.ndarray         # int64 [P]: sample-local Q tiles, ascending per row
    full_idx: np.ndarray            # int64 [F]
    payload: np.ndarray             # uint32 [P, T_KV, ceil(T_Q/32)]
    dq_write_order: np.ndarray      # int64 [P]
    dq_write_order_full: np.ndarray  # int64 [F]
    fwd_rows: int

    @property
    def header(self):
        return [self.k_rows, int(self.partial_idx.size), int(self.full_idx.size)]


def _tile_classes(vis: np.ndarray, T_Q: int, T_KV: int, nq: int, nk: int):
    """Dense visibility [q_len, k_len] -> (tiles bool [nq, T_Q, nk, T_KV], class [nq, nk])
    with class 0 empty, 1 partial, 2 full."""
    q_len, k_len = vis.shape
    d = np.zeros((nq * T_Q, nk * T_KV), dtype=bool)
    d[:q_len, :k_len] = vis
    tiles = d.reshape(nq, T_Q, nk, T_KV)
    anyv = tiles.any(axis=(1, 3))
    allv = tiles.all(axis=(1, 3))
    cls = np.where(allv, 2, np.where(anyv, 1, 0))
    return tiles, cls


def build_backward_view(w, T_Q: int = 128, T_KV: int = 128) -> BackwardView:
    """K2Q view, its payload and the dQ write order, by dense expansion of the mask."""
    bounds = w.sample_bounds()
    B = len(bounds)
    k_rows_b = np.array([-(-kl // T_KV) for (_, _, _, kl) in bounds], dtype=np.int64)
    q_rows_b = np.array([-(-ql // T_Q) for (_, ql, _, _) in bounds], dtype=np.int64)
    cu_k_rows = np.concatenate([[0], np.cumsum(k_rows_b)]).astype(np.int64)
    k_rows = int(cu_k_rows[-1])
    krow_batch = np.repeat(np.arange(B), k_rows_b)
    krow_nblock = np.concatenate([np.arange(n) for n in k_rows_b]) if k_rows else np.zeros(0, np.int64)
    nw = -(-T_Q // 32)
    p_cnt = np.zeros((w.Hmask, k_rows), np.int64)
    f_cnt = np.zeros((w.Hmask, k_rows), np.int64)
    p_lists, f_lists, pays, p_ord, f_ord = [], [], [], [], []
    for hm in range(w.Hmask):
        for b, (q_off, q_len, k_off, k_len) in enumerate(bounds):
            nq, nk = int(q_rows_b[b]), int(k_rows_b[b])
            if nk == 0:
                continue
            vis = M.visible_rows(w, hm, b, np.arange(q_len)) if q_len else np.zeros((0, k_len), bool)
            tiles, cls = _tile_classes(vis, T_Q, T_KV, nq, nk)
            # rank of K tile j among the non-empty K tiles of Q tile i (ascending K)
            nonempty = cls > 0
            rank = np.cumsum(nonempty, axis=1) - 1
            for j in range(nk):
                r = int(cu_k_rows[b]) + j
                pi = np.nonzero(cls[:, j] == 1)[0]
                fi = np.nonzero(cls[:, j] == 2)[0]
                p_cnt[hm, r], f_cnt[hm, r] = pi.size, fi.size
                p_lists.append(pi)
                f_lists.append(fi)
                p_ord.append(rank[pi, j])
                f_ord.append(rank[fi, j])
                for i in pi:
                    t = tiles[i, :, j, :]                       # [T_Q rows, T_KV keys]
                    padded = np.zeros((T_KV, nw * 32), dtype=bool)
                    padded[:, :T_Q] = t.T                       # key-major
                    words = np.packbits(padded, axis=1, bitorder="little").view("<u4")
                    pays.append(words.reshape(T_KV, nw).astype(np.uint32))

    def _csr(cnt):
        off = np.zeros(cnt.size + 1, np.int64)
        off[1:] = np.cumsum(cnt.reshape(-1))
        return off

    cat = lambda xs: np.concatenate(xs).astype(np.int64) if xs else np.zeros(0, np.int64)
    payload = np.stack(pays) if pays else np.zeros((0, T_KV, nw), np.uint32)
    fwd_rows = int(q_rows_b.sum())
    return BackwardView(T_Q, T_KV, w.Hmask, k_rows, cu_k_rows, krow_batch, krow_nblock, _csr(p_cnt),
                        _csr(f_cnt), cat(p_lists), cat(f_lists), payload, cat(p_ord), cat(f_ord),
                        fwd_rows)


def visible_from_k2q(v: BackwardView, hm: int, b: int, q_len: int, k_len: int) -> np.ndarray:
    """Dense visibility of (mask head hm, sample b) rebuilt from the K2Q view alone."""
    T_Q, T_KV = v.T_Q, v.T_KV
    nk = int(v.cu_k_rows[b + 1] - v.cu_k_rows[b])
    nq = -(-q_len // T_Q)
    out = np.zeros((nq * T_Q, nk * T_KV), dtype=bool)
    bits = np.arange(32, dtype=np.uint32)
    for j in range(nk):
        flat = hm * v.k_rows + int(v.cu_k_rows[b]) + j
        for e in range(int(v.full_offset[flat]), int(v.full_offset[flat + 1])):
            i = int(v.full_idx[e])
            out[i * T_Q:(i + 1) * T_Q, j * T_KV:(j + 1) * T_KV] = True
        for e in range(int(v.partial_offset[flat]), int(v.partial_offset[flat + 1])):
            i = int(v.partial_idx[e])
            words = v.payload[e]                                   # [T_KV keys, nw]
            dense = ((words[:, :, None] >> bits[None, None, :]) & 1).astype(bool).reshape(T_KV, -1)
            out[i * T_Q:(i + 1) * T_Q, j * T_KV:(j + 1) * T_KV] |= dense[:, :T_Q].T
    return out[:q_len, :k_len]


def attention_grad_dense(q, k, v, do, vis, q_pos, scale, softcap=0.0, slope=None):
    """One (sample, head) in fp64: q [n, d], k/v [m, d], do [n, d], vis [n, m].

    Returns (dq [n, d], dk [m, d], dv [m, d], O [n, d], LSE [n]).
    """
    s = (q @ k.T) * scale
    if softcap and softcap > 0.0:
        th = np.tanh(s / softcap)
        z = softcap * th
        dz_ds = 1.0 - th * th
    else:
        z = s
        dz_ds = np.ones_like(s)
    if slope is not None:
        kpos = np.arange(k.shape[0], dtype=np.float64)
        z = z + float(slope) * (kpos[None, :] - np.asarray(q_pos, np.float64)[:, None])
    z = np.where(vis, z, -np.inf)
    m = z.max(axis=1, initial=-np.inf)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.exp(z - m_safe[:, None])
    l = e.sum(axis=1)
    p = e / np.where(has, l, 1.0)[:, None]
    p[~has] = 0.0
    o = p @ v
    lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    dv = p.T @ do
    dp = do @ v.T
    delta = (do * o).sum(axis=1)
    dz = p * (dp - delta[:, None])
    ds = dz * dz_ds
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, o, lse


def attention_grad_full(w, dout):
    """Gradients of every Q/K/V element (small workloads only), fp64, shaped
    like w.q / w.k / w.v; K/V gradients sum over the Q heads of their group."""
    dq = np.zeros(tuple(w.q.shape), np.float64)
    dk = np.zeros(tuple(w.k.shape), np.float64)
    dv = np.zeros(tuple(w.v.shape), np.float64)
    do_all = as_f64(dout)
    group = w.Hq // w.Hk
    for b, (q_off, q_len, k_off, k_len) in enumerate(w.sample_bounds()):
        for h in range(w.Hq):
            qh, kh, vh = head_slice(w, b, h)
            hm = 0 if w.Hmask == 1 else h
            rows = np.arange(q_len)
            vis = M.visible_rows(w, hm, b, rows)
            do = do_all[b, :, h, :] if w.layout == 0 else do_all[q_off:q_off + q_len, h, :]
            slope = None if w.alibi_slopes is None else float(w.alibi_slopes[h])
            gq, gk, gv, _, _ = attention_grad_dense(qh, kh, vh, do, vis, rows, w.scale, w.softcap, slope)
            hk = h // group
            if w.layout == 0:
                dq[b, :, h, :] = gq
                dk[b, :, hk, :] += gk
                dv[b, :, hk, :] += gv
            else:
                dq[q_off:q_off + q_len, h, :] = gq
                dk[k_off:k_off + k_len, hk, :] += gk
                dv[k_off:k_off + k_len, hk, :] += gv
    return dq, dk, dv
