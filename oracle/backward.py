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


def build_backward_view(w, T_Q: int = 128, T_KV: int = 128, mask_heads=None) -> BackwardView:
    """K2Q view, its payload and the dQ write order, by dense expansion of the
    mask one Q tile strip at a time (every element of every tile is tested).

    ``mask_heads`` restricts the build to those heads, in that order (for
    building large views one head per process)."""
    bounds = w.sample_bounds()
    B = len(bounds)
    heads = list(range(w.Hmask)) if mask_heads is None else list(mask_heads)
    k_rows_b = np.array([-(-kl // T_KV) for (_, _, _, kl) in bounds], dtype=np.int64)
    q_rows_b = np.array([-(-ql // T_Q) for (_, ql, _, _) in bounds], dtype=np.int64)
    cu_k_rows = np.concatenate([[0], np.cumsum(k_rows_b)]).astype(np.int64)
    k_rows = int(cu_k_rows[-1])
    krow_batch = np.repeat(np.arange(B), k_rows_b)
    krow_nblock = np.concatenate([np.arange(n) for n in k_rows_b]) if k_rows else np.zeros(0, np.int64)
    nw = -(-T_Q // 32)
    # per (head slot, K row): lists of (Q tile, rank, payload or None) in ascending Q tile order
    plist = [[[] for _ in range(k_rows)] for _ in heads]
    flist = [[[] for _ in range(k_rows)] for _ in heads]
    for slot, hm in enumerate(heads):
        for b, (q_off, q_len, k_off, k_len) in enumerate(bounds):
            nq, nk = int(q_rows_b[b]), int(k_rows_b[b])
            for i in range(nq):
                rows = np.arange(i * T_Q, min((i + 1) * T_Q, q_len))
                vis = M.visible_rows(w, hm, b, rows)
                strip = np.zeros((T_Q, nk * T_KV), dtype=bool)
                strip[:rows.size, :k_len] = vis
                tiles = strip.reshape(T_Q, nk, T_KV)
                anyv = tiles.any(axis=(0, 2))
                allv = tiles.all(axis=(0, 2))
                rank = np.cumsum(anyv) - 1         # rank among the strip's non-empty K tiles
                for j in np.nonzero(anyv)[0]:
                    r = int(cu_k_rows[b]) + int(j)
                    if allv[j]:
                        flist[slot][r].append((i, int(rank[j])))
                    else:
                        padded = np.zeros((T_KV, nw * 32), dtype=bool)
                        padded[:, :T_Q] = tiles[:, j, :].T      # key-major
                        words = np.packbits(padded, axis=1, bitorder="little").view("<u4")
                        plist[slot][r].append((i, int(rank[j]), words.reshape(T_KV, nw).astype(np.uint32)))

    def _csr(lists):
        cnt = np.array([[len(x) for x in per] for per in lists], np.int64).reshape(-1)
        off = np.zeros(cnt.size + 1, np.int64)
        off[1:] = np.cumsum(cnt)
        return off

    flat_p = [e for per in plist for row in per for e in row]
    flat_f = [e for per in flist for row in per for e in row]
    payload = (np.stack([e[2] for e in flat_p]) if flat_p else np.zeros((0, T_KV, nw), np.uint32))
    return BackwardView(T_Q, T_KV, len(heads), k_rows, cu_k_rows, krow_batch, krow_nblock, _csr(plist),
                        _csr(flist), np.array([e[0] for e in flat_p], np.int64),
                        np.array([e[0] for e in flat_f], np.int64), payload,
                        np.array([e[1] for e in flat_p], np.int64), np.array([e[1] for e in flat_f], np.int64),
                        int(q_rows_b.sum()))


def _one_head(args):
    w, T_Q, T_KV, hm = args
    return build_backward_view(w, T_Q, T_KV, mask_heads=[hm])


def build_backward_view_by_heads(w, T_Q: int = 128, T_KV: int = 128, processes: int = 8) -> BackwardView:
    """Same result as build_backward_view(w), one mask head per spawned worker
    (``w`` mask-only); per-head parts concatenate in head order, the layout
    of the row-major (mask head, K row) CSR."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes) as pool:
        parts = pool.map(_one_head, [(w, T_Q, T_KV, hm) for hm in range(w.Hmask)])
    first = parts[0]

    def _merge(offs):
        out, base = [np.zeros(1, np.int64)], 0
        for o in offs:
            out.append(o[1:] + base)
            base += int(o[-1])
        return np.concatenate(out)

    cat = lambda f: np.concatenate([getattr(q, f) for q in parts])
    return BackwardView(T_Q, T_KV, w.Hmask, first.k_rows, first.cu_k_rows, first.krow_batch,
                        first.krow_nblock, _merge([q.partial_offset for q in parts]),
                        _merge([q.full_offset for q in parts]), cat("partial_idx"), cat("full_idx"),
                        cat("payload"), cat("dq_write_order"), cat("dq_write_order_full"), first.fwd_rows)


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


def dq_rows(w, b: int, h: int, rows, dout):
    """dQ of sample b, Q head h at sample-local rows only (fp64): a row's dQ
    depends on its own visible keys and its own softmax, so full-size
    workloads can be checked row by row."""
    qh, kh, vh = head_slice(w, b, h)
    rows = np.asarray(rows, np.int64)
    hm = 0 if w.Hmask == 1 else h
    vis = M.visible_rows(w, hm, b, rows)
    q_off = w.sample_bounds()[b][0]
    do_all = as_f64(dout)
    do = do_all[b, rows, h, :] if w.layout == 0 else do_all[q_off + rows, h, :]
    slope = None if w.alibi_slopes is None else float(w.alibi_slopes[h])
    gq, _, _, _, _ = attention_grad_dense(qh[rows], kh, vh, do, vis, rows, w.scale, w.softcap, slope)
    return gq
