"""Brute-force MaskPlan (oracle, test infrastructure).

Follows "Flex Attention Mask Plan Design":

* §4.2 compact row prefixes: each sample contributes ceil(q_len / T_Q) Q plan
  rows; ``cu_q_rows`` is their prefix sum.
* §4.3 Q2K classification: every (Q plan row, sample-local K tile) pair is
  exactly one of empty (no valid visible element), full (the whole T_Q x T_KV
  tile lies inside the sample and every element is visible) or partial
  (anything else: some visible element, or visible but needing Q/K tail
  protection).
* §4.5 header: {forward Q rows, partial nnz, full nnz, 0, 0, 0, 0, error}.
* §4.6 independent partial and full CSR lists per (mask head, Q plan row);
  indices are sample-local K tiles in ascending order.
* §5 packed predicate payload, one per partial entry.  Layout of this
  library's consumer (one TMEM lane = one score row): payload[e, r, w] is a
  uint32 whose bit l is 1 iff element (row r, column 32*w + l) of the tile is
  visible; padding and out-of-sample elements are 0.  With it goes
  halves[e]: bit s is 1 iff some element in columns [s*T_KV/2, (s+1)*T_KV/2)
  of the tile is visible (the consumer skips an empty half), and quads[e]
  for the tile's four quadrants (row half a, column half s, quadrant index
  2a + s): bit 2a+s is 1 iff some element of the quadrant is visible, bit
  4+2a+s iff every element of it is (so the quadrant lies inside the sample).
  A consumer that works on one half-height row block at a time reads which
  column halves it must visit, and which need no predicate, from it.
* §4.8 schedule: ``sequence_desc[B, 8]`` = (q_offset, k_offset, q_len, k_len,
  Q-plan-row begin, Q-plan-row count, K tile count, 0) and
  ``work_desc[tasks, 4]`` = (m_block, head, batch, q_valid_rows), one task per
  (valid Q plan row, Q head); cost = partial + full count.  Positive-cost
  tasks are ordered by L2 section (the (sample, K/V head) pair whose K/V the
  task reads), then descending cost, then the tie order (head, m_block);
  zero-cost tasks follow in (batch, head, m_block) order.
* Consumer order ``lpt[tasks]``: for interval masks, the positions of
  work_desc sorted by task cost, descending, ties in work_desc order (a
  stable sort), so zero-cost tasks stay last: the longest-first order in
  which a consumer with few tasks per SM takes the tasks.  For block masks,
  work_desc's own order (the identity): their consumers keep the section
  order, under which a (sample, K/V head)'s K/V stays in L2 (§4.8 fixes the
  task list; the traversal is the consumer's).

The classification here is computed by expanding each Q tile into a dense
boolean matrix and testing every element, which is independent of the GPU's
interval / bitset reduction.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import mask as M


@dataclasses.dataclass
class Plan:
    T_Q: int
    T_KV: int
    Hmask: int
    Hq: int
    Hk: int
    rows: int                      # valid Q plan rows over all samples
    cu_q_rows: np.ndarray          # int64 [B+1]
    k_tiles: np.ndarray            # int64 [B]
    row_batch: np.ndarray          # int64 [rows]
    row_mblock: np.ndarray         # int64 [rows]
    row_qvalid: np.ndarray         # int64 [rows]
    partial_count: np.ndarray      # int64 [Hmask, rows]
    full_count: np.ndarray         # int64 [Hmask, rows]
    partial_offset: np.ndarray     # int64 [Hmask*rows + 1]
    full_offset: np.ndarray        # int64 [Hmask*rows + 1]
    partial_idx: np.ndarray        # int64 [P]
    full_idx: np.ndarray           # int64 [F]
    payload: np.ndarray            # uint32 [P, T_Q, ceil(T_KV/32)]
    halves: np.ndarray             # uint8 [P]: bit s = some element of column half s is visible
    quads: np.ndarray              # uint8 [P]: bit 2a+s any / bit 4+2a+s all of quadrant (a, s) visible
    sequence_desc: np.ndarray      # int64 [B, 8]
    work_desc: np.ndarray          # int64 [tasks, 4]
    visible_pairs: int             # |visible (q, k)| summed over mask heads and samples
    lpt: np.ndarray                # int64 [tasks]: work_desc positions, cost descending (stable)             # |visible (q, k)| summed over mask heads and samples

    @property
    def header(self):
        return [self.rows, int(self.partial_idx.size), int(self.full_idx.size), 0, 0, 0, 0, 0]


def _classify_tile_row(vis_rows: np.ndarray, T_Q: int, T_KV: int, nk: int):
    """Classify one Q tile given its dense visibility rows [tq <= T_Q, k_len].

    Returns (visible[nk], full[nk], tiles[T_Q, nk, T_KV]) where elements outside
    the sample are False.
    """
    tq, k_len = vis_rows.shape
    tiles = np.zeros((T_Q, nk * T_KV), dtype=bool)
    tiles[:tq, :k_len] = vis_rows
    tiles = tiles.reshape(T_Q, nk, T_KV)
    visible = tiles.any(axis=(0, 2))
    # full: every element of the whole T_Q x T_KV tile is visible; tail
    # elements are False above, so a tile needing tail protection is never full.
    full = tiles.all(axis=(0, 2))
    return visible, full, tiles


def _quadrant_bits(tiles: np.ndarray) -> np.ndarray:
    """bool [T_Q, n, T_KV] -> uint8 [n]: quadrant (a, s) = rows [a*T_Q/2, (a+1)*T_Q/2)
    x columns [s*T_KV/2, (s+1)*T_KV/2); bit 2a+s = any element visible, bit
    4+2a+s = all elements visible."""
    T_Q, n, T_KV = tiles.shape
    rq, cq = T_Q // 2, T_KV // 2
    out = np.zeros(n, np.uint8)
    for a in range(2):
        for s in range(2):
            quad = tiles[a * rq:(a + 1) * rq, :, s * cq:(s + 1) * cq]
            out |= (quad.any(axis=(0, 2)).astype(np.uint8) << (2 * a + s))
            out |= (quad.all(axis=(0, 2)).astype(np.uint8) << (4 + 2 * a + s))
    return out


def _pack_tiles(tiles: np.ndarray) -> np.ndarray:
    """bool [T_Q, n, T_KV] -> uint32 [n, T_Q, ceil(T_KV/32)]; bit l of word w = column 32w+l."""
    T_Q, n, T_KV = tiles.shape
    nw = -(-T_KV // 32)
    padded = np.zeros((n, T_Q, nw * 32), dtype=bool)
    padded[:, :, :T_KV] = tiles.transpose(1, 0, 2)
    # little bit order: column 32w+l -> byte 4w + l//8, bit l%8 -> bit l of the LE word w
    packed = np.packbits(padded, axis=2, bitorder="little")
    return np.ascontiguousarray(packed).view("<u4").reshape(n, T_Q, nw).astype(np.uint32)


def build_plan(w, T_Q: int = 128, T_KV: int = 128, with_payload: bool = True,
               mask_heads=None) -> Plan:
    """Build the plan for workload ``w`` by dense expansion (raises MaskError on bad input).

    ``mask_heads`` restricts the build to those mask heads (the result then
    covers only them, in the given order, and carries no schedule); it exists
    so that large plans can be built one head per process and merged.
    """
    bounds = w.sample_bounds()
    B = len(bounds)
    if w.layout == 1:
        M.validate_seqlens(w.cu_seqlens_q, w.cu_seqlens_k, w.total_q, w.total_k, w.Sq, w.Sk)
    if w.mask_kind == "intervals":
        Hm, nf, tq_all = w.mask_func.shape
        if tq_all != w.total_q:
            raise M.MaskError("mask_func rows != total_q")
        for (q_off, q_len, k_off, k_len) in bounds:
            M.validate_endpoints(w.mask_func[:, :, q_off:q_off + q_len].transpose(1, 0, 2)
                                 .reshape(nf, -1), k_len)
    Hmask = w.Hmask
    if Hmask not in (1, w.Hq):
        raise M.MaskError("Hmask must be 1 or Hq")
    heads = list(range(Hmask)) if mask_heads is None else list(mask_heads)

    q_rows = np.array([-(-ql // T_Q) for (_, ql, _, _) in bounds], dtype=np.int64)
    k_tiles = np.array([-(-kl // T_KV) for (_, _, _, kl) in bounds], dtype=np.int64)
    cu_q_rows = np.concatenate([[0], np.cumsum(q_rows)]).astype(np.int64)
    rows = int(cu_q_rows[-1])
    row_batch = np.repeat(np.arange(B), q_rows)
    row_mblock = np.concatenate([np.arange(n) for n in q_rows]) if rows else np.zeros(0, np.int64)
    row_qvalid = np.array([min(T_Q, bounds[b][1] - m * T_Q) for b, m in zip(row_batch, row_mblock)],
                          dtype=np.int64)

    p_cnt = np.zeros((len(heads), rows), np.int64)
    f_cnt = np.zeros((len(heads), rows), np.int64)
    p_lists, f_lists, payloads, halves, quads = [], [], [], [], []
    visible_pairs = 0
    for slot, hm in enumerate(heads):
        for r in range(rows):
            b, m = int(row_batch[r]), int(row_mblock[r])
            q_off, q_len, k_off, k_len = bounds[b]
            q_local = np.arange(m * T_Q, min((m + 1) * T_Q, q_len))
            vis = M.visible_rows(w, hm, b, q_local)
            visible_pairs += int(vis.sum())
            visible, full, tiles = _classify_tile_row(vis, T_Q, T_KV, int(k_tiles[b]))
            partial = visible & ~full
            pi = np.nonzero(partial)[0]
            fi = np.nonzero(full)[0]
            p_cnt[slot, r] = pi.size
            f_cnt[slot, r] = fi.size
            p_lists.append(pi)
            f_lists.append(fi)
            if with_payload and pi.size:
                payloads.append(_pack_tiles(tiles[:, pi, :]))
            if pi.size:
                hcut = T_KV // 2
                lo = tiles[:, pi, :hcut].any(axis=(0, 2))
                hi = tiles[:, pi, hcut:].any(axis=(0, 2))
                halves.append((lo.astype(np.uint8) | (hi.astype(np.uint8) << 1)))
                quads.append(_quadrant_bits(tiles[:, pi, :]))

    def _csr(cnt):
        off = np.zeros(cnt.size + 1, np.int64)
        off[1:] = np.cumsum(cnt.reshape(-1))
        return off

    partial_idx = np.concatenate(p_lists).astype(np.int64) if p_lists else np.zeros(0, np.int64)
    full_idx = np.concatenate(f_lists).astype(np.int64) if f_lists else np.zeros(0, np.int64)
    nw = -(-T_KV // 32)
    payload = (np.concatenate(payloads) if payloads else np.zeros((0, T_Q, nw), np.uint32))
    halves_arr = np.concatenate(halves) if halves else np.zeros(0, np.uint8)
    quads_arr = np.concatenate(quads) if quads else np.zeros(0, np.uint8)

    seq = np.zeros((B, 8), np.int64)
    for b, (q_off, q_len, k_off, k_len) in enumerate(bounds):
        seq[b] = (q_off, k_off, q_len, k_len, cu_q_rows[b], q_rows[b], k_tiles[b], 0)

    if mask_heads is None:
        work = schedule(row_batch, row_mblock, row_qvalid, p_cnt, f_cnt, w.Hq, w.Hk, Hmask)
    else:
        work = np.zeros((0, 4), np.int64)
    return Plan(T_Q, T_KV, len(heads), w.Hq, w.Hk, rows, cu_q_rows, k_tiles, row_batch, row_mblock,
                row_qvalid, p_cnt, f_cnt, _csr(p_cnt), _csr(f_cnt), partial_idx, full_idx,
                payload, halves_arr, quads_arr, seq, work, visible_pairs,
                consumer_order(work, seq, p_cnt, f_cnt, Hmask, w.mask_kind))


def schedule(row_batch, row_mblock, row_qvalid, p_cnt, f_cnt, Hq, Hk, Hmask) -> np.ndarray:
    """Forward task order of §4.8 (see module docstring), as work_desc [tasks, 4]."""
    rows = row_batch.size
    group = Hq // Hk
    tasks = []   # (batch, head, m_block, row)
    for r in range(rows):
        for h in range(Hq):
            tasks.append((int(row_batch[r]), h, int(row_mblock[r]), r))
    # base (tie) order: batch, head, m_block
    tasks.sort(key=lambda t: (t[0], t[1], t[2]))

    def cost(t):
        hm = 0 if Hmask == 1 else t[1]
        return int(p_cnt[hm, t[3]] + f_cnt[hm, t[3]])

    def section(t):
        return t[0] * Hk + t[1] // group

    pos = [t for t in tasks if cost(t) > 0]
    zero = [t for t in tasks if cost(t) == 0]
    pos.sort(key=lambda t: (section(t), -cost(t)))  # Python's sort is stable: keeps tie order
    out = np.array([(t[2], t[1], t[0], int(row_qvalid[t[3]])) for t in pos + zero],
                   dtype=np.int64).reshape(-1, 4)
    return out


def consumer_order(work, sequence_desc, p_cnt, f_cnt, Hmask, mask_kind) -> np.ndarray:
    """Interval masks: positions of work_desc by task cost (partial + full
    entries of the task's Q plan row), descending, ties in work_desc order.
    Block masks: work_desc order."""
    if mask_kind != "intervals":
        return np.arange(len(work), dtype=np.int64)
    cost = np.zeros(len(work), np.int64)
    for i, (m, h, b, _) in enumerate(np.asarray(work).tolist()):
        hm, r = (0 if Hmask == 1 else h), int(sequence_desc[b, 4]) + m
        cost[i] = int(p_cnt[hm, r]) + int(f_cnt[hm, r])
    return np.argsort(-cost, kind="stable").astype(np.int64)


def visible_from_plan(p: Plan, hm: int, b: int, q_len: int, k_len: int) -> np.ndarray:
    """Reconstruct the dense visibility of (hm, sample b) from a plan's CSR + payload.

    Used to check that a plan preserves E(M) exactly under any physical tiling.
    """
    T_Q, T_KV = p.T_Q, p.T_KV
    nk = int(p.k_tiles[b])
    out = np.zeros((int(p.cu_q_rows[b + 1] - p.cu_q_rows[b]) * T_Q, nk * T_KV), dtype=bool)
    bits = (np.arange(32, dtype=np.uint32))
    for r in range(int(p.cu_q_rows[b]), int(p.cu_q_rows[b + 1])):
        m = r - int(p.cu_q_rows[b])
        flat = hm * p.rows + r
        for e in range(int(p.full_offset[flat]), int(p.full_offset[flat + 1])):
            j = int(p.full_idx[e])
            out[m * T_Q:(m + 1) * T_Q, j * T_KV:(j + 1) * T_KV] = True
        for e in range(int(p.partial_offset[flat]), int(p.partial_offset[flat + 1])):
            j = int(p.partial_idx[e])
            words = p.payload[e]                              # [T_Q, nw]
            dense = ((words[:, :, None] >> bits[None, None, :]) & 1).astype(bool)
            dense = dense.reshape(T_Q, -1)[:, :T_KV]
            out[m * T_Q:(m + 1) * T_Q, j * T_KV:(j + 1) * T_KV] |= dense
    return out[:q_len, :k_len]


def _one_head(args):
    w, T_Q, T_KV, hm = args
    return build_plan(w, T_Q, T_KV, True, mask_heads=[hm])


def build_plan_by_heads(w, T_Q: int = 128, T_KV: int = 128, processes: int = 8) -> Plan:
    """Same result as build_plan(w), one mask head per worker process (spawned).

    ``w`` should be a mask-only workload (see Workload.mask_only) so that it
    pickles cheaply.  Per-head plans are concatenated in head order, which is
    exactly the row-major (mask head, row) layout of the CSR.
    """
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes) as pool:
        parts = pool.map(_one_head, [(w, T_Q, T_KV, hm) for hm in range(w.Hmask)])
    first = parts[0]
    p_cnt = np.concatenate([q.partial_count for q in parts])
    f_cnt = np.concatenate([q.full_count for q in parts])

    def _csr(cnt):
        off = np.zeros(cnt.size + 1, np.int64)
        off[1:] = np.cumsum(cnt.reshape(-1))
        return off

    work = schedule(first.row_batch, first.row_mblock, first.row_qvalid, p_cnt, f_cnt, w.Hq, w.Hk,
                    w.Hmask)
    return Plan(T_Q, T_KV, w.Hmask, w.Hq, w.Hk, first.rows, first.cu_q_rows, first.k_tiles,
                first.row_batch, first.row_mblock, first.row_qvalid, p_cnt, f_cnt, _csr(p_cnt),
                _csr(f_cnt), np.concatenate([q.partial_idx for q in parts]),
                np.concatenate([q.full_idx for q in parts]),
                np.concatenate([q.payload for q in parts]),
                np.concatenate([q.halves for q in parts]),
                np.concatenate([q.quads for q in parts]), first.sequence_desc, work,
                sum(q.visible_pairs for q in parts),
                consumer_order(work, first.sequence_desc, p_cnt, f_cnt, w.Hmask, w.mask_kind))
