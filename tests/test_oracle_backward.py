"""Pins for oracle.backward: gradients against autograd through a library
attention routine and against finite differences; the K2Q view against the
dense mask (invariant 7 of "Flex Attention Mask Plan Design" §9), against the
Q2K view, and its dQ write order and payload bit positions."""
import math

import numpy as np
import pytest
import torch

from oracle import backward as OB
from oracle import mask as M
from oracle import plan as P
from block_sparse_masked_gb300 import workloads as W


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


@pytest.mark.parametrize("kind", ["all", "causal", "random", "empty_rows"])
def test_grad_matches_sdpa_autograd(kind):
    n, m, d = 37, 53, 16
    q, k, v, do = _rand((n, d), 1), _rand((m, d), 2), _rand((m, d), 3), _rand((n, d), 4)
    if kind == "all":
        vis = np.ones((n, m), bool)
    elif kind == "causal":
        vis = np.arange(m)[None, :] <= np.arange(n)[:, None]
    else:
        vis = np.random.default_rng(5).random((n, m)) < 0.3
        if kind == "empty_rows":
            vis[[0, 7, 20]] = False
    scale = 1 / math.sqrt(d)
    dq, dk, dv, o, lse = OB.attention_grad_dense(q.numpy(), k.numpy(), v.numpy(), do.numpy(), vis,
                                                 np.arange(n), scale)
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    has = vis.any(axis=1)
    mask = torch.from_numpy(vis | ~has[:, None])  # SDPA needs one visible key per row
    ot = torch.nn.functional.scaled_dot_product_attention(qt[None], kt[None], vt[None],
                                                          attn_mask=mask[None], scale=scale)[0]
    ot = ot * torch.from_numpy(has)[:, None]       # rows without keys: O = 0, no gradient
    (ot * do).sum().backward()
    assert np.allclose(o, ot.detach().numpy(), atol=1e-12)
    assert np.allclose(dq, qt.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, kt.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, vt.grad.numpy(), atol=1e-11)
    assert np.all(dq[~has] == 0)


def test_grad_softcap_alibi_autograd_and_finite_differences():
    n, m, d = 19, 23, 8
    q, k, v, do = _rand((n, d), 11), _rand((m, d), 12), _rand((m, d), 13), _rand((n, d), 14)
    q = q * 3.0  # scores of a few units, where the softcap's curvature matters
    vis = np.random.default_rng(6).random((n, m)) < 0.6
    vis[:, 0] = True
    scale, cap, slope = 1 / math.sqrt(d), 2.0, 0.3
    pos = np.arange(n) + 4
    dq, dk, dv, o, _ = OB.attention_grad_dense(q.numpy(), k.numpy(), v.numpy(), do.numpy(), vis, pos,
                                               scale, cap, slope)

    # autograd through the forward written with torch operations
    def fwd(qq, kk, vv):
        s = (qq @ kk.T) * scale
        z = cap * torch.tanh(s / cap) + slope * (torch.arange(m, dtype=torch.float64)[None, :]
                                                 - torch.from_numpy(pos).double()[:, None])
        z = z.masked_fill(~torch.from_numpy(vis), float("-inf"))
        return torch.softmax(z, dim=1) @ vv

    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    (fwd(qt, kt, vt) * do).sum().backward()
    assert np.allclose(dq, qt.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, kt.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, vt.grad.numpy(), atol=1e-11)
    # central differences on a few coordinates
    f = lambda qq, kk, vv: float((fwd(qq, kk, vv) * do).sum())
    h = 1e-6
    for (arr, grad, idx) in ((q, dq, (3, 2)), (k, dk, (5, 7)), (v, dv, (0, 1))):
        a1, a2 = arr.clone(), arr.clone()
        a1[idx] += h
        a2[idx] -= h
        args1 = [q, k, v]
        args2 = [q, k, v]
        which = 0 if arr is q else (1 if arr is k else 2)
        args1[which], args2[which] = a1, a2
        fd = (f(*args1) - f(*args2)) / (2 * h)
        assert abs(fd - grad[idx]) < 1e-6


def _interval_case():
    lens = np.array([300, 1, 129, 200])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    mf = W.random_intervals(7, len(lens), 0, 0, 3, 2, lens_q=lens, lens_k=lens)
    z = torch.zeros(int(lens.sum()), 2, 0, dtype=torch.bfloat16)
    return W.Workload("v", W.LAYOUT_THD, len(lens), 300, 300, 2, 2, 8, z, z, z, 1.0, "intervals",
                      mask_func=mf, cu_seqlens_q=cu, cu_seqlens_k=cu.copy())


def _block_case():
    S = 333
    bm = W.random_block_mask(9, 2, -(-S // 64), -(-S // 64), 0.25)
    z = torch.zeros(1, S, 2, 0, dtype=torch.bfloat16)
    return W.Workload("b", W.LAYOUT_BSHD, 1, S, S, 2, 2, 8, z, z, z, 1.0, "blocks", block_mask=bm,
                      block_q=64, block_kv=64)


@pytest.mark.parametrize("case", ["intervals", "blocks"])
@pytest.mark.parametrize("T", [(128, 128), (64, 32)])
def test_k2q_view_reproduces_mask_and_transposes_q2k(case, T):
    w = _interval_case() if case == "intervals" else _block_case()
    v = OB.build_backward_view(w, *T)
    fwd = P.build_plan(w, *T)
    for hm in range(w.Hmask):
        for b, (qo, ql, ko, kl) in enumerate(w.sample_bounds()):
            dense = M.visible_rows(w, hm, b, np.arange(ql)) if ql else np.zeros((0, kl), bool)
            assert np.array_equal(OB.visible_from_k2q(v, hm, b, ql, kl), dense)
    # same block relation as the Q2K view: {(i, j, class)} sets agree
    q2k, k2q = set(), set()
    for hm in range(w.Hmask):
        for r in range(fwd.rows):
            b, i = int(fwd.row_batch[r]), int(fwd.row_mblock[r])
            f = hm * fwd.rows + r
            for e in range(int(fwd.partial_offset[f]), int(fwd.partial_offset[f + 1])):
                q2k.add((hm, b, i, int(fwd.partial_idx[e]), 1))
            for e in range(int(fwd.full_offset[f]), int(fwd.full_offset[f + 1])):
                q2k.add((hm, b, i, int(fwd.full_idx[e]), 2))
        for r in range(v.k_rows):
            b, j = int(v.krow_batch[r]), int(v.krow_nblock[r])
            f = hm * v.k_rows + r
            lst = v.partial_idx[v.partial_offset[f]:v.partial_offset[f + 1]].tolist()
            assert lst == sorted(lst)
            for i in lst:
                k2q.add((hm, b, i, j, 1))
            for i in v.full_idx[v.full_offset[f]:v.full_offset[f + 1]].tolist():
                k2q.add((hm, b, i, j, 2))
    assert q2k == k2q and len(k2q) == fwd.partial_idx.size + fwd.full_idx.size
    assert v.header[1:] == [fwd.partial_idx.size, fwd.full_idx.size]


def test_dq_write_order_is_ascending_k_rank():
    w = _interval_case()
    v = OB.build_backward_view(w)
    fwd = P.build_plan(w)
    contrib = {}
    for hm in range(w.Hmask):
        for r in range(v.k_rows):
            b, j = int(v.krow_batch[r]), int(v.krow_nblock[r])
            f = hm * v.k_rows + r
            for lst, ords, off in ((v.partial_idx, v.dq_write_order, v.partial_offset),
                                   (v.full_idx, v.dq_write_order_full, v.full_offset)):
                for e in range(int(off[f]), int(off[f + 1])):
                    contrib.setdefault((hm, b, int(lst[e])), []).append((j, int(ords[e])))
    for (hm, b, i), items in contrib.items():
        items.sort()
        assert [o for _, o in items] == list(range(len(items)))   # ranks 0..n-1 in K order
        r = int(fwd.cu_q_rows[b]) + i
        f = hm * fwd.rows + r
        n = (fwd.partial_offset[f + 1] - fwd.partial_offset[f]) + (fwd.full_offset[f + 1] - fwd.full_offset[f])
        assert len(items) == n


def test_k2q_payload_single_element():
    """One visible element at (query row 5, key 70) of a tile: K2Q payload
    word 0 of key 70 has bit 5 set, nothing else."""
    S = 128
    ends = np.zeros((1, 3, S), np.int32)
    ends[0, 1, 5] = 70
    ends[0, 2, 5] = 71
    z = torch.zeros(1, S, 1, 0, dtype=torch.bfloat16)
    w = W.Workload("one", W.LAYOUT_BSHD, 1, S, S, 1, 1, 8, z, z, z, 1.0, "intervals", mask_func=ends)
    v = OB.build_backward_view(w)
    assert v.partial_idx.tolist() == [0] and v.full_idx.size == 0
    want = np.zeros((128, 4), np.uint32)
    want[70, 0] = 1 << 5
    assert np.array_equal(v.payload[0], want)
    assert v.dq_write_order.tolist() == [0]


def test_backward_view_by_heads_equals_single_pass():
    w = _interval_case()
    one = OB.build_backward_view(w)
    merged = OB.build_backward_view_by_heads(w.mask_only(), processes=2)
    for f in ("partial_offset", "full_offset", "partial_idx", "full_idx", "payload", "dq_write_order",
              "dq_write_order_full", "cu_k_rows"):
        assert np.array_equal(getattr(one, f), getattr(merged, f)), f
    assert one.k_rows == merged.k_rows


def test_dq_rows_equals_full_gradient_rows():
    n, d = 70, 16
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn(1, n, 2, d, generator=g).bfloat16() for _ in range(3))
    mf = W.random_intervals(4, 1, n, n, 3, 1)
    w = W.Workload("t", W.LAYOUT_BSHD, 1, n, n, 2, 2, d, q, k, v, 0.25, "intervals", mask_func=mf)
    w.softcap = 3.0
    w.alibi_slopes = W.alibi_slopes(2)
    dout = torch.randn(1, n, 2, d, generator=g).bfloat16()
    fq, _, _ = OB.attention_grad_full(w, dout)
    rows = np.array([0, 5, 33, 69])
    assert np.allclose(OB.dq_rows(w, 0, 1, rows, dout), fq[0, rows, 1, :], atol=1e-12)
