"""Pins for oracle.attention: special cases that reduce to torch's
scaled_dot_product_attention in fp64, and closed forms."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle import mask as M
from block_sparse_masked_gb300 import workloads as W


def _rand(n, m, d, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal((n, d)), g.standard_normal((m, d)), g.standard_normal((m, d))


def _sdpa(q, k, v, bool_mask=None, bias=None, scale=None):
    qt, kt, vt = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    am = None
    if bool_mask is not None:
        am = torch.from_numpy(bool_mask)[None, None]
    if bias is not None:
        am = torch.from_numpy(bias)[None, None]
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, scale=scale)
    return o[0, 0].numpy()


def _lse_ref(q, k, vis, scale):
    s = torch.from_numpy(q @ k.T * scale).masked_fill(~torch.from_numpy(vis), -math.inf)
    return torch.logsumexp(s, dim=1).numpy()


@pytest.mark.parametrize("n,m,d", [(7, 7, 8), (33, 50, 16), (64, 128, 64)])
def test_all_visible_equals_sdpa(n, m, d):
    q, k, v = _rand(n, m, d, n + m)
    vis = np.ones((n, m), bool)
    o, lse = A.attention_dense(q, k, v, vis, np.arange(n), 1 / math.sqrt(d))
    assert np.allclose(o, _sdpa(q, k, v), atol=1e-12, rtol=1e-12)
    assert np.allclose(lse, _lse_ref(q, k, vis, 1 / math.sqrt(d)), atol=1e-12)


def test_causal_equals_sdpa_is_causal():
    q, k, v = _rand(40, 40, 16, 3)
    vis = np.tril(np.ones((40, 40), bool))
    o, _ = A.attention_dense(q, k, v, vis, np.arange(40), 0.25)
    qt, kt, vt = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.25)[0, 0].numpy()
    assert np.allclose(o, ref, atol=1e-12)


def test_random_mask_equals_sdpa_bool_mask():
    q, k, v = _rand(50, 70, 16, 4)
    vis = np.random.default_rng(1).random((50, 70)) < 0.3
    vis[:, 0] = True   # SDPA returns NaN on fully masked rows; those are pinned separately
    o, lse = A.attention_dense(q, k, v, vis, np.arange(50), 0.3)
    assert np.allclose(o, _sdpa(q, k, v, bool_mask=vis, scale=0.3), atol=1e-12)
    assert np.allclose(lse, _lse_ref(q, k, vis, 0.3), atol=1e-12)


def test_alibi_equals_sdpa_with_additive_bias():
    # ALiBi slope * (k - q) as an additive float mask of the library routine
    q, k, v = _rand(30, 45, 8, 5)
    slope = 0.37
    qpos = np.arange(10, 40)
    bias = slope * (np.arange(45)[None, :] - qpos[:, None]).astype(np.float64)
    vis = np.ones((30, 45), bool)
    o, lse = A.attention_dense(q, k, v, vis, qpos, 0.5, slope=slope)
    assert np.allclose(o, _sdpa(q, k, v, bias=bias, scale=0.5), atol=1e-12)
    s = q @ k.T * 0.5 + bias
    assert np.allclose(lse, torch.logsumexp(torch.from_numpy(s), 1).numpy(), atol=1e-12)


def test_empty_row_zero_and_neg_inf():
    q, k, v = _rand(4, 6, 8, 6)
    vis = np.zeros((4, 6), bool)
    vis[1, 2] = True
    o, lse = A.attention_dense(q, k, v, vis, np.arange(4), 1.0)
    for r in (0, 2, 3):
        assert np.all(o[r] == 0.0) and lse[r] == -np.inf
    assert np.isfinite(lse[1])


def test_single_visible_key_closed_form():
    q, k, v = _rand(5, 9, 8, 8)
    vis = np.zeros((5, 9), bool)
    cols = [0, 3, 8, 4, 4]
    for r, c in enumerate(cols):
        vis[r, c] = True
    o, lse = A.attention_dense(q, k, v, vis, np.arange(5), 0.7)
    for r, c in enumerate(cols):
        assert np.allclose(o[r], v[c], atol=1e-15)
        assert np.isclose(lse[r], 0.7 * float(q[r] @ k[c]), atol=1e-12)


def test_equal_scores_mean_and_log_count():
    # q = 0 makes every score 0: O = mean of visible V rows, LSE = ln(count)
    _, k, v = _rand(1, 20, 8, 9)
    q = np.zeros((3, 8))
    vis = np.zeros((3, 20), bool)
    vis[0, :5] = True
    vis[1, ::3] = True
    vis[2, :] = True
    o, lse = A.attention_dense(q, k, v, vis, np.arange(3), 1.0)
    for r in range(3):
        idx = np.nonzero(vis[r])[0]
        assert np.allclose(o[r], v[idx].mean(axis=0), atol=1e-14)
        assert np.isclose(lse[r], math.log(idx.size), atol=1e-14)


def test_convex_hull():
    q, k, v = _rand(30, 40, 16, 10)
    vis = np.random.default_rng(2).random((30, 40)) < 0.5
    vis[:, 5] = True
    o, _ = A.attention_dense(q * 3, k, v, vis, np.arange(30), 1.0, softcap=2.0, slope=0.1)
    for r in range(30):
        vv = v[vis[r]]
        assert np.all(o[r] <= vv.max(axis=0) + 1e-12) and np.all(o[r] >= vv.min(axis=0) - 1e-12)


def test_softcap_saturates_at_cap_after_scaling():
    # one visible key with a huge score: mod(s) -> +-cap, so LSE -> +-cap.
    # (applying the cap before the scale would saturate at cap * scale instead)
    d = 8
    q = np.full((2, d), 10.0)
    k = np.vstack([np.full(d, 10.0), np.full(d, -10.0)])
    v = np.eye(2, d)
    vis = np.array([[True, False], [False, True]])
    _, lse = A.attention_dense(q, k, v, vis, np.arange(2), 0.5, softcap=5.0)
    assert np.isclose(lse[0], 5.0, atol=1e-9) and np.isclose(lse[1], -5.0, atol=1e-9)


def test_softcap_then_alibi_order():
    # softcap first, ALiBi added after: a saturated score plus slope*(k - q)
    d = 8
    q = np.full((1, d), 10.0)
    k = np.full((1, d), 10.0)
    v = np.ones((1, d))
    vis = np.ones((1, 1), bool)
    _, lse = A.attention_dense(q, k, v, vis, np.array([100]), 1.0, softcap=5.0, slope=1.0)
    assert np.isclose(lse[0], 5.0 - 100.0, atol=1e-9)


def test_softcap_limits():
    q, k, v = _rand(20, 30, 16, 11)
    vis = np.random.default_rng(3).random((20, 30)) < 0.6
    vis[:, 0] = True
    # very large cap: identical to unmodified attention (library routine)
    o, _ = A.attention_dense(q, k, v, vis, np.arange(20), 0.25, softcap=1e9)
    assert np.allclose(o, _sdpa(q, k, v, bool_mask=vis, scale=0.25), atol=1e-9)
    # tiny cap: all scores ~0, so O = mean of the visible V and LSE = ln(count)
    o, lse = A.attention_dense(q, k, v, vis, np.arange(20), 0.25, softcap=1e-9)
    for r in range(20):
        assert np.allclose(o[r], v[vis[r]].mean(axis=0), atol=1e-8)
        assert np.isclose(lse[r], math.log(vis[r].sum()), atol=1e-8)


def test_softcap_bound():
    q, k, v = _rand(16, 16, 8, 12)
    vis = np.eye(16, dtype=bool)
    _, lse = A.attention_dense(q * 50, k * 50, v, vis, np.arange(16), 1.0, softcap=3.0)
    assert np.all(np.abs(lse) <= 3.0)        # tanh saturates to exactly +-1 in fp64
    _, lse = A.attention_dense(q, k, v, vis, np.arange(16), 0.1, softcap=3.0)
    assert np.all(np.abs(lse) < 3.0)


def test_alibi_row_constant_shift_leaves_o():
    # Moving every query position by +7 adds the row constant -slope*7 to all
    # ALiBi terms slope*(k - q): O is unchanged and LSE drops by slope*7.
    q, k, v = _rand(6, 10, 8, 13)
    vis = np.ones((6, 10), bool)
    o0, l0 = A.attention_dense(q, k, v, vis, np.arange(6), 0.5)
    o1, l1 = A.attention_dense(q, k, v, vis, np.arange(6) + 7, 0.5, slope=0.0)
    assert np.allclose(o0, o1) and np.allclose(l0, l1)
    o2, l2 = A.attention_dense(q, k, v, vis, np.arange(6), 0.5, slope=0.3)
    o3, l3 = A.attention_dense(q, k, v, vis, np.arange(6) + 7, 0.5, slope=0.3)
    assert np.allclose(o2, o3, atol=1e-12)
    assert np.allclose(l3, l2 - 0.3 * 7, atol=1e-12)


def test_varlen_equals_per_document_causal_sdpa():
    w = W.varlen_doc_causal(2, total=1200, ndocs=4, H=2, d=16, min_len=100)
    o, lse = A.attention_full(w)
    for b in range(4):
        a, e = int(w.cu_seqlens_q[b]), int(w.cu_seqlens_q[b + 1])
        for h in range(2):
            qh = w.q[a:e, h].double()[None, None]
            kh = w.k[a:e, h].double()[None, None]
            vh = w.v[a:e, h].double()[None, None]
            ref = F.scaled_dot_product_attention(qh, kh, vh, is_causal=True, scale=w.scale)[0, 0]
            assert np.allclose(o[a:e, h], ref.numpy(), atol=1e-12)


def test_block_mask_workload_equals_sdpa():
    w = W.video_block_sparse(4, B=1, H=2, S=512, d=16, block=64, density=0.3)
    o, lse = A.attention_full(w)
    for h in range(2):
        vis = M.block_visible_rows(w.block_mask, 64, 64, h, np.arange(512), 512)
        ref = _sdpa(w.q[0, :, h].double().numpy(), w.k[0, :, h].double().numpy(),
                    w.v[0, :, h].double().numpy(), bool_mask=vis, scale=w.scale)
        assert np.allclose(o[0, :, h], ref, atol=1e-12)


def test_brute_force_triple_loop():
    """Naive per-element loops on a tiny problem with all mods."""
    g = np.random.default_rng(14)
    n, m, d = 5, 7, 3
    q, k, v = g.standard_normal((n, d)), g.standard_normal((m, d)), g.standard_normal((m, d))
    vis = g.random((n, m)) < 0.6
    vis[0] = False
    qpos = np.array([3, 4, 5, 6, 7])
    o, lse = A.attention_dense(q, k, v, vis, qpos, 0.9, softcap=1.5, slope=0.2)
    for i in range(n):
        w_, tot = [], 0.0
        for j in range(m):
            if vis[i, j]:
                s = 0.0
                for t in range(d):
                    s += q[i, t] * k[j, t]
                s = 1.5 * math.tanh(s * 0.9 / 1.5) + 0.2 * (j - qpos[i])
                w_.append((j, math.exp(s)))
                tot += math.exp(s)
        if not w_:
            assert lse[i] == -math.inf and np.all(o[i] == 0)
            continue
        assert math.isclose(lse[i], math.log(tot), abs_tol=1e-12)
        for t in range(d):
            ref = sum(p * v[j, t] for j, p in w_) / tot
            assert math.isclose(o[i, t], ref, abs_tol=1e-12)


def test_gqa_heads_and_per_head_masks_equal_sdpa():
    """Q head h reads K/V head h // (Hq / Hk) and, with one mask per Q head,
    its own intervals: per-head sliding windows of different widths, checked
    against fp64 SDPA on explicitly selected K/V heads (a mapping by h % Hk,
    or every head reading mask 0, fails)."""
    B, S, Hq, Hk, d = 2, 40, 6, 2, 8
    gen = torch.Generator().manual_seed(23)
    q = torch.randn(B, S, Hq, d, generator=gen).bfloat16()
    k = torch.randn(B, S, Hk, d, generator=gen).bfloat16()
    v = torch.randn(B, S, Hk, d, generator=gen).bfloat16()
    qi = np.arange(S)
    wins = [3 + 4 * h for h in range(Hq)]
    mf = np.zeros((Hq, 3, B * S), np.int32)
    for h, win in enumerate(wins):
        lo = np.maximum(0, qi + 1 - win)
        mf[h, 1] = np.tile(lo, B)                # [0,0) U [lo, q+1)
        mf[h, 2] = np.tile(qi + 1, B)
    w = W.Workload("gqa", W.LAYOUT_BSHD, B, S, S, Hq, Hk, d, q, k, v, 0.3, "intervals",
                   mask_func=mf)
    kk = np.arange(S)
    for b in range(B):
        for h in range(Hq):
            o, lse = A.attention_rows(w, b, h)
            vis = (kk[None, :] <= qi[:, None]) & (kk[None, :] >= qi[:, None] + 1 - wins[h])
            qh = q[b, :, h].double().numpy()
            kh = k[b, :, h // (Hq // Hk)].double().numpy()
            vh = v[b, :, h // (Hq // Hk)].double().numpy()
            assert np.allclose(o, _sdpa(qh, kh, vh, bool_mask=vis, scale=0.3), atol=1e-12)
            assert np.allclose(lse, _lse_ref(qh, kh, vis, 0.3), atol=1e-12)


def test_varlen_unequal_q_and_k_lengths_equal_sdpa():
    """THD samples whose Q and K lengths differ (cu_seqlens_q != cu_seqlens_k):
    sample b's rows read keys [cu_k[b], cu_k[b+1]) with sample-local
    positions; a mask that ends every row's keys at q + 1 + (k_len - q_len)
    (queries aligned to the end of their keys) is checked against fp64 SDPA
    on explicitly sliced keys."""
    lq, lk = np.array([5, 17, 1, 9]), np.array([12, 17, 30, 9])
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    H, d = 2, 8
    gen = torch.Generator().manual_seed(29)
    q = torch.randn(int(lq.sum()), H, d, generator=gen).bfloat16()
    k = torch.randn(int(lk.sum()), H, d, generator=gen).bfloat16()
    v = torch.randn(int(lk.sum()), H, d, generator=gen).bfloat16()
    F0 = np.concatenate([np.arange(n) + 1 + (m - n) for n, m in zip(lq, lk)]).astype(np.int32)
    w = W.Workload("varlen_qk", W.LAYOUT_THD, len(lq), int(lq.max()), int(lk.max()), H, H, d, q, k, v,
                   0.35, "intervals", mask_func=F0[None, None, :], cu_seqlens_q=cq, cu_seqlens_k=ck)
    for b in range(len(lq)):
        n, m = int(lq[b]), int(lk[b])
        vis = np.arange(m)[None, :] < (np.arange(n) + 1 + (m - n))[:, None]
        for h in range(H):
            o, lse = A.attention_rows(w, b, h)
            qh = q[cq[b]:cq[b + 1], h].double().numpy()
            kh = k[ck[b]:ck[b + 1], h].double().numpy()
            vh = v[ck[b]:ck[b + 1], h].double().numpy()
            assert np.allclose(o, _sdpa(qh, kh, vh, bool_mask=vis, scale=0.35), atol=1e-12)
            assert np.allclose(lse, _lse_ref(qh, kh, vis, 0.35), atol=1e-12)
