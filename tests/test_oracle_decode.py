"""Pins for oracle.decode (decoding over a paged KV cache).

* identity paging with the causal decode mask equals torch's
  scaled_dot_product_attention (fp64) over the sequence's keys, and with
  the sliding-window + sink mask equals SDPA under a boolean mask that the
  test builds from the window's definition;
* a random page permutation gives the same rows as pages laid out in order
  (paging relocates keys; it changes nothing else);
* a decode row equals the training-time oracle row of the same sequence at
  position q = offset (the mask converted for inference is the training
  mask at the absolute position);
* the endpoint rows of the decode generator are the training generator's
  rows at q + offset;
* a sequence whose query sees no key gives O = 0 and LSE = -inf."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from block_sparse_masked_gb300 import workloads as W
from oracle import attention as A
from oracle import decode as D


def _contiguous(seed, B, Hq, Hk, d, k_lens, page_size, q_len=1, mask="causal", window=64, sink=4,
                permute=False):
    """A decode workload whose sequence b's logical K/V are also returned
    contiguously, laid out in pages either in order or permuted."""
    w = W.decode_paged(seed, B=B, Hq=Hq, Hk=Hk, d=d, page_size=page_size, q_len=q_len, mask=mask,
                       window=window, sink=sink, k_lens=k_lens, spare_pages=3)
    gen = torch.Generator().manual_seed(seed + 100)
    logical = [(torch.randn((int(n), Hk, d), generator=gen).bfloat16(),
                torch.randn((int(n), Hk, d), generator=gen).bfloat16()) for n in w.k_lens]
    rng = np.random.default_rng(seed + 7)
    order = rng.permutation(w.num_pages) if permute else np.arange(w.num_pages)
    table = np.full_like(w.page_table, -1)
    kc = torch.full_like(w.k_cache, float("nan"))
    vc = torch.full_like(w.v_cache, float("nan"))
    at = 0
    for b, (kl, vl) in enumerate(logical):
        n = int(w.k_lens[b])
        for pj in range(-(-n // page_size)):
            pg = int(order[at])
            at += 1
            table[b, pj] = pg
            r = slice(pj * page_size, min(n, (pj + 1) * page_size))
            kc[pg, :r.stop - r.start] = kl[r]
            vc[pg, :r.stop - r.start] = vl[r]
    w.page_table, w.k_cache, w.v_cache = table, kc, vc
    return w, logical


def _sdpa(q, k, v, scale, bool_mask=None):
    qt, kt, vt = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    am = None if bool_mask is None else torch.from_numpy(bool_mask)[None, None]
    return F.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, scale=scale)[0, 0].numpy()


@pytest.mark.parametrize("page_size", [16, 64, 128])
@pytest.mark.parametrize("q_len", [1, 3])
def test_identity_paging_causal_equals_sdpa(page_size, q_len):
    w, logical = _contiguous(1, B=3, Hq=4, Hk=2, d=16, k_lens=[5, 130, 300], page_size=page_size,
                             q_len=q_len)
    for b in range(w.B):
        n = int(w.k_lens[b])
        kb, vb = (A.as_f64(t) for t in logical[b])
        # query row i sits at absolute position n - q_len + i and sees keys <= it
        causal = np.arange(n)[None, :] <= (n - q_len + np.arange(q_len))[:, None]
        for h in range(w.Hq):
            o, _ = D.decode_rows(w, b, h)
            q = A.as_f64(w.q[b * q_len:(b + 1) * q_len, h])
            ref = _sdpa(q, kb[:, h // 2], vb[:, h // 2], w.scale, causal)
            np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_identity_paging_sliding_window_equals_sdpa():
    window, sink = 40, 3
    w, logical = _contiguous(2, B=2, Hq=2, Hk=1, d=8, k_lens=[200, 37], page_size=16, mask="sliding",
                             window=window, sink=sink)
    for b in range(w.B):
        n = int(w.k_lens[b])
        pos = n - 1
        j = np.arange(n)
        vis = ((j < sink) | ((j > pos - window) & (j <= pos)))[None, :]
        kb, vb = (A.as_f64(t) for t in logical[b])
        for h in range(w.Hq):
            o, lse = D.decode_rows(w, b, h)
            q = A.as_f64(w.q[b:b + 1, h])
            np.testing.assert_allclose(o, _sdpa(q, kb[:, 0], vb[:, 0], w.scale, vis), rtol=0, atol=1e-12)
            s = torch.from_numpy(q @ kb[:, 0].T * w.scale).masked_fill(~torch.from_numpy(vis), -math.inf)
            np.testing.assert_allclose(lse, torch.logsumexp(s, dim=1).numpy(), rtol=0, atol=1e-12)


def test_page_permutation_changes_nothing():
    a, _ = _contiguous(3, B=3, Hq=4, Hk=4, d=16, k_lens=[100, 64, 257], page_size=32, permute=False)
    b, _ = _contiguous(3, B=3, Hq=4, Hk=4, d=16, k_lens=[100, 64, 257], page_size=32, permute=True)
    assert not np.array_equal(a.page_table, b.page_table)
    oa, la = D.decode_full(a)
    ob, lb = D.decode_full(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


@pytest.mark.parametrize("mask,mods", [("causal", False), ("sliding", False), ("causal", True),
                                       ("sliding", True)])
def test_decode_row_equals_training_row_at_offset(mask, mods):
    window, sink = 50, 4
    w, logical = _contiguous(4, B=2, Hq=2, Hk=2, d=16, k_lens=[180, 77], page_size=16, mask=mask,
                             window=window, sink=sink)
    if mods:  # the score_mod converted for inference: ALiBi at the absolute position, softcap
        w.softcap, w.alibi_slopes = 3.0, W.alibi_slopes(w.Hq)
    for b in range(w.B):
        n = int(w.k_lens[b])
        kb, vb = logical[b]
        # the same sequence as a training problem: Q row `offset` holds the decode query
        q = torch.zeros((1, n, w.Hq, w.d), dtype=torch.bfloat16)
        q[0, n - 1] = w.q[b]
        if mask == "causal":
            mf = W.causal_rows(np.arange(n))
        else:
            mf = W.sliding_sink_rows(np.arange(n), window, sink)
        tw = W.Workload("train", W.LAYOUT_BSHD, 1, n, n, w.Hq, w.Hk, w.d, q, kb[None], vb[None], w.scale,
                        "intervals", mask_func=mf.astype(np.int32)[None], softcap=w.softcap,
                        alibi_slopes=w.alibi_slopes)
        for h in range(w.Hq):
            o_dec, l_dec = D.decode_rows(w, b, h)
            o_tr, l_tr = A.attention_rows(tw, 0, h, np.array([n - 1]))
            np.testing.assert_allclose(o_dec, o_tr, rtol=0, atol=1e-13)
            np.testing.assert_allclose(l_dec, l_tr, rtol=0, atol=1e-13)


def test_decode_endpoints_are_training_endpoints_at_offset():
    w = W.decode_paged(5, B=6, Hq=2, Hk=1, d=8, kmin=10, kmax=3000, mask="sliding", window=1024, sink=4)
    tr = W.sliding_sink(0, B=1, H=1, S=3000, d=8)
    for b in range(w.B):
        pos = int(w.k_lens[b]) - 1
        assert np.array_equal(w.mask_func[0][:, b], tr.mask_func[0][:, pos])
    c = W.decode_paged(5, B=6, Hq=2, Hk=1, d=8, kmin=10, kmax=3000)
    assert np.array_equal(c.mask_func[0][0], c.k_lens)  # causal: every key up to the query


def test_query_without_visible_keys():
    w, _ = _contiguous(6, B=2, Hq=2, Hk=1, d=8, k_lens=[40, 70], page_size=16, mask="sliding",
                       window=1, sink=0)
    w.mask_func = np.zeros_like(w.mask_func)  # F0 = F1 = F2 = 0: no interval is non-empty
    o, lse = D.decode_full(w)
    assert np.all(o == 0.0) and np.all(lse == -np.inf)


def test_generator_hides_unused_rows_behind_nan():
    w = W.decode_paged(7, B=4, Hq=4, Hk=2, d=16, kmin=50, kmax=300, page_size=64)
    for b in range(w.B):
        n = int(w.k_lens[b])
        last = w.page_table[b, (n - 1) // 64]
        tail = n % 64
        if tail:
            assert torch.isnan(w.k_cache[last, tail:].float()).all()
        assert np.isfinite(D.gather_logical(w.k_cache, w.page_table[b], n, 64)).all()
    o, lse = D.decode_full(w)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_per_head_masks_follow_their_own_rows():
    # mask heads = Q heads (no GQA): head h sees a window of 8 + 24 h keys
    w, logical = _contiguous(8, B=2, Hq=3, Hk=3, d=8, k_lens=[150, 61], page_size=16)
    windows = [8 + 24 * h for h in range(w.Hq)]
    pos = w.k_lens - 1
    w.mask_func = np.stack([W.sliding_sink_rows(pos, win, 0) for win in windows]).astype(np.int32)
    for b in range(w.B):
        n = int(w.k_lens[b])
        kb, vb = (A.as_f64(t) for t in logical[b])
        j = np.arange(n)
        for h in range(w.Hq):
            vis = ((j > n - 1 - windows[h]) & (j <= n - 1))[None, :]
            o, _ = D.decode_rows(w, b, h)
            ref = _sdpa(A.as_f64(w.q[b:b + 1, h]), kb[:, h], vb[:, h], w.scale, vis)
            np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_alibi_decode_equals_sdpa_with_additive_bias():
    # identity paging, causal, ALiBi only: SDPA with the bias slope * (k - pos)
    w, logical = _contiguous(9, B=2, Hq=4, Hk=2, d=16, k_lens=[150, 33], page_size=16)
    w.alibi_slopes = W.alibi_slopes(w.Hq)
    for b in range(w.B):
        n = int(w.k_lens[b])
        kb, vb = (A.as_f64(t) for t in logical[b])
        for h in range(w.Hq):
            bias = (float(w.alibi_slopes[h]) * (np.arange(n) - (n - 1)))[None, :]
            q = A.as_f64(w.q[b:b + 1, h])
            qt, kt, vt = (torch.from_numpy(x)[None, None] for x in (q, kb[:, h // 2], vb[:, h // 2]))
            ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(bias)[None, None],
                                                 scale=w.scale)[0, 0].numpy()
            o, _ = D.decode_rows(w, b, h)
            np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
