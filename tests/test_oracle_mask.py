"""Pins for oracle.mask: the pages' worked example, closed forms and
independent formulations of each workload's mask."""
import os

import numpy as np
import pytest

from oracle import mask as M
from block_sparse_masked_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ranges(vis_row):
    """Half-open [a, b) runs of True in a bool vector (pure Python)."""
    out, start = [], None
    for i, x in enumerate(list(vis_row) + [False]):
        if x and start is None:
            start = i
        if not x and start is not None:
            out += [start, i]
            start = None
    return out


def test_worked_example_golden():
    # "Flex Attention Mask Plan Design" §2: endpoints [32, 64, 96] -> [0,32) U [64,96)
    with open(os.path.join(GOLDEN, "worked_example_intervals.txt")) as f:
        line = [l for l in f if l.startswith("endpoints:")][0]
    left, right = line.split("|")
    ends = [int(x) for x in left.split(":")[1].split()]
    want = [int(x) for x in right.split(":")[1].split()]
    for k_len in (96, 97, 128, 300):
        vis = M.interval_visible(np.array(ends).reshape(-1, 1), k_len)[0]
        assert _ranges(vis) == want


@pytest.mark.parametrize("ends,k_len,want", [
    ([5, 5, 5], 10, [0, 5]),          # equal neighbours: empty middle interval
    ([0, 0, 0], 10, []),              # nothing visible
    ([0], 10, []),
    ([10], 10, [0, 10]),              # whole row
    ([3, 3, 7], 10, [0, 7]),          # gap of width 0 merges the intervals
    ([2, 4, 6, 8, 10], 10, [0, 2, 4, 6, 8, 10]),
    ([0, 4, 4], 10, []),              # second interval empty too
    ([0, 4, 10], 10, [4, 10]),
])
def test_closed_form_intervals(ends, k_len, want):
    vis = M.interval_visible(np.array(ends).reshape(-1, 1), k_len)[0]
    assert _ranges(vis) == want


def test_brute_force_intervals():
    """Random endpoints against a per-element pure-Python reading of §2."""
    rng = np.random.default_rng(7)
    for nfunc in (1, 3, 5, 7):
        for _ in range(40):
            k_len = int(rng.integers(0, 40))
            F = np.sort(rng.integers(0, k_len + 1, size=nfunc))
            vis = M.interval_visible(F.reshape(-1, 1), k_len)[0]
            for kk in range(k_len):
                inside = kk < F[0]
                for i in range(1, nfunc, 2):
                    inside = inside or (F[i] <= kk < F[i + 1])
                assert vis[kk] == inside


@pytest.mark.parametrize("F,k_len", [
    ([[-1]], 8), ([[9]], 8), ([[3], [2], [5]], 8), ([[1], [2]], 8), ([[1], [2], [9]], 8)])
def test_validation_rejects(F, k_len):
    with pytest.raises(M.MaskError):
        M.validate_endpoints(np.array(F), k_len)


def test_validation_accepts_edges():
    M.validate_endpoints(np.array([[0], [0], [8]]), 8)
    M.validate_endpoints(np.array([[8], [8], [8]]), 8)


@pytest.mark.parametrize("cu_q,cu_k,tq,tk,mq,mk", [
    ([1, 5, 10], [0, 5, 10], 10, 10, 8, 8),      # does not start at 0
    ([0, 5, 9], [0, 5, 10], 10, 10, 8, 8),       # does not end at total
    ([0, 6, 5, 10], [0, 5, 6, 10], 10, 10, 8, 8),  # decreasing
    ([0, 1, 10], [0, 1, 10], 10, 10, 8, 8),      # longer than max_seqlen
    ([0, 10], [0, 5, 10], 10, 10, 10, 10),       # shapes differ
])
def test_seqlens_rejects(cu_q, cu_k, tq, tk, mq, mk):
    with pytest.raises(M.MaskError):
        M.validate_seqlens(cu_q, cu_k, tq, tk, mq, mk)


# Independent formulations of each workload's mask (FlexAttention mask_mod
# examples: causal q >= kv; sliding window; prefix_lm = or(prefix, causal);
# block masks via a Kronecker expansion of M).

def test_causal_equals_q_ge_k():
    w = W.tiny_causal(0)
    vis = M.visible_rows(w, 0, 0, np.arange(256))
    q = np.arange(256)[:, None]
    k = np.arange(256)[None, :]
    assert np.array_equal(vis, q >= k)


def test_sliding_sink_formulation():
    w = W.sliding_sink(0, B=2, H=1, S=2048, d=8)
    for b in range(2):
        vis = M.visible_rows(w, 0, b, np.arange(2048))
        q = np.arange(2048)[:, None]
        k = np.arange(2048)[None, :]
        want = (k <= q) & ((k < 4) | (q - k <= 1023))
        assert np.array_equal(vis, want)


def test_prefix_lm_formulation():
    w = W.prefix_alibi_softcap(3, B=2, H=2, S=2048, d=8, pmin=100, pmax=1500)
    for b in range(2):
        P = int(w.prefix[b])
        vis = M.visible_rows(w, 0, b, np.arange(2048))
        q = np.arange(2048)[:, None]
        k = np.arange(2048)[None, :]
        assert np.array_equal(vis, (k < P) | (q >= k))


def test_varlen_document_formulation():
    w = W.varlen_doc_causal(1, total=4096, ndocs=5, H=1, d=8, min_len=100)
    lens = np.diff(w.cu_seqlens_q)
    assert lens.sum() == 4096 and lens.min() >= 100
    doc = np.repeat(np.arange(5), lens)
    pos = np.arange(4096)
    # document mask over the packed sequence (FlexAttention document_id form) and causal
    dense = (doc[:, None] == doc[None, :]) & (pos[:, None] >= pos[None, :])
    for b in range(5):
        o = int(w.cu_seqlens_q[b])
        n = int(lens[b])
        vis = M.visible_rows(w, 0, b, np.arange(n))
        assert np.array_equal(vis, dense[o:o + n, o:o + n])


def test_block_mask_is_kron():
    bm = W.random_block_mask(5, 3, 6, 5, 0.3)
    for hm in range(3):
        full = np.kron(bm[hm], np.ones((64, 64), dtype=np.uint8)).astype(bool)
        for q_len, k_len in ((384, 320), (350, 300)):
            vis = M.block_visible_rows(bm, 64, 64, hm, np.arange(q_len), k_len)
            assert np.array_equal(vis, full[:q_len, :k_len])


def test_block_mask_has_diagonal_and_density():
    bm = W.random_block_mask(0, 24, 512, 512, 0.1)
    assert np.all(bm[:, np.arange(512), np.arange(512)] == 1)
    dens = bm.mean()
    assert 0.1 < dens < 0.105
