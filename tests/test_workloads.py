"""Pins for the seeded input generators that both the CUDA path and the
oracle consume: values the workload statements fix in closed form."""
import math

import numpy as np

from block_sparse_masked_gb300 import workloads as W


def test_alibi_slopes_closed_form_for_32_heads():
    """The prefix-LM + ALiBi + softcap workload states slope_h = 2^(-8(h+1)/32)
    for 0-based h over 32 heads, i.e. 2^(-(h+1)/4): every fourth head is an
    exact power of two (1/2 at h=3 down to 1/256 at h=31), and consecutive
    slopes differ by the factor 2^(-1/4)."""
    s = W.alibi_slopes(32)
    assert s.dtype == np.float32 and s.shape == (32,)
    for j in range(1, 9):
        assert s[4 * j - 1] == np.float32(0.5 ** j)          # exact powers of two
    ratio = 2.0 ** -0.25
    for h in range(31):
        assert abs(float(s[h + 1]) / float(s[h]) - ratio) < 2e-7
    assert abs(float(s[0]) - 0.8408964152537145) < 1e-7      # 2^(-1/4)
    w = W.prefix_alibi_softcap(0, B=1, H=32, S=64, pmin=8, pmax=16)
    assert np.array_equal(w.alibi_slopes, s)


def test_video_block_mask_density_and_diagonal():
    """Block pairs active i.i.d. at 10% plus the diagonal, regenerated per seed."""
    m0 = W.random_block_mask(0, 24, 512, 512, 0.1)
    m1 = W.random_block_mask(1, 24, 512, 512, 0.1)
    assert m0.shape == (24, 512, 512) and m0.dtype == np.uint8
    assert np.all(m0[:, np.arange(512), np.arange(512)] == 1)
    off = ~np.eye(512, dtype=bool)
    dens = m0[:, off].mean()
    assert abs(dens - 0.1) < 3 * math.sqrt(0.1 * 0.9 / m0[:, off].size) + 1e-4
    assert not np.array_equal(m0, m1)


def test_doc_lengths_sum_and_minimum():
    for seed in (0, 1, 2):
        L = W.doc_lengths(seed)
        assert L.sum() == 16384 and L.min() >= 256 and L.size == 8
