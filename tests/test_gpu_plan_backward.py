"""GPU planner backward views (FA_PLAN_BACKWARD) against the oracle: K2Q
CSR lists, key-major predicate payload and dQ write order bit-exact, the
extended header, and the forward view unchanged ("Flex Attention Mask Plan
Design" §4.4, §4.5, §4.7)."""
import numpy as np
import pytest
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import runner
from block_sparse_masked_gb300 import workloads as W
from oracle import backward as OB
from oracle import plan as OP

import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    PT.ensure_built()


def compare_backward(gpu: dict, ref: OB.BackwardView, fwd: OP.Plan):
    hdr = gpu["header"]
    assert list(hdr[3:7]) == [fwd.rows, ref.k_rows, ref.partial_idx.size, ref.full_idx.size]
    assert hdr[7] == 0
    assert np.array_equal(gpu["cu_k_rows"], ref.cu_k_rows)
    assert np.array_equal(gpu["partial_offset"], ref.partial_offset)
    assert np.array_equal(gpu["full_offset"], ref.full_offset)
    assert np.array_equal(gpu["partial_idx"], ref.partial_idx)
    assert np.array_equal(gpu["full_idx"], ref.full_idx)
    assert np.array_equal(gpu["dq_write_order"], ref.dq_write_order)
    assert np.array_equal(gpu["dq_write_order_full"], ref.dq_write_order_full)
    assert np.array_equal(gpu["payload"], ref.payload)


def _check(w, ref=None, fwd=None):
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, backward=True)
    m = w.mask_only()
    fwd = OP.build_plan(m) if fwd is None else fwd
    ref = OB.build_backward_view(m) if ref is None else ref
    PT.compare_plan(fa.fa_plan_export(plan), fwd)
    compare_backward(fa.fa_plan_export_backward(plan), ref, fwd)
    plan.free()


@pytest.mark.parametrize("name", ["tiny_causal", "sliding_sink", "varlen_doc_causal",
                                  "prefix_alibi_softcap"])
def test_backward_view_interval_workloads(name):
    _check(W.make(name, 0))


def test_backward_view_video_block_sparse():
    w = W.make("video_block_sparse", 0).mask_only()
    _check(w, ref=OB.build_backward_view_by_heads(w, processes=16),
           fwd=OP.build_plan_by_heads(w, processes=16))


@pytest.mark.parametrize("seed", range(3))
def test_backward_view_fuzz_varlen_unequal(seed):
    lq = np.array([70, 300, 1, 129, 0, 260, 513])
    lk = np.array([200, 300, 517, 0, 64, 130, 129])
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    mf = W.random_intervals(60 + seed, len(lq), 0, 0, 5, 4, lens_q=lq, lens_k=lk)
    zq = torch.zeros(int(lq.sum()), 4, 64, dtype=torch.bfloat16)
    zk = torch.zeros(int(lk.sum()), 2, 64, dtype=torch.bfloat16)
    w = W.Workload("vqk", W.LAYOUT_THD, len(lq), int(lq.max()), int(lk.max()), 4, 2, 64, zq, zk, zk,
                   1.0, "intervals", mask_func=mf, cu_seqlens_q=cq, cu_seqlens_k=ck)
    _check(w)


@pytest.mark.parametrize("geom", [(64, 64), (48, 80), (128, 32)])
def test_backward_view_block_geometries(geom):
    S = 700
    bm = W.random_block_mask(70, 2, -(-S // geom[0]), -(-S // geom[1]), 0.3)
    z = torch.zeros(2, S, 2, 64, dtype=torch.bfloat16)
    w = W.Workload("blk", W.LAYOUT_BSHD, 2, S, S, 2, 2, 64, z, z, z, 1.0, "blocks", block_mask=bm,
                   block_q=geom[0], block_kv=geom[1])
    _check(w)


def test_forward_only_plan_has_no_backward_view():
    w = W.make("tiny_causal", 0)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    assert list(fa.fa_plan_info_get(plan)["header"][3:7]) == [0, 0, 0, 0]
    with pytest.raises(fa.FaError) as ei:
        fa.fa_plan_export_backward(plan)
    assert ei.value.code == fa.FA_ERR_INVALID_ARG
    plan.free()


def test_backward_view_more_samples_than_staged():
    """1102 samples (more sample prefixes than the front stage keeps in shared
    memory for the K2Q offset scan), empty ones at both ends."""
    lens = np.array([0] + [int(x) for x in np.random.default_rng(11).integers(0, 300, 1100)] + [0])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    mf = W.random_intervals(4, len(lens), 0, 0, 3, 1, lens_q=lens, lens_k=lens)
    z = torch.zeros(int(lens.sum()), 2, 128, dtype=torch.bfloat16)
    mx = int(lens.max())
    w = W.Workload("many", W.LAYOUT_THD, len(lens), mx, mx, 2, 2, 128, z, z, z, 1.0, "intervals",
                   mask_func=mf, cu_seqlens_q=cu, cu_seqlens_k=cu.copy())
    _check(w)
