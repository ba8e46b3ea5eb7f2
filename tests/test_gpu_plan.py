"""GPU planner vs oracle: bit-exact plans (tile classes, CSR lists, packed
predicate bits, schedule) on every workload and on random small masks, plus
the error paths of the single header readback."""
import numpy as np
import pytest
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import runner
from block_sparse_masked_gb300 import workloads as W
from oracle import plan as OP

import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    PT.ensure_built()


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name", ["tiny_causal", "sliding_sink", "varlen_doc_causal",
                                  "prefix_alibi_softcap"])
def test_plan_parity_interval_workloads(name, seed):
    w = W.make(name, seed)
    dp, plan = PT.gpu_plan(w)
    PT.compare_plan(fa.fa_plan_export(plan), OP.build_plan(w.mask_only()))
    plan.free()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_plan_parity_video_block_sparse(seed):
    # the block mask is regenerated per seed
    w = W.make("video_block_sparse", seed)
    dp, plan = PT.gpu_plan(w)
    ref = OP.build_plan_by_heads(w.mask_only(), processes=16)
    PT.compare_plan(fa.fa_plan_export(plan), ref)
    info = fa.fa_plan_info_get(plan, count_visible=True)
    assert info["visible_pairs"] == ref.visible_pairs
    plan.free()


def _interval_workload(seed, B, S, nfunc, Hmask=1, H=2, lens=None, Sk=None):
    Sk = S if Sk is None else Sk
    if lens is None:
        mf = W.random_intervals(seed, B, S, Sk, nfunc, Hmask)
        z = torch.zeros(B, S, H, 64, dtype=torch.bfloat16)
        zk = torch.zeros(B, Sk, H, 64, dtype=torch.bfloat16)
        return W.Workload("fuzz", W.LAYOUT_BSHD, B, S, Sk, H, H, 64, z, zk, zk, 1.0, "intervals",
                          mask_func=mf)
    lens = np.array(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tot = int(lens.sum())
    mf = W.random_intervals(seed, len(lens), 0, 0, nfunc, Hmask, lens_q=lens, lens_k=lens)
    z = torch.zeros(tot, H, 64, dtype=torch.bfloat16)
    mx = int(lens.max())
    return W.Workload("fuzz_varlen", W.LAYOUT_THD, len(lens), mx, mx, H, H, 64, z, z, z, 1.0,
                      "intervals", mask_func=mf, cu_seqlens_q=cu, cu_seqlens_k=cu.copy())


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("shape", [
    dict(B=1, S=300, nfunc=1), dict(B=2, S=513, nfunc=3), dict(B=1, S=1000, nfunc=5, Hmask=2),
    dict(B=3, S=128, nfunc=7), dict(B=1, S=257, nfunc=3, Sk=4500),
    dict(B=0, S=0, nfunc=3, lens=[70, 1, 129, 0, 300, 4100]),
    dict(B=0, S=0, nfunc=1, Hmask=2, lens=[256, 255, 257]),
])
def test_plan_parity_fuzz(seed, shape):
    w = _interval_workload(seed, **shape)
    dp, plan = PT.gpu_plan(w)
    PT.compare_plan(fa.fa_plan_export(plan), OP.build_plan(w))
    plan.free()


@pytest.mark.parametrize("seed", range(2))
@pytest.mark.parametrize("shape", [
    # more endpoints per row than the back stage keeps in shared memory
    dict(B=1, S=400, nfunc=17), dict(B=2, S=300, nfunc=15),
    # more samples than the front stage's last CTA has threads, empty ones at
    # both ends and in runs (rows of a sample found by binary search)
    dict(B=0, S=0, nfunc=3, lens=[0, 0] + [int(x) for x in
                                           np.random.default_rng(5).integers(0, 300, 297)] + [0, 0]),
])
def test_plan_parity_wide(seed, shape):
    w = _interval_workload(seed, **shape)
    dp, plan = PT.gpu_plan(w)
    PT.compare_plan(fa.fa_plan_export(plan), OP.build_plan(w))
    plan.free()


def _many_samples(seed, Hmask):
    """More samples than the planner stages in shared memory (1024 sample
    prefixes): the offset scans read the sample prefixes from global memory.
    Empty samples at both ends."""
    lens = [0] + [int(x) for x in np.random.default_rng(9).integers(0, 260, 1100)] + [0]
    return _interval_workload(seed, B=0, S=0, nfunc=3, Hmask=Hmask, lens=lens)


@pytest.mark.parametrize("Hmask", [1, 2])
def test_plan_parity_more_samples_than_staged(Hmask):
    w = _many_samples(3, Hmask)
    dp, plan = PT.gpu_plan(w)
    PT.compare_plan(fa.fa_plan_export(plan), OP.build_plan(w))
    plan.free()


@pytest.mark.parametrize("Hk", [32, 1])
def test_plan_parity_schedule_outside_shared_memory(Hk):
    """2,000 short samples x 32 Q heads: the schedule stage's task buckets
    (one per Q tile row and Q head) exceed its shared memory and live in the
    workspace; with 32 K/V heads (one section per sample and K/V head) its
    histogram and cursors do too."""
    lens = np.random.default_rng(12).integers(1, 129, 2000)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    mf = W.random_intervals(6, len(lens), 0, 0, 3, 1, lens_q=lens, lens_k=lens)
    z = torch.zeros(int(lens.sum()), Hk, 64, dtype=torch.bfloat16)
    zq = torch.zeros(int(lens.sum()), 32, 64, dtype=torch.bfloat16)
    mx = int(lens.max())
    w = W.Workload("short_docs", W.LAYOUT_THD, len(lens), mx, mx, 32, Hk, 64, zq, z, z, 1.0, "intervals",
                   mask_func=mf, cu_seqlens_q=cu, cu_seqlens_k=cu.copy())
    dp, plan = PT.gpu_plan(w)
    PT.compare_plan(fa.fa_plan_export(plan), OP.build_plan(w))
    plan.free()


@pytest.mark.parametrize("geom", [(64, 64), (48, 80), (128, 32), (200, 300), (16, 128), (256, 256), (128, 384)])
@pytest.mark.parametrize("S", [700, 1024])
def test_block_plan_parity_geometries(geom, S):
    BQ, BKV = geom
    bm = W.random_block_mask(S + BQ, 2, -(-S // BQ), -(-S // BKV), 0.3)
    z = torch.zeros(1, S, 2, 64, dtype=torch.bfloat16)
    w = W.Workload("blk", W.LAYOUT_BSHD, 1, S, S, 2, 2, 64, z, z, z, 1.0, "blocks",
                   block_mask=bm, block_q=BQ, block_kv=BKV)
    dp, plan = PT.gpu_plan(w)
    ref = OP.build_plan(w)
    PT.compare_plan(fa.fa_plan_export(plan), ref)
    assert fa.fa_plan_info_get(plan, count_visible=True)["visible_pairs"] == ref.visible_pairs
    plan.free()


def test_bad_endpoints_raise_without_plan():
    w = _interval_workload(1, B=1, S=300, nfunc=3)
    for row, f, val in [(5, 2, 301), (7, 0, -1), (9, 1, None)]:
        mf = w.mask_func.copy()
        if val is None:           # out of order: F1 < F0
            mf[0, 0, row], mf[0, 1, row] = 50, 10
        else:
            mf[0, f, row] = val
        w2 = W.Workload(**{**w.__dict__, "mask_func": mf})
        dp = runner.to_device(w2)
        with pytest.raises(fa.FaError) as ei:
            runner.build_plan(dp)
        assert ei.value.code == fa.FA_ERR_INVALID_MASK


@pytest.mark.parametrize("cu", [[1, 100, 200], [0, 150, 199], [0, 120, 100, 200], [0, 200, 200]])
def test_bad_seqlens_raise(cu):
    lens_ok = np.array([100, 100])
    w = _interval_workload(2, B=0, S=0, nfunc=1, lens=lens_ok)
    cu = np.array(cu, np.int32)
    B = cu.size - 1
    mx = 150
    dev_cu = torch.from_numpy(cu).cuda()
    g = fa.geometry(fa.FA_LAYOUT_THD, B, mx, mx, 2, 2, 64, total_q=200, total_k=200,
                    cu_seqlens_q=dev_cu, cu_seqlens_k=dev_cu)
    mf = torch.zeros(1, 1, 200, dtype=torch.int32, device="cuda")
    with pytest.raises(fa.FaError) as ei:
        fa.fa_plan_build_intervals(g, mf, 1, 1)
    assert ei.value.code == fa.FA_ERR_INVALID_SEQLENS


def test_plan_owns_cloned_seqlens_and_mask():
    w = _interval_workload(3, B=0, S=0, nfunc=3, lens=[300, 200])
    dp, plan = PT.gpu_plan(w)
    before = fa.fa_plan_export(plan)
    dp.cu_q.fill_(0)       # caller mutates its tensors after the build
    dp.mask.fill_(0)
    after = fa.fa_plan_export(plan)
    for k in before:
        assert np.array_equal(before[k], after[k])
    plan.free()


def test_empty_query_geometry():
    z = torch.zeros(2, 0, 2, 64, dtype=torch.bfloat16)
    zk = torch.zeros(2, 300, 2, 64, dtype=torch.bfloat16)
    w = W.Workload("empty", W.LAYOUT_BSHD, 2, 0, 300, 2, 2, 64, z, zk, zk, 1.0, "intervals",
                   mask_func=np.zeros((1, 1, 0), np.int32))
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    assert fa.fa_plan_info_get(plan)["header"][:3] == [0, 0, 0]
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    plan.free()


def test_plan_parity_schedule_counts_in_global_memory():
    # 256 K/V heads x 81 cost buckets: the schedule's counting arrays (2 x 20736
    # ints) exceed what it keeps in shared memory and live in the workspace
    B, Sq, Sk, H = 1, 128, 10240, 256
    mf = W.random_intervals(31, B, Sq, Sk, 3, 1)
    q = torch.zeros(B, Sq, H, 64, dtype=torch.bfloat16)
    kv = torch.zeros(1, 1, 1, 1, dtype=torch.bfloat16).expand(B, Sk, H, 64)
    w = W.Workload("many_heads", W.LAYOUT_BSHD, B, Sq, Sk, H, H, 64, q, kv, kv, 1.0, "intervals",
                   mask_func=mf)
    dp, plan = PT.gpu_plan(w)
    PT.compare_plan(fa.fa_plan_export(plan), OP.build_plan(w))
    plan.free()


def _quads_to_payload(quads: np.ndarray) -> np.ndarray:
    """Predicate words [P][128][4] of entries whose quadrants are each wholly
    visible or wholly masked, from their 'all visible' quadrant bits."""
    out = np.zeros((len(quads), 128, 4), np.uint32)
    for a in range(2):
        for s in range(2):
            on = ((quads >> (4 + 2 * a + s)) & 1).astype(bool)
            out[on, 64 * a:64 * (a + 1), 2 * s:2 * s + 2] = 0xFFFFFFFF
    return out


@pytest.mark.parametrize("seed", [0])
def test_quadrant_payload_plan_video_block_sparse(seed):
    # 64x64 logical blocks over S = 32768: every quadrant is all or nothing,
    # so the plan keeps the quadrant bits and no predicate words
    w = W.make("video_block_sparse", seed)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, quadrant_payload=True)
    info = fa.fa_plan_info_get(plan, count_visible=True)
    assert info["payload_bytes"] == 0
    gpu = fa.fa_plan_export(plan)
    ref = OP.build_plan_by_heads(w.mask_only(), processes=16)
    assert gpu["payload"].size == 0
    gpu["payload"] = _quads_to_payload(gpu["quads"])  # the words the quadrant bits stand for
    PT.compare_plan(gpu, ref)
    assert info["visible_pairs"] == ref.visible_pairs
    plan.free()


def test_quadrant_payload_flag_without_exact_quadrants_builds_words():
    # 64-aligned blocks but a length that is not a multiple of 64: the flag has no effect
    gen = torch.Generator().manual_seed(3)
    S = 700
    z = torch.zeros(1, S, 2, 64, dtype=torch.bfloat16)
    bm = W.random_block_mask(3, 2, -(-S // 64), -(-S // 64), 0.3)
    w = W.Workload("blk", W.LAYOUT_BSHD, 1, S, S, 2, 2, 64, z, z, z, 1.0, "blocks", block_mask=bm,
                   block_q=64, block_kv=64)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, quadrant_payload=True)
    assert fa.fa_plan_info_get(plan)["payload_bytes"] > 0
    PT.compare_plan(fa.fa_plan_export(plan), OP.build_plan(w.mask_only()))
    plan.free()
