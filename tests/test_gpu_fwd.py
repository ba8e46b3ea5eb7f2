"""GPU forward vs the fp64 oracle through the C ABI: O max-abs <= 2e-2 and
|LSE error| <= 1e-3.  Small problems are compared on every row; the full
workloads on sampled rows (tile edges, sample tails and random rows)."""
import math

import numpy as np
import pytest
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import runner
from block_sparse_masked_gb300 import workloads as W

import parity as PT
from oracle import plan as OP

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    PT.ensure_built()


def run(w):
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    return dp, plan


def all_rows(w):
    return {(b, h): list(range(ql)) for b, (_, ql, _, _) in enumerate(w.sample_bounds())
            for h in range(w.Hq) if ql > 0}


def test_tiny_causal_all_rows():
    w = W.tiny_causal(0)
    dp, plan = run(w)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


def _random_problem(seed, B, S, H, d, nfunc, Hk=None, Hmask=1, lens=None, softcap=0.0,
                    alibi=False, Sk=None):
    gen = torch.Generator().manual_seed(seed)
    Hk = H if Hk is None else Hk
    Sk = S if Sk is None else Sk
    if lens is None:
        q = torch.randn(B, S, H, d, generator=gen).bfloat16()
        k = torch.randn(B, Sk, Hk, d, generator=gen).bfloat16()
        v = torch.randn(B, Sk, Hk, d, generator=gen).bfloat16()
        mf = W.random_intervals(seed, B, S, Sk, nfunc, Hmask)
        w = W.Workload("rand", W.LAYOUT_BSHD, B, S, Sk, H, Hk, d, q, k, v, 1 / math.sqrt(d),
                       "intervals", mask_func=mf)
    else:
        lens = np.array(lens)
        tot = int(lens.sum())
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        q = torch.randn(tot, H, d, generator=gen).bfloat16()
        k = torch.randn(tot, Hk, d, generator=gen).bfloat16()
        v = torch.randn(tot, Hk, d, generator=gen).bfloat16()
        mf = W.random_intervals(seed, len(lens), 0, 0, nfunc, Hmask, lens_q=lens, lens_k=lens)
        mx = int(lens.max())
        w = W.Workload("rand_varlen", W.LAYOUT_THD, len(lens), mx, mx, H, Hk, d, q, k, v,
                       1 / math.sqrt(d), "intervals", mask_func=mf, cu_seqlens_q=cu,
                       cu_seqlens_k=cu.copy())
    w.softcap = softcap
    if alibi:
        w.alibi_slopes = W.alibi_slopes(H)
    return w


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", [
    dict(seed=1, B=2, S=300, H=2, nfunc=1),
    dict(seed=2, B=1, S=513, H=2, nfunc=3),
    dict(seed=3, B=1, S=400, H=4, Hk=2, nfunc=5, Hmask=4),       # GQA + per-head masks
    dict(seed=4, B=1, S=260, H=2, nfunc=3, Sk=700),              # Sq != Sk
    dict(seed=5, B=0, S=0, H=2, nfunc=3, lens=[70, 1, 129, 0, 300, 260]),
    dict(seed=6, B=1, S=384, H=2, nfunc=3, softcap=5.0),
    dict(seed=7, B=1, S=384, H=2, nfunc=3, alibi=True),
    dict(seed=8, B=2, S=333, H=2, nfunc=1, softcap=50.0, alibi=True),
    # the softcap's tanh is evaluated three ways, chosen per warp from the
    # largest |scale * s / softcap| it holds: below 0.125, below 0.5, above;
    # unit-variance scores put softcap 50 in the first, 12 in the second and
    # 2 in the third
    dict(seed=13, B=1, S=384, H=2, nfunc=3, softcap=12.0),
    dict(seed=14, B=1, S=384, H=2, nfunc=3, softcap=2.0, alibi=True),
])
def test_random_small_all_rows(d, case):
    w = _random_problem(d=d, **case)
    dp, plan = run(w)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


@pytest.mark.parametrize("d", [64, 128])
def test_block_mask_small_all_rows(d):
    S, BQ, BKV = 700, 48, 80
    gen = torch.Generator().manual_seed(9)
    q, k, v = (torch.randn(1, S, 2, d, generator=gen).bfloat16() for _ in range(3))
    bm = W.random_block_mask(9, 2, -(-S // BQ), -(-S // BKV), 0.25)
    w = W.Workload("blk", W.LAYOUT_BSHD, 1, S, S, 2, 2, d, q, k, v, 1 / math.sqrt(d), "blocks",
                   block_mask=bm, block_q=BQ, block_kv=BKV)
    dp, plan = run(w)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mods", [False, True])
def test_block_mask_64_blocks_all_rows(d, mods):
    # 64x64 logical blocks under 128x128 tiles at low density: most visited
    # tiles have one live 64-key half, and the forward runs two such tiles per
    # step (an odd count leaves the last one alone); two samples, GQA, a
    # ragged last tile, per-head masks, and softcap + ALiBi positions per half
    B, S, H, Hk, blk = 2, 1000, 4, 2, 64
    gen = torch.Generator().manual_seed(21)
    q = torch.randn(B, S, H, d, generator=gen).bfloat16()
    k, v = (torch.randn(B, S, Hk, d, generator=gen).bfloat16() for _ in range(2))
    nb = -(-S // blk)
    bm = W.random_block_mask(21, H, nb, nb, 0.12)
    w = W.Workload("blk64", W.LAYOUT_BSHD, B, S, S, H, Hk, d, q, k, v, 1 / math.sqrt(d), "blocks",
                   block_mask=bm, block_q=blk, block_kv=blk)
    if mods:
        w.softcap = 20.0
        w.alibi_slopes = W.alibi_slopes(H)
    dp, plan = run(w)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


def test_heads_at_limit_with_alibi():
    # 256 Q heads (the largest count the forward's parameters hold slopes
    # for) sharing 8 K/V heads, per-head masks, ALiBi slope per head
    w = _random_problem(31, B=1, S=130, H=256, Hk=8, d=64, nfunc=3, Hmask=256, alibi=True)
    dp, plan = run(w)
    rows = {(0, h): list(range(0, 130, 7)) + [127, 128, 129] for h in range(0, 256, 5)}
    PT.check_rows(w, dp.o, dp.lse, rows)
    plan.free()


@pytest.mark.parametrize("mods", [False, True])
def test_block_mask_unequal_lengths(mods):
    # Sq != Sk with ragged last tiles on both axes: one-half tiles of the
    # last K tile pair with others, rows past Sq stay out of the output
    B, Sq, Sk, H, blk, d = 2, 700, 1100, 2, 64, 128
    gen = torch.Generator().manual_seed(33)
    q = torch.randn(B, Sq, H, d, generator=gen).bfloat16()
    k, v = (torch.randn(B, Sk, H, d, generator=gen).bfloat16() for _ in range(2))
    bm = W.random_block_mask(33, H, -(-Sq // blk), -(-Sk // blk), 0.15, diagonal=False)
    w = W.Workload("blk_qk", W.LAYOUT_BSHD, B, Sq, Sk, H, H, d, q, k, v, 1 / math.sqrt(d), "blocks",
                   block_mask=bm, block_q=blk, block_kv=blk)
    if mods:
        w.softcap = 30.0
        w.alibi_slopes = W.alibi_slopes(H)
    dp, plan = run(w)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


@pytest.mark.parametrize("d,mods", [(64, False), (128, False), (128, True)])
def test_varlen_unequal_q_and_k_lengths(d, mods):
    # THD samples whose Q and K lengths differ (cu_seqlens_q != cu_seqlens_k),
    # including a sample with no keys and one with no queries; GQA; the plan
    # is compared bit-exactly and every row's output
    lq, lk = np.array([70, 300, 1, 129, 0, 260]), np.array([200, 300, 517, 0, 64, 130])
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    H, Hk = 4, 2
    gen = torch.Generator().manual_seed(41)
    q = torch.randn(int(lq.sum()), H, d, generator=gen).bfloat16()
    k = torch.randn(int(lk.sum()), Hk, d, generator=gen).bfloat16()
    v = torch.randn(int(lk.sum()), Hk, d, generator=gen).bfloat16()
    mf = W.random_intervals(41, len(lq), 0, 0, 3, 1, lens_q=lq, lens_k=lk)
    w = W.Workload("vqk", W.LAYOUT_THD, len(lq), int(lq.max()), int(lk.max()), H, Hk, d, q, k, v,
                   1 / math.sqrt(d), "intervals", mask_func=mf, cu_seqlens_q=cq, cu_seqlens_k=ck)
    if mods:
        w.softcap = 20.0
        w.alibi_slopes = W.alibi_slopes(H)
    dp, plan = run(w)
    PT.compare_plan(fa.fa_plan_export(plan), OP.build_plan(w))
    rows = {(b, h): list(range(int(lq[b]))) for b in range(len(lq)) for h in range(H) if lq[b] > 0}
    PT.check_rows(w, dp.o, dp.lse, rows)
    plan.free()


def test_rows_without_visible_keys():
    w = _random_problem(10, B=1, S=300, H=2, d=64, nfunc=3)
    w.mask_func[:] = 0               # nothing visible anywhere
    w.mask_func[0, :, 130] = [0, 5, 7]  # except two keys of row 130
    dp, plan = run(w)
    lse = dp.lse.cpu()
    assert torch.all(torch.isinf(lse[:, :130])) and torch.all(lse[:, :130] < 0)
    assert torch.all(dp.o.float().cpu()[0, :130] == 0)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


def test_plan_reuse_with_new_values_and_mismatch():
    w = _random_problem(11, B=1, S=300, H=2, d=64, nfunc=3)
    dp, plan = run(w)
    gen = torch.Generator().manual_seed(12)
    w2 = W.Workload(**{**w.__dict__, "q": torch.randn(1, 300, 2, 64, generator=gen).bfloat16(),
                       "v": torch.randn(1, 300, 2, 64, generator=gen).bfloat16()})
    dp2 = runner.to_device(w2)
    runner.forward(dp2, plan)
    torch.cuda.synchronize()
    PT.check_rows(w2, dp2.o, dp2.lse, all_rows(w2))
    g_bad = fa.geometry(fa.FA_LAYOUT_BSHD, 1, 301, 300, 2, 2, 64)
    with pytest.raises(fa.FaError) as ei:
        fa.fa_fwd(plan, dp.q, dp.k, dp.v, dp.o, dp.lse, g_bad, 0.125)
    assert ei.value.code == fa.FA_ERR_PLAN_MISMATCH
    plan.free()


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name,per_head", [
    ("sliding_sink", 256),
    ("varlen_doc_causal", 256),
    ("prefix_alibi_softcap", 128),
    ("video_block_sparse", 128),
])
def test_full_workload_sampled_rows(name, per_head, seed):
    # every head of every sample; the inputs and (block-sparse) mask of each seed
    w = W.make(name, seed)
    dp, plan = run(w)
    rows = PT.sample_rows(w, per_head, seed=seed + 1)
    eo, el = PT.check_rows(w, dp.o, dp.lse, rows)
    print(f"{name} seed {seed}: O max-abs {eo:.3e}, LSE max-abs {el:.3e}")
    plan.free()


def _block_problem(seed, B, S, H, Hk, blk_q, blk_kv, density, diagonal=True, Sk=None, d=128):
    Sk = S if Sk is None else Sk
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, S, H, d, generator=gen).bfloat16()
    k, v = (torch.randn(B, Sk, Hk, d, generator=gen).bfloat16() for _ in range(2))
    bm = W.random_block_mask(seed, H, -(-S // blk_q), -(-Sk // blk_kv), density, diagonal=diagonal)
    return W.Workload("blk", W.LAYOUT_BSHD, B, S, Sk, H, Hk, d, q, k, v, 1 / math.sqrt(d), "blocks",
                      block_mask=bm, block_q=blk_q, block_kv=blk_kv)


@pytest.mark.parametrize("geom", [(128, 64), (64, 192), (128, 128), (256, 256), (128, 384)])
def test_block_mask_64_multiple_geometries(geom):
    # logical blocks that are multiples of 64 run one 64-row half of a Q tile
    # against pairs of its live 64x64 quadrants; ragged tails on both axes
    w = _block_problem(51, B=1, S=777, H=2, Hk=2, blk_q=geom[0], blk_kv=geom[1], density=0.3, Sk=650)
    dp, plan = run(w)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


def test_block_mask_empty_block_rows():
    # whole logical block rows without an active block (no diagonal): the Q
    # halves see no key at all (O = 0, LSE = -inf), next to halves that do
    w = _block_problem(52, B=2, S=640, H=2, Hk=1, blk_q=64, blk_kv=64, density=0.2, diagonal=False)
    w.block_mask[:, 1, :] = 0      # rows 64-127 of tile 0: its second half
    w.block_mask[:, 2:4, :] = 0    # all of tile 1
    w.block_mask[0, 7, :] = 0
    dp, plan = run(w)
    lse = dp.lse.cpu()
    assert torch.all(lse[:, 64:128] == -math.inf) and torch.all(lse[:, 640 + 128:640 + 256] == -math.inf)
    assert torch.all(dp.o.float().cpu()[:, 128:256] == 0)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


def test_block_mask_growing_scores_rescale():
    # key blocks of growing magnitude along each row's list: column maxima
    # move by far more than 2^8 between steps, so the running sums and O are
    # rescaled many times inside a task
    w = _block_problem(53, B=1, S=1024, H=2, Hk=2, blk_q=64, blk_kv=64, density=0.5)
    k = w.k.float()
    for j in range(1024 // 64):
        k[:, 64 * j:64 * (j + 1)] *= 1.0 + 0.45 * j
    w.k = k.bfloat16()
    w.q = (w.q.float() * 2.0).bfloat16()
    dp, plan = run(w)
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    plan.free()


@pytest.mark.parametrize("name,choice", [
    ("blocks64", fa.FA_FWD_COARSENED),   # Coarsened 128x128 tiles instead of the Direct 64x64 steps
    ("intervals", fa.FA_FWD_ONE_TILE),   # one Q tile per task instead of two
])
def test_plan_choices_agree_with_the_oracle(name, choice):
    if name == "blocks64":
        w = _block_problem(61, B=1, S=700, H=2, Hk=1, blk_q=64, blk_kv=128, density=0.3, Sk=650)
    else:
        w = _random_problem(62, B=2, S=500, H=2, d=128, nfunc=3)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    rows = all_rows(w)
    for c in (0, choice):
        runner.forward(dp, plan, choice=c)
        torch.cuda.synchronize()
        assert fa.fa_device_error_flags() == 0
        PT.check_rows(w, dp.o, dp.lse, rows)
    plan.free()


def test_quadrant_payload_plan_forward():
    # a plan with quadrant bits only (64-aligned blocks, 64-multiple lengths)
    # runs the Direct 64x64 forward; the Coarsened choice and mods are refused
    w = _block_problem(63, B=2, S=640, H=2, Hk=1, blk_q=64, blk_kv=192, density=0.3, Sk=576)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, quadrant_payload=True)
    assert fa.fa_plan_info_get(plan)["payload_bytes"] == 0
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    PT.check_rows(w, dp.o, dp.lse, all_rows(w))
    with pytest.raises(fa.FaError):
        runner.forward(dp, plan, choice=fa.FA_FWD_COARSENED)
    with pytest.raises(fa.FaError):
        fa.fa_fwd(plan, dp.q, dp.k, dp.v, dp.o, dp.lse, dp.geom, w.scale, softcap=30.0)
    plan.free()
