"""GPU backward (fa_bwd) against the fp64 oracle gradients through the C ABI.

Tolerance (the pages state none for gradients): the kernels round P and dS
to bf16 (relative 2^-9) before the accumulating products and accumulate in
fp32, so each gradient element carries an error of a few 2^-9 of the
magnitudes it sums; the test bounds the max-abs error by 2e-2 times
max(1, max |reference|) per tensor, the forward's O tolerance scaled to the
gradient's size."""
import math

import numpy as np
import pytest
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import runner
from block_sparse_masked_gb300 import workloads as W
from oracle import backward as OB

import parity as PT

pytestmark = pytest.mark.gpu
GRAD_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    PT.ensure_built()


def run_bwd(w, seed=0):
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, backward=True)
    runner.forward(dp, plan)
    gen = torch.Generator().manual_seed(1000 + seed)
    dout = torch.randn(tuple(w.q.shape), generator=gen).bfloat16()
    dq, dk, dv = runner.backward(dp, plan, dout.cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    rq, rk, rv = OB.attention_grad_full(w, dout)
    worst = {}
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        gg = g.float().cpu().double().numpy()
        assert np.all(np.isfinite(gg)), name
        err = float(np.abs(gg - r).max())
        bound = GRAD_TOL * max(1.0, float(np.abs(r).max()))
        worst[name] = (err, bound)
        assert err <= bound, f"{name}: max-abs error {err:.3e} > {bound:.3e}"
    plan.free()
    return worst


def _interval_problem(seed, B, S, H, nfunc, Hk=None, Hmask=1, Sk=None, lens=None, lens_k=None,
                      softcap=0.0, alibi=False, d=128):
    gen = torch.Generator().manual_seed(seed)
    Hk = H if Hk is None else Hk
    if lens is None:
        Sk = S if Sk is None else Sk
        q = torch.randn(B, S, H, d, generator=gen).bfloat16()
        k = torch.randn(B, Sk, Hk, d, generator=gen).bfloat16()
        v = torch.randn(B, Sk, Hk, d, generator=gen).bfloat16()
        mf = W.random_intervals(seed, B, S, Sk, nfunc, Hmask)
        w = W.Workload("rand", W.LAYOUT_BSHD, B, S, Sk, H, Hk, d, q, k, v, 1 / math.sqrt(d), "intervals",
                       mask_func=mf)
    else:
        lq = np.array(lens)
        lk = lq if lens_k is None else np.array(lens_k)
        cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
        ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
        q = torch.randn(int(lq.sum()), H, d, generator=gen).bfloat16()
        k = torch.randn(int(lk.sum()), Hk, d, generator=gen).bfloat16()
        v = torch.randn(int(lk.sum()), Hk, d, generator=gen).bfloat16()
        mf = W.random_intervals(seed, len(lq), 0, 0, nfunc, Hmask, lens_q=lq, lens_k=lk)
        w = W.Workload("rand_varlen", W.LAYOUT_THD, len(lq), int(lq.max()), int(lk.max()), H, Hk, d, q, k,
                       v, 1 / math.sqrt(d), "intervals", mask_func=mf, cu_seqlens_q=cq, cu_seqlens_k=ck)
    w.softcap = softcap
    if alibi:
        w.alibi_slopes = W.alibi_slopes(H)
    return w


@pytest.mark.parametrize("case", [
    dict(seed=1, B=2, S=300, H=2, nfunc=1),
    dict(seed=2, B=1, S=513, H=2, nfunc=3),
    dict(seed=3, B=1, S=400, H=4, Hk=2, nfunc=5, Hmask=4),        # GQA + per-head masks
    dict(seed=4, B=1, S=260, H=2, nfunc=3, Sk=700),               # Sq != Sk
    dict(seed=5, B=0, S=0, H=2, nfunc=3, lens=[70, 1, 129, 0, 300, 260]),
    dict(seed=6, B=0, S=0, H=4, Hk=2, nfunc=3, lens=[70, 300, 1, 129, 0, 260],
         lens_k=[200, 300, 517, 0, 64, 130]),                      # unequal Q/K lengths per sample
    dict(seed=7, B=1, S=384, H=2, nfunc=3, softcap=5.0),
    dict(seed=8, B=1, S=384, H=2, nfunc=3, alibi=True),
    dict(seed=9, B=2, S=333, H=2, nfunc=1, softcap=50.0, alibi=True),
])
def test_backward_random_intervals(case):
    w = _interval_problem(**case)
    print(run_bwd(w, case["seed"]))


@pytest.mark.parametrize("geom", [(64, 64), (48, 80), (128, 128)])
def test_backward_block_masks(geom):
    S, H, Hk = 700, 4, 2
    gen = torch.Generator().manual_seed(11)
    q = torch.randn(1, S, H, 128, generator=gen).bfloat16()
    k, v = (torch.randn(1, S, Hk, 128, generator=gen).bfloat16() for _ in range(2))
    bm = W.random_block_mask(11, H, -(-S // geom[0]), -(-S // geom[1]), 0.3)
    w = W.Workload("blk", W.LAYOUT_BSHD, 1, S, S, H, Hk, 128, q, k, v, 1 / math.sqrt(128), "blocks",
                   block_mask=bm, block_q=geom[0], block_kv=geom[1])
    print(run_bwd(w))


def test_backward_rows_and_keys_without_visible_pairs():
    w = _interval_problem(12, B=1, S=300, H=2, nfunc=3)
    w.mask_func[:] = 0                    # nothing visible ...
    w.mask_func[0, :, 130] = [0, 5, 7]    # ... except keys 5 and 6 for row 130
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, backward=True)
    runner.forward(dp, plan)
    dout = torch.randn(tuple(w.q.shape)).bfloat16()
    dq, dk, dv = runner.backward(dp, plan, dout.cuda())
    torch.cuda.synchronize()
    dqc, dkc, dvc = dq.float().cpu(), dk.float().cpu(), dv.float().cpu()
    assert torch.all(dqc[0, :130] == 0) and torch.all(dqc[0, 131:] == 0)
    assert torch.all(dkc[0, 7:] == 0) and torch.all(dvc[0, 7:] == 0) and torch.all(dvc[0, :5] == 0)
    rq, rk, rv = OB.attention_grad_full(w, dout)
    for g, r in ((dqc, rq), (dkc, rk), (dvc, rv)):
        assert float(np.abs(g.double().numpy() - r).max()) <= GRAD_TOL * max(1.0, float(np.abs(r).max()))
    plan.free()


def test_backward_needs_backward_plan():
    w = _interval_problem(13, B=1, S=128, H=2, nfunc=1)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    runner.forward(dp, plan)
    with pytest.raises(fa.FaError) as ei:
        runner.backward(dp, plan, torch.zeros_like(dp.q))
    assert ei.value.code == fa.FA_ERR_PLAN_MISMATCH
    plan.free()


@pytest.mark.parametrize("name", ["sliding_sink", "varlen_doc_causal", "prefix_alibi_softcap"])
def test_backward_full_workload_sampled_dq_rows(name):
    """Full-size workloads: dQ of sampled rows (tile edges, sample tails,
    random rows) against the oracle; a dQ row needs only its own visible
    keys (and the row's own softmax), so any size can be checked."""
    w = W.make(name, 0)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, backward=True)
    runner.forward(dp, plan)
    gen = torch.Generator().manual_seed(77)
    dout = torch.randn(tuple(w.q.shape), generator=gen).bfloat16()
    dq, dk, dv = runner.backward(dp, plan, dout.cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    dqc = dq.float().cpu().double().numpy()
    assert np.all(np.isfinite(dqc))
    rows = PT.sample_rows(w, 24, seed=5, heads=[0, w.Hq - 1])
    worst = 0.0
    for (b, h), rr in rows.items():
        rr = np.array(sorted(set(int(x) for x in rr)))
        ref = OB.dq_rows(w, b, h, rr, dout)
        q_off = w.sample_bounds()[b][0]
        got = dqc[b, rr, h, :] if w.layout == 0 else dqc[q_off + rr, h, :]
        worst = max(worst, float(np.abs(got - ref).max()) / max(1.0, float(np.abs(ref).max())))
    assert worst <= GRAD_TOL, worst
    plan.free()
