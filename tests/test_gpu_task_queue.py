"""The forward schedules its tasks on the device (one CTA per task; running
CTAs take over CTAs that have not started), with no state kept between
launches.  Repeated launches on one stream, launches on two streams at once,
the two forward kernels one after the other on the same stream, and a graph
replayed several times must all give the output of the first launch bit for
bit (each task is computed by one CTA in a fixed order, so the forward is
deterministic), and that output must match the oracle: a task handled twice
or not at all would show."""
import math

import pytest
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import runner
from block_sparse_masked_gb300 import workloads as W

import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    PT.ensure_built()


def _problem(seed, mods=False):
    gen = torch.Generator().manual_seed(seed)
    B, S, H, d = 1, 700, 4, 128
    q, k, v = (torch.randn(B, S, H, d, generator=gen).bfloat16() for _ in range(3))
    mf = W.random_intervals(seed, B, S, S, 3, 1)
    w = W.Workload("queue", W.LAYOUT_BSHD, B, S, S, H, H, d, q, k, v, 1 / math.sqrt(d), "intervals",
                   mask_func=mf)
    if mods:  # score mods route to the one-tile kernel; plain intervals to the two-tile one
        w.softcap = 20.0
    return w


def _rows(w):
    return {(0, h): list(range(0, w.Sq, 7)) for h in range(w.Hq)}


@pytest.mark.parametrize("mods", [False, True])
def test_repeated_launches_one_stream(mods):
    w = _problem(21, mods)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    ref = dp.o.clone()
    PT.check_rows(w, dp.o, dp.lse, _rows(w))
    for _ in range(5):
        dp.o.zero_()
        runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert torch.equal(dp.o, ref)
    assert fa.fa_device_error_flags() == 0
    plan.free()


def test_both_kernels_alternating_on_one_stream():
    wa, wb = _problem(22, False), _problem(23, True)
    da, db = runner.to_device(wa), runner.to_device(wb)
    pa, pb = runner.build_plan(da), runner.build_plan(db)
    runner.forward(da, pa)
    runner.forward(db, pb)
    torch.cuda.synchronize()
    ra, rb = da.o.clone(), db.o.clone()
    for _ in range(3):
        da.o.zero_()
        db.o.zero_()
        runner.forward(da, pa)
        runner.forward(db, pb)
    torch.cuda.synchronize()
    assert torch.equal(da.o, ra) and torch.equal(db.o, rb)
    PT.check_rows(wa, da.o, da.lse, _rows(wa))
    PT.check_rows(wb, db.o, db.lse, _rows(wb))
    pa.free()
    pb.free()


def test_two_streams_at_once():
    w = _problem(24)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    ref = dp.o.clone()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1, o2 = torch.empty_like(dp.o), torch.empty_like(dp.o)
    l1, l2 = torch.empty_like(dp.lse), torch.empty_like(dp.lse)
    for _ in range(4):
        for s, o, l in ((s1, o1, l1), (s2, o2, l2)):
            with torch.cuda.stream(s):
                fa.fa_fwd(plan, dp.q, dp.k, dp.v, o, l, dp.geom, w.scale, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(o1, ref) and torch.equal(o2, ref)
    assert fa.fa_device_error_flags() == 0
    plan.free()


def test_graph_replays():
    w = _problem(25)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    ref = dp.o.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fa.fa_fwd(plan, dp.q, dp.k, dp.v, dp.o, dp.lse, dp.geom, w.scale, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        dp.o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dp.o, ref)
    # an ordinary launch after the capture
    dp.o.zero_()
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert torch.equal(dp.o, ref)
    assert fa.fa_device_error_flags() == 0
    del g
    plan.free()
