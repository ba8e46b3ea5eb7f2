"""Failure detection without a GPU fault: a bounded in-kernel wait that can
never complete gives up, reports through the device error flags, and leaves
the context usable for the next forward."""
import numpy as np
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


def test_bounded_wait_times_out_and_context_survives():
    assert fa.fa_device_error_flags() == 0
    fa.fa_selftest_wait_timeout(1_000_000)          # 1 ms
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() & 1           # the wait gave up and said so
    assert fa.fa_device_error_flags() == 0          # reading clears the bits
    w = W.tiny_causal(0)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    rows = {(0, h): list(range(256)) for h in range(2)}
    PT.check_rows(w, dp.o, dp.lse, rows)
    plan.free()


def test_selftest_argument_range():
    with pytest.raises(fa.FaError) as ei:
        fa.fa_selftest_wait_timeout(10)
    assert ei.value.code == fa.FA_ERR_INVALID_ARG


class CountingAllocator:
    """A caller allocator (fa_allocator) on torch's caching allocator that
    counts calls, can refuse its k-th request, and checks every free."""

    def __init__(self, fail_at=None):
        self.calls = 0
        self.frees = 0
        self.fail_at = fail_at
        self.live = {}
        self.errors = []
        self.obj = fa.Allocator(self.alloc, self.free)

    def alloc(self, n, st):
        k = self.calls
        self.calls += 1
        if self.fail_at is not None and k == self.fail_at:
            return 0
        p = torch.cuda.caching_allocator_alloc(n, torch.cuda.current_device(), st)
        self.live[p] = n
        return p

    def free(self, p, n, st):
        if self.live.pop(p, None) != n:
            self.errors.append((p, n))
            return
        self.frees += 1
        torch.cuda.caching_allocator_delete(p)


def _small_block_problem():
    import math
    gen = torch.Generator().manual_seed(3)
    S, H, d = 700, 2, 64
    q, k, v = (torch.randn(1, S, H, d, generator=gen).bfloat16() for _ in range(3))
    bm = W.random_block_mask(3, H, -(-S // 64), -(-S // 64), 0.2)
    return W.Workload("blk", W.LAYOUT_BSHD, 1, S, S, H, H, d, q, k, v, 1 / math.sqrt(d), "blocks",
                      block_mask=bm, block_q=64, block_kv=64)


@pytest.mark.parametrize("kind", ["intervals", "blocks"])
def test_failing_allocator_every_call(kind):
    """"Flex Attention Mask Plan Design" §8: plan memory comes from the
    caller's allocator.  A build whose k-th allocation is refused returns
    FA_ERR_ALLOC, yields no plan and gives back everything it took, for
    every k; the build after it succeeds with the same allocator."""
    w = W.varlen_doc_causal(0) if kind == "intervals" else _small_block_problem()
    dp = runner.to_device(w)
    ok = CountingAllocator()
    plan = runner.build_plan(dp, allocator=ok.obj)
    torch.cuda.synchronize()
    n_calls = ok.calls
    assert n_calls >= 2 and len(ok.live) == 1 and not ok.errors  # the workspace went back
    plan.free()
    torch.cuda.synchronize()
    assert not ok.live and ok.frees == n_calls and not ok.errors
    for k in range(n_calls):
        bad = CountingAllocator(fail_at=k)
        with pytest.raises(fa.FaError) as ei:
            runner.build_plan(dp, allocator=bad.obj)
        assert ei.value.code == fa.FA_ERR_ALLOC
        torch.cuda.synchronize()
        assert bad.calls == k + 1 and not bad.live and bad.frees == k and not bad.errors
    # the library is still usable, and the next build succeeds
    plan = runner.build_plan(dp, allocator=ok.obj)
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    plan.free()


def test_caller_allocator_on_the_block_sparse_workload():
    """The whole 24-head, 32768-token block-sparse plan built from a caller
    allocator is the same plan (bit for bit) as one from the library's pool,
    and the forward over it gives bit-identical O and LSE."""
    w = W.video_block_sparse(0)
    dp = runner.to_device(w)
    ref = runner.build_plan(dp)
    runner.forward(dp, ref)
    o_ref, l_ref = dp.o.clone(), dp.lse.clone()
    al = CountingAllocator()
    plan = runner.build_plan(dp, allocator=al.obj)
    dp.o.zero_()
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    a, b = fa.fa_plan_export(ref), fa.fa_plan_export(plan)
    for key in a:
        assert np.array_equal(a[key], b[key]), key
    assert torch.equal(dp.o, o_ref) and torch.equal(dp.lse, l_ref)
    ref.free()
    plan.free()
    torch.cuda.synchronize()
    assert not al.live and not al.errors and al.frees == al.calls
