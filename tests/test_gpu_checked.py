"""The bounds-checked debug build (libbsm_fa_checked.so, -DBSM_CHECKED).

In that build every plan-derived global index of the planner, forward and
backward kernels goes through a check against the plan's exact sizes (P, F,
tasks, heads, samples, rows; the backward view's P' and F'); a violation
sets bit 2 of the device error word and the access is redirected to index 0
(reads) or skipped (writes), so nothing faults.

test_small_cases_run_clean builds the checked library and re-runs the small
GPU parity tests in a child process that loads it (BSM_FA_CHECKED=1): every
one must pass with no error bit set (the tests assert fa_device_error_flags()
== 0 after each launch).  The tests below it run only in that child: they
overwrite the head or sample of one task of a plan's work_desc with a value
one past its range and check that each kernel family reports the violation
instead of using it."""
import math
import os
import subprocess
import sys

import pytest
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import build as fb
from block_sparse_masked_gb300 import runner
from block_sparse_masked_gb300 import workloads as W

import parity as PT

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEVERR_BOUNDS = 4
IN_CHILD = os.environ.get("BSM_FA_CHECKED") == "1"

SMALL_SUITES = ["tests/test_gpu_plan.py", "tests/test_gpu_fwd.py", "tests/test_gpu_plan_backward.py",
                "tests/test_gpu_decode.py",
                "tests/test_gpu_bwd.py", "tests/test_gpu_checked.py"]


@pytest.mark.skipif(IN_CHILD, reason="runs the child process itself")
def test_small_cases_run_clean():
    fb.build(checked=True)
    env = dict(os.environ, BSM_FA_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           *SMALL_SUITES, "-k", "not full_workload and not sampled and not video and not parity_interval_workloads"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = r.stdout[-6000:] + r.stderr[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail


def _poked(w, field, value, backward=False):
    """Build the plan of w and run the forward on it (clean), overwrite one
    task's field, then run the forward again, or only the backward; return
    the device error bits of that second run."""
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, backward=backward)
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0  # the plan as built runs clean
    fa.fa_debug_set_work_desc(plan, 0, field, value)
    if backward:
        runner.backward(dp, plan, torch.ones_like(dp.q))
    else:
        runner.forward(dp, plan)
    torch.cuda.synchronize()
    flags = fa.fa_device_error_flags()
    plan.free()
    return flags


def _intervals(d, alibi=False):
    gen = torch.Generator().manual_seed(7)
    B, S, H = 2, 384, 2
    q, k, v = (torch.randn(B, S, H, d, generator=gen).bfloat16() for _ in range(3))
    mf = W.random_intervals(7, B, S, S, 3, 1)
    w = W.Workload("poke", W.LAYOUT_BSHD, B, S, S, H, H, d, q, k, v, 1 / math.sqrt(d), "intervals",
                   mask_func=mf)
    if alibi:
        w.alibi_slopes = W.alibi_slopes(H)
    return w


def _blocks64():
    gen = torch.Generator().manual_seed(8)
    B, S, H = 1, 512, 2
    q, k, v = (torch.randn(B, S, H, 128, generator=gen).bfloat16() for _ in range(3))
    bm = W.random_block_mask(8, H, S // 64, S // 64, 0.3, diagonal=True)
    return W.Workload("poke_blk", W.LAYOUT_BSHD, B, S, S, H, H, 128, q, k, v, 1 / math.sqrt(128),
                      "blocks", block_mask=bm, block_q=64, block_kv=64)


@pytest.mark.skipif(not IN_CHILD, reason="needs the bounds-checked library (runs in the child process)")
@pytest.mark.parametrize("case", ["pair", "one_tile", "keys_major", "backward"])
@pytest.mark.parametrize("field", [1, 2])
def test_out_of_range_task_is_reported(case, field):
    PT.ensure_built()
    assert fa.checked_build()
    if case == "pair":          # interval mask, d = 128: two Q tiles per task
        w, bwd = _intervals(128), False
    elif case == "one_tile":    # score mods: one Q tile per task
        w, bwd = _intervals(128, alibi=True), False
    elif case == "keys_major":  # 64x64 logical blocks: keys-major quadrant steps
        w, bwd = _blocks64(), False
    else:                       # the dQ kernel reads work_desc too
        w, bwd = _intervals(128), True
    value = w.Hq if field == 1 else w.B
    flags = _poked(w, field, value, backward=bwd)
    assert flags & DEVERR_BOUNDS, flags
