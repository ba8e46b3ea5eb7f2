"""The allocation-free sizing entry point (fa_plan_header_noalloc).

It serves callers that cannot allocate device memory at all, for example
code inside a memory manager that owns every device byte and must not
re-enter cudaMalloc, or latency-bound loops where allocation calls (which may
synchronise the device) are forbidden.  It must return the same 8-value
header as the allocating build (fa_plan_build_intervals), call after call,
using only its fixed per-device scratch array.  This file is collected last
so that a failure here cannot hide the results of the other tests.
"""
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


def _cases():
    out = [W.make("tiny_causal", 0).mask_only(), W.make("sliding_sink", 0).mask_only(),
           W.make("varlen_doc_causal", 0).mask_only()]
    lens = np.array([70, 1, 129, 0, 300, 260])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tot = int(lens.sum())
    mf = W.random_intervals(5, len(lens), 0, 0, 5, 2, lens_q=lens, lens_k=lens)
    z = torch.zeros(tot, 2, 0, dtype=torch.bfloat16)
    out.append(W.Workload("fuzz", W.LAYOUT_THD, len(lens), 300, 300, 2, 2, 64, z, z, z, 1.0,
                          "intervals", mask_func=mf, cu_seqlens_q=cu, cu_seqlens_k=cu.copy()))
    # per-sample Q and K lengths that differ, with a sample without keys and
    # one without queries
    lq, lk = np.array([70, 150, 1, 129, 0, 60]), np.array([200, 150, 300, 0, 64, 130])
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    mf = W.random_intervals(17, len(lq), 0, 0, 3, 2, lens_q=lq, lens_k=lk)
    zq = torch.zeros(int(lq.sum()), 2, 0, dtype=torch.bfloat16)
    zk = torch.zeros(int(lk.sum()), 2, 0, dtype=torch.bfloat16)
    out.append(W.Workload("vqk", W.LAYOUT_THD, len(lq), int(lq.max()), int(lk.max()), 2, 2, 64,
                          zq, zk, zk, 1.0, "intervals", mask_func=mf, cu_seqlens_q=cq,
                          cu_seqlens_k=ck))
    return out


@pytest.mark.parametrize("case", range(5))
def test_noalloc_header_matches_allocating_build(case):
    w = _cases()[case]
    if w.d == 0:
        w.d = 128 if w.name != "tiny_causal" else 64
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    want = fa.fa_plan_info_get(plan)["header"]
    plan.free()
    Hm, nf = w.mask_func.shape[:2]
    for _ in range(2):  # two calls in a row share (and reuse) the scratch array
        out = torch.full((8,), -7, dtype=torch.int64, device="cuda")
        fa.fa_plan_header_noalloc(dp.geom, dp.mask, Hm, nf, out)
        torch.cuda.synchronize()
        assert out.cpu().tolist() == list(want)


def test_noalloc_reports_bad_endpoints_in_header():
    w = _cases()[3]
    w.d = 64
    mf = w.mask_func.copy()
    mf[0, 2, 10] = 10_000              # beyond the sample's k_len
    bad = W.Workload(**{**w.__dict__, "mask_func": mf})
    dp = runner.to_device(bad)
    with pytest.raises(fa.FaError) as ei:
        runner.build_plan(dp)
    assert ei.value.code == fa.FA_ERR_INVALID_MASK
    out = torch.zeros(8, dtype=torch.int64, device="cuda")
    fa.fa_plan_header_noalloc(dp.geom, dp.mask, 2, 5, out)
    torch.cuda.synchronize()
    assert int(out[7]) & 1
    # the next call starts from a clean error word
    good = runner.to_device(w)
    fa.fa_plan_header_noalloc(good.geom, good.mask, 2, 5, out)
    torch.cuda.synchronize()
    assert int(out[7]) == 0


def test_noalloc_rejects_scratch_beyond_limit():
    # 32 mask heads x 4096 Q tiles x 8 words of 32 K tiles: about 10 MiB of scratch
    g = fa.geometry(fa.FA_LAYOUT_BSHD, 32, 16384, 32768, 32, 32, 128)
    mf = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(8, dtype=torch.int64, device="cuda")
    with pytest.raises(fa.FaError) as ei:
        fa.fa_plan_header_noalloc(g, mf, 32, 1, out)
    assert ei.value.code == fa.FA_ERR_UNSUPPORTED
    assert "scratch" in fa.fa_last_error()
