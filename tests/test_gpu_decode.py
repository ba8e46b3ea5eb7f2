"""GPU decoding over a paged KV cache (fa_decode_paged) against the fp64
oracle (oracle.decode) through the C ABI: O max-abs <= 2e-2 and |LSE error|
<= 1e-3, the forward's tolerances (bf16 inputs, P rounded to bf16, fp32
accumulation).  Unused cache rows hold NaN in every case, so a kernel that
read them would fail."""
import numpy as np
import pytest
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import runner
from block_sparse_masked_gb300 import workloads as W
from oracle import decode as OD

import parity as PT

pytestmark = pytest.mark.gpu
DEVERR_PAGE = 8


@pytest.fixture(scope="module", autouse=True)
def _built():
    PT.ensure_built()


def run(w):
    dp = runner.decode_to_device(w)
    plan = runner.decode_plan(dp)
    runner.decode(dp, plan)
    torch.cuda.synchronize()
    flags = fa.fa_device_error_flags()
    plan.free()
    return dp, flags


def check(w, dp, seqs=None, heads=None):
    o = dp.o.float().cpu().numpy()
    lse = dp.lse.cpu().numpy()
    worst_o = worst_l = 0.0
    for b in (range(w.B) if seqs is None else seqs):
        for h, (ob, lb) in OD.decode_sequence(w, b, heads).items():
            got_o, got_l = o[b, h], lse[h, b]
            if np.isinf(lb[0]):
                assert got_l == -np.inf and np.all(got_o == 0.0), (b, h)
                continue
            worst_o = max(worst_o, float(np.abs(got_o - ob[0]).max()))
            worst_l = max(worst_l, abs(float(got_l) - float(lb[0])))
    assert worst_o <= PT.O_ATOL and worst_l <= PT.LSE_ATOL, (worst_o, worst_l)


@pytest.mark.parametrize("Hq,Hk", [(8, 8), (16, 4), (32, 4), (64, 2), (64, 1)])
def test_gqa_groups(Hq, Hk):
    # N (query columns per K/V head) = 16, 16, 16, 32, 64
    w = W.decode_paged(11, B=5, Hq=Hq, Hk=Hk, kmin=1, kmax=900, page_size=64)
    dp, flags = run(w)
    assert flags == 0
    check(w, dp)


@pytest.mark.parametrize("page_size", [16, 32, 128, 256, 512])
def test_page_sizes(page_size):
    w = W.decode_paged(12, B=6, Hq=8, Hk=2, kmin=1, kmax=1300, page_size=page_size)
    dp, flags = run(w)
    assert flags == 0
    check(w, dp)


@pytest.mark.parametrize("k_lens", [[1], [127, 128, 129], [255, 256, 257, 383, 384, 385], [5000, 3, 64]])
def test_ragged_lengths(k_lens):
    w = W.decode_paged(13, B=len(k_lens), Hq=8, Hk=4, page_size=64, k_lens=k_lens)
    dp, flags = run(w)
    assert flags == 0
    check(w, dp)


@pytest.mark.parametrize("window,sink", [(1, 0), (100, 4), (1024, 4), (4096, 0)])
def test_sliding_window_skips_tiles(window, sink):
    w = W.decode_paged(14, B=8, Hq=16, Hk=4, kmin=1, kmax=6000, page_size=64, mask="sliding",
                       window=window, sink=sink)
    dp, flags = run(w)
    assert flags == 0
    check(w, dp)


def test_many_units_per_sequence():
    # long sequences on few heads: each list splits into many units, merged per row
    w = W.decode_paged(15, B=2, Hq=4, Hk=1, page_size=128, k_lens=[60000, 33333])
    dp, flags = run(w)
    assert flags == 0
    check(w, dp)


def test_per_head_masks():
    w = W.decode_paged(16, B=4, Hq=6, Hk=6, kmin=100, kmax=3000, page_size=32)
    pos = w.k_lens - 1
    w.mask_func = np.stack([W.sliding_sink_rows(pos, 16 + 200 * h, h) for h in range(w.Hq)]).astype(np.int32)
    dp, flags = run(w)
    assert flags == 0
    check(w, dp)


def test_rows_without_visible_keys():
    w = W.decode_paged(17, B=4, Hq=8, Hk=2, kmin=1, kmax=400, page_size=16, mask="sliding", window=8, sink=0)
    w.mask_func[0][:, 1] = 0  # sequence 1: every interval empty
    w.mask_func[0][:, 3] = 0
    dp, flags = run(w)
    assert flags == 0
    o, lse = dp.o.float().cpu(), dp.lse.cpu()
    for b in (1, 3):
        assert torch.all(o[b] == 0) and torch.all(torch.isneginf(lse[:, b]))
    check(w, dp)


def test_bad_page_number_is_reported():
    w = W.decode_paged(18, B=3, Hq=8, Hk=2, kmin=300, kmax=600, page_size=64)
    w.page_table[1, 2] = w.num_pages + 5  # a page the cache does not have
    dp, flags = run(w)
    assert flags & DEVERR_PAGE
    assert torch.isfinite(dp.o.float()).all()
    check(w, dp, seqs=[0, 2])  # the other sequences are unaffected


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_workload_sampled(seed):
    w = W.decode_paged(seed)
    dp, flags = run(w)
    assert flags == 0
    # every sequence, four heads spread over the K/V groups
    check(w, dp, heads=[0, 9, 18, 31])


def test_repeat_is_bitwise_stable():
    w = W.decode_paged(19, B=6, Hq=16, Hk=4, kmin=1000, kmax=9000, page_size=64)
    dp = runner.decode_to_device(w)
    plan = runner.decode_plan(dp)
    runner.decode(dp, plan)
    first_o, first_l = dp.o.clone(), dp.lse.clone()
    for _ in range(3):
        runner.decode(dp, plan)
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    assert torch.equal(first_o, dp.o) and torch.equal(first_l, dp.lse)
    plan.free()


def test_rejects_unsupported_inputs():
    w = W.decode_paged(20, B=2, Hq=4, Hk=2, kmin=100, kmax=200, page_size=64)
    dp = runner.decode_to_device(w)
    plan = runner.decode_plan(dp)
    with pytest.raises(fa.FaError):
        fa.fa_decode_paged(plan, dp.q, dp.k_cache, dp.v_cache, dp.page_table, 48, dp.o, dp.lse, dp.geom, w.scale)
    plan.free()


@pytest.mark.parametrize("softcap,alibi", [(30.0, False), (0.0, True), (20.0, True)])
def test_score_mods_at_the_absolute_position(softcap, alibi):
    w = W.decode_paged(21, B=6, Hq=16, Hk=4, kmin=1, kmax=3000, page_size=64, mask="sliding", window=1000,
                       sink=4)
    w.softcap = softcap
    if alibi:
        w.alibi_slopes = W.alibi_slopes(w.Hq)
    dp, flags = run(w)
    assert flags == 0
    check(w, dp)


def test_score_mods_on_the_decode_workload():
    w = W.decode_paged(1, B=8)
    w.softcap, w.alibi_slopes = 50.0, W.alibi_slopes(w.Hq)
    dp, flags = run(w)
    assert flags == 0
    check(w, dp, heads=[0, 13, 31])
