"""Pins for oracle.plan: brute force on tiny inputs, E(M) preservation under
several physical tilings, class invariants and the schedule order."""
import functools

import numpy as np
import pytest

from oracle import mask as M
from oracle import plan as P
from block_sparse_masked_gb300 import workloads as W


def _tiny_interval_workload(seed, B, S, nfunc, Hmask=1, H=2, varlen_lens=None):
    import torch
    if varlen_lens is None:
        mf = W.random_intervals(seed, B, S, S, nfunc, Hmask)
        w = W.Workload("fuzz", W.LAYOUT_BSHD, B, S, S, H, H, 8,
                       torch.zeros(B, S, H, 8, dtype=torch.bfloat16),
                       torch.zeros(B, S, H, 8, dtype=torch.bfloat16),
                       torch.zeros(B, S, H, 8, dtype=torch.bfloat16), 1.0, "intervals",
                       mask_func=mf)
        return w
    lens = np.array(varlen_lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tot = int(lens.sum())
    mf = W.random_intervals(seed, len(lens), 0, 0, nfunc, Hmask, lens_q=lens, lens_k=lens)
    mx = int(lens.max())
    return W.Workload("fuzz_varlen", W.LAYOUT_THD, len(lens), mx, mx, H, H, 8,
                      torch.zeros(tot, H, 8, dtype=torch.bfloat16),
                      torch.zeros(tot, H, 8, dtype=torch.bfloat16),
                      torch.zeros(tot, H, 8, dtype=torch.bfloat16), 1.0, "intervals",
                      mask_func=mf, cu_seqlens_q=cu, cu_seqlens_k=cu.copy())


def _brute_plan(w, T_Q, T_KV):
    """Per-element Python loops: classes, ascending CSR lists and payload words."""
    out = {}
    for hm in range(w.Hmask):
        for b, (qo, ql, ko, kl) in enumerate(w.sample_bounds()):
            vis = M.visible_rows(w, hm, b, np.arange(ql))
            nq, nk = -(-ql // T_Q), -(-kl // T_KV)
            for i in range(nq):
                plist, flist, pays = [], [], []
                for j in range(nk):
                    cnt, inb = 0, 0
                    words = []
                    for r in range(T_Q):
                        row_words = []
                        for wd in range(-(-T_KV // 32)):
                            word = 0
                            for l in range(32):
                                c = wd * 32 + l
                                qq, kk = i * T_Q + r, j * T_KV + c
                                if c < T_KV and qq < ql and kk < kl:
                                    inb += 1
                                    if vis[qq, kk]:
                                        cnt += 1
                                        word |= 1 << l
                            row_words.append(word)
                        words.append(row_words)
                    if cnt == 0:
                        continue
                    if cnt == T_Q * T_KV:
                        flist.append(j)
                    else:
                        plist.append(j)
                        pays.append(words)
                out[(hm, b, i)] = (plist, flist, pays)
    return out


@pytest.mark.parametrize("T", [(64, 64), (128, 128), (64, 32)])
@pytest.mark.parametrize("case", [
    dict(seed=1, B=1, S=200, nfunc=1),
    dict(seed=2, B=2, S=130, nfunc=3),
    dict(seed=3, B=1, S=257, nfunc=5, Hmask=2),
    dict(seed=4, B=0, S=0, nfunc=3, varlen_lens=[70, 1, 129, 64]),
])
def test_plan_matches_brute_force(T, case):
    w = _tiny_interval_workload(**case)
    p = P.build_plan(w, *T)
    ref = _brute_plan(w, *T)
    for hm in range(w.Hmask):
        for r in range(p.rows):
            b, m = int(p.row_batch[r]), int(p.row_mblock[r])
            plist, flist, pays = ref[(hm, b, m)]
            f = hm * p.rows + r
            pi = p.partial_idx[p.partial_offset[f]:p.partial_offset[f + 1]].tolist()
            fi = p.full_idx[p.full_offset[f]:p.full_offset[f + 1]].tolist()
            assert pi == plist and fi == flist
            got = p.payload[p.partial_offset[f]:p.partial_offset[f + 1]].tolist()
            assert got == pays
    assert p.header[:3] == [p.rows, p.partial_idx.size, p.full_idx.size]


@pytest.mark.parametrize("T", [(64, 64), (128, 128), (128, 64), (64, 128), (32, 96)])
@pytest.mark.parametrize("geom", [(64, 64), (48, 80), (128, 32)])
def test_block_plan_preserves_EM(T, geom):
    """"A plan built from block geometry reproduces E(M) exactly under any physical tiling."""
    import torch
    BQ, BKV = geom
    S = 700
    nbq, nbk = -(-S // BQ), -(-S // BKV)
    bm = W.random_block_mask(11, 2, nbq, nbk, 0.3)
    w = W.Workload("blk", W.LAYOUT_BSHD, 1, S, S, 2, 2, 8,
                   torch.zeros(1, S, 2, 8), torch.zeros(1, S, 2, 8), torch.zeros(1, S, 2, 8),
                   1.0, "blocks", block_mask=bm, block_q=BQ, block_kv=BKV)
    p = P.build_plan(w, *T)
    for hm in range(2):
        rec = P.visible_from_plan(p, hm, 0, S, S)
        em = np.kron(bm[hm], np.ones((BQ, BKV), np.uint8))[:S, :S].astype(bool)
        assert np.array_equal(rec, em)


@pytest.mark.parametrize("geom", [(256, 256), (128, 384), (384, 128)])
@pytest.mark.parametrize("S", [1024, 1000])
def test_refined_geometry_has_no_partial_tile_away_from_tails(geom, S):
    """Logical blocks that are whole multiples of the 128x128 tile (the
    Refined mapping of "Decoupling Logical Masks from GPU Execution for
    Dynamic Block-Sparse Attention", physical tiles inside logical blocks):
    every tile lies inside one block, so it is empty or fully visible; only
    a tile that the sequence end cuts can be partial, and the plan still
    reproduces E(M)."""
    import torch
    BQ, BKV = geom
    nbq, nbk = -(-S // BQ), -(-S // BKV)
    bm = W.random_block_mask(17, 2, nbq, nbk, 0.4)
    w = W.Workload("blk", W.LAYOUT_BSHD, 1, S, S, 2, 2, 8,
                   torch.zeros(1, S, 2, 8), torch.zeros(1, S, 2, 8), torch.zeros(1, S, 2, 8),
                   1.0, "blocks", block_mask=bm, block_q=BQ, block_kv=BKV)
    p = P.build_plan(w)
    last_q, last_k = (S - 1) // 128, (S - 1) // 128
    tail = S % 128 != 0
    for hm in range(2):
        for r in range(p.rows):
            f = hm * p.rows + r
            for kt in p.partial_idx[p.partial_offset[f]:p.partial_offset[f + 1]].tolist():
                assert tail and (r == last_q or kt == last_k), (hm, r, kt)
        em = np.kron(bm[hm], np.ones((BQ, BKV), np.uint8))[:S, :S].astype(bool)
        assert np.array_equal(P.visible_from_plan(p, hm, 0, S, S), em)
    if not tail:
        assert p.partial_idx.size == 0 and p.full_idx.size > 0


def test_interval_plan_preserves_visibility_and_counts():
    w = _tiny_interval_workload(seed=9, B=0, S=0, nfunc=5, Hmask=2,
                                varlen_lens=[300, 5, 128, 257])
    p = P.build_plan(w, 128, 128)
    total = 0
    for hm in range(2):
        for b, (qo, ql, ko, kl) in enumerate(w.sample_bounds()):
            vis = M.visible_rows(w, hm, b, np.arange(ql))
            assert np.array_equal(P.visible_from_plan(p, hm, b, ql, kl), vis)
            total += int(vis.sum())
    # sum over full tiles of T_Q*T_KV plus payload popcount == visible pairs
    pop = int(np.unpackbits(p.payload.view(np.uint8)).sum())
    assert p.full_idx.size * 128 * 128 + pop == total == p.visible_pairs


def test_each_tile_exactly_one_class_and_tail_never_full():
    w = _tiny_interval_workload(seed=12, B=0, S=0, nfunc=3,
                                varlen_lens=[129, 256, 200, 1, 383])
    p = P.build_plan(w, 128, 128)
    for r in range(p.rows):
        b = int(p.row_batch[r])
        pi = set(p.partial_idx[p.partial_offset[r]:p.partial_offset[r + 1]].tolist())
        fi = set(p.full_idx[p.full_offset[r]:p.full_offset[r + 1]].tolist())
        assert not (pi & fi)
        assert all(0 <= j < p.k_tiles[b] for j in pi | fi)
        kl = w.sample_bounds()[b][3]
        if p.row_qvalid[r] < 128:
            assert not fi
        for j in fi:
            assert (j + 1) * 128 <= kl
        lst = p.partial_idx[p.partial_offset[r]:p.partial_offset[r + 1]].tolist()
        assert lst == sorted(lst)


def test_halves_match_payload_columns():
    w = _tiny_interval_workload(seed=13, B=0, S=0, nfunc=5, varlen_lens=[300, 129, 257])
    p = P.build_plan(w, 128, 128)
    for e in range(p.partial_idx.size):
        words = p.payload[e]
        want = int(np.any(words[:, :2] != 0)) | (int(np.any(words[:, 2:] != 0)) << 1)
        assert p.halves[e] == want and want != 0


def test_payload_bit_layout_single_element():
    """One visible element at (row 5, col 70) of a tile lands in word 2, bit 6."""
    import torch
    S = 128
    ends = np.zeros((1, 3, S), np.int32)
    ends[0, :, :] = 0
    ends[0, 1, 5] = 70     # row 5: [0,0) U [70,71)
    ends[0, 2, 5] = 71
    ends[0, 1, :] = np.maximum(ends[0, 1, :], ends[0, 0, :])
    ends[0, 2, :] = np.maximum(ends[0, 2, :], ends[0, 1, :])
    w = W.Workload("one", W.LAYOUT_BSHD, 1, S, S, 1, 1, 8, torch.zeros(1, S, 1, 8),
                   torch.zeros(1, S, 1, 8), torch.zeros(1, S, 1, 8), 1.0, "intervals",
                   mask_func=ends)
    p = P.build_plan(w)
    assert p.partial_idx.tolist() == [0] and p.full_idx.size == 0
    want = np.zeros((128, 4), np.uint32)
    want[5, 2] = 1 << 6
    assert np.array_equal(p.payload[0], want)
    assert p.halves.tolist() == [2]  # column 70 is in the upper half


def test_malformed_inputs_raise():
    w = _tiny_interval_workload(seed=1, B=1, S=64, nfunc=3)
    w.mask_func[0, 1, 10] = w.mask_func[0, 0, 10] - 1 if w.mask_func[0, 0, 10] > 0 else 65
    with pytest.raises(M.MaskError):
        P.build_plan(w)
    w = _tiny_interval_workload(seed=1, B=1, S=64, nfunc=1)
    w.mask_func[0, 0, 3] = 65
    with pytest.raises(M.MaskError):
        P.build_plan(w)


def test_schedule_brute_force_comparator():
    w = _tiny_interval_workload(seed=21, B=0, S=0, nfunc=3, Hmask=2, H=2,
                                varlen_lens=[300, 40, 520])
    p = P.build_plan(w, 128, 128)
    # enumerate tasks and compare with a comparator written from the §4.8 rules
    items = []
    for r in range(p.rows):
        for h in range(2):
            c = int(p.partial_count[h, r] + p.full_count[h, r])
            items.append((int(p.row_batch[r]), h, int(p.row_mblock[r]), c, int(p.row_qvalid[r])))

    def cmp(a, b):
        if (a[3] > 0) != (b[3] > 0):
            return -1 if a[3] > 0 else 1
        if a[3] > 0:
            sa, sb = a[0] * 2 + a[1], b[0] * 2 + b[1]
            if sa != sb:
                return -1 if sa < sb else 1
            if a[3] != b[3]:
                return -1 if a[3] > b[3] else 1
        ta, tb = (a[0], a[1], a[2]), (b[0], b[1], b[2])
        return (ta > tb) - (ta < tb)

    items.sort(key=functools.cmp_to_key(cmp))
    want = [(m, h, b, qv) for (b, h, m, c, qv) in items]
    assert [tuple(x) for x in p.work_desc.tolist()] == want


def _longest_first_violations(order, cost):
    """Pairs (i, j), i < j, of the order that break "each task before every
    cheaper task and before the later tasks of equal cost"."""
    bad = []
    for i in range(len(order)):
        for j in range(i + 1, len(order)):
            a, c = order[i], order[j]
            if not (cost[a] > cost[c] or (cost[a] == cost[c] and a < c)):
                bad.append((i, j))
    return bad


def _task_costs(p, Hmask):
    cost = []
    for (m, h, b, _) in p.work_desc.tolist():
        hm, r = (0 if Hmask == 1 else h), int(p.cu_q_rows[b]) + m
        cost.append(int(p.partial_count[hm, r] + p.full_count[hm, r]))
    return cost


@pytest.mark.parametrize("seed,Hmask", [(21, 2), (22, 1)])
def test_consumer_order_is_longest_first(seed, Hmask):
    """The consumer order lists every work_desc position once, each task
    before every task of smaller cost and before the tasks of equal cost
    that come later in work_desc (checked pair by pair from the task costs
    read off the CSR counts, not through a sort)."""
    w = _tiny_interval_workload(seed=seed, B=0, S=0, nfunc=3, Hmask=Hmask, H=2,
                                varlen_lens=[300, 40, 520, 129])
    p = P.build_plan(w, 128, 128)
    T = p.work_desc.shape[0]
    assert sorted(p.lpt.tolist()) == list(range(T))
    cost = _task_costs(p, Hmask)
    assert len(set(cost)) > 2  # the ordering is exercised
    assert _longest_first_violations(p.lpt.tolist(), cost) == []


def test_consumer_order_pin_catches_planted_mistakes():
    """Orders with a plausible mistake fail the pin: equal costs in reverse
    work_desc order (an unstable or descending-index sort), and costs
    ascending."""
    w = _tiny_interval_workload(seed=21, B=0, S=0, nfunc=3, Hmask=2, H=2,
                                varlen_lens=[300, 40, 520, 129])
    p = P.build_plan(w, 128, 128)
    cost = _task_costs(p, 2)
    assert any(cost.count(c) > 1 for c in set(cost))  # ties exist
    T = len(cost)
    reversed_ties = sorted(range(T), key=lambda i: (-cost[i], -i))
    ascending = sorted(range(T), key=lambda i: (cost[i], i))
    assert _longest_first_violations(reversed_ties, cost) != []
    assert _longest_first_violations(ascending, cost) != []


def test_block_plan_consumer_order_is_work_desc_order():
    """Block-mask plans keep work_desc's section order (the identity), even
    where task costs differ, so each (sample, K/V head) section's tasks stay
    together."""
    w = _small_block_workload(H=2, S=1000, BQ=64, BKV=64, seed=5, density=0.3)
    p = P.build_plan(w, 128, 128)
    T = p.work_desc.shape[0]
    costs = {int(p.partial_count[h, r] + p.full_count[h, r]) for h in range(2) for r in range(p.rows)}
    assert len(costs) > 2
    assert p.lpt.tolist() == list(range(T))

def test_sequence_desc_and_workload_shapes():
    w = W.varlen_doc_causal(0)
    lens = np.diff(w.cu_seqlens_q)
    assert w.total_q == 16384 and lens.min() >= 256 and len(lens) == 8
    w2 = W.tiny_causal(0)
    p = P.build_plan(w2)
    assert p.sequence_desc.tolist() == [[0, 0, 256, 256, 0, 2, 2, 0]]
    assert p.partial_idx.tolist() == [0, 1] and p.full_idx.tolist() == [0]
    assert p.visible_pairs == 256 * 257 // 2


def test_plan_unequal_q_and_k_lengths():
    """THD with cu_seqlens_q != cu_seqlens_k (a sample without keys, one
    without queries): the plan equals the per-element brute force, its tiles
    reproduce the dense visibility, and K tiles count from each sample's keys."""
    import torch
    lq, lk = np.array([70, 150, 1, 129, 0, 60]), np.array([200, 150, 300, 0, 64, 130])
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    mf = W.random_intervals(17, len(lq), 0, 0, 3, 2, lens_q=lq, lens_k=lk)
    zq = torch.zeros(int(lq.sum()), 2, 8, dtype=torch.bfloat16)
    zk = torch.zeros(int(lk.sum()), 2, 8, dtype=torch.bfloat16)
    w = W.Workload("vqk", W.LAYOUT_THD, len(lq), int(lq.max()), int(lk.max()), 2, 2, 8, zq, zk, zk,
                   1.0, "intervals", mask_func=mf, cu_seqlens_q=cq, cu_seqlens_k=ck)
    for T in ((64, 64), (128, 128)):
        p = P.build_plan(w, *T)
        ref = _brute_plan(w, *T)
        for hm in range(2):
            for r in range(p.rows):
                b, m = int(p.row_batch[r]), int(p.row_mblock[r])
                plist, flist, pays = ref[(hm, b, m)]
                f = hm * p.rows + r
                assert p.partial_idx[p.partial_offset[f]:p.partial_offset[f + 1]].tolist() == plist
                assert p.full_idx[p.full_offset[f]:p.full_offset[f + 1]].tolist() == flist
                assert p.payload[p.partial_offset[f]:p.partial_offset[f + 1]].tolist() == pays
            for b in range(len(lq)):
                vis = M.visible_rows(w, hm, b, np.arange(lq[b]))
                assert np.array_equal(P.visible_from_plan(p, hm, b, int(lq[b]), int(lk[b])), vis)
        assert p.rows == sum(-(-int(n) // T[0]) for n in lq)
        assert [int(x) for x in p.sequence_desc[:, 6]] == [-(-int(m) // T[1]) for m in lk]


def _small_block_workload(H, S, BQ, BKV, seed, density=0.25):
    import torch
    nbq, nbk = -(-S // BQ), -(-S // BKV)
    bm = W.random_block_mask(seed, H, nbq, nbk, density)
    z = torch.zeros(1, S, H, 0, dtype=torch.bfloat16)
    return W.Workload("blk", W.LAYOUT_BSHD, 1, S, S, H, H, 8, z, z, z, 1.0, "blocks",
                      block_mask=bm, block_q=BQ, block_kv=BKV)


def _assert_same_plan(a, b):
    for f in ("rows", "Hmask", "visible_pairs"):
        assert getattr(a, f) == getattr(b, f), f
    for f in ("cu_q_rows", "k_tiles", "row_batch", "row_mblock", "row_qvalid", "partial_count",
              "full_count", "partial_offset", "full_offset", "partial_idx", "full_idx", "payload",
              "halves", "quads", "sequence_desc", "work_desc", "lpt"):
        x, y = getattr(a, f), getattr(b, f)
        assert x.shape == y.shape and np.array_equal(x, y), f


@pytest.mark.parametrize("kind", ["blocks", "intervals"])
def test_plan_by_heads_equals_single_process_plan(kind):
    """The per-head merge used for the large block-sparse plan gives, array
    for array, the plan built in one pass: the CSR of "Flex Attention Mask
    Plan Design" §4.6 is row-major over (mask head, row), so per-head parts
    concatenated in head order must reproduce offsets, lists, payloads and
    halves, and the §4.8 schedule built from the merged counts is the same."""
    if kind == "blocks":
        w = _small_block_workload(3, 333, 64, 64, seed=5)
    else:
        w = _tiny_interval_workload(seed=31, B=0, S=0, nfunc=3, Hmask=3, H=3,
                                    varlen_lens=[260, 1, 129, 75])
    one = P.build_plan(w)
    merged = P.build_plan_by_heads(w.mask_only(), processes=2)
    _assert_same_plan(one, merged)
    # and it is not a trivial match: the heads differ from one another
    assert one.partial_count[0].tolist() != one.partial_count[1].tolist() or \
        one.partial_idx.size != 0


def _gqa_workload(Hmask):
    import torch
    lens = np.array([300, 40, 520, 129])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tot = int(lens.sum())
    mf = W.random_intervals(23, len(lens), 0, 0, 3, Hmask, lens_q=lens, lens_k=lens)
    zq = torch.zeros(tot, 4, 0, dtype=torch.bfloat16)
    zk = torch.zeros(tot, 2, 0, dtype=torch.bfloat16)
    return W.Workload("gqa", W.LAYOUT_THD, len(lens), int(lens.max()), int(lens.max()), 4, 2, 8,
                      zq, zk, zk, 1.0, "intervals", mask_func=mf, cu_seqlens_q=cu,
                      cu_seqlens_k=cu.copy())


@pytest.mark.parametrize("Hmask", [1, 4])
def test_schedule_gqa_sections(Hmask):
    """§4.8 order with grouped-query heads (Hq=4, Hk=2): the L2 section of a
    task is (sample, K/V head) and Q heads 2g and 2g+1 share K/V head g, so
    they must be interleaved by cost inside one section; a `sample*Hq + head`
    section would split them.  The expected order is built here by explicit
    grouping: sections in (sample, K/V head) order, inside each the positive
    cost tasks by descending cost with ties in (head, m_block) order, then all
    zero-cost tasks in (sample, head, m_block) order."""
    w = _gqa_workload(Hmask)
    p = P.build_plan(w, 128, 128)
    Hq, Hk = 4, 2
    cost = {}
    for r in range(p.rows):
        b, m = int(p.row_batch[r]), int(p.row_mblock[r])
        for h in range(Hq):
            hm = 0 if Hmask == 1 else h
            cost[(b, h, m)] = (int(p.partial_count[hm, r] + p.full_count[hm, r]), int(p.row_qvalid[r]))
    want = []
    for b in range(w.B):
        for g in range(Hk):
            sect = [(c, h, m, qv) for (bb, h, m), (c, qv) in cost.items()
                    if bb == b and h // (Hq // Hk) == g and c > 0]
            by_cost = {}
            for c, h, m, qv in sect:
                by_cost.setdefault(c, []).append((h, m, qv))
            for c in sorted(by_cost, reverse=True):
                for h, m, qv in sorted(by_cost[c]):
                    want.append((m, h, b, qv))
    zero = sorted((b, h, m, qv) for (b, h, m), (c, qv) in cost.items() if c == 0)
    want += [(m, h, b, qv) for (b, h, m, qv) in zero]
    got = [tuple(x) for x in p.work_desc.tolist()]
    assert got == want
    # both Q heads of a group appear inside one section run
    first = got[:sum(1 for v in cost.values() if v[0] > 0)]
    secs = [(b, h // 2) for (m, h, b, qv) in first]
    assert secs == sorted(secs)
    assert any(h % 2 == 1 for (m, h, b, qv) in first) and any(h % 2 == 0 for (m, h, b, qv) in first)


@pytest.mark.parametrize("T", [(128, 128), (64, 32)])
@pytest.mark.parametrize("kind", ["intervals", "blocks64", "blocks48"])
def test_quads_brute_force(T, kind):
    """Quadrant bits of every partial entry by per-element loops: quadrant
    (a, s) covers tile rows [a*T_Q/2, (a+1)*T_Q/2) and columns
    [s*T_KV/2, (s+1)*T_KV/2); bit 2a+s says one of its elements is visible,
    bit 4+2a+s that all are (elements outside the sample are not visible)."""
    if kind == "intervals":
        w = _tiny_interval_workload(seed=19, B=0, S=0, nfunc=1, varlen_lens=[300, 129, 70, 257])
        # causal rows: diagonal tiles have a full lower-left quadrant
        for b, (qo, ql, _, _) in enumerate(w.sample_bounds()):
            w.mask_func[0, 0, qo:qo + ql] = np.arange(1, ql + 1)
    elif kind == "blocks64":
        w = _small_block_workload(2, 333, 64, 64, seed=7, density=0.3)
    else:
        w = _small_block_workload(2, 301, 48, 80, seed=8, density=0.3)
    T_Q, T_KV = T
    p = P.build_plan(w, T_Q, T_KV)
    bounds = w.sample_bounds()
    seen_full = seen_partial_quad = 0
    for hm in range(w.Hmask):
        for r in range(p.rows):
            b, m = int(p.row_batch[r]), int(p.row_mblock[r])
            _, ql, _, kl = bounds[b]
            vis = M.visible_rows(w, hm, b, np.arange(ql))
            f = hm * p.rows + r
            for e in range(int(p.partial_offset[f]), int(p.partial_offset[f + 1])):
                j = int(p.partial_idx[e])
                want = 0
                for a in range(2):
                    for s_ in range(2):
                        anyv, allv = False, True
                        for rr in range(a * T_Q // 2, (a + 1) * T_Q // 2):
                            for cc in range(s_ * T_KV // 2, (s_ + 1) * T_KV // 2):
                                q, k = m * T_Q + rr, j * T_KV + cc
                                v = q < ql and k < kl and bool(vis[q, k])
                                anyv |= v
                                allv &= v
                        want |= (int(anyv) << (2 * a + s_)) | (int(allv) << (4 + 2 * a + s_))
                assert int(p.quads[e]) == want, (hm, r, j)
                seen_full += bin(want >> 4).count("1")
                seen_partial_quad += bin((want & 15) & ~(want >> 4)).count("1")
    assert p.partial_idx.size > 0
    if T == (128, 128):  # both kinds of quadrant occur at the consumer's tile
        assert seen_full > 0 and seen_partial_quad > 0
