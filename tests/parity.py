"""Shared helpers of the GPU parity tests: build + run through the C ABI,
compare with the oracle.  Tolerances are those of the masked-attention
forward for bf16 inputs with fp32 accumulation: O max-abs <= 2e-2 and
|LSE error| <= 1e-3; plans (classes, CSR, payload bits, schedule) bit-exact."""
import numpy as np
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import build as fb
from block_sparse_masked_gb300 import runner
from oracle import attention as OA
from oracle import plan as OP

O_ATOL = 2e-2
LSE_ATOL = 1e-3


def ensure_built():
    # the bounds-checked debug library when BSM_FA_CHECKED=1 selected it
    fb.build(checked=fa.LIB_PATH.endswith("_checked.so"))
    fa.lib()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def compare_plan(gpu: dict, ref: OP.Plan):
    """Bit-exact comparison of an exported GPU plan with the oracle plan."""
    assert list(gpu["header"][:3]) == ref.header[:3]
    assert gpu["header"][7] == 0
    assert np.array_equal(gpu["cu_q_rows"], ref.cu_q_rows)
    assert np.array_equal(gpu["sequence_desc"], ref.sequence_desc)
    assert np.array_equal(gpu["partial_offset"], ref.partial_offset)
    assert np.array_equal(gpu["full_offset"], ref.full_offset)
    assert np.array_equal(gpu["partial_idx"], ref.partial_idx)
    assert np.array_equal(gpu["full_idx"], ref.full_idx)
    assert np.array_equal(gpu["payload"], ref.payload)
    assert np.array_equal(gpu["halves"], ref.halves)
    assert np.array_equal(gpu["quads"], ref.quads)
    assert np.array_equal(gpu["work_desc"], ref.work_desc)
    assert np.array_equal(gpu["lpt"], ref.lpt)


def gpu_plan(w):
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    return dp, plan


def check_rows(w, o_gpu: torch.Tensor, lse_gpu: torch.Tensor, rows_by_bh: dict):
    """Compare GPU O/LSE with the oracle on {(b, h): sample-local rows}."""
    worst_o = worst_l = 0.0
    o_cpu = o_gpu.float().cpu()
    l_cpu = lse_gpu.cpu()
    for (b, h), rows in rows_by_bh.items():
        rows = np.asarray(sorted(set(int(r) for r in rows)), np.int64)
        if rows.size == 0:
            continue
        q_off, q_len, _, _ = w.sample_bounds()[b]
        o_ref, l_ref = OA.attention_rows(w, b, h, rows)
        if w.layout == 0:
            og = o_cpu[b, rows, h, :].double().numpy()
        else:
            og = o_cpu[q_off + rows, h, :].double().numpy()
        lg = l_cpu[h, q_off + rows].double().numpy()
        assert np.all(np.isfinite(og)), "non-finite O"
        fin = np.isfinite(l_ref)
        assert np.array_equal(np.isfinite(lg), fin), "LSE -inf pattern differs"
        assert np.all(lg[~fin] == -np.inf)
        assert np.all(og[~fin] == 0.0)
        eo = float(np.abs(og - o_ref).max())
        el = float(np.abs(lg[fin] - l_ref[fin]).max()) if fin.any() else 0.0
        worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    assert worst_o <= O_ATOL, f"O max-abs error {worst_o}"
    assert worst_l <= LSE_ATOL, f"LSE max-abs error {worst_l}"
    return worst_o, worst_l


def sample_rows(w, per_head: int, seed: int = 0, heads=None):
    """Rows per (sample, head): tile-edge rows, each sample's last rows and random ones."""
    rng = np.random.default_rng(seed)
    out = {}
    heads = range(w.Hq) if heads is None else heads
    for b, (q_off, q_len, _, _) in enumerate(w.sample_bounds()):
        if q_len == 0:
            continue
        edges = [r for t in range(0, q_len, 128) for r in (t, t + 127) if r < q_len]
        tail = [q_len - 1, q_len - 2] if q_len > 1 else [0]
        for h in heads:
            # up to half of the rows are tile-edge rows spread over the whole
            # sample (a different subset per head), the sample's last rows
            # always, the rest random
            n_edge = min(len(edges), per_head // 2)
            pick = rng.choice(len(edges), size=n_edge, replace=False) if n_edge else []
            chosen = [edges[i] for i in pick] + tail
            extra = rng.integers(0, q_len, size=max(0, per_head - len(chosen)))
            out[(b, h)] = chosen + list(extra)
    return out
