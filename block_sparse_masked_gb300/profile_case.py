"""Run a few forward (and optionally backward) launches of one workload, for
use under a profiler: ``python -m block_sparse_masked_gb300.profile_case
--workload video_block_sparse --heads 4 --launches 4``.

The workload is the seeded synthetic one of ``workloads.py``; ``--heads``
keeps its per-head structure with fewer heads so that a capture holds a few
GB at most.  ``--workload decode_paged`` runs fa_decode_paged instead
(``--heads`` then sets the number of sequences).  The plan is built once; the launches follow it back to back;
the last one is timed with CUDA events and printed (not a benchmark number:
see ``bench.py``).
"""
from __future__ import annotations

import argparse

import torch

from . import build as fb


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="video_block_sparse")
    ap.add_argument("--heads", type=int, default=0, help="0: the workload's own head count")
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--backward", action="store_true", help="also run fa_bwd after each forward")
    args = ap.parse_args()
    fb.build()
    import block_sparse_masked_gb300 as fa
    from . import runner
    from . import workloads as W

    if args.workload == "decode_paged":
        w = W.decode_paged(0, **({"B": args.heads} if args.heads > 0 else {}))
        dp = runner.decode_to_device(w)
        plan = runner.decode_plan(dp)
        for _ in range(args.launches):
            runner.decode(dp, plan)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        runner.decode(dp, plan)
        e1.record()
        torch.cuda.synchronize()
        print(f"decode_paged B={w.B}: last call {e0.elapsed_time(e1):.4f} ms, "
              f"device error flags {fa.fa_device_error_flags()}")
        plan.free()
        return
    kw = {}
    if args.heads > 0:
        kw["H"] = args.heads
    w = W.make(args.workload, 0, **kw)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp, backward=args.backward)
    dout = torch.randn(dp.q.shape, device="cuda").to(torch.bfloat16) if args.backward else None
    for _ in range(args.launches):
        runner.forward(dp, plan)
        if args.backward:
            runner.backward(dp, plan, dout)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    runner.forward(dp, plan)
    if args.backward:
        runner.backward(dp, plan, dout)
    e1.record()
    torch.cuda.synchronize()
    print(f"{args.workload} heads={w.Hq}: last launch(es) {e0.elapsed_time(e1):.4f} ms, "
          f"device error flags {fa.fa_device_error_flags()}")
    plan.free()


if __name__ == "__main__":
    main()
