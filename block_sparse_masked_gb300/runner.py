"""Convenience marshalling for a Workload: device copies, geometry, plan, forward.

Used by the tests, the smoke check and the benchmark.  It only moves tensors
and forwards arguments to the C ABI; all computation is in the library.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import (FA_LAYOUT_BSHD, FA_LAYOUT_THD, FaGeometry, Plan, fa_bwd, fa_decode_paged, fa_fwd,
               fa_plan_build_blocks, fa_plan_build_intervals, geometry)
from .workloads import DecodeWorkload, Workload


@dataclasses.dataclass
class DeviceProblem:
    w: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    mask: torch.Tensor
    cu_q: Optional[torch.Tensor]
    cu_k: Optional[torch.Tensor]
    geom: FaGeometry
    o: torch.Tensor
    lse: torch.Tensor


def to_device(w: Workload, device="cuda") -> DeviceProblem:
    q, k, v = (t.to(device).contiguous() for t in (w.q, w.k, w.v))
    if w.mask_kind == "intervals":
        mask = torch.from_numpy(np.ascontiguousarray(w.mask_func)).to(device)
    else:
        mask = torch.from_numpy(np.ascontiguousarray(w.block_mask)).to(device)
    cu_q = cu_k = None
    if w.layout == FA_LAYOUT_BSHD:
        g = geometry(FA_LAYOUT_BSHD, w.B, w.Sq, w.Sk, w.Hq, w.Hk, w.d)
    else:
        cu_q = torch.from_numpy(w.cu_seqlens_q.astype(np.int32)).to(device)
        cu_k = torch.from_numpy(w.cu_seqlens_k.astype(np.int32)).to(device)
        g = geometry(w.layout, w.B, w.Sq, w.Sk, w.Hq, w.Hk, w.d, total_q=w.total_q,
                     total_k=w.total_k, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    o = torch.empty_like(q)
    lse = torch.empty(w.Hq, w.total_q, dtype=torch.float32, device=device)
    return DeviceProblem(w, q, k, v, mask, cu_q, cu_k, g, o, lse)


def build_plan(dp: DeviceProblem, stream=None, allocator=None, backward: bool = False,
               quadrant_payload: bool = False) -> Plan:
    """The workload's plan; quadrant_payload asks block plans for quadrant bits only."""
    w = dp.w
    if w.mask_kind == "intervals":
        return fa_plan_build_intervals(dp.geom, dp.mask, w.mask_func.shape[0], w.mask_func.shape[1],
                                       stream=stream, allocator=allocator, backward=backward)
    return fa_plan_build_blocks(dp.geom, dp.mask, w.block_mask.shape[0], w.block_q, w.block_kv,
                                stream=stream, allocator=allocator, backward=backward,
                                quadrant_payload=quadrant_payload)


def forward(dp: DeviceProblem, plan: Plan, stream=None, choice: int = 0):
    """fa_fwd on the problem; choice: FA_FWD_* plan-choice bits."""
    w = dp.w
    fa_fwd(plan, dp.q, dp.k, dp.v, dp.o, dp.lse, dp.geom, w.scale, softcap=w.softcap,
           alibi_slopes=w.alibi_slopes, stream=stream, choice=choice)
    return dp.o, dp.lse


def backward(dp: DeviceProblem, plan: Plan, dout: torch.Tensor, stream=None):
    """Gradients for the forward outputs dp.o / dp.lse: returns (dq, dk, dv)."""
    w = dp.w
    dq, dk, dv = torch.empty_like(dp.q), torch.empty_like(dp.k), torch.empty_like(dp.v)
    fa_bwd(plan, dp.q, dp.k, dp.v, dp.o, dout, dp.lse, dq, dk, dv, dp.geom, w.scale, softcap=w.softcap,
           alibi_slopes=w.alibi_slopes, stream=stream)
    return dq, dk, dv


@dataclasses.dataclass
class DecodeProblem:
    w: DecodeWorkload
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_table: torch.Tensor
    mask: torch.Tensor
    cu_q: torch.Tensor
    cu_k: torch.Tensor
    geom: FaGeometry
    o: torch.Tensor
    lse: torch.Tensor


def decode_to_device(w: DecodeWorkload, device="cuda") -> DecodeProblem:
    """Device copies of a decode workload and its THD geometry over the
    logical keys (one query row per sequence, k_len keys each)."""
    q, kc, vc = (t.to(device).contiguous() for t in (w.q, w.k_cache, w.v_cache))
    table = torch.from_numpy(np.ascontiguousarray(w.page_table, dtype=np.int32)).to(device)
    mask = torch.from_numpy(np.ascontiguousarray(w.mask_func)).to(device)
    cu_q = torch.from_numpy(w.cu_seqlens_q).to(device)
    cu_k = torch.from_numpy(w.cu_seqlens_k).to(device)
    total_k = int(w.cu_seqlens_k[-1])
    g = geometry(FA_LAYOUT_THD, w.B, w.q_len, int(w.k_lens.max()) if w.B else 0, w.Hq, w.Hk, w.d,
                 total_q=w.B * w.q_len, total_k=total_k, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    o = torch.empty_like(q)
    lse = torch.empty(w.Hq, w.B * w.q_len, dtype=torch.float32, device=device)
    return DecodeProblem(w, q, kc, vc, table, mask, cu_q, cu_k, g, o, lse)


def decode_plan(dp: DecodeProblem, stream=None, allocator=None) -> Plan:
    """The plan of the decode rows' endpoints over the logical keys."""
    w = dp.w
    return fa_plan_build_intervals(dp.geom, dp.mask, w.mask_func.shape[0], w.mask_func.shape[1],
                                   stream=stream, allocator=allocator)


def decode(dp: DecodeProblem, plan: Plan, stream=None):
    w = dp.w
    fa_decode_paged(plan, dp.q, dp.k_cache, dp.v_cache, dp.page_table, w.page_size, dp.o, dp.lse, dp.geom,
                    w.scale, softcap=w.softcap, alibi_slopes=w.alibi_slopes, stream=stream)
    return dp.o, dp.lse
