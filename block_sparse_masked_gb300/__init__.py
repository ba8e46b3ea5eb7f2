"""Python binding of the C ABI in ``include/fa.h`` (argument marshalling only).

Every step of the masked-attention path runs in ``libbsm_fa.so`` (sm_103a
CUDA).  PyTorch is used only to own device memory and streams: tensors are
passed as raw device pointers.  If the shared library is missing the calls
raise; there is no other implementation to fall back to.

Names follow the C entry points:

    fa_plan_build_intervals(geom, mask_func, Hmask, nfunc) -> Plan
    fa_plan_build_blocks(geom, block_mask, Hmask, block_q, block_kv) -> Plan
    fa_plan_free(plan)
    fa_fwd(plan, q, k, v, o, lse, geom, scale, mods=None)
    fa_bwd(plan, q, k, v, o, dout, lse, dq, dk, dv, geom, scale, mods=None)
    fa_decode_paged(plan, q, k_cache, v_cache, page_table, page_size, o, lse, geom, scale)
    fa_plan_info_get(plan, count_visible=False) -> dict
    fa_plan_export(plan) -> dict of numpy arrays
    fa_last_error(), fa_device_error_flags(), fa_version()
    fa_debug_set_work_desc(plan, task, field, value)   (bounds-checked build only)
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# BSM_FA_CHECKED=1 selects the bounds-checked debug build of the same library
# (build(checked=True)); it must be chosen before the first call.
LIB_PATH = os.path.join(_HERE, "libbsm_fa_checked.so" if os.environ.get("BSM_FA_CHECKED") == "1"
                        else "libbsm_fa.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "fa.h")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_INVALID_MASK = -2
FA_ERR_INVALID_SEQLENS = -3
FA_ERR_PLAN_MISMATCH = -4
FA_ERR_ALLOC = -5
FA_ERR_CUDA = -6
FA_ERR_DEVICE_TIMEOUT = -7
FA_ERR_UNSUPPORTED = -8

FA_LAYOUT_BSHD = 0
FA_LAYOUT_THD = 1
FA_DTYPE_BF16 = 0
FA_PLAN_BACKWARD = 1
FA_PLAN_QUADRANT_PAYLOAD = 2  # block plans: keep only the quadrant bits when they are exact
FA_MOD_SOFTCAP = 1
FA_MOD_ALIBI = 2
FA_FWD_ONE_TILE = 16    # plan choice: one Q tile per task for interval plans
FA_FWD_COARSENED = 32   # plan choice: 128x128 tiles for 64-aligned block plans
FA_TILE_Q = 128
FA_TILE_K = 128
FA_PAYLOAD_WORDS = 4

_c = ctypes
_i32, _i64, _u32, _u64, _vp = _c.c_int32, _c.c_int64, _c.c_uint32, _c.c_uint64, _c.c_void_p


class FaGeometry(_c.Structure):
    _fields_ = [("layout", _i32), ("batch", _i32), ("seqlen_q", _i32), ("seqlen_k", _i32),
                ("total_q", _i32), ("total_k", _i32), ("cu_seqlens_q", _vp), ("cu_seqlens_k", _vp),
                ("heads_q", _i32), ("heads_k", _i32), ("head_dim", _i32), ("dtype", _i32)]


class FaAllocator(_c.Structure):
    _fields_ = [("alloc", _vp), ("free", _vp), ("ctx", _vp)]


class FaMods(_c.Structure):
    _fields_ = [("flags", _i32), ("softcap", _c.c_float), ("alibi_slopes", _vp)]


class FaPlanInfo(_c.Structure):
    _fields_ = [("header", _i64 * 8), ("tile_q", _i32), ("tile_k", _i32), ("mask_heads", _i32),
                ("batch", _i32), ("heads_q", _i32), ("heads_k", _i32), ("head_dim", _i32),
                ("layout", _i32), ("num_tasks", _i64), ("payload_bytes", _i64),
                ("plan_bytes", _i64), ("visible_pairs", _i64), ("signature", _u64),
                ("build_us", _c.c_double)]


class FaPlanBwdHostView(_c.Structure):
    _fields_ = [("cu_k_rows", _vp), ("partial_offset", _vp), ("partial_idx", _vp),
                ("full_offset", _vp), ("full_idx", _vp), ("payload", _vp), ("dq_write_order", _vp),
                ("dq_write_order_full", _vp)]


class FaPlanHostView(_c.Structure):
    _fields_ = [("cu_q_rows", _vp), ("sequence_desc", _vp), ("partial_offset", _vp),
                ("partial_idx", _vp), ("full_offset", _vp), ("full_idx", _vp), ("payload", _vp),
                ("work_desc", _vp), ("halves", _vp), ("quads", _vp), ("lpt", _vp)]


class FaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_LIB = None


def lib():
    """Load libbsm_fa.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m block_sparse_masked_gb300.build`"
                               + (" --checked" if LIB_PATH.endswith("_checked.so") else ""))
        L = _c.CDLL(LIB_PATH)
        P = _c.POINTER
        L.fa_plan_build_intervals.argtypes = [P(FaGeometry), _vp, _i32, _i32, P(FaAllocator), _vp,
                                              P(_vp)]
        L.fa_plan_build_blocks.argtypes = [P(FaGeometry), _vp, _i32, _i32, _i32, P(FaAllocator),
                                           _vp, P(_vp)]
        L.fa_plan_build_intervals_ex.argtypes = [P(FaGeometry), _vp, _i32, _i32, _u32, P(FaAllocator),
                                                 _vp, P(_vp)]
        L.fa_plan_build_blocks_ex.argtypes = [P(FaGeometry), _vp, _i32, _i32, _i32, _u32,
                                              P(FaAllocator), _vp, P(_vp)]
        L.fa_plan_export_backward.argtypes = [_vp, P(FaPlanBwdHostView)]
        L.fa_plan_free.argtypes = [_vp, _vp]
        L.fa_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, P(FaGeometry), _c.c_float,
                             P(FaMods), _vp]
        L.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, P(FaGeometry), _c.c_float, P(FaMods), _vp]
        L.fa_decode_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _c.c_int64, _vp, _vp,
                                      P(FaGeometry), _c.c_float, P(FaMods), _vp]
        L.fa_plan_info_get.argtypes = [_vp, _i32, _vp, P(FaPlanInfo)]
        L.fa_plan_export.argtypes = [_vp, P(FaPlanHostView)]
        L.fa_device_error_flags.argtypes = [_vp, P(_u32)]
        L.fa_plan_header_noalloc.argtypes = [P(FaGeometry), _vp, _i32, _i32, _vp, _vp]
        L.fa_selftest_wait_timeout.argtypes = [_u64, _vp]
        L.fa_debug_set_work_desc.argtypes = [_vp, _c.c_int64, _i32, _i32, _vp]
        L.fa_last_error.restype = _c.c_char_p
        L.fa_version.restype = _c.c_char_p
        for f in ("fa_plan_build_intervals", "fa_plan_build_blocks", "fa_plan_build_intervals_ex",
                  "fa_plan_build_blocks_ex", "fa_plan_export_backward", "fa_plan_free", "fa_fwd", "fa_bwd",
                  "fa_plan_info_get", "fa_plan_export", "fa_device_error_flags",
                  "fa_plan_header_noalloc", "fa_selftest_wait_timeout", "fa_debug_set_work_desc",
                  "fa_decode_paged"):
            getattr(L, f).restype = _c.c_int
        _LIB = L
    return _LIB


def header_functions() -> list:
    """Names of the entry points declared in include/fa.h."""
    src = open(HEADER_PATH).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_]+)\s*\(", src)))


def _check(code: int):
    if code != FA_OK:
        raise FaError(code, lib().fa_last_error().decode())


def fa_last_error() -> str:
    return lib().fa_last_error().decode()


def fa_version() -> str:
    return lib().fa_version().decode()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def geometry(layout: int, batch: int, seqlen_q: int, seqlen_k: int, heads_q: int, heads_k: int,
             head_dim: int, total_q: int = 0, total_k: int = 0, cu_seqlens_q=None,
             cu_seqlens_k=None) -> FaGeometry:
    """Build the fa_geometry struct; cu_seqlens_* are device int32 tensors (THD)."""
    g = FaGeometry()
    g.layout, g.batch, g.seqlen_q, g.seqlen_k = layout, batch, seqlen_q, seqlen_k
    g.total_q, g.total_k = total_q, total_k
    g.cu_seqlens_q, g.cu_seqlens_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)
    g.heads_q, g.heads_k, g.head_dim, g.dtype = heads_q, heads_k, head_dim, FA_DTYPE_BF16
    g._keep = (cu_seqlens_q, cu_seqlens_k)  # keep tensors alive with the struct
    return g


class Plan:
    """Owner of an fa_plan* handle."""

    def __init__(self, handle: int, allocator=None):
        self.handle = handle
        self.allocator = allocator  # frees the plan's memory: keep it alive with the plan

    def free(self, stream=None):
        if self.handle:
            _check(lib().fa_plan_free(self.handle, _stream_handle(stream)))
            self.handle = None

    def __del__(self):
        try:
            if self.handle and _LIB is not None:
                _LIB.fa_plan_free(self.handle, None)
        except Exception:
            pass


_ALLOC_FN = _c.CFUNCTYPE(_vp, _c.c_size_t, _vp, _vp)
_FREE_FN = _c.CFUNCTYPE(None, _vp, _c.c_size_t, _vp, _vp)


class Allocator:
    """A caller allocator for plan and workspace memory (the fa_allocator
    struct): ``alloc(bytes, stream) -> device address or 0`` and
    ``free(address, bytes, stream)``, both called in stream order.  A plan
    built with it keeps a reference, because the plan frees through it."""

    def __init__(self, alloc, free):
        self._alloc = _ALLOC_FN(lambda n, st, ctx: alloc(int(n), st or 0) or None)
        self._free = _FREE_FN(lambda ptr, n, st, ctx: free(int(ptr), int(n), st or 0))
        self.struct = FaAllocator(_c.cast(self._alloc, _vp), _c.cast(self._free, _vp), None)


def _alloc_arg(allocator: Optional[Allocator]):
    return _c.byref(allocator.struct) if allocator is not None else None


def fa_plan_build_intervals(geom: FaGeometry, mask_func, Hmask: int, nfunc: int,
                            stream=None, allocator: Optional[Allocator] = None,
                            backward: bool = False) -> Plan:
    """fa_plan_build_intervals, or fa_plan_build_intervals_ex with FA_PLAN_BACKWARD."""
    out = _vp()
    if backward:
        _check(lib().fa_plan_build_intervals_ex(_c.byref(geom), _ptr(mask_func), Hmask, nfunc,
                                                FA_PLAN_BACKWARD, _alloc_arg(allocator),
                                                _stream_handle(stream), _c.byref(out)))
    else:
        _check(lib().fa_plan_build_intervals(_c.byref(geom), _ptr(mask_func), Hmask, nfunc,
                                             _alloc_arg(allocator), _stream_handle(stream),
                                             _c.byref(out)))
    return Plan(out.value, allocator)


def fa_plan_build_blocks(geom: FaGeometry, block_mask, Hmask: int, block_q: int, block_kv: int,
                         stream=None, allocator: Optional[Allocator] = None,
                         backward: bool = False, quadrant_payload: bool = False) -> Plan:
    """fa_plan_build_blocks, or fa_plan_build_blocks_ex with FA_PLAN_BACKWARD
    and/or FA_PLAN_QUADRANT_PAYLOAD."""
    out = _vp()
    flags = (FA_PLAN_BACKWARD if backward else 0) | (FA_PLAN_QUADRANT_PAYLOAD if quadrant_payload else 0)
    if flags:
        _check(lib().fa_plan_build_blocks_ex(_c.byref(geom), _ptr(block_mask), Hmask, block_q,
                                             block_kv, flags, _alloc_arg(allocator),
                                             _stream_handle(stream), _c.byref(out)))
    else:
        _check(lib().fa_plan_build_blocks(_c.byref(geom), _ptr(block_mask), Hmask, block_q, block_kv,
                                          _alloc_arg(allocator), _stream_handle(stream),
                                          _c.byref(out)))
    return Plan(out.value, allocator)


def fa_plan_free(plan: Plan, stream=None):
    plan.free(stream)


def fa_fwd(plan: Plan, q, k, v, o, lse, geom: FaGeometry, scale: float, softcap: float = 0.0,
           alibi_slopes=None, stream=None, choice: int = 0):
    """Launch the forward; alibi_slopes is a host float32 array of heads_q
    values or None; choice holds FA_FWD_* plan-choice bits."""
    mods = None
    keep = None
    flags = int(choice)
    if softcap and softcap > 0:
        flags |= FA_MOD_SOFTCAP
    if alibi_slopes is not None:
        flags |= FA_MOD_ALIBI
        keep = np.ascontiguousarray(alibi_slopes, dtype=np.float32)
    if flags:
        mods = FaMods(flags, float(softcap or 0.0),
                      keep.ctypes.data if keep is not None else None)
    _check(lib().fa_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                        _c.byref(geom), float(scale), _c.byref(mods) if mods else None,
                        _stream_handle(stream)))


def fa_decode_paged(plan: Plan, q, k_cache, v_cache, page_table, page_size: int, o, lse,
                    geom: FaGeometry, scale: float, softcap: float = 0.0, alibi_slopes=None, stream=None):
    """Decoding over a paged KV cache (see fa.h): q [batch, heads_q, d],
    k_cache / v_cache [num_pages, page_size, heads_k, d], page_table
    [batch, pages_per_seq] int32, all on the device; score mods as fa_fwd,
    at the queries' absolute positions."""
    mods, keep = _mods(softcap, alibi_slopes)
    _check(lib().fa_decode_paged(plan.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                 int(page_table.shape[1]), int(page_size), int(k_cache.shape[0]),
                                 _ptr(o), _ptr(lse), _c.byref(geom), float(scale),
                                 _c.byref(mods) if mods else None, _stream_handle(stream)))
    del keep


def _mods(softcap, alibi_slopes):
    flags = 0
    keep = None
    if softcap and softcap > 0:
        flags |= FA_MOD_SOFTCAP
    if alibi_slopes is not None:
        flags |= FA_MOD_ALIBI
        keep = np.ascontiguousarray(alibi_slopes, dtype=np.float32)
    if not flags:
        return None, None
    return FaMods(flags, float(softcap or 0.0), keep.ctypes.data if keep is not None else None), keep


def fa_bwd(plan: Plan, q, k, v, o, dout, lse, dq, dk, dv, geom: FaGeometry, scale: float,
           softcap: float = 0.0, alibi_slopes=None, stream=None):
    """Launch the backward (plan built with backward=True); dq, dk, dv are written."""
    mods, keep = _mods(softcap, alibi_slopes)
    _check(lib().fa_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                        _ptr(dq), _ptr(dk), _ptr(dv), _c.byref(geom), float(scale),
                        _c.byref(mods) if mods else None, _stream_handle(stream)))
    del keep


def fa_plan_info_get(plan: Plan, count_visible: bool = False, stream=None) -> dict:
    info = FaPlanInfo()
    _check(lib().fa_plan_info_get(plan.handle, int(count_visible), _stream_handle(stream),
                                  _c.byref(info)))
    d = {f: getattr(info, f) for f, _ in FaPlanInfo._fields_}
    d["header"] = list(info.header)
    return d


def fa_plan_export_backward(plan: Plan) -> dict:
    """Debug snapshot of the backward views (K2Q lists, key-major payload, dQ order)."""
    info = fa_plan_info_get(plan)
    KR, KP, KF = info["header"][4], info["header"][5], info["header"][6]
    B, Hm = info["batch"], info["mask_heads"]
    arrs = {
        "cu_k_rows": np.zeros(B + 1, np.int32),
        "partial_offset": np.zeros(Hm * KR + 1, np.int32),
        "partial_idx": np.zeros(KP, np.int32),
        "full_offset": np.zeros(Hm * KR + 1, np.int32),
        "full_idx": np.zeros(KF, np.int32),
        "payload": np.zeros((KP, FA_TILE_K, FA_PAYLOAD_WORDS), np.uint32),
        "dq_write_order": np.zeros(KP, np.int32),
        "dq_write_order_full": np.zeros(KF, np.int32),
    }
    view = FaPlanBwdHostView(*[a.ctypes.data if a.size else None for a in arrs.values()])
    _check(lib().fa_plan_export_backward(plan.handle, _c.byref(view)))
    arrs["header"] = np.array(info["header"], np.int64)
    return arrs


def fa_plan_export(plan: Plan) -> dict:
    """Debug snapshot: every plan array copied to host numpy arrays."""
    info = fa_plan_info_get(plan)
    R, P, F = info["header"][0], info["header"][1], info["header"][2]
    B, Hm, T = info["batch"], info["mask_heads"], info["num_tasks"]
    arrs = {
        "cu_q_rows": np.zeros(B + 1, np.int32),
        "sequence_desc": np.zeros((B, 8), np.int32),
        "partial_offset": np.zeros(Hm * R + 1, np.int32),
        "partial_idx": np.zeros(P, np.int32),
        "full_offset": np.zeros(Hm * R + 1, np.int32),
        "full_idx": np.zeros(F, np.int32),
        # empty for a plan that keeps only quadrant bits (FA_PLAN_QUADRANT_PAYLOAD)
        "payload": np.zeros((P if info["payload_bytes"] else 0, FA_TILE_Q, FA_PAYLOAD_WORDS), np.uint32),
        "work_desc": np.zeros((T, 4), np.int32),
        "halves": np.zeros(P, np.uint8),
        "quads": np.zeros(P, np.uint8),
        "lpt": np.zeros(T, np.int32),
    }
    view = FaPlanHostView(*[a.ctypes.data if a.size else None for a in arrs.values()])
    _check(lib().fa_plan_export(plan.handle, _c.byref(view)))
    arrs["header"] = np.array(info["header"], np.int64)
    return arrs


def fa_selftest_wait_timeout(timeout_ns: int = 1_000_000, stream=None):
    """Launch the never-completing bounded wait (see fa.h); read the result with fa_device_error_flags."""
    _check(lib().fa_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream)))


def fa_debug_set_work_desc(plan: "Plan", task: int, field: int, value: int, stream=None):
    """Debug build only (see fa.h): overwrite one work_desc field of a plan."""
    _check(lib().fa_debug_set_work_desc(plan.handle, int(task), int(field), int(value), _stream_handle(stream)))


def checked_build() -> bool:
    """True when the bounds-checked debug library is the one loaded."""
    return b"bounds-checked" in lib().fa_version()


def fa_device_error_flags(stream=None) -> int:
    v = _u32(0)
    _check(lib().fa_device_error_flags(_stream_handle(stream), _c.byref(v)))
    return v.value


def fa_plan_header_noalloc(geom: FaGeometry, mask_func, Hmask: int, nfunc: int, header_out,
                           stream=None):
    """Allocation-free plan sizing: writes the 8-value header into header_out (device int64[8])."""
    _check(lib().fa_plan_header_noalloc(_c.byref(geom), _ptr(mask_func), Hmask, nfunc,
                                        _ptr(header_out), _stream_handle(stream)))
