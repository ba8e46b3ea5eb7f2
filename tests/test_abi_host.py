"""Host-only checks of the C ABI: the library builds, loads and exports every
entry point declared in include/fa.h, and structural argument errors are
reported before any GPU work (no GPU needed)."""
import ctypes

import pytest

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import build as fb


@pytest.fixture(scope="module")
def L():
    fb.build()
    return fa.lib()


def test_exports_every_header_symbol(L):
    names = fa.header_functions()
    assert {"fa_plan_build_intervals", "fa_plan_build_blocks", "fa_plan_free", "fa_fwd"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_version(L):
    assert "sm_103a" in fa.fa_version()


def _geom(**kw):
    base = dict(layout=fa.FA_LAYOUT_BSHD, batch=1, seqlen_q=256, seqlen_k=256, heads_q=2,
                heads_k=2, head_dim=64)
    base.update(kw)
    return fa.geometry(**base)


def _build_intervals(L, g, Hmask=1, nfunc=1, mask=1):
    out = ctypes.c_void_p()
    rc = L.fa_plan_build_intervals(ctypes.byref(g) if g is not None else None, mask, Hmask, nfunc,
                                   None, None, ctypes.byref(out))
    return rc, out.value


@pytest.mark.parametrize("kw,nfunc,Hmask,code", [
    (dict(), 2, 1, fa.FA_ERR_INVALID_ARG),              # even nfunc
    (dict(), 0, 1, fa.FA_ERR_INVALID_ARG),              # nfunc < 1
    (dict(), 1, 3, fa.FA_ERR_INVALID_ARG),              # Hmask not in {1, Hq}
    (dict(head_dim=96), 1, 1, fa.FA_ERR_UNSUPPORTED),
    (dict(heads_q=3, heads_k=2), 1, 1, fa.FA_ERR_INVALID_ARG),
    (dict(batch=0), 1, 1, fa.FA_ERR_INVALID_ARG),
    (dict(layout=7), 1, 1, fa.FA_ERR_INVALID_ARG),
    (dict(layout=fa.FA_LAYOUT_THD), 1, 1, fa.FA_ERR_INVALID_ARG),  # no cu_seqlens
    (dict(heads_q=512, heads_k=512), 1, 1, fa.FA_ERR_UNSUPPORTED),
])
def test_structural_errors(L, kw, nfunc, Hmask, code):
    rc, plan = _build_intervals(L, _geom(**kw), Hmask=Hmask, nfunc=nfunc)
    assert rc == code and plan is None
    assert fa.fa_last_error() != ""


@pytest.mark.parametrize("kw", [
    dict(batch=(1 << 26) + 1, seqlen_q=1, seqlen_k=1),               # Q tiles above 2^26
    dict(seqlen_q=1 << 30, seqlen_k=128, heads_q=256, heads_k=256),  # Q tiles x Q heads at 2^31
])
def test_size_limits_rejected_before_any_gpu_work(L, kw):
    rc, plan = _build_intervals(L, _geom(**kw))
    assert rc == fa.FA_ERR_UNSUPPORTED and plan is None
    assert "too many Q tiles" in fa.fa_last_error()


def test_null_geometry_and_mask(L):
    rc, plan = _build_intervals(L, None)
    assert rc == fa.FA_ERR_INVALID_ARG and plan is None
    rc, plan = _build_intervals(L, _geom(), mask=None)
    assert rc == fa.FA_ERR_INVALID_ARG and plan is None


def test_block_mask_needs_fixed_length(L):
    g = _geom(layout=fa.FA_LAYOUT_THD, total_q=10, total_k=10)
    g.cu_seqlens_q = g.cu_seqlens_k = 8  # never dereferenced: rejected first
    out = ctypes.c_void_p()
    rc = L.fa_plan_build_blocks(ctypes.byref(g), 1, 1, 64, 64, None, None, ctypes.byref(out))
    assert rc == fa.FA_ERR_UNSUPPORTED and out.value is None
    rc = L.fa_plan_build_blocks(ctypes.byref(_geom()), 1, 1, 0, 64, None, None, ctypes.byref(out))
    assert rc == fa.FA_ERR_INVALID_ARG


def test_fwd_and_free_argument_checks(L):
    g = _geom()
    assert L.fa_fwd(None, 16, 16, 16, 16, None, ctypes.byref(g), 1.0, None, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_plan_free(None, None) == fa.FA_OK
    info = fa.FaPlanInfo()
    assert L.fa_plan_info_get(None, 0, None, ctypes.byref(info)) == fa.FA_ERR_INVALID_ARG
    assert L.fa_plan_export(None, None) == fa.FA_ERR_INVALID_ARG


def test_struct_sizes_match_header():
    # fa_geometry: 6 int32, 2 pointers, 4 int32; fa_plan_info ends with a double
    assert ctypes.sizeof(fa.FaGeometry) == 56
    assert ctypes.sizeof(fa.FaMods) == 16
    assert ctypes.sizeof(fa.FaPlanInfo) == 144
    assert ctypes.sizeof(fa.FaPlanHostView) == 88  # eleven array pointers
