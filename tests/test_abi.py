"""C-ABI contract tests that need no GPU: the library loads, exports every symbol that
include/pisa.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import pyramid_top_selection_gb300 as pisa
from pyramid_top_selection_gb300 import _pisa
from oracle import pisa_oracle as po

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pisa.h")).read()
    return sorted(set(re.findall(r"\b(pisa_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    L = pisa.lib()
    decl = _declared()
    assert len(decl) >= 12
    for name in decl:
        assert hasattr(L, name), name
    assert set(decl) == set(_pisa.EXPORTS)
    hdr = int(re.search(r"#define PISA_VERSION (\d+)", open(os.path.join(ROOT, "include", "pisa.h")).read()).group(1))
    assert L.pisa_version() == hdr == _pisa.ABI_VERSION


@pytest.mark.parametrize("N,C", [(4096, 64), (65536, 64), (262144, 64), (1, 64), (65, 64), (130, 64)])
def test_layout_matches_oracle_geometry(N, C):
    n, off, nodes = pisa.pyramid_layout(pisa.make_shape(1, N, 4, 1, 64, C, 8))
    sizes = po.level_sizes(N, C)
    assert n == len(sizes)
    assert nodes == sum(sizes)
    assert off == [sum(sizes[:l]) for l in range(len(sizes))]


def _rc(fn, *args):
    rc = fn(*args)
    return rc, pisa.lib().pisa_last_error().decode()


def test_host_validation_before_any_cuda_call():
    L = pisa.lib()
    A = 1 << 20        # fake, 16-byte aligned addresses: must never be dereferenced
    good = pisa.make_shape(1, 4096, 4, 1, 64, 64, 8)
    ws = pisa.workspace_size(good, _pisa.OP_SELECT)
    cases = [
        (pisa.make_shape(1, 4096, 4, 1, 96, 64, 8), _pisa.PISA_EUNSUPPORTED, "head dim"),
        (pisa.make_shape(1, 4096, 4, 1, 64, 32, 8), _pisa.PISA_EUNSUPPORTED, "leaf block"),
        (pisa.make_shape(1, 4096, 4, 1, 64, 64, 8, g=3), _pisa.PISA_EUNSUPPORTED, "fan-out"),
        (pisa.make_shape(1, 4096, 4, 1, 64, 64, 33), _pisa.PISA_EUNSUPPORTED, "K=33"),
        (pisa.make_shape(1, 4096, 6, 4, 64, 64, 8), _pisa.PISA_EINVAL, "multiple"),
        (pisa.make_shape(1, 4096, 32, 1, 64, 64, 8), _pisa.PISA_EUNSUPPORTED, "GQA group"),
        (pisa.make_shape(0, 4096, 4, 1, 64, 64, 8), _pisa.PISA_EINVAL, "positive"),
        (pisa.make_shape(1, 4096, 4, 1, 64, 64, 8, scale=-1.0), _pisa.PISA_EINVAL, "scale"),
    ]
    for shape, code, text in cases:
        rc, msg = _rc(L.pisa_select, ctypes.byref(shape), A, A, A, A, None, None, A, 1 << 40, None)
        assert rc == code and text in msg, (rc, msg)
    rc, msg = _rc(L.pisa_select, ctypes.byref(good), None, A, A, A, None, None, A, ws, None)
    assert rc == _pisa.PISA_EINVAL and "Q is NULL" in msg
    rc, msg = _rc(L.pisa_select, ctypes.byref(good), A + 8, A, A, A, None, None, A, ws, None)
    assert rc == _pisa.PISA_EINVAL and "aligned" in msg
    rc, msg = _rc(L.pisa_select, ctypes.byref(good), A, A, A, A, None, None, A, ws - 1, None)
    assert rc == _pisa.PISA_EWORKSPACE
    rc, msg = _rc(L.pisa_select, ctypes.byref(good), A, A, A, A, None, None, None, ws, None)
    assert rc == _pisa.PISA_EWORKSPACE
    rc, msg = _rc(L.pisa_select, ctypes.byref(good), A, A, A, A, None, A + 4, A, ws, None)
    assert rc == _pisa.PISA_EINVAL and "head_lse" in msg
    # the PISA-1 ablation entry validates like pisa_select (same shape checks, workspace op)
    for shape, code, text in cases[:4]:
        rc, msg = _rc(L.pisa_select_mean, ctypes.byref(shape), A, A, A, A, None, A, 1 << 40, None)
        assert rc == code and text in msg, (rc, msg)
    rc, msg = _rc(L.pisa_select_mean, ctypes.byref(good), A, A, A, None, None, A, ws, None)
    assert rc == _pisa.PISA_EINVAL and "idx is NULL" in msg
    ws_mean = pisa.workspace_size(good, _pisa.OP_SELECT_MEAN)
    assert 0 < ws_mean < ws            # no grouping and no per-head terms on the PISA-1 path
    rc, msg = _rc(L.pisa_select_mean, ctypes.byref(good), A, A, A, A, None, A, ws_mean - 1, None)
    assert rc == _pisa.PISA_EWORKSPACE
    ws_mv = pisa.workspace_size(good, _pisa.OP_SELECT_MEANVAR)
    rc, msg = _rc(L.pisa_select_meanvar, ctypes.byref(good), A, A, A, A, None, A, ws_mv - 1, None)
    assert rc == _pisa.PISA_EWORKSPACE
    rc, msg = _rc(L.pisa_select_meanvar, ctypes.byref(cases[0][0]), A, A, A, A, None, A, 1 << 40, None)
    assert rc == _pisa.PISA_EUNSUPPORTED and "head dim" in msg
    rc, msg = _rc(L.pisa_sparse_attn_fwd, ctypes.byref(good), A, A, None, A, None, A, A, A, 1 << 40, None)
    assert rc == _pisa.PISA_EINVAL and "V is NULL" in msg
    rc, msg = _rc(L.pisa_build_pyramid, None, A, A, None)
    assert rc == _pisa.PISA_EINVAL
    dshape = pisa.make_decode_shape(2, 1000, 8, 2, 128, 64, 16)
    rc, msg = _rc(L.pisa_decode_step, ctypes.byref(dshape), A, A, A, A, A, A, A, A, A, None, None, None)
    assert rc == _pisa.PISA_EINVAL and "status" in msg
    rc, msg = _rc(L.pisa_workspace_size, ctypes.byref(good), 7, ctypes.byref(ctypes.c_size_t()))
    assert rc == _pisa.PISA_EINVAL
    # fan-out 4: at most 64 candidates, and only where a descent is built for it
    rc, msg = _rc(L.pisa_select, ctypes.byref(pisa.make_shape(1, 4096, 4, 1, 64, 64, 17, g=4)), A, A, A, A,
                  None, None, A, 1 << 40, None)
    assert rc == _pisa.PISA_EUNSUPPORTED and "g*K" in msg
    g4 = pisa.make_shape(1, 4096, 4, 1, 64, 64, 16, g=4)
    rc, msg = _rc(L.pisa_select_mean, ctypes.byref(g4), A, A, A, A, None, A, 1 << 40, None)
    assert rc == _pisa.PISA_EUNSUPPORTED and "fan-out" in msg
    rc, msg = _rc(L.pisa_select_meanvar, ctypes.byref(g4), A, A, A, A, None, A, 1 << 40, None)
    assert rc == _pisa.PISA_EUNSUPPORTED and "fan-out" in msg
    rc, msg = _rc(L.pisa_decode_step, ctypes.byref(pisa.make_decode_shape(2, 1000, 8, 2, 128, 64, 8, g=4)),
                  A, A, A, A, A, A, A, A, A, None, A, None)
    assert rc == _pisa.PISA_EUNSUPPORTED and "fan-out" in msg
    bad = pisa.make_shape(1, 4096, 4, 1, 64, 64, 8)
    bad.per_head = 2
    rc, msg = _rc(L.pisa_select, ctypes.byref(bad), A, A, A, A, None, None, A, 1 << 40, None)
    assert rc == _pisa.PISA_EINVAL and "per_head" in msg
    # a per-head selection has Hq units: its workspace grows with Hq, its pyramid does not
    ph = pisa.make_shape(1, 4096, 8, 2, 64, 64, 8, per_head=True)
    sh = pisa.make_shape(1, 4096, 8, 2, 64, 64, 8)
    assert pisa.workspace_size(ph, _pisa.OP_SELECT) > pisa.workspace_size(sh, _pisa.OP_SELECT)
    assert pisa.pyramid_layout(ph) == pisa.pyramid_layout(sh)
    # the wait limit and the test stall are host-only settings: no CUDA call, always accepted
    assert L.pisa_set_wait_limit(5_000_000) == _pisa.PISA_OK and L.pisa_set_wait_limit(0) == _pisa.PISA_OK
    assert L.pisa_test_stall(1) == _pisa.PISA_OK and L.pisa_test_stall(0) == _pisa.PISA_OK


def test_workspace_sizes_grow_with_problem():
    a = pisa.make_shape(1, 4096, 16, 2, 128, 64, 16)
    b = pisa.make_shape(1, 65536, 16, 2, 128, 64, 16)
    for op in range(6):
        assert 256 < pisa.workspace_size(a, op) < pisa.workspace_size(b, op)   # past the status block


def test_noalloc_select_rejects_shapes_beyond_its_scratch_on_the_host():
    # The 32 MiB fixed scratch holds the selection workspace of about 63K (query, KV head) units
    # at K = 16, G = 8 and 70K at G = 4 (the header's figures). Shapes past that are rejected
    # before any CUDA call, so fake addresses are safe here; shapes within it would launch, and
    # are left to the GPU tests.
    f = pisa.lib().pisa_select_noalloc
    A = 1 << 20
    for Hq, Hkv, N in ((16, 2, 32768), (8, 2, 36864), (16, 2, 1 << 20)):
        shape = pisa.make_shape(1, N, Hq, Hkv, 128, 64, 16)
        rc = f(ctypes.byref(shape), A, A, A, A, None, None)
        assert rc == _pisa.PISA_EUNSUPPORTED, (Hq, Hkv, N, rc)
        assert "scratch" in pisa.lib().pisa_last_error().decode()
