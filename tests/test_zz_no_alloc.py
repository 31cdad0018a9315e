"""pisa_select_noalloc: the selection entry point for callers that cannot give the library
device memory at call time (an engine that owns a fixed device arena and allows no
allocation while serving, or a plugin host without an allocator). It must return what
pisa_select returns with a caller workspace, call after call, although every call reuses
the same fixed scratch array inside the library.

Collected last on purpose; it needs no state from other tests."""
import ctypes

import pytest
import torch

import pisa_synth as syn
import pyramid_top_selection_gb300 as pisa
from pyramid_top_selection_gb300 import _pisa
from _parity import SCORE_ATOL

pytestmark = pytest.mark.gpu


def _entry():
    f = pisa.lib().pisa_select_noalloc
    f.argtypes = [ctypes.POINTER(_pisa.Shape)] + [ctypes.c_void_p] * 6
    f.restype = ctypes.c_int
    return f


def _run_both(f, B, N, Hq, Hkv, d, K, seed):
    dev = torch.device("cuda", 0)
    Q, Kt, _ = syn.make_prefill(B, N, Hq, Hkv, d, C=64, seed=seed, needles=True, device=dev)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, 64, K, qtile=4)
    pyr = pisa.build_pyramid(Kt, shape)
    idx_ref, score_ref = pisa.select(Q, Kt, pyr, shape)            # caller-provided workspace
    idx = torch.full_like(idx_ref, -7)
    score = torch.full_like(score_ref, float("nan"))
    stream = torch.cuda.current_stream(dev).cuda_stream
    rc = f(ctypes.byref(shape), Q.data_ptr(), Kt.data_ptr(), pyr.data_ptr(), idx.data_ptr(),
           score.data_ptr(), stream)
    assert rc == 0, pisa.lib().pisa_last_error().decode()
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_ref)
    torch.testing.assert_close(score, score_ref, atol=SCORE_ATOL, rtol=0)


def test_noalloc_select_matches_workspace_select_on_consecutive_calls():
    f = _entry()
    # two calls in a row on different inputs and shapes share the one scratch array
    _run_both(f, 1, 4096, 16, 2, 128, 16, seed=0)
    _run_both(f, 2, 3000, 8, 2, 64, 8, seed=1)


def test_noalloc_select_rejects_shapes_beyond_its_scratch():
    f = _entry()
    shape = pisa.make_shape(1, 1 << 20, 16, 2, 128, 64, 16)
    A = 1 << 20     # never dereferenced: the size check comes first
    rc = f(ctypes.byref(shape), A, A, A, A, None, None)
    assert rc == _pisa.PISA_EUNSUPPORTED
    assert "scratch" in pisa.lib().pisa_last_error().decode()
