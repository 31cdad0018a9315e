"""ctypes binding of libpisa.so: argument marshalling only.

Every step of the PISA hot path runs in the library's CUDA kernels. PyTorch supplies the
device memory (outputs and workspaces are torch tensors), the current CUDA stream and
the dtype/shape bookkeeping. There is no fallback: if the library cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpisa.so")

PISA_OK, PISA_EINVAL, PISA_EUNSUPPORTED, PISA_EWORKSPACE, PISA_ECUDA, PISA_ETIMEOUT = range(6)
OP_SELECT, OP_SELECT_FLAT, OP_ATTN_FWD, OP_ATTN_BWD, OP_SELECT_MEAN, OP_SELECT_MEANVAR = range(6)
STATUS_POS_RANGE, STATUS_TIMEOUT = 1, 2
MAX_LEVELS = 32
ABI_VERSION = 4          # PISA_VERSION of the header these argument lists follow

EXPORTS = (
    "pisa_version", "pisa_last_error", "pisa_pyramid_layout", "pisa_workspace_size",
    "pisa_build_pyramid", "pisa_select", "pisa_select_flat", "pisa_sparse_attn_fwd",
    "pisa_sparse_attn_bwd", "pisa_decode_pyramid_layout", "pisa_decode_build_pyramid",
    "pisa_decode_step", "pisa_profile_start", "pisa_profile_stop", "pisa_profile_read",
    "pisa_select_noalloc", "pisa_select_mean", "pisa_set_wait_limit", "pisa_test_stall",
    "pisa_select_meanvar",
)


class PisaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"PISA error {code}: {msg}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "N", "Hq", "Hkv", "d", "C", "K", "g", "qtile")] + \
               [("scale", ctypes.c_float), ("per_head", ctypes.c_int32)]


class ProfileEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_double)]


class DecodeShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "Ncap", "Hq", "Hkv", "d", "C", "K", "g")] + \
               [("scale", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpisa.so (built by pyramid_top_selection_gb300.build) or raise."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libpisa.so not built at {LIB_PATH}: run pyramid_top_selection_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        P = ctypes.POINTER
        L.pisa_version.restype = ctypes.c_int
        if L.pisa_version() != ABI_VERSION:
            raise ImportError(f"libpisa.so has ABI version {L.pisa_version()}, this binding needs {ABI_VERSION}: "
                              "rebuild with pyramid_top_selection_gb300/build.py")
        L.pisa_last_error.restype = ctypes.c_char_p
        L.pisa_pyramid_layout.argtypes = [P(Shape), P(i32), P(i64), P(i64)]
        L.pisa_workspace_size.argtypes = [P(Shape), ctypes.c_int, P(sz)]
        L.pisa_build_pyramid.argtypes = [P(Shape), vp, vp, vp]
        L.pisa_select.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.pisa_select_flat.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, sz, vp]
        L.pisa_select_mean.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, sz, vp]
        L.pisa_select_meanvar.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, sz, vp]
        L.pisa_sparse_attn_fwd.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.pisa_sparse_attn_bwd.argtypes = [P(Shape)] + [vp] * 10 + [vp, sz, vp]
        L.pisa_decode_pyramid_layout.argtypes = [P(DecodeShape), P(i32), P(i64), P(i64)]
        L.pisa_decode_build_pyramid.argtypes = [P(DecodeShape), vp, vp, vp, vp]
        L.pisa_decode_step.argtypes = [P(DecodeShape)] + [vp] * 11 + [vp]
        L.pisa_profile_start.argtypes = []
        L.pisa_profile_stop.argtypes = []
        L.pisa_profile_read.argtypes = [P(ProfileEntry), i32, P(i32)]
        L.pisa_set_wait_limit.argtypes = [ctypes.c_uint64]
        L.pisa_test_stall.argtypes = [ctypes.c_int]
        for f in EXPORTS:
            if f not in ("pisa_version", "pisa_last_error"):
                getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != PISA_OK:
        raise PisaError(rc, lib().pisa_last_error().decode())


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def make_shape(B, N, Hq, Hkv, d, C=64, K=16, g=2, qtile=1, scale=0.0, per_head=False) -> Shape:
    return Shape(B, N, Hq, Hkv, d, C, K, g, qtile, float(scale), 1 if per_head else 0)


def shape_of(Q: torch.Tensor, Kt: torch.Tensor, C=64, K=16, g=2, qtile=1, scale=0.0, per_head=False) -> Shape:
    B, N, Hq, d = Q.shape
    return make_shape(B, N, Hq, Kt.shape[2], d, C, K, g, qtile, scale, per_head)


def _units(shape: Shape) -> int:
    """Selection units per batch: the KV heads, or the query heads of a per-head selection."""
    return shape.Hq if shape.per_head else shape.Hkv


def pyramid_layout(shape: Shape):
    n = ctypes.c_int32()
    off = (ctypes.c_int64 * MAX_LEVELS)()
    nodes = ctypes.c_int64()
    _check(lib().pisa_pyramid_layout(ctypes.byref(shape), ctypes.byref(n), off, ctypes.byref(nodes)))
    return n.value, list(off[:n.value]), nodes.value


def workspace_size(shape: Shape, op: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().pisa_workspace_size(ctypes.byref(shape), op, ctypes.byref(b)))
    return b.value


def workspace(shape: Shape, op: int, device) -> torch.Tensor:
    """A device workspace of the size `op` needs (uint8 tensor)."""
    return _workspace(shape, op, device)


def _workspace(shape: Shape, op: int, device) -> torch.Tensor:
    return torch.empty(max(workspace_size(shape, op), 256), dtype=torch.uint8, device=device)


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor (got {t.dtype}, "
                         f"cuda={t.is_cuda}, contiguous={t.is_contiguous()})")


def build_pyramid(Kt: torch.Tensor, shape: Shape, out: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 key sums [B, Hkv, nodes, d] of K [B, N, Hkv, d] bf16."""
    _need(Kt, torch.bfloat16, "K")
    _, _, nodes = pyramid_layout(shape)
    pyr = out if out is not None else torch.empty(shape.B, shape.Hkv, nodes, shape.d, dtype=torch.float32,
                                                  device=Kt.device)
    _check(lib().pisa_build_pyramid(ctypes.byref(shape), _ptr(Kt), _ptr(pyr), _stream(Kt.device)))
    return pyr


def _select_out(Q, shape, want_score, idx, score):
    dev = Q.device
    if idx is None:
        idx = torch.empty(shape.B, _units(shape), shape.N, shape.K, dtype=torch.int32, device=dev)
    if score is None and want_score:
        score = torch.empty(shape.B, _units(shape), shape.N, shape.K, dtype=torch.float32, device=dev)
    return idx, score


def _select_in(Q, Kt, pyr):
    _need(Q, torch.bfloat16, "Q")
    _need(Kt, torch.bfloat16, "K")
    _need(pyr, torch.float32, "pyr_sum")


def select(Q, Kt, pyr, shape: Shape, ws=None, want_score=True, idx=None, score=None,
           want_head_lse=False, head_lse=None):
    """Pyramid Top-K selection: idx [B,Hkv,N,K] int32 (ascending, -1 pad), score fp32.

    With want_head_lse (or a head_lse buffer) also returns the per-head leaf LSEs
    [B,Hq,N,K] fp32 that sparse_attn_fwd takes to skip its normalisation pass."""
    _select_in(Q, Kt, pyr)
    dev = Q.device
    idx, score = _select_out(Q, shape, want_score, idx, score)
    if head_lse is None and want_head_lse:
        head_lse = torch.empty(shape.B, shape.Hq, shape.N, shape.K, dtype=torch.float32, device=dev)
    if ws is None:
        ws = _workspace(shape, OP_SELECT, dev)
    _check(lib().pisa_select(ctypes.byref(shape), _ptr(Q), _ptr(Kt), _ptr(pyr), _ptr(idx), _ptr(score),
                             _ptr(head_lse), _ptr(ws), ws.numel(), _stream(dev)))
    if head_lse is not None:
        return idx, score, head_lse
    return idx, score


def select_flat(Q, Kt, pyr, shape: Shape, ws=None, want_score=True, idx=None, score=None):
    """Flat O(N^2/C) block selection (comparator)."""
    _select_in(Q, Kt, pyr)
    dev = Q.device
    idx, score = _select_out(Q, shape, want_score, idx, score)
    if ws is None:
        ws = _workspace(shape, OP_SELECT_FLAT, dev)
    _check(lib().pisa_select_flat(ctypes.byref(shape), _ptr(Q), _ptr(Kt), _ptr(pyr), _ptr(idx), _ptr(score),
                                  _ptr(ws), ws.numel(), _stream(dev)))
    return idx, score


def select_mean(Q, Kt, pyr, shape: Shape, ws=None, want_score=True, idx=None, score=None):
    """PISA-1 ablation selection: the pyramid descent with every block scored by its mean key."""
    _select_in(Q, Kt, pyr)
    dev = Q.device
    idx, score = _select_out(Q, shape, want_score, idx, score)
    if ws is None:
        ws = _workspace(shape, OP_SELECT_MEAN, dev)
    _check(lib().pisa_select_mean(ctypes.byref(shape), _ptr(Q), _ptr(Kt), _ptr(pyr), _ptr(idx), _ptr(score),
                                  _ptr(ws), ws.numel(), _stream(dev)))
    return idx, score


def select_meanvar(Q, Kt, pyr, shape: Shape, ws=None, want_score=True, idx=None, score=None):
    """PISA-2 ablation selection: the pyramid descent with every block scored by mean + variance."""
    _select_in(Q, Kt, pyr)
    dev = Q.device
    idx, score = _select_out(Q, shape, want_score, idx, score)
    if ws is None:
        ws = _workspace(shape, OP_SELECT_MEANVAR, dev)
    _check(lib().pisa_select_meanvar(ctypes.byref(shape), _ptr(Q), _ptr(Kt), _ptr(pyr), _ptr(idx), _ptr(score),
                                     _ptr(ws), ws.numel(), _stream(dev)))
    return idx, score


def sparse_attn_fwd(Q, Kt, V, idx, shape: Shape, ws=None, out=None, lse=None, head_lse=None):
    """Causal attention over the selected leaves: O [B,N,Hq,d] bf16, lse [B,Hq,N] fp32.

    head_lse: the selection's per-head leaf LSEs for these idx (optional)."""
    for t, n in ((Q, "Q"), (Kt, "K"), (V, "V")):
        _need(t, torch.bfloat16, n)
    _need(idx, torch.int32, "idx")
    if head_lse is not None:
        _need(head_lse, torch.float32, "head_lse")
    dev = Q.device
    O = out if out is not None else torch.empty_like(Q)
    lse = lse if lse is not None else torch.empty(shape.B, shape.Hq, shape.N, dtype=torch.float32, device=dev)
    if ws is None:
        ws = _workspace(shape, OP_ATTN_FWD, dev)
    _check(lib().pisa_sparse_attn_fwd(ctypes.byref(shape), _ptr(Q), _ptr(Kt), _ptr(V), _ptr(idx),
                                      _ptr(head_lse), _ptr(O), _ptr(lse), _ptr(ws), ws.numel(), _stream(dev)))
    return O, lse


def sparse_attn_bwd(Q, Kt, V, O, lse, dO, idx, shape: Shape, ws=None):
    """Gradients through the selected attention only: dQ, dK, dV (bf16)."""
    for t, n in ((Q, "Q"), (Kt, "K"), (V, "V"), (O, "O"), (dO, "dO")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    _need(idx, torch.int32, "idx")
    dev = Q.device
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(Kt), torch.empty_like(V)
    if ws is None:
        ws = _workspace(shape, OP_ATTN_BWD, dev)
    _check(lib().pisa_sparse_attn_bwd(ctypes.byref(shape), _ptr(Q), _ptr(Kt), _ptr(V), _ptr(O),
                                      _ptr(lse), _ptr(dO), _ptr(idx), _ptr(dQ), _ptr(dK), _ptr(dV),
                                      _ptr(ws), ws.numel(), _stream(dev)))
    return dQ, dK, dV


def make_decode_shape(B, Ncap, Hq, Hkv, d, C=64, K=16, g=2, scale=0.0) -> DecodeShape:
    return DecodeShape(B, Ncap, Hq, Hkv, d, C, K, g, float(scale))


def decode_pyramid_layout(shape: DecodeShape):
    n = ctypes.c_int32()
    off = (ctypes.c_int64 * MAX_LEVELS)()
    nodes = ctypes.c_int64()
    _check(lib().pisa_decode_pyramid_layout(ctypes.byref(shape), ctypes.byref(n), off, ctypes.byref(nodes)))
    return n.value, list(off[:n.value]), nodes.value


def decode_build_pyramid(Kcache, length, shape: DecodeShape) -> torch.Tensor:
    """Cached pyramid over Ncap from the first length[b] keys of each sequence."""
    _need(Kcache, torch.bfloat16, "Kcache")
    _need(length, torch.int32, "len")
    _, _, nodes = decode_pyramid_layout(shape)
    pyr = torch.empty(shape.B, shape.Hkv, nodes, shape.d, dtype=torch.float32, device=Kcache.device)
    _check(lib().pisa_decode_build_pyramid(ctypes.byref(shape), _ptr(Kcache), _ptr(length), _ptr(pyr),
                                           _stream(Kcache.device)))
    return pyr


def decode_step(shape: DecodeShape, pos, Kcache, Vcache, pyr, q, k_new, v_new, o=None, idx=None,
                score=None, status=None):
    """One fused decode step (append + ancestor update + select + attend) for all sequences."""
    dev = q.device
    o = o if o is not None else torch.empty_like(q)
    idx = idx if idx is not None else torch.empty(shape.B, shape.Hkv, shape.K, dtype=torch.int32, device=dev)
    status = status if status is not None else torch.zeros(4, dtype=torch.int32, device=dev)
    _check(lib().pisa_decode_step(ctypes.byref(shape), _ptr(pos), _ptr(Kcache), _ptr(Vcache), _ptr(pyr),
                                  _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(o), _ptr(idx), _ptr(score),
                                  _ptr(status), _stream(dev)))
    return o, idx, score, status


def workspace_status(ws: torch.Tensor) -> int:
    """The status word of the last call that used workspace `ws` (its first 4 bytes, read after
    the current stream has passed the call): 0, or STATUS_* bits."""
    torch.cuda.current_stream(ws.device).synchronize()
    return int(ws[:4].view(torch.int32).item())


def check_status(ws: torch.Tensor) -> None:
    """Raise PisaError(PISA_ETIMEOUT) when the last call on `ws` reported a wait that gave up."""
    st = workspace_status(ws)
    if st & STATUS_TIMEOUT:
        raise PisaError(PISA_ETIMEOUT, f"a bounded device wait gave up (status word {st}); outputs are poisoned")


def set_wait_limit(ns: int) -> None:
    """Bound of every device-side pipeline wait in nanoseconds (0 restores the one-second default)."""
    _check(lib().pisa_set_wait_limit(int(ns)))


def set_test_stall(on: bool) -> None:
    """Test aid: make the tensor-core kernels wait on a barrier nothing signals (see pisa.h)."""
    _check(lib().pisa_test_stall(1 if on else 0))


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def profile_start() -> None:
    """Record CUDA events around every kernel launch of the library (on its stream)."""
    _check(lib().pisa_profile_start())


def profile_stop() -> None:
    _check(lib().pisa_profile_stop())


def profile_read() -> dict:
    """{kernel name: (launches, total ms)} since the last read; waits for the events."""
    buf = (ProfileEntry * 64)()
    n = ctypes.c_int32()
    _check(lib().pisa_profile_read(buf, 64, ctypes.byref(n)))
    return {buf[k].name.decode(): (buf[k].launches, buf[k].total_ms) for k in range(n.value)}
