"""A bounded device wait that runs out: the tensor-core kernels of the selection and of the
attention forward give up, drain what they issued, and report PISA_STATUS_TIMEOUT in the
workspace's status word; the outputs are poisoned. The wait is made to run out by the
library's test stall (a barrier nothing signals) under a short wait limit, so no GPU fault,
trap or hang is involved; afterwards the same calls run normally again."""
import pytest
import torch

import pisa_synth as syn
import pyramid_top_selection_gb300 as pisa
from pyramid_top_selection_gb300 import _pisa

pytestmark = pytest.mark.gpu


@pytest.fixture
def stalled():
    pisa.set_wait_limit(2_000_000)          # 2 ms
    pisa.set_test_stall(True)
    try:
        yield
    finally:
        pisa.set_test_stall(False)
        pisa.set_wait_limit(0)              # back to the default


def _problem(N):
    B, Hq, Hkv, d, K = 1, 8, 2, 128, 8
    Q, Kt, V = (x.cuda() for x in syn.make_prefill(B, N, Hq, Hkv, d, C=64, seed=4, needles=True))
    shape = pisa.make_shape(B, N, Hq, Hkv, d, 64, K, qtile=4)
    return Q, Kt, V, shape


def _normal_run(Q, Kt, V, shape):
    pyr = pisa.build_pyramid(Kt, shape)
    ws_s = pisa.workspace(shape, _pisa.OP_SELECT, Q.device)
    idx, score, hl = pisa.select(Q, Kt, pyr, shape, ws=ws_s, want_head_lse=True)
    ws_a = pisa.workspace(shape, _pisa.OP_ATTN_FWD, Q.device)
    O, lse = pisa.sparse_attn_fwd(Q, Kt, V, idx, shape, ws=ws_a, head_lse=hl)
    assert pisa.workspace_status(ws_s) == 0 and pisa.workspace_status(ws_a) == 0
    return pyr, idx, score, hl, O, lse


# 6000 and 32768 (query, KV head) units: the top-K finish runs its warp and its thread-per-query
# version, and both must poison
@pytest.mark.parametrize("N", [3000, 16384])
def test_wait_that_runs_out_is_reported_and_poisons_outputs(stalled, N):
    Q, Kt, V, shape = _problem(N)
    pisa.set_test_stall(False)
    pisa.set_wait_limit(0)
    pyr, idx0, score0, hl0, O0, lse0 = _normal_run(Q, Kt, V, shape)
    pisa.set_wait_limit(2_000_000)
    pisa.set_test_stall(True)
    # selection: the leaf-scoring kernel gives up before its first MMA
    ws_s = pisa.workspace(shape, _pisa.OP_SELECT, Q.device)
    idx, score, hl = pisa.select(Q, Kt, pyr, shape, ws=ws_s, want_head_lse=True)
    st = pisa.workspace_status(ws_s)
    assert st & pisa.STATUS_TIMEOUT, st
    assert bool((idx == -1).all()) and bool(score.isnan().all()) and bool(hl.isnan().all())
    with pytest.raises(pisa.PisaError):
        pisa.check_status(ws_s)
    # attention forward (its own block-LSE pass and its output pass both stall)
    ws_a = pisa.workspace(shape, _pisa.OP_ATTN_FWD, Q.device)
    O, lse = pisa.sparse_attn_fwd(Q, Kt, V, idx0, shape, ws=ws_a)
    st = pisa.workspace_status(ws_a)
    assert st & pisa.STATUS_TIMEOUT, st
    assert bool(O.isnan().all()) and bool(lse.isnan().all())
    # attention backward (the tensor-core kernel, d = 128)
    dO = syn.make_grad_out(*Q.shape[:3], Q.shape[3], seed=4).cuda()
    ws_b = pisa.workspace(shape, _pisa.OP_ATTN_BWD, Q.device)
    dQ, dK, dV = pisa.sparse_attn_bwd(Q, Kt, V, O0, lse0, dO, idx0, shape, ws=ws_b)
    st = pisa.workspace_status(ws_b)
    assert st & pisa.STATUS_TIMEOUT, st
    assert bool(dQ.isnan().all()) and bool(dK.isnan().all()) and bool(dV.isnan().all())
    # the context is intact: the same calls run normally again and reproduce the results
    pisa.set_test_stall(False)
    pisa.set_wait_limit(0)
    _, idx1, score1, hl1, O1, lse1 = _normal_run(Q, Kt, V, shape)
    assert torch.equal(idx1, idx0) and torch.equal(score1, score0) and torch.equal(hl1, hl0)
    assert torch.equal(lse1, lse0)
    # block contributions are added in a run-dependent order: equal up to fp32 rounding
    torch.testing.assert_close(O1.float(), O0.float(), atol=1e-2, rtol=1e-2)
    dQ1, dK1, dV1 = pisa.sparse_attn_bwd(Q, Kt, V, O0, lse0, dO, idx0, shape, ws=ws_b)
    assert pisa.workspace_status(ws_b) == 0
    assert not (dQ1.isnan().any() or dK1.isnan().any() or dV1.isnan().any())
