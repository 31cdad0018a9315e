"""GPU parity of the sparse-attention backward (through the C ABI) against the fp64 oracle.
The selection is an input here: the oracle's own selection, or a seeded random valid one."""
import numpy as np
import pytest
import torch

import pisa_synth as syn
import pyramid_top_selection_gb300 as pisa
from oracle import pisa_oracle as po
from _parity import check_close

pytestmark = pytest.mark.gpu
C = 64


@pytest.mark.parametrize("B,N,Hq,Hkv,d,K,seed", [
    (1, 500, 8, 2, 128, 4, 0),      # G = 4, ragged N
    (2, 300, 2, 2, 64, 3, 1),       # G = 1, d = 64
    (1, 700, 16, 2, 128, 16, 2),    # G = 8, K >= visible leaves for early queries
    (1, 420, 4, 2, 64, 4, 3),       # G = 2, d = 64
    (1, 390, 8, 2, 64, 5, 4),       # G = 4, d = 64
    (1, 333, 8, 1, 64, 3, 5),       # G = 8, d = 64, ragged
    (2, 260, 2, 2, 128, 3, 6),      # G = 1, d = 128
    (1, 450, 4, 2, 128, 6, 7),      # G = 2, d = 128
])
def test_backward_vs_oracle(B, N, Hq, Hkv, d, K, seed):
    Q, Kt, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=seed, needles=True)
    dO = syn.make_grad_out(B, N, Hq, d, seed=seed)
    idx = po.select(Q, Kt, C, K)["idx"]
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K)
    Qg, Kg, Vg, dOg = Q.cuda(), Kt.cuda(), V.cuda(), dO.cuda()
    ig = torch.from_numpy(idx).cuda()
    O, lse = pisa.sparse_attn_fwd(Qg, Kg, Vg, ig, shape)
    dQ, dK, dV = pisa.sparse_attn_bwd(Qg, Kg, Vg, O, lse, dOg, ig, shape)
    torch.cuda.synchronize()
    rq, rk, rv = po.sparse_attn_bwd(Q, Kt, V, dO, idx, C)
    check_close(dQ.float().cpu().numpy(), rq, what="dQ")
    check_close(dK.float().cpu().numpy(), rk, what="dK")
    check_close(dV.float().cpu().numpy(), rv, what="dV")


def test_backward_training_shape_sampled():
    # The training workload (B=4, N=16384, Hq=16, Hkv=4, d=128, K=16) at full size; the oracle
    # evaluates dQ of sampled queries and dK/dV of sampled leaf blocks.
    B, N, Hq, Hkv, d, K = 4, 16384, 16, 4, 128, 16
    Q, Kt, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=0, needles=False)
    dO = syn.make_grad_out(B, N, Hq, d, seed=0)
    idx = syn.random_selection(B, Hkv, N, C, K, seed=5)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=4)
    Qg, Kg, Vg, dOg, ig = Q.cuda(), Kt.cuda(), V.cuda(), dO.cuda(), idx.cuda()
    O, lse = pisa.sparse_attn_fwd(Qg, Kg, Vg, ig, shape)
    dQ, dK, dV = pisa.sparse_attn_bwd(Qg, Kg, Vg, O, lse, dOg, ig, shape)
    torch.cuda.synchronize()
    qs = [(0, 0), (1, 777), (2, 8191), (3, N - 1)]
    ls = [(0, 0, 0), (1, 2, 100), (3, 3, 255)]
    sq, sk, sv = po.sparse_attn_bwd_sampled(Q, Kt, V, dO, idx.numpy(), C, queries=qs, leaves=ls)
    for (b, i) in qs:
        check_close(dQ[b, i].float().cpu().numpy(), sq[(b, i)], what=f"dQ {b},{i}")
    for (b, kv, t) in ls:
        s0, e0 = po.node_range(0, t, C, N)
        check_close(dK[b, s0:e0, kv].float().cpu().numpy(), sk[(b, kv, t)], what=f"dK {b},{kv},{t}")
        check_close(dV[b, s0:e0, kv].float().cpu().numpy(), sv[(b, kv, t)], what=f"dV {b},{kv},{t}")
    Oref, lref = po.sparse_attn_fwd(Q, Kt, V, idx.numpy(), C, queries=[i for _, i in qs])
    for (b, i) in qs:
        check_close(O[b, i].float().cpu().numpy(), Oref[b, i], what="O")


def test_unselected_leaf_gets_zero_key_gradients():
    B, N, Hq, Hkv, d, K = 1, 256, 4, 1, 64, 1
    Q, Kt, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=9)
    dO = syn.make_grad_out(B, N, Hq, d, seed=9)
    idx = torch.zeros(B, Hkv, N, K, dtype=torch.int32)       # everyone selects leaf 0 only
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K)
    Qg, Kg, Vg, dOg, ig = Q.cuda(), Kt.cuda(), V.cuda(), dO.cuda(), idx.cuda()
    O, lse = pisa.sparse_attn_fwd(Qg, Kg, Vg, ig, shape)
    dQ, dK, dV = pisa.sparse_attn_bwd(Qg, Kg, Vg, O, lse, dOg, ig, shape)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dK[:, C:]) == 0 and torch.count_nonzero(dV[:, C:]) == 0
    rq, rk, rv = po.sparse_attn_bwd(Q, Kt, V, dO, idx.numpy(), C)
    check_close(dK.float().cpu().numpy(), rk, what="dK")
    check_close(dV.float().cpu().numpy(), rv, what="dV")
    check_close(dQ.float().cpu().numpy(), rq, what="dQ")
