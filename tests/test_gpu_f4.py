"""GPU parity of the per-head (unshared) selection and of fan-out g = 4, through the C ABI,
against the fp64 oracle on the same seeded bf16 inputs: the selections, and the sparse
attention forward and backward over a per-head selection. Needs a GB300 and the built library."""
import numpy as np
import pytest
import torch

import pisa_synth as syn
import pyramid_top_selection_gb300 as pisa
from oracle import pisa_oracle as po
from _parity import SCORE_ATOL, check_close, check_selection

pytestmark = pytest.mark.gpu
C = 64

PER_HEAD_CASES = [
    ("ph_g4_d128", 1, 1500, 8, 2, 128, 6),
    ("ph_g4_d64_b2", 2, 700, 4, 1, 64, 4),
    ("ph_g2_d128_k16", 1, 2300, 4, 2, 128, 16),
]


def _inputs(B, N, Hq, Hkv, d, seed=0):
    Q, K, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=seed, needles=True)
    return (Q, K, V), (Q.cuda(), K.cuda(), V.cuda())


@pytest.mark.parametrize("case", PER_HEAD_CASES, ids=[c[0] for c in PER_HEAD_CASES])
def test_per_head_selections_and_attention_vs_oracle(case):
    _, B, N, Hq, Hkv, d, K = case
    (Q, Kt, V), (Qg, Kg, Vg) = _inputs(B, N, Hq, Hkv, d)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=1, per_head=True)
    pyr = pisa.build_pyramid(Kg, shape)
    idx, score, hl = pisa.select(Qg, Kg, pyr, shape, want_head_lse=True)
    idx4, score4 = pisa.select(Qg, Kg, pyr, pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=4, per_head=True))
    torch.cuda.synchronize()
    assert idx.shape == (B, Hq, N, K) and torch.equal(idx, idx4) and torch.equal(score, score4)
    ora = po.select(Q, Kt, C, K, per_head=True)
    st = check_selection(idx.cpu().numpy(), score.cpu().numpy(), ora, range(N), C, K, N)
    assert st["strict"] + st["exempt"] == st["units"] and st["strict"] >= 0.98 * st["units"], st
    gi = idx.cpu().numpy()
    want = po.selected_head_lse(Q, Kt, gi, C)
    got = hl.cpu().numpy()
    assert np.array_equal(np.isneginf(got), np.isneginf(want))
    f = np.isfinite(want)
    check_close(got[f], want[f], atol=SCORE_ATOL, rtol=0, what="per-head head_lse")
    # a per-head selection's score is its own head's leaf LSE
    check_close(score.cpu().numpy()[gi >= 0], got[gi >= 0], atol=1e-6, rtol=0, what="score = head_lse")
    # the per-head PISA-1, PISA-2 and flat selections
    for fn, ofn in ((pisa.select_mean, po.select_mean), (pisa.select_meanvar, po.select_meanvar),
                    (pisa.select_flat, po.select_flat)):
        i2, s2 = fn(Qg, Kg, pyr, shape)
        o2 = ofn(Q, Kt, C, K, per_head=True)
        st2 = check_selection(i2.cpu().numpy(), s2.cpu().numpy(), o2, range(N), C, K, N)
        assert st2["strict"] + st2["exempt"] == st2["units"] and st2["strict"] >= 0.9 * st2["units"], (fn, st2)
    # attention over the per-head selection, normalised by its head_lse and by its own LSE pass
    Oref, lref = po.sparse_attn_fwd(Q, Kt, V, gi, C)
    for kw in ({"head_lse": hl}, {}):
        O, lse = pisa.sparse_attn_fwd(Qg, Kg, Vg, idx, shape, **kw)
        check_close(O.float().cpu().numpy(), Oref, what=f"O {list(kw)}")
        check_close(lse.cpu().numpy(), lref, atol=1e-3, rtol=0, what=f"lse {list(kw)}")


@pytest.mark.parametrize("B,N,Hq,Hkv,d,K,seed", [(1, 600, 8, 2, 128, 5, 0), (1, 450, 4, 1, 64, 3, 1)])
def test_per_head_backward_vs_oracle(B, N, Hq, Hkv, d, K, seed):
    Q, Kt, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=seed, needles=True)
    dO = syn.make_grad_out(B, N, Hq, d, seed=seed)
    idx = syn.random_selection(B, Hq, N, C, K, seed=seed + 9)          # a different selection per head
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, per_head=True)
    Qg, Kg, Vg, dOg, ig = Q.cuda(), Kt.cuda(), V.cuda(), dO.cuda(), idx.cuda()
    O, lse = pisa.sparse_attn_fwd(Qg, Kg, Vg, ig, shape)
    dQ, dK, dV = pisa.sparse_attn_bwd(Qg, Kg, Vg, O, lse, dOg, ig, shape)
    torch.cuda.synchronize()
    rq, rk, rv = po.sparse_attn_bwd(Q, Kt, V, dO, idx.numpy(), C)
    check_close(dQ.float().cpu().numpy(), rq, what="dQ")
    check_close(dK.float().cpu().numpy(), rk, what="dK")
    check_close(dV.float().cpu().numpy(), rv, what="dV")


G4_CASES = [
    ("g4_4k_d64", 1, 4096, 4, 1, 64, 8),
    ("g4_ragged_d128", 1, 3000, 8, 2, 128, 5),
    ("g4_k1_b2", 2, 1300, 4, 2, 64, 1),
    ("g4_per_head", 1, 2000, 4, 2, 128, 4),
]


@pytest.mark.parametrize("case", G4_CASES, ids=[c[0] for c in G4_CASES])
def test_fanout4_selection_vs_oracle(case):
    name, B, N, Hq, Hkv, d, K = case
    per_head = name.endswith("per_head")
    (Q, Kt, _), (Qg, Kg, _) = _inputs(B, N, Hq, Hkv, d, seed=2)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, g=4, qtile=4, per_head=per_head)
    pyr = pisa.build_pyramid(Kg, shape)
    idx, score = pisa.select(Qg, Kg, pyr, shape)
    ora = po.select(Q, Kt, C, K, g=4, per_head=per_head)
    st = check_selection(idx.cpu().numpy(), score.cpu().numpy(), ora, range(N), C, K, N)
    assert st["strict"] + st["exempt"] == st["units"] and st["strict"] >= 0.98 * st["units"], st


def test_fanout4_sampled_at_16k():
    # 256 leaves, K = 16: 64 candidates at the pruning steps (the 64-candidate routing and top-K)
    B, N, Hq, Hkv, d, K = 1, 16384, 16, 2, 128, 16
    Q, Kt, _ = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=3, needles=True)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, g=4, qtile=4)
    pyr = pisa.build_pyramid(Kt.cuda(), shape)
    idx, score = pisa.select(Q.cuda(), Kt.cuda(), pyr, shape)
    qs = sorted(set(range(0, N, 211)) | {N - 1})
    ora = po.select(Q, Kt, C, K, g=4, queries=qs)
    st = check_selection(idx.cpu().numpy(), score.cpu().numpy(), ora, qs, C, K, N)
    print(f"g=4 N={N} K={K}: {st}")
    assert st["strict"] + st["exempt"] == st["units"] and st["strict"] >= 0.95 * st["units"], st
