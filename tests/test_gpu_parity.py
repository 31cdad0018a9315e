"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded bf16 inputs, plus GPU self-invariants. Needs a GB300 and the built library."""
import numpy as np
import pytest
import torch

import pisa_synth as syn
import pyramid_top_selection_gb300 as pisa
from oracle import pisa_oracle as po
from _parity import SCORE_ATOL, check_close, check_selection

pytestmark = pytest.mark.gpu
C = 64

# name, B, N, Hq, Hkv, d, K, needles
CASES = [
    ("prefill_4k_gqa4_d64", 1, 4096, 4, 1, 64, 8, False),     # the 4K / 64-leaf / 7-level workload
    ("ragged_g4_d128", 1, 1000, 8, 2, 128, 4, True),
    ("g8_d128_needles", 1, 2048, 16, 2, 128, 16, True),
    ("g1_b2_d64", 2, 777, 2, 2, 64, 3, False),
    ("g2_keep_all", 1, 1500, 4, 2, 64, 32, False),
    ("k1_d128", 1, 1300, 8, 1, 128, 1, True),
    # K = 1 at G = 4: the first scored level's child dots come from the prefix pass, and a level
    # kept whole after it (the kept node's right child not yet visible) must load its own
    ("k1_g4_d128", 1, 1300, 4, 1, 128, 1, True),
    ("single_partial_leaf", 1, 63, 4, 1, 64, 4, False),
    ("one_token", 1, 1, 2, 1, 128, 4, False),
    ("two_leaves_b2", 2, 65, 8, 1, 128, 1, False),
    ("g1_d128", 1, 1200, 2, 2, 128, 6, True),                 # G = 1 with d = 128
    ("g8_d64", 1, 1100, 8, 1, 64, 5, True),                   # G = 8 with d = 64
    ("g2_d128", 1, 1100, 4, 2, 128, 6, True),                 # G = 2 with d = 128
]


def _inputs(B, N, Hq, Hkv, d, needles, seed=0):
    Q, K, V = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=seed, needles=needles)
    return (Q, K, V), (Q.cuda(), K.cuda(), V.cuda())


def _check_head_lse(got, want, what="head_lse"):
    """Per-head leaf LSEs: -inf exactly on the padded slots, SCORE_ATOL elsewhere."""
    assert np.array_equal(np.isneginf(got), np.isneginf(want)), what
    f = np.isfinite(want)
    check_close(got[f], want[f], atol=SCORE_ATOL, rtol=0, what=what)


def _pyr_levels(pyr, shape):
    _, off, _ = pisa.pyramid_layout(shape)
    return off


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_pyramid_select_flat_attention_vs_oracle(case):
    _, B, N, Hq, Hkv, d, K, needles = case
    (Q, Kt, V), (Qg, Kg, Vg) = _inputs(B, N, Hq, Hkv, d, needles)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=1)
    pyr = pisa.build_pyramid(Kg, shape)
    # A1 pyramid: fp32 sums against the oracle's direct range sums
    off = _pyr_levels(pyr, shape)
    K64 = Kt.double().numpy()
    pg = pyr.cpu().double().numpy()
    for b in range(B):
        for kv in range(Hkv):
            ref = po.pyramid_sums(K64[b, :, kv, :], C)
            for l, S in enumerate(ref):
                cnt = np.array([po.node_range(l, m, C, N)[1] - po.node_range(l, m, C, N)[0] for m in range(len(S))])
                got = pg[b, kv, off[l]:off[l] + len(S)]
                assert np.all(np.abs(got - S) <= 1e-6 * cnt[:, None] + 1e-6 * np.abs(S)), (b, kv, l)
    # A2-A4 selection (with the per-head leaf terms, as the prefill path runs it)
    idx, score, hl = pisa.select(Qg, Kg, pyr, shape, want_head_lse=True)
    idx4, score4 = pisa.select(Qg, Kg, pyr, pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=4))
    torch.cuda.synchronize()
    assert torch.equal(idx, idx4) and torch.equal(score, score4)      # qtile is scheduling only
    gi = idx.cpu().numpy()
    _check_head_lse(hl.cpu().numpy(), po.selected_head_lse(Q, Kt, gi, C))
    ora = po.select(Q, Kt, C, K)
    st = check_selection(idx.cpu().numpy(), score.cpu().numpy(), ora, range(N), C, K, N)
    assert st["strict"] + st["exempt"] == st["units"]
    assert st["strict"] >= 0.98 * st["units"], st
    # A8 flat comparator
    fidx, fscore = pisa.select_flat(Qg, Kg, pyr, shape)
    fora = po.select_flat(Q, Kt, C, K)
    check_selection(fidx.cpu().numpy(), fscore.cpu().numpy(), fora, range(N), C, K, N)
    # A5 attention over the oracle's selection (block LSEs computed by the call itself)
    oidx = torch.from_numpy(ora["idx"]).cuda()
    O, lse = pisa.sparse_attn_fwd(Qg, Kg, Vg, oidx, shape)
    Oref, lref = po.sparse_attn_fwd(Q, Kt, V, ora["idx"], C)
    check_close(O.float().cpu().numpy(), Oref, what="O")
    check_close(lse.cpu().numpy(), lref, atol=1e-3, rtol=0, what="lse")
    # ... and over the GPU's own selection, normalised by the selection's head_lse
    O2, lse2 = pisa.sparse_attn_fwd(Qg, Kg, Vg, idx, shape, head_lse=hl)
    Oref2, lref2 = po.sparse_attn_fwd(Q, Kt, V, gi, C)
    check_close(O2.float().cpu().numpy(), Oref2, what="O (head_lse)")
    check_close(lse2.cpu().numpy(), lref2, atol=1e-3, rtol=0, what="lse (head_lse)")


def test_select_is_independent_of_pyramid_height():
    # A shorter sequence inside a longer pyramid: query i's selection must not change when
    # tokens after it are appended (extra top levels never prune).
    B, N, Hq, Hkv, d, K = 1, 3000, 8, 2, 128, 4
    (Q, Kt, V), (Qg, Kg, Vg) = _inputs(B, N, Hq, Hkv, d, True, seed=3)
    n_short = 700
    full = pisa.make_shape(B, N, Hq, Hkv, d, C, K)
    short = pisa.make_shape(B, n_short, Hq, Hkv, d, C, K)
    i_full, s_full = pisa.select(Qg, Kg, pisa.build_pyramid(Kg, full), full)
    Qs, Ks = Qg[:, :n_short].contiguous(), Kg[:, :n_short].contiguous()
    i_short, s_short = pisa.select(Qs, Ks, pisa.build_pyramid(Ks, short), short)
    assert torch.equal(i_full[:, :, :n_short], i_short)
    torch.testing.assert_close(s_full[:, :, :n_short], s_short, atol=1e-4, rtol=0)


def test_attention_random_selection_vs_oracle():
    # attention on an arbitrary valid selection drawn from a seeded generator
    B, N, Hq, Hkv, d, K = 2, 900, 8, 2, 128, 5
    (Q, Kt, V), (Qg, Kg, Vg) = _inputs(B, N, Hq, Hkv, d, False, seed=7)
    gen = torch.Generator().manual_seed(11)
    idx = torch.full((B, Hkv, N, K), -1, dtype=torch.int32)
    for b in range(B):
        for kv in range(Hkv):
            for i in range(N):
                nv = i // C + 1
                pick = torch.randperm(nv, generator=gen)[:K].sort().values
                idx[b, kv, i, :len(pick)] = pick.to(torch.int32)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K)
    O, lse = pisa.sparse_attn_fwd(Qg, Kg, Vg, idx.cuda(), shape)
    Oref, lref = po.sparse_attn_fwd(Q, Kt, V, idx.numpy(), C)
    check_close(O.float().cpu().numpy(), Oref, what="O")
    check_close(lse.cpu().numpy(), lref, atol=1e-3, rtol=0, what="lse")
    # the same selection with caller-supplied block LSEs (the oracle's, rounded to fp32)
    hl = torch.from_numpy(po.selected_head_lse(Q, Kt, idx.numpy(), C)).float().cuda()
    O2, lse2 = pisa.sparse_attn_fwd(Qg, Kg, Vg, idx.cuda(), shape, head_lse=hl)
    check_close(O2.float().cpu().numpy(), Oref, what="O (head_lse)")
    check_close(lse2.cpu().numpy(), lref, atol=1e-3, rtol=0, what="lse (head_lse)")
    # the same leaves in shuffled slots (padding interleaved): the output pass, which takes
    # sibling leaves together, finds a row's siblings wherever its slots hold them
    perm = torch.argsort(torch.rand((B, Hkv, N, K), generator=gen), dim=-1)
    idx_s = torch.gather(idx, -1, perm)
    hl_s = torch.from_numpy(po.selected_head_lse(Q, Kt, idx_s.numpy(), C)).float().cuda()
    O3, lse3 = pisa.sparse_attn_fwd(Qg, Kg, Vg, idx_s.cuda(), shape, head_lse=hl_s)
    check_close(O3.float().cpu().numpy(), Oref, what="O (shuffled slots)")
    check_close(lse3.cpu().numpy(), lref, atol=1e-3, rtol=0, what="lse (shuffled slots)")


@pytest.mark.parametrize("name,Hq,Hkv,N", [("prefill_64k_gqa8", 16, 2, 65536), ("sweep_64k_gqa4", 32, 8, 65536)])
def test_full_size_sampled_vs_oracle(name, Hq, Hkv, N):
    # The 64K workloads at full size, launched as the benchmark launches them; the oracle
    # checks a deterministic sample of queries (units are independent once the pyramid is
    # fixed).
    B, d, K = 1, 128, 16
    (Q, Kt, V), (Qg, Kg, Vg) = _inputs(B, N, Hq, Hkv, d, True)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=4)
    pyr = pisa.build_pyramid(Kg, shape)
    idx, score, hl = pisa.select(Qg, Kg, pyr, shape, want_head_lse=True)
    fidx, fscore = pisa.select_flat(Qg, Kg, pyr, shape)
    O, lse = pisa.sparse_attn_fwd(Qg, Kg, Vg, idx, shape, head_lse=hl)
    O_own, lse_own = pisa.sparse_attn_fwd(Qg, Kg, Vg, idx, shape)     # block LSEs recomputed
    torch.cuda.synchronize()
    qs = sorted(set(range(0, N, 4099)) | {0, 1, 63, 64, 4095, 4096, N - 2, N - 1})
    ora = po.select(Q, Kt, C, K, queries=qs)
    gi = idx.cpu().numpy()
    check_selection(gi, score.cpu().numpy(), ora, qs, C, K, N)
    hl_ref = po.selected_head_lse(Q, Kt, gi, C, queries=qs)
    _check_head_lse(hl.cpu().numpy()[:, :, qs], hl_ref[:, :, qs])
    fora = po.select_flat(Q, Kt, C, K, queries=qs)
    check_selection(fidx.cpu().numpy(), fscore.cpu().numpy(), fora, qs, C, K, N)
    # attention of the GPU path's own selection, re-derived by the oracle from the oracle's
    # idx where they agree (exempt units are skipped)
    same = [i for i in qs if np.array_equal(gi[:, :, i], ora["idx"][:, :, i])]
    Oref, lref = po.sparse_attn_fwd(Q, Kt, V, ora["idx"], C, queries=same)
    for Og, lg, tag in ((O, lse, "head_lse"), (O_own, lse_own, "own LSE pass")):
        check_close(Og.float().cpu().numpy()[:, same], Oref[:, same], what=f"O ({tag})")
        check_close(lg.cpu().numpy()[:, :, same], lref[:, :, same], atol=1e-3, rtol=0, what=f"lse ({tag})")


# ------------------------------------------------------------------------------- decode
def _decode_run(B, Ncap, L0, Hq, Hkv, d, K, steps, device="cpu", seed=0):
    Kc = syn.randn_bf16((B, Ncap, Hkv, d), seed + 1, device)
    Vc = syn.randn_bf16((B, Ncap, Hkv, d), seed + 2, device)
    qs, ks, vs = syn.make_decode_stream(B, steps, Hq, Hkv, d, seed=seed, device=device)
    return Kc, Vc, qs, ks, vs


def test_decode_vs_oracle_and_prefill():
    B, Ncap, Hq, Hkv, d, K, steps = 2, 1000, 8, 2, 128, 8, 6
    L0 = [700, 937]
    Kc, Vc, qs, ks, vs = _decode_run(B, Ncap, L0, Hq, Hkv, d, K, steps)
    shape = pisa.make_decode_shape(B, Ncap, Hq, Hkv, d, C, K)
    Kg, Vg = Kc.cuda(), Vc.cuda()
    length = torch.tensor(L0, dtype=torch.int32, device="cuda")
    pyr = pisa.decode_build_pyramid(Kg, length, shape)
    states = [po.DecodeState(Kc[b:b + 1], Vc[b:b + 1], L0[b], C) for b in range(B)]
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    last_margin = [None] * B
    for t in range(steps):
        score = torch.empty(B, Hkv, K, device="cuda")
        o, idx, _, _ = pisa.decode_step(shape, length, Kg, Vg, pyr, qs[t].cuda(), ks[t].cuda(), vs[t].cuda(),
                                        score=score, status=status)
        torch.cuda.synchronize()
        for b in range(B):
            oo, oi, osc, om = states[b].step(qs[t][b:b + 1], ks[t][b:b + 1], vs[t][b:b + 1], K)
            last_margin[b] = om[0]
            p = L0[b] + t
            gi = idx.cpu().numpy()[b:b + 1, :, None, :]
            gs = score.cpu().numpy()[b:b + 1, :, None, :]
            # compare as a one-query selection at "query index" p
            full_i = np.full((1, Hkv, p + 1, K), -1, np.int32)
            full_s = np.full((1, Hkv, p + 1, K), np.nan)
            full_i[:, :, p], full_s[:, :, p] = gi[:, :, 0], gs[:, :, 0]
            ofull = dict(idx=np.full((1, Hkv, p + 1, K), -1, np.int32), score=np.full((1, Hkv, p + 1, K), np.nan),
                         margin=np.full((1, Hkv, p + 1), np.inf))
            ofull["idx"][:, :, p] = oi
            ofull["score"][:, :, p] = osc
            ofull["margin"][:, :, p] = om
            check_selection(full_i, full_s, ofull, [p], C, K, p + 1)
            if np.array_equal(gi[:, :, 0], oi):
                check_close(o[b].float().cpu().numpy(), oo[0], what=f"decode o step {t} seq {b}")
        assert int(status.sum()) == 0
        length += 1
    # the incrementally updated pyramid equals a rebuilt one, bit for bit
    rebuilt = pisa.decode_build_pyramid(Kg, length, shape)
    assert torch.equal(pyr, rebuilt)
    # and equals the prefill build over tokens 0..p on every node the prefill pyramid has
    n_lv, off_d, _ = pisa.decode_pyramid_layout(shape)
    for b in range(B):
        p1 = int(length[b])
        pshape = pisa.make_shape(1, p1, Hq, Hkv, d, C, K)
        pp = pisa.build_pyramid(Kg[b:b + 1, :p1].contiguous(), pshape)
        n_lp, off_p, _ = pisa.pyramid_layout(pshape)
        sizes = po.level_sizes(p1, C)
        for l in range(n_lp):
            assert torch.equal(pp[0, :, off_p[l]:off_p[l] + sizes[l]], pyr[b, :, off_d[l]:off_d[l] + sizes[l]]), (b, l)
    # decode(p) equals prefill's query p (same GPU library, two code paths); units whose
    # oracle margin is below the exemption threshold may differ
    for b in range(B):
        p = int(length[b]) - 1
        Qp = torch.zeros(1, p + 1, Hq, d, dtype=torch.bfloat16, device="cuda")
        Qp[0, p] = qs[steps - 1][b].cuda()
        pshape = pisa.make_shape(1, p + 1, Hq, Hkv, d, C, K)
        Kp = Kg[b:b + 1, :p + 1].contiguous()
        pi, ps = pisa.select(Qp, Kp, pisa.build_pyramid(Kp, pshape), pshape)
        for kv in range(Hkv):
            if torch.equal(pi[0, kv, p], idx[b, kv]):
                torch.testing.assert_close(ps[0, kv, p], score[b, kv], atol=1e-4, rtol=0)
            else:
                assert last_margin[b][kv] < 1e-3, (b, kv, pi[0, kv, p], idx[b, kv])


def test_decode_rejects_out_of_range_position_without_fault():
    B, Ncap, Hq, Hkv, d, K = 2, 300, 4, 1, 64, 4
    Kc, Vc, qs, ks, vs = _decode_run(B, Ncap, None, Hq, Hkv, d, K, 1)
    shape = pisa.make_decode_shape(B, Ncap, Hq, Hkv, d, C, K)
    Kg, Vg = Kc.cuda(), Vc.cuda()
    length = torch.tensor([10, Ncap], dtype=torch.int32, device="cuda")     # seq 1 is full
    pyr = pisa.decode_build_pyramid(Kg, length, shape)
    before = (Kg.clone(), pyr.clone())
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    pisa.decode_step(shape, length, Kg, Vg, pyr, qs[0].cuda(), ks[0].cuda(), vs[0].cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 1
    assert torch.equal(Kg[1], before[0][1]) and torch.equal(pyr[1], before[1][1])
    assert not torch.equal(Kg[0], before[0][0])      # the valid sequence advanced


def test_decode_full_size_sampled():
    # The batch-32 decode workload over a 131072-token cache, 4 steps; the oracle follows two
    # of the 32 sequences.
    B, Ncap, Hq, Hkv, d, K, L0, steps = 32, 131328, 32, 8, 128, 16, 131072, 4
    Kc, Vc, qs, ks, vs = _decode_run(B, Ncap, L0, Hq, Hkv, d, K, steps, device="cuda")
    shape = pisa.make_decode_shape(B, Ncap, Hq, Hkv, d, C, K)
    length = torch.full((B,), L0, dtype=torch.int32, device="cuda")
    pyr = pisa.decode_build_pyramid(Kc, length, shape)
    follow = [0, 17]
    states = [po.DecodeState(Kc[b:b + 1].cpu(), Vc[b:b + 1].cpu(), L0, C) for b in follow]
    for t in range(steps):
        score = torch.empty(B, Hkv, K, device="cuda")
        o, idx, _, status = pisa.decode_step(shape, length, Kc, Vc, pyr, qs[t], ks[t], vs[t], score=score)
        torch.cuda.synchronize()
        assert int(status.sum()) == 0
        for st, b in zip(states, follow):
            oo, oi, osc, om = st.step(qs[t][b:b + 1].cpu(), ks[t][b:b + 1].cpu(), vs[t][b:b + 1].cpu(), K)
            gi = idx[b].cpu().numpy()
            for kv in range(Hkv):
                if np.array_equal(gi[kv], oi[0, kv]):
                    np.testing.assert_allclose(score[b, kv].cpu().numpy(), osc[0, kv], atol=SCORE_ATOL, rtol=0)
                    G = Hq // Hkv
                    check_close(o[b, kv * G:(kv + 1) * G].float().cpu().numpy(), oo[0, kv * G:(kv + 1) * G],
                                what="decode o")
                else:
                    assert om[0, kv] < 1e-3, (t, b, kv, gi[kv], oi[0, kv])
        length += 1
