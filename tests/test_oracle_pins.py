"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: values the pages print,
closed forms, a textbook library routine, brute force on tiny inputs, finite differences,
or an invariant. A plausible slip in the oracle (a dropped term, a wrong index or sign, a
transposed operand, a wrong tie rule, a non-causal summary) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import pisa_oracle as po

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    r = np.random.default_rng(seed)
    # bf16-exact values, like the real inputs
    return torch.from_numpy(r.standard_normal(shape) * scale).to(torch.bfloat16).to(torch.float64).numpy()


# ---------------------------------------------------------------- pyramid geometry
def test_level_counts_match_printed_values():
    with open(os.path.join(GOLD, "level_counts.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        sizes = po.level_sizes(c["N"], c["C"])
        if "levels" in c:
            assert len(sizes) == c["levels"]
            assert sizes[0] == c["leaves"]
        if "pooled_levels" in c:
            assert len(sizes) - 1 == c["pooled_levels"]
            assert len(sizes) - 1 == math.ceil(math.log2(c["N"] / c["C"]))


@pytest.mark.parametrize("N,C", [(64, 4), (67, 4), (40, 8), (8, 8), (1, 8), (129, 16)])
def test_pyramid_sums_are_direct_range_means(N, C):
    K = _rand((N, 5), 1)
    sums = po.pyramid_sums(K, C)
    # merge factor 2: a parent is the sum of its two children (closed form)
    for l in range(1, len(sums)):
        for m in range(len(sums[l])):
            kids = [c for c in (2 * m, 2 * m + 1) if c < len(sums[l - 1])]
            np.testing.assert_allclose(sums[l][m], sum(sums[l - 1][c] for c in kids), rtol=1e-12, atol=1e-12)
    # leaf means against pure-Python token loops
    for t in range(len(sums[0])):
        toks = [j for j in range(N) if j // C == t]
        ref = [sum(K[j, k] for j in toks) / len(toks) for k in range(5)]
        np.testing.assert_allclose(sums[0][t] / len(toks), ref, rtol=1e-12, atol=1e-12)
    assert len(sums[-1]) == 1
    np.testing.assert_allclose(sums[-1][0], K.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_mean_pooling_equals_library_avg_pool():
    N, C, d = 256, 8, 6
    K = _rand((N, d), 2)
    sums = po.pyramid_sums(K, C)
    x = torch.from_numpy(K.T.copy()).unsqueeze(0)             # [1, d, N]
    for l in range(len(sums)):
        pooled = torch.nn.functional.avg_pool1d(x, kernel_size=C << l, stride=C << l)[0].T.numpy()
        np.testing.assert_allclose(sums[l] / (C << l), pooled, rtol=1e-12, atol=1e-12)


def test_causal_means_match_direct_prefix_means():
    N, C, d = 45, 4, 3
    K = _rand((N, d), 3)
    summ = po.CausalKeySummaries(K, C)
    for l, n in enumerate(summ.sizes):
        for m in range(n):
            s, e = po.node_range(l, m, C, N)
            for i in range(N):
                if s > i:
                    assert not summ.visible(l, m, i)
                    continue
                assert summ.visible(l, m, i)
                ref = K[s:min(e, i + 1)].mean(axis=0)
                np.testing.assert_allclose(summ.means(l, np.array([m]), i)[0], ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- descent vs brute force
def _bf_mean(K, l, m, i, C):
    N = K.shape[0]
    toks = [j for j in range(m * (C << l), min((m + 1) * (C << l), N)) if j <= i]
    return [sum(K[j, k] for j in toks) / len(toks) for k in range(K.shape[1])]


def _bf_score(q, K, l, m, i, C, s):
    """Independent scalar-loop enumerator of S_i(l, m)."""
    N = K.shape[0]
    tot = 0.0
    for h in range(q.shape[0]):
        if l == 0:
            vals = [s * sum(q[h, k] * K[j, k] for k in range(K.shape[1]))
                    for j in range(m * C, min((m + 1) * C, N)) if j <= i]
        else:
            vals = []
            for c in (2 * m, 2 * m + 1):
                if c * (C << (l - 1)) <= i and c * (C << (l - 1)) < N:
                    mu = _bf_mean(K, l - 1, c, i, C)
                    vals.append(s * sum(q[h, k] * mu[k] for k in range(K.shape[1])))
        mx = max(vals)
        tot += mx + math.log(sum(math.exp(v - mx) for v in vals))
    return tot


def _bf_mean_score(q, K, l, m, i, C, s):
    """PISA-1 score by token loops: sum_h s q_h . mean of the node's keys j <= i."""
    N = K.shape[0]
    toks = [j for j in range(m * (C << l), min((m + 1) * (C << l), N)) if j <= i]
    tot = 0.0
    for h in range(q.shape[0]):
        tot += s * sum(q[h, k] * sum(K[j, k] for j in toks) / len(toks) for k in range(K.shape[1]))
    return tot


def _bf_select(q, K, i, C, Ksel, s, score_fn=None):
    score_fn = score_fn or _bf_score
    N = K.shape[0]
    n = [-(-N // C)]
    while n[-1] > 1:
        n.append(-(-n[-1] // 2))
    table = {}
    for l in range(len(n)):
        for m in range(n[l]):
            if m * (C << l) <= i:
                table[(l, m)] = score_fn(q, K, l, m, i, C, s)
    kept = {0}
    for l in range(len(n) - 2, -1, -1):
        cand = sorted({c for a in kept for c in (2 * a, 2 * a + 1) if (l, c) in table})
        if len(cand) > Ksel or l == 0:
            cand.sort(key=lambda c: (-table[(l, c)], c))
            kept = set(cand[:Ksel])
        else:
            kept = set(cand)
    if len(n) == 1:
        kept = {0}
    leaves = sorted(kept)
    return leaves, [table[(0, t)] for t in leaves]


@pytest.mark.parametrize("N,C,Ksel,G,seed", [
    (64, 4, 1, 1, 0), (64, 4, 2, 2, 1), (96, 4, 3, 2, 2), (72, 8, 2, 1, 3),
    (128, 8, 3, 2, 4), (61, 4, 2, 2, 5), (200, 8, 1, 2, 6), (256, 4, 3, 1, 7)])
def test_descent_matches_brute_force(N, C, Ksel, G, seed):
    d = 4
    Q = _rand((1, N, G, d), 10 + seed, scale=2.0)
    K = _rand((1, N, 1, d), 20 + seed, scale=2.0)
    s = 0.7
    out = po.select(Q, K, C, Ksel, scale=s)
    rng = np.random.default_rng(seed)
    for i in sorted(set(rng.integers(0, N, 12).tolist()) | {0, N - 1}):
        leaves, scores = _bf_select(Q[0, i], K[0, :, 0, :], i, C, Ksel, s)
        got = out["idx"][0, 0, i]
        assert list(got[got >= 0]) == leaves, (i, got, leaves)
        np.testing.assert_allclose(out["score"][0, 0, i, :len(leaves)], scores, rtol=1e-12, atol=1e-12)
        assert np.all(out["score"][0, 0, i, len(leaves):] == -np.inf)


@pytest.mark.parametrize("N,C,Ksel,G,seed", [
    (64, 4, 1, 1, 0), (96, 4, 3, 2, 2), (128, 8, 3, 2, 4), (61, 4, 2, 2, 5), (200, 8, 1, 2, 6)])
def test_pisa1_descent_matches_brute_force(N, C, Ksel, G, seed):
    d = 4
    Q = _rand((1, N, G, d), 40 + seed, scale=2.0)
    K = _rand((1, N, 1, d), 50 + seed, scale=2.0)
    s = 0.7
    out = po.select_mean(Q, K, C, Ksel, scale=s)
    rng = np.random.default_rng(seed)
    for i in sorted(set(rng.integers(0, N, 12).tolist()) | {0, N - 1}):
        leaves, scores = _bf_select(Q[0, i], K[0, :, 0, :], i, C, Ksel, s, _bf_mean_score)
        got = out["idx"][0, 0, i]
        assert list(got[got >= 0]) == leaves, (i, got, leaves)
        np.testing.assert_allclose(out["score"][0, 0, i, :len(leaves)], scores, rtol=1e-12, atol=1e-12)
        assert np.all(out["score"][0, 0, i, len(leaves):] == -np.inf)


def test_pisa1_keep_all_and_no_pruning_cases():
    N, C, G, d = 96, 8, 2, 6
    Q = _rand((1, N, G, d), 60)
    K = _rand((1, N, 1, d), 61)
    n0 = -(-N // C)
    # K >= n0: every visible leaf, in order
    out = po.select_mean(Q, K, C, n0)
    for i in range(N):
        got = out["idx"][0, 0, i]
        assert list(got[got >= 0]) == list(range(i // C + 1))
    # 2K >= n0: no intermediate level prunes, so the leaf stage sees every visible leaf and
    # PISA-1 is the flat top-K of the mean scores
    Ksel = -(-n0 // 2)
    a = po.select_mean(Q, K, C, Ksel)
    b = po.select_flat(Q, K, C, Ksel)
    np.testing.assert_array_equal(a["idx"], b["idx"])


def test_descent_invariants():
    N, C, Ksel, G, d = 512, 4, 3, 2, 4
    Q = _rand((1, N, G, d), 30)
    K = _rand((1, N, 1, d), 31)
    summ = po.CausalKeySummaries(K[0, :, 0, :], C)
    for i in range(0, N, 7):
        u = po.select_unit(Q[0, i], i, summ, Ksel, 0.5)
        assert all(c <= 2 * Ksel for c in u.cand_sizes)            # at most gK candidates per level
        assert np.all(u.leaves <= i // C) and np.all(np.diff(u.leaves) > 0)
        assert set(u.leaves.tolist()) <= set(u.leaf_candidates.tolist())
        parents = {int(t) // 2 for t in u.leaf_candidates}
        assert len(parents) <= Ksel                                 # candidates are children of <= K kept nodes
        assert len(u.leaves) == min(Ksel, i // C + 1)


# ---------------------------------------------------------------- special cases
def test_zero_query_closed_form():
    with open(os.path.join(GOLD, "zero_query.json")) as f:
        g = json.load(f)
    sh = g["shape"]
    Q = np.zeros((1, sh["N"], sh["G"], sh["d"]))
    K = _rand((1, sh["N"], 1, sh["d"]), 40)
    for c in g["cases"]:
        out = po.select(Q, K, sh["C"], c["K"], queries=[c["i"]])
        got = out["idx"][0, 0, c["i"]]
        assert list(got[got >= 0]) == c["leaves"]
        want = [eval(x, {"log": math.log}) for x in c["scores"]]
        np.testing.assert_allclose(out["score"][0, 0, c["i"], :len(want)], want, rtol=0, atol=1e-12)


def test_keep_all_returns_every_visible_leaf():
    with open(os.path.join(GOLD, "keep_all.json")) as f:
        g = json.load(f)
    sh = g["shape"]
    Q = _rand((1, sh["N"], sh["G"], sh["d"]), 41)
    K = _rand((1, sh["N"], 1, sh["d"]), 42)
    out = po.select(Q, K, sh["C"], sh["K"])
    flat = po.select_flat(Q, K, sh["C"], sh["K"])
    for c in g["cases"]:
        for o in (out, flat):
            got = o["idx"][0, 0, c["i"]]
            assert list(got[got >= 0]) == c["leaves"]
    # and for every query of a larger random case
    N, C = 300, 8
    Q = _rand((1, N, 2, 8), 43)
    K = _rand((1, N, 1, 8), 44)
    out = po.select(Q, K, C, 38)
    for i in range(N):
        got = out["idx"][0, 0, i]
        assert list(got[got >= 0]) == list(range(i // C + 1))


def test_no_intermediate_pruning_equals_exhaustive():
    # K >= number of level-1 nodes: no intermediate level prunes, so the leaf stage sees
    # every visible leaf and PISA reduces to exhaustive exact scoring + top-K.
    N, C, G, d = 128, 4, 2, 4
    Ksel = 16                      # n0 = 32, n1 = 16
    Q = _rand((1, N, G, d), 50, 1.5)
    K = _rand((1, N, 1, d), 51, 1.5)
    a = po.select(Q, K, C, Ksel)
    b = po.select_exhaustive(Q, K, C, Ksel)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_allclose(a["score"], b["score"], rtol=1e-12, atol=1e-12)


def test_planted_block_wins():
    N, C, G, d = 256, 8, 2, 8
    Q = _rand((1, N, G, d), 60)
    K = _rand((1, N, 1, d), 61) * 0.1
    direction = Q[0, N - 1].sum(axis=0)
    star = 13
    K[0, star * C:(star + 1) * C, 0, :] += 4.0 * direction / np.linalg.norm(direction)
    out = po.select(Q, K, C, 1, queries=[N - 1])
    assert list(out["idx"][0, 0, N - 1]) == [star]


def test_exact_ties_go_to_lower_index():
    N, C, G, d = 128, 4, 2, 4
    Q = _rand((1, N, G, d), 70)
    blk = _rand((C, d), 71)
    K = np.tile(blk, (N // C, 1))[None, :, None, :]      # every leaf holds the same keys
    out = po.select(Q, K, C, 3, queries=[N - 1, 77])
    assert list(out["idx"][0, 0, N - 1]) == [0, 1, 2]
    assert list(out["idx"][0, 0, 77]) == [0, 1, 2]


def test_constant_leaves_closed_forms():
    # Keys constant inside each leaf: mu_i(0,t) = k_t, so the flat score is s sum_h q_h.k_t
    # and the exact leaf score is sum_h (s q_h.k_t + log n_t), n_t = visible keys of t.
    N, C, G, d, Ksel = 96, 8, 2, 6, 3
    Q = _rand((1, N, G, d), 80)
    kt = _rand((N // C, d), 81)
    K = np.repeat(kt, C, axis=0)[None, :, None, :]
    s = 0.4
    qs = [5, 40, 95]
    flat = po.select_flat(Q, K, C, Ksel, scale=s, queries=qs)
    exh = po.select_exhaustive(Q, K, C, Ksel, scale=s, queries=qs)
    for i in qs:
        vis = np.arange(i // C + 1)
        base = s * torch.from_numpy(Q[0, i]).sum(0).numpy() @ kt[vis].T          # library matmul
        n_t = np.array([min((t + 1) * C, i + 1) - t * C for t in vis])
        exact = base + G * np.log(n_t)
        for o, sc in ((flat, base), (exh, exact)):
            order = sorted(range(len(vis)), key=lambda r: (-sc[r], r))[:Ksel]
            got = o["idx"][0, 0, i]
            assert list(got[got >= 0]) == sorted(order)
            np.testing.assert_allclose(o["score"][0, 0, i, :len(order)], sc[sorted(order)], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- attention
def _sdpa_dense(Q, K, V, s):
    G = Q.shape[2] // K.shape[2]
    q = torch.from_numpy(Q).permute(0, 2, 1, 3)
    k = torch.from_numpy(K).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    v = torch.from_numpy(V).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    return q, k, v


def test_attention_all_selected_equals_sdpa():
    B, N, Hq, Hkv, d, C = 2, 70, 4, 2, 8, 8
    Q, K, V = _rand((B, N, Hq, d), 90), _rand((B, N, Hkv, d), 91), _rand((B, N, Hkv, d), 92)
    s = 0.3
    n0 = -(-N // C)
    idx = np.tile(np.arange(n0, dtype=np.int32), (B, Hkv, N, 1))
    O, lse = po.sparse_attn_fwd(Q, K, V, idx, C, scale=s)
    q, k, v = _sdpa_dense(Q, K, V, s)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=s)
    np.testing.assert_allclose(O, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12)
    logits = (q @ k.transpose(-1, -2)) * s
    logits = logits.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(logits, dim=-1).numpy(), rtol=1e-12, atol=1e-12)


def _random_idx(B, Hkv, N, C, Ksel, seed):
    """Random ascending leaf lists of visible leaves, -1 padded, some rows short."""
    r = np.random.default_rng(seed)
    idx = np.full((B, Hkv, N, Ksel), -1, dtype=np.int32)
    for b in range(B):
        for kv in range(Hkv):
            for i in range(N):
                vis = i // C + 1
                n = min(vis, int(r.integers(1, Ksel + 1)))
                idx[b, kv, i, :n] = np.sort(r.choice(vis, size=n, replace=False))
    return idx


def test_selected_head_lse_equals_masked_dense_logsumexp():
    # Per-head block LSE against torch.logsumexp over dense logits with a block-and-causal mask.
    B, N, Hq, Hkv, d, C, Ksel = 1, 45, 4, 2, 8, 8, 3
    Q, K = _rand((B, N, Hq, d), 120), _rand((B, N, Hkv, d), 121)
    s = 0.7
    idx = _random_idx(B, Hkv, N, C, Ksel, 122)
    got = po.selected_head_lse(Q, K, idx, C, scale=s)
    q, k, _ = _sdpa_dense(Q, K, K, s)
    logits = (q @ k.transpose(-1, -2)) * s                    # [B, Hq, N, N]
    j = torch.arange(N)
    for h in range(Hq):
        for i in range(N):
            for slot in range(Ksel):
                t = int(idx[0, h // (Hq // Hkv), i, slot])
                if t < 0:
                    assert got[0, h, i, slot] == -np.inf
                    continue
                keep = (j // C == t) & (j <= i)
                ref = torch.logsumexp(logits[0, h, i].masked_fill(~keep, float("-inf")), dim=0)
                assert abs(got[0, h, i, slot] - ref.item()) < 1e-12


def test_block_lses_combine_to_attention_lse():
    # LSE over a disjoint union of key sets = LSE of the per-set LSEs.
    B, N, Hq, Hkv, d, C, Ksel = 2, 40, 4, 1, 8, 8, 4
    Q, K, V = _rand((B, N, Hq, d), 123), _rand((B, N, Hkv, d), 124), _rand((B, N, Hkv, d), 125)
    idx = _random_idx(B, Hkv, N, C, Ksel, 126)
    hl = po.selected_head_lse(Q, K, idx, C, scale=0.4)
    _, lse = po.sparse_attn_fwd(Q, K, V, idx, C, scale=0.4)
    np.testing.assert_allclose(torch.logsumexp(torch.from_numpy(hl), dim=-1).numpy(), lse, rtol=1e-12, atol=1e-12)


def test_head_lse_of_the_selection_sums_to_its_scores():
    # The selection's leaf score is the group sum of the per-head leaf LSEs.
    B, N, Hq, Hkv, d, C, Ksel = 1, 96, 4, 2, 8, 8, 3
    Q, K = _rand((B, N, Hq, d), 127), _rand((B, N, Hkv, d), 128)
    o = po.select(Q, K, C, Ksel, scale=0.5)
    hl = po.selected_head_lse(Q, K, o["idx"], C, scale=0.5)
    G = Hq // Hkv
    summed = hl.reshape(B, Hkv, G, N, Ksel).sum(axis=2)
    ok = o["idx"] >= 0
    np.testing.assert_allclose(summed[ok], o["score"][ok], rtol=1e-12, atol=1e-12)
    assert np.all(np.isneginf(summed[~ok]))


def test_attention_masks_unselected_blocks():
    # Only leaf 1 selected: the output must be the softmax over exactly its visible keys.
    B, N, Hq, Hkv, d, C = 1, 32, 2, 1, 4, 8
    Q, K, V = _rand((B, N, Hq, d), 93), _rand((B, N, Hkv, d), 94), _rand((B, N, Hkv, d), 95)
    idx = np.full((B, Hkv, N, 2), -1, dtype=np.int32)
    idx[..., 0] = 1
    O, _ = po.sparse_attn_fwd(Q, K, V, idx, C, scale=1.0, queries=[12, 31])
    for i in (12, 31):
        J = list(range(8, min(16, i + 1)))
        for h in range(Hq):
            w = np.exp([Q[0, i, h] @ K[0, j, 0] for j in J])
            w /= w.sum()
            np.testing.assert_allclose(O[0, i, h], w @ V[0, J, 0], rtol=1e-12, atol=1e-12)


def test_backward_all_selected_equals_autograd():
    B, N, Hq, Hkv, d, C = 1, 40, 4, 2, 8, 8
    Q, K, V = _rand((B, N, Hq, d), 100), _rand((B, N, Hkv, d), 101), _rand((B, N, Hkv, d), 102)
    dO = _rand((B, N, Hq, d), 103)
    s = 0.35
    idx = np.tile(np.arange(N // C, dtype=np.int32), (B, Hkv, N, 1))
    dQ, dK, dV = po.sparse_attn_bwd(Q, K, V, dO, idx, C, scale=s)
    q = torch.from_numpy(Q).requires_grad_()
    k = torch.from_numpy(K).requires_grad_()
    v = torch.from_numpy(V).requires_grad_()
    G = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        q.permute(0, 2, 1, 3), k.repeat_interleave(G, 2).permute(0, 2, 1, 3),
        v.repeat_interleave(G, 2).permute(0, 2, 1, 3), is_causal=True, scale=s)
    (o.permute(0, 2, 1, 3) * torch.from_numpy(dO)).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_backward_finite_differences_sparse():
    B, N, Hq, Hkv, d, C = 1, 24, 2, 1, 4, 4
    Q, K, V = _rand((B, N, Hq, d), 110), _rand((B, N, Hkv, d), 111), _rand((B, N, Hkv, d), 112)
    dO = _rand((B, N, Hq, d), 113)
    sel = po.select(Q, K, C, 2)
    idx = sel["idx"]
    dQ, dK, dV = po.sparse_attn_bwd(Q, K, V, dO, idx, C, scale=0.5)

    def loss(Q_, K_, V_):
        O, _ = po.sparse_attn_fwd(Q_, K_, V_, idx, C, scale=0.5)
        return float((O * dO).sum())

    eps = 1e-6
    rng = np.random.default_rng(0)
    for name, X, G_ in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        for _ in range(6):
            pos = tuple(int(rng.integers(0, n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[pos] += eps
            Xm[pos] -= eps
            args_p = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
            args_m = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - G_[pos]) < 1e-6 * max(1.0, abs(fd)), (name, pos, fd, G_[pos])


# ---------------------------------------------------------------- decode
def test_decode_incremental_pyramid_equals_rebuilt_and_prefill():
    B, Ncap, Hq, Hkv, d, C, Ksel = 2, 96, 4, 2, 4, 4, 2
    L0, steps = 37, 11
    Kc, Vc = _rand((B, Ncap, Hkv, d), 120), _rand((B, Ncap, Hkv, d), 121)
    Kc[:, L0:] = 0.0
    Vc[:, L0:] = 0.0
    qs, ks, vs = _rand((steps, B, Hq, d), 122), _rand((steps, B, Hkv, d), 123), _rand((steps, B, Hkv, d), 124)
    st = po.DecodeState(Kc, Vc, L0, C)
    for t in range(steps):
        o, idx, score, _ = st.step(qs[t], ks[t], vs[t], Ksel, scale=0.5)
        p = L0 + t
        # the incrementally maintained pyramid equals one rebuilt from the cache
        rb = po.DecodeState(st.K, st.V, p + 1, C)
        for l in range(len(st.sums)):
            np.testing.assert_allclose(st.sums[l], rb.sums[l], rtol=1e-12, atol=1e-12)
        # decode at step p equals prefill's query p (a shorter pyramid: height invariance)
        Qp = np.zeros((B, p + 1, Hq, d))
        Qp[:, p] = qs[t]
        pre = po.select(Qp, st.K[:, :p + 1], C, Ksel, scale=0.5, queries=[p])
        np.testing.assert_array_equal(idx, pre["idx"][:, :, p])
        np.testing.assert_allclose(score, pre["score"][:, :, p], rtol=1e-10, atol=1e-10)
        Op, _ = po.sparse_attn_fwd(Qp, st.K[:, :p + 1], st.V[:, :p + 1], pre["idx"], C, scale=0.5, queries=[p])
        np.testing.assert_allclose(o, Op[:, p], rtol=1e-10, atol=1e-12)


def test_sampled_backward_equals_full_backward():
    B, N, Hq, Hkv, d, C = 2, 50, 4, 2, 4, 8
    Q, K, V = _rand((B, N, Hq, d), 130), _rand((B, N, Hkv, d), 131), _rand((B, N, Hkv, d), 132)
    dO = _rand((B, N, Hq, d), 133)
    idx = po.select(Q, K, C, 2)["idx"]
    dQ, dK, dV = po.sparse_attn_bwd(Q, K, V, dO, idx, C, scale=0.4)
    qs = [(0, 0), (1, 17), (0, 49)]
    ls = [(0, 0, 0), (1, 1, 3), (0, 1, 6)]
    sq, sk, sv = po.sparse_attn_bwd_sampled(Q, K, V, dO, idx, C, scale=0.4, queries=qs, leaves=ls)
    for (b, i) in qs:
        np.testing.assert_allclose(sq[(b, i)], dQ[b, i], rtol=1e-12, atol=1e-13)
    for (b, kv, t) in ls:
        s0, e0 = po.node_range(0, t, C, N)
        np.testing.assert_allclose(sk[(b, kv, t)], dK[b, s0:e0, kv], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sv[(b, kv, t)], dV[b, s0:e0, kv], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- pruning margin
# The oracle reports, per unit, the smallest gap between the K-th and (K+1)-th ranked scores
# over every level that prunes (its candidate set holds more than K). The GPU parity tests
# exempt a unit from the exact index match when that margin is below 1e-3, so the margin
# itself is pinned here: against a brute-force descent that records the gap of every level
# from its own score table, and against closed forms.
def _bf_descent_gaps(q, K, i, C, Ksel, s, score_fn=None):
    """Brute-force descent (scores from the scalar enumerator) that also returns the
    K-th vs (K+1)-th gap of every level whose candidate set exceeds K, keyed by level."""
    score_fn = score_fn or _bf_score
    N = K.shape[0]
    n = [-(-N // C)]
    while n[-1] > 1:
        n.append(-(-n[-1] // 2))
    table = {(l, m): score_fn(q, K, l, m, i, C, s)
             for l in range(len(n)) for m in range(n[l]) if m * (C << l) <= i}
    kept, gaps = {0}, {}
    for l in range(len(n) - 2, -1, -1):
        cand = sorted({c for a in kept for c in (2 * a, 2 * a + 1) if (l, c) in table})
        ranked = sorted(cand, key=lambda c: (-table[(l, c)], c))
        if len(cand) > Ksel:
            gaps[l] = table[(l, ranked[Ksel - 1])] - table[(l, ranked[Ksel])]
        kept = set(ranked[:Ksel]) if (len(cand) > Ksel or l == 0) else set(cand)
    return gaps


MARGIN_CASES = [(64, 4, 1, 1, 0), (96, 4, 3, 2, 2), (128, 8, 3, 2, 4), (200, 8, 1, 2, 6),
                (256, 4, 3, 1, 7), (256, 4, 2, 2, 8)]


def _check_margins(select_fn, score_fn, seed_base):
    """Raises AssertionError where select_fn's margin differs from the brute-force minimum gap.
    Returns which levels supplied the minimum (to show that both kinds are exercised)."""
    sources = set()
    for N, C, Ksel, G, seed in MARGIN_CASES:
        d = 4
        Q = _rand((1, N, G, d), seed_base + seed, scale=2.0)
        K = _rand((1, N, 1, d), seed_base + 50 + seed, scale=2.0)
        s = 0.7
        rng = np.random.default_rng(seed)
        qs = sorted(set(rng.integers(0, N, 10).tolist()) | {N - 1})
        out = select_fn(Q, K, C, Ksel, scale=s, queries=qs)
        for i in qs:
            gaps = _bf_descent_gaps(Q[0, i], K[0, :, 0, :], i, C, Ksel, s, score_fn)
            want = min(gaps.values()) if gaps else np.inf
            got = out["margin"][0, 0, i]
            assert (got == want) if not np.isfinite(want) else abs(got - want) <= 1e-12, (N, C, Ksel, i, got, want)
            if gaps:
                sources.add("leaf" if min(gaps, key=gaps.get) == 0 else "intermediate")
    return sources


def test_margin_matches_brute_force_gaps_of_every_pruning_level():
    sources = _check_margins(po.select, _bf_score, 200)
    assert sources == {"leaf", "intermediate"}       # the minimum comes from both kinds of level


def test_pisa1_margin_matches_brute_force_gaps():
    sources = _check_margins(po.select_mean, _bf_mean_score, 300)
    assert sources == {"leaf", "intermediate"}


def test_margin_constant_leaves_closed_form():
    # Constant keys inside each leaf and K >= n1 (only the leaf level prunes): the exact leaf
    # score is sum_h (s q_h.k_t + log n_t) and the flat score s sum_h q_h.k_t, so each margin
    # is the gap between the K-th and (K+1)-th of those closed forms.
    N, C, G, d = 128, 8, 2, 6
    n0 = N // C
    Ksel = n0 // 2                                   # = n1: no intermediate level prunes
    Q = _rand((1, N, G, d), 90)
    kt = _rand((n0, d), 91)
    K = np.repeat(kt, C, axis=0)[None, :, None, :]
    s = 0.45
    qs = [Ksel * C + 3, 100, N - 1]                  # more than K visible leaves
    sel = po.select(Q, K, C, Ksel, scale=s, queries=qs)
    flat = po.select_flat(Q, K, C, Ksel, scale=s, queries=qs)
    for i in qs:
        vis = np.arange(i // C + 1)
        base = s * torch.from_numpy(Q[0, i]).sum(0).numpy() @ kt[vis].T
        n_t = np.array([min((t + 1) * C, i + 1) - t * C for t in vis])
        for o, sc in ((sel, base + G * np.log(n_t)), (flat, base)):
            ranked = np.sort(sc)[::-1]
            assert abs(o["margin"][0, 0, i] - (ranked[Ksel - 1] - ranked[Ksel])) <= 1e-12
    # fewer than K + 1 visible leaves anywhere: nothing is pruned, the margin is infinite
    few = po.select(Q, K, C, n0, scale=s, queries=[N - 1])
    assert few["margin"][0, 0, N - 1] == np.inf


def test_margin_pins_catch_planted_mistakes(monkeypatch):
    # Mistakes planted in the oracle (on the CPU) must fail the pins above.
    real = po._top_k

    def unsorted_margin(cand, scores, K):
        kept, m = real(cand, scores, K)
        return kept, (np.inf if len(cand) <= K else float(scores[K - 1] - scores[K]))

    def flipped_sign(cand, scores, K):
        kept, m = real(cand, scores, K)
        return kept, -m

    def next_gap(cand, scores, K):
        kept, m = real(cand, scores, K)
        if len(cand) <= K + 1:
            return kept, m
        r = np.sort(scores)[::-1]
        return kept, float(r[K] - r[K + 1])

    for bad in (unsorted_margin, flipped_sign, next_gap):
        monkeypatch.setattr(po, "_top_k", bad)
        with pytest.raises(AssertionError):
            _check_margins(po.select, _bf_score, 200)
    monkeypatch.setattr(po, "_top_k", real)
    # A margin taken at the leaf level only, or over the intermediate levels only, differs
    # from the minimum over all pruning levels for some unit of the pinned cases, so an
    # oracle that computed it would fail the brute-force pin.
    leaf_only = inter_only = False
    for N, C, Ksel, G, seed in MARGIN_CASES:
        Q = _rand((1, N, G, 4), 200 + seed, scale=2.0)
        K = _rand((1, N, 1, 4), 250 + seed, scale=2.0)
        rng = np.random.default_rng(seed)
        for i in sorted(set(rng.integers(0, N, 10).tolist()) | {N - 1}):
            gaps = _bf_descent_gaps(Q[0, i], K[0, :, 0, :], i, C, Ksel, 0.7)
            if not gaps:
                continue
            true = min(gaps.values())
            leaf_only |= gaps.get(0, np.inf) != true
            inter_only |= min([v for l, v in gaps.items() if l > 0], default=np.inf) != true
    assert leaf_only and inter_only


# ---------------------------------------------------------------- PISA-2 ablation (R23)
def _bf_meanvar_score(q, K, l, m, i, C, s):
    """PISA-2 score by token loops: mean, then the two-pass population variance per dimension."""
    N, d = K.shape
    toks = [j for j in range(m * (C << l), min((m + 1) * (C << l), N)) if j <= i]
    mu = [sum(K[j, k] for j in toks) / len(toks) for k in range(d)]
    var = [sum((K[j, k] - mu[k]) ** 2 for j in toks) / len(toks) for k in range(d)]
    tot = 0.0
    for h in range(q.shape[0]):
        tot += s * sum(q[h, k] * mu[k] for k in range(d)) + 0.5 * s * s * sum(q[h, k] ** 2 * var[k] for k in range(d))
    return tot


@pytest.mark.parametrize("N,C,Ksel,G,seed", [
    (64, 4, 1, 1, 0), (96, 4, 3, 2, 2), (128, 8, 3, 2, 4), (61, 4, 2, 2, 5), (200, 8, 1, 2, 6)])
def test_pisa2_descent_matches_brute_force(N, C, Ksel, G, seed):
    d = 4
    Q = _rand((1, N, G, d), 400 + seed, scale=2.0)
    K = _rand((1, N, 1, d), 450 + seed, scale=2.0)
    s = 0.7
    rng = np.random.default_rng(seed)
    qs = sorted(set(rng.integers(0, N, 12).tolist()) | {0, N - 1})
    out = po.select_meanvar(Q, K, C, Ksel, scale=s, queries=qs)
    for i in qs:
        leaves, scores = _bf_select(Q[0, i], K[0, :, 0, :], i, C, Ksel, s, _bf_meanvar_score)
        got = out["idx"][0, 0, i]
        assert list(got[got >= 0]) == leaves, (i, got, leaves)
        np.testing.assert_allclose(out["score"][0, 0, i, :len(leaves)], scores, rtol=1e-10, atol=1e-10)
        gaps = _bf_descent_gaps(Q[0, i], K[0, :, 0, :], i, C, Ksel, s, _bf_meanvar_score)
        want = min(gaps.values()) if gaps else np.inf
        assert out["margin"][0, 0, i] == want if not np.isfinite(want) else abs(out["margin"][0, 0, i] - want) < 1e-10


def test_pisa2_is_the_second_order_cumulant_expansion_of_the_block_lse():
    # For a block whose keys are mu + (+-a, +-b) (uncorrelated dimensions, symmetric), the
    # exact log-mean-exp of s q.k equals s q.mu + (s^2/2)(q1^2 a^2 + q2^2 b^2) + O(s^4): the
    # PISA-2 score minus the exact leaf LSE (less log n) must shrink like s^4, not s^2 or s^3.
    mu, a, b = np.array([0.3, -0.2]), 0.9, 1.7
    keys = np.array([mu + [sa * a, sb * b] for sa in (1, -1) for sb in (1, -1)])   # one leaf, C = 4
    q = np.array([[1.3, -0.8]])
    summ = po.CausalKeySummaries(keys, 4)
    errs = []
    for s in (0.2, 0.1, 0.05):
        pisa2 = po.meanvar_scores(q, 3, 0, np.array([0]), summ, s)[0]
        exact = po.leaf_scores(q, 3, np.array([0]), keys, 4, s)[0][0] - math.log(4)
        errs.append(abs(exact - pisa2))
        assert abs(pisa2 - (s * q[0] @ mu + 0.5 * s * s * (q[0, 0] ** 2 * a * a + q[0, 1] ** 2 * b * b))) < 1e-14
    assert errs[0] / errs[1] > 12 and errs[1] / errs[2] > 14           # fourth order: ratio -> 16


def test_pisa2_keep_all_and_zero_variance_leaves():
    N, C, G, d = 96, 8, 2, 6
    Q = _rand((1, N, G, d), 460)
    kt = _rand((N // C, d), 461)
    K = np.repeat(kt, C, axis=0)[None, :, None, :]     # constant keys inside each leaf: variance 0
    n0 = N // C
    out = po.select_meanvar(Q, K, C, n0)
    for i in range(N):
        got = out["idx"][0, 0, i]
        assert list(got[got >= 0]) == list(range(i // C + 1))
    # with zero leaf variance the PISA-2 leaf scores are the PISA-1 ones
    Ksel = 3
    a = po.select_meanvar(Q, K, C, Ksel, queries=[N - 1, 50])
    b = po.select_mean(Q, K, C, Ksel, queries=[N - 1, 50])
    for i in (N - 1, 50):
        common = [t for t in a["idx"][0, 0, i] if t in set(b["idx"][0, 0, i].tolist()) and t >= 0]
        for t in common:
            sa = a["score"][0, 0, i][list(a["idx"][0, 0, i]).index(t)]
            sb = b["score"][0, 0, i][list(b["idx"][0, 0, i]).index(t)]
            assert abs(sa - sb) < 1e-12


# ---------------------------------------------------------------- fan-out g = 4 (R24)
def _bf_select_g4(q, K, i, C, Ksel, s):
    """Brute-force descent with fan-out 4 over the scalar enumerator's full score table:
    visible grandchildren of the kept nodes at every step, one level for the last step when
    two would pass the leaves."""
    N = K.shape[0]
    n = [-(-N // C)]
    while n[-1] > 1:
        n.append(-(-n[-1] // 2))
    table = {(l, m): _bf_score(q, K, l, m, i, C, s)
             for l in range(len(n)) for m in range(n[l]) if m * (C << l) <= i}
    kept, l = [0], len(n) - 1
    while l > 0:
        nl = max(l - 2, 0)
        cand = sorted({c for a in kept for c in range(a << (l - nl), (a + 1) << (l - nl)) if (nl, c) in table})
        assert len(cand) <= 4 * Ksel
        l = nl
        if len(cand) > Ksel or l == 0:
            kept = sorted(cand, key=lambda c: (-table[(l, c)], c))[:Ksel]
        else:
            kept = cand
    leaves = sorted(kept)
    return leaves, [table[(0, t)] for t in leaves]


@pytest.mark.parametrize("N,C,Ksel,G,seed", [
    (64, 4, 1, 1, 0), (96, 4, 2, 2, 1), (128, 4, 3, 2, 2), (200, 8, 1, 2, 3), (256, 4, 2, 1, 4), (61, 4, 2, 2, 5)])
def test_g4_descent_matches_brute_force(N, C, Ksel, G, seed):
    d = 4
    Q = _rand((1, N, G, d), 500 + seed, scale=2.0)
    K = _rand((1, N, 1, d), 550 + seed, scale=2.0)
    s = 0.7
    rng = np.random.default_rng(seed)
    qs = sorted(set(rng.integers(0, N, 12).tolist()) | {0, N - 1})
    out = po.select(Q, K, C, Ksel, scale=s, queries=qs, g=4)
    for i in qs:
        leaves, scores = _bf_select_g4(Q[0, i], K[0, :, 0, :], i, C, Ksel, s)
        got = out["idx"][0, 0, i]
        assert list(got[got >= 0]) == leaves, (i, got, leaves)
        np.testing.assert_allclose(out["score"][0, 0, i, :len(leaves)], scores, rtol=1e-12, atol=1e-12)


def test_g4_invariants_and_keep_all():
    N, C, Ksel, G, d = 512, 4, 3, 2, 4
    Q = _rand((1, N, G, d), 560)
    K = _rand((1, N, 1, d), 561)
    summ = po.CausalKeySummaries(K[0, :, 0, :], C)
    for i in range(0, N, 9):
        u = po.select_unit(Q[0, i], i, summ, Ksel, 0.5, g=4)
        assert all(c <= 4 * Ksel for c in u.cand_sizes)            # at most gK candidates per step
        assert len(u.cand_sizes) == -(-(len(summ.sizes) - 1) // 2)  # ceil(top / 2) steps to the leaves
        assert len(u.leaves) == min(Ksel, i // C + 1) and np.all(u.leaves <= i // C)
        assert set(u.leaves.tolist()) <= set(u.leaf_candidates.tolist())
    out = po.select(Q, K, C, -(-N // C), g=4)
    for i in range(0, N, 5):
        got = out["idx"][0, 0, i]
        assert list(got[got >= 0]) == list(range(i // C + 1))


# ---------------------------------------------------------------- per-head selection (R25)
def test_per_head_selection_matches_single_head_brute_force():
    N, C, Ksel, Hq, Hkv, d = 128, 4, 2, 4, 2, 4
    Q = _rand((1, N, Hq, d), 570, scale=2.0)
    K = _rand((1, N, Hkv, d), 571, scale=2.0)
    s = 0.6
    qs = [0, 17, 63, 100, N - 1]
    out = po.select(Q, K, C, Ksel, scale=s, queries=qs, per_head=True)
    assert out["idx"].shape == (1, Hq, N, Ksel) and out["head_lse"].shape == (1, Hq, N, Ksel)
    for h in range(Hq):
        for i in qs:
            leaves, scores = _bf_select(Q[0, i, h:h + 1], K[0, :, h // (Hq // Hkv), :], i, C, Ksel, s)
            got = out["idx"][0, h, i]
            assert list(got[got >= 0]) == leaves, (h, i)
            np.testing.assert_allclose(out["score"][0, h, i, :len(leaves)], scores, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(out["head_lse"][0, h, i, :len(leaves)], scores, rtol=1e-12, atol=1e-12)


def test_per_head_equals_shared_when_the_group_queries_coincide():
    # identical queries in every head of a group: the shared score is G times a per-head
    # score, so both rankings (and tie rules) agree
    N, C, Ksel, Hq, Hkv, d = 160, 8, 3, 6, 2, 6
    q = _rand((1, N, Hkv, d), 580)
    Q = np.repeat(q, Hq // Hkv, axis=2)
    K = _rand((1, N, Hkv, d), 581)
    shared = po.select(Q, K, C, Ksel)
    per = po.select(Q, K, C, Ksel, per_head=True)
    for h in range(Hq):
        np.testing.assert_array_equal(per["idx"][0, h], shared["idx"][0, h // (Hq // Hkv)])


def _dense_masked_attention(Q, K, V, idx, C, s):
    """Per head: torch softmax over dense logits masked to the head's own selected leaves."""
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, N, Hq, d))
    j = torch.arange(N)
    for b in range(B):
        for h in range(Hq):
            logits = torch.from_numpy(Q[b, :, h, :] @ K[b, :, h // G, :].T) * s          # [N, N]
            rows = idx[b, h] if idx.shape[1] == Hq else idx[b, h // G]
            keep = torch.zeros(N, N, dtype=torch.bool)
            for i in range(N):
                for t in rows[i]:
                    if t >= 0:
                        keep[i] |= (j // C == int(t)) & (j <= i)
            O[b, :, h, :] = (torch.softmax(logits.masked_fill(~keep, float("-inf")), dim=-1) @
                             torch.from_numpy(V[b, :, h // G, :])).numpy()
    return O


def test_per_head_attention_and_backward():
    B, N, Hq, Hkv, d, C = 1, 40, 4, 2, 4, 8
    Q, K, V = _rand((B, N, Hq, d), 590), _rand((B, N, Hkv, d), 591), _rand((B, N, Hkv, d), 592)
    dO = _rand((B, N, Hq, d), 593)
    idx = _random_idx(B, Hq, N, C, 2, 594)                    # a different selection per query head
    s = 0.5
    O, lse = po.sparse_attn_fwd(Q, K, V, idx, C, scale=s)
    np.testing.assert_allclose(O, _dense_masked_attention(Q, K, V, idx, C, s), rtol=1e-10, atol=1e-12)
    hl = po.selected_head_lse(Q, K, idx, C, scale=s)
    np.testing.assert_allclose(torch.logsumexp(torch.from_numpy(hl), dim=-1).numpy(), lse, rtol=1e-12, atol=1e-12)
    dQ, dK, dV = po.sparse_attn_bwd(Q, K, V, dO, idx, C, scale=s)

    def loss(Q_, K_, V_):
        O_, _ = po.sparse_attn_fwd(Q_, K_, V_, idx, C, scale=s)
        return float((O_ * dO).sum())

    eps = 1e-6
    rng = np.random.default_rng(1)
    for name, X, G_ in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        for _ in range(5):
            pos = tuple(int(rng.integers(0, n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[pos] += eps
            Xm[pos] -= eps
            args_p = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
            args_m = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - G_[pos]) < 1e-6 * max(1.0, abs(fd)), (name, pos, fd, G_[pos])
    sq, sk, sv = po.sparse_attn_bwd_sampled(Q, K, V, dO, idx, C, scale=s, queries=[(0, 7), (0, 39)],
                                            leaves=[(0, 0, 0), (0, 1, 3)])
    for (b, i) in ((0, 7), (0, 39)):
        np.testing.assert_allclose(sq[(b, i)], dQ[b, i], rtol=1e-12, atol=1e-13)
    for (b, kv, t) in ((0, 0, 0), (0, 1, 3)):
        s0, e0 = po.node_range(0, t, C, N)
        np.testing.assert_allclose(sk[(b, kv, t)], dK[b, s0:e0, kv], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sv[(b, kv, t)], dV[b, s0:e0, kv], rtol=1e-12, atol=1e-13)


def test_per_head_flat_mean_meanvar_decompose_into_single_head_problems():
    # a per-head selection of head h is the shared selection of the one-head problem (q_h, its KV head)
    N, C, Ksel, Hq, Hkv, d = 96, 8, 3, 4, 2, 6
    Q = _rand((1, N, Hq, d), 600)
    K = _rand((1, N, Hkv, d), 601)
    qs = [5, 40, 95]
    for fn in (po.select_flat, po.select_mean, po.select_meanvar, po.select):
        per = fn(Q, K, C, Ksel, queries=qs, per_head=True)
        for h in range(Hq):
            one = fn(Q[:, :, h:h + 1], K[:, :, h // 2:h // 2 + 1], C, Ksel, queries=qs)
            np.testing.assert_array_equal(per["idx"][0, h, qs], one["idx"][0, 0, qs])
            np.testing.assert_allclose(per["score"][0, h, qs], one["score"][0, 0, qs], rtol=0, atol=0)
