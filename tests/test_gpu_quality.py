"""Selection quality on the GPU path: the quality workload's own library calls (pyramid
selection, its PISA-1 ablation, the flat comparator) on a small needle case, measured with the
benchmark's measuring stick (dense exact leaf LSEs, pinned against the oracle on CPU in
test_bench_tools.py and here again on three queries), and the invariants its figures must
satisfy. Needs a GB300 and the built library."""
import math
import os
import sys

import numpy as np
import pytest
import torch

import pisa_synth as syn
import pyramid_top_selection_gb300 as pisa
from oracle import pisa_oracle as po

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


def test_quality_figures_and_their_invariants():
    dev = torch.device("cuda", 0)
    B, N, Hq, Hkv, d, C, K = 1, 2048, 8, 2, 128, 64, 8
    G, n0 = Hq // Hkv, N // C
    cfg = dict(C=C, K=K, g=2, qtile=4)
    Q, Kt, _ = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=5, needles=True, device=dev)
    needles = syn.needle_leaves(B, Hkv, n0, 5 + 3, device=dev)
    sels = bench.quality_selections(Q, Kt, cfg)
    stats = bench.quality_stats(sels, Q, Kt, C, K, needles)
    print(stats)
    for name, st in stats.items():
        for v in st.values():
            assert 0.0 <= v <= 1.0 + 1e-6, (name, st)
    assert stats["exact"]["recall_exact_topk"] == 1.0
    # per-query invariants against the measuring stick
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=4)
    idx, score = pisa.select(Q, Kt, pisa.build_pyramid(Kt, shape), shape)
    scale = 1.0 / math.sqrt(d)
    for kv in range(Hkv):
        ll = bench.exact_leaf_lse(Q[0, :, kv * G:(kv + 1) * G, :], Kt[0, :, kv, :], 0, N, C, scale)   # [N, G, n0]
        # the stick against the oracle's exact leaf LSEs on three queries
        for i in (0, 777, N - 1):
            leaves = np.arange(i // C + 1)
            _, per_head = po.leaf_scores(Q[0, i, kv * G:(kv + 1) * G].double().cpu().numpy(), i, leaves,
                                         Kt[0, :, kv, :].double().cpu().numpy(), C, scale)
            np.testing.assert_allclose(ll[i, :, :len(leaves)].double().cpu().numpy(), per_head.T, atol=2e-5, rtol=0)
        tot = ll.sum(1).double().cpu().numpy()                                                      # [N, n0]
        full = torch.logsumexp(ll, dim=-1).double().cpu().numpy()                                   # [N, G]
        lld = ll.double().cpu().numpy()
        gi, gs = idx[0, kv].cpu().numpy(), score[0, kv].cpu().numpy()
        for i in range(N):
            vis = i // C + 1
            if vis <= K:
                # every visible leaf is selected by every method, and holds the whole softmax mass
                for name, sel in sels.items():
                    row = sel[0, kv, i].cpu().numpy()
                    assert list(row[row >= 0]) == list(range(vis)), (name, i, row)
                mass = np.exp(lld[i, :, :vis] - full[i][:, None]).sum(-1)
                np.testing.assert_allclose(mass, 1.0, atol=1e-5)
            if vis <= 2 * K:
                # no intermediate level prunes: the pyramid selection is the exact top-K
                order = sorted(range(vis), key=lambda t: (-tot[i, t], t))
                if vis > K and tot[i, order[K - 1]] - tot[i, order[K]] < 1e-3:
                    continue                                       # a near tie may fall either way
                assert list(gi[i][gi[i] >= 0]) == sorted(order[:K]), (kv, i)
            sel_t = gi[i][gi[i] >= 0]
            np.testing.assert_allclose(gs[i, :len(sel_t)], tot[i, sel_t], atol=1e-3, rtol=0)
