"""The benchmark's measuring code on CPU (not the product): the dense exact leaf scores that the
selection-quality workload compares the library's selections with."""
import os
import sys

import numpy as np
import torch

from oracle import pisa_oracle as po

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_exact_leaf_lse_matches_oracle_leaf_scores():
    N, G, d, C, s = 200, 3, 8, 16, 0.6
    r = np.random.default_rng(7)
    Q = torch.from_numpy(r.standard_normal((N, G, d))).to(torch.bfloat16)
    K = torch.from_numpy(r.standard_normal((N, d))).to(torch.bfloat16)
    q0, q1 = 37, 131
    got = bench.exact_leaf_lse(Q, K, q0, q1, C, s).double().numpy()        # [q, G, leaves]
    K64 = K.double().numpy()
    for i in range(q0, q1):
        leaves = np.arange(i // C + 1)
        tot, per_head = po.leaf_scores(Q[i].double().numpy(), i, leaves, K64, C, s)
        np.testing.assert_allclose(got[i - q0, :, :len(leaves)], per_head.T, rtol=0, atol=2e-5)
        assert np.all(np.isneginf(got[i - q0, :, len(leaves):]))            # leaves past the query
        np.testing.assert_allclose(got[i - q0, :, :len(leaves)].sum(0), tot, rtol=0, atol=5e-5)
