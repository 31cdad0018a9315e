"""GPU parity on the shapes the narrower cases leave out: K = 24 and 32 with real pruning at
every level (the 64-candidate routing, top-K and flat-merge paths), and the selection sweep's
128K and 256K shapes (Hq = 32, Hkv = 8) at full size on a deterministic query sample. The
oracle evaluates only the sampled units, one (batch, KV head, query) at a time, from the same
bf16 inputs. Needs a GB300 and the built library."""
import math

import numpy as np
import pytest
import torch

import pisa_synth as syn
import pyramid_top_selection_gb300 as pisa
from oracle import pisa_oracle as po
from _parity import check_selection

pytestmark = pytest.mark.gpu
C = 64


def _oracle_units(Q, Kt, Ksel, qs, kind):
    """The oracle's selection of the sampled queries: idx/score/margin arrays [B,Hkv,N,...]
    filled on the sampled units only. Q, Kt: CPU bf16 tensors."""
    B, N, Hq, d = Q.shape
    Hkv = Kt.shape[2]
    G = Hq // Hkv
    s = po.default_scale(d)
    idx = np.full((B, Hkv, N, Ksel), -1, np.int32)
    score = np.full((B, Hkv, N, Ksel), np.nan)
    margin = np.full((B, Hkv, N), np.nan)
    for b in range(B):
        for kv in range(Hkv):
            summ = po.CausalKeySummaries(Kt[b, :, kv, :].double().numpy(), C)
            for i in qs:
                q = Q[b, i, kv * G:(kv + 1) * G, :].double().numpy()
                if kind == "pyramid":
                    u = po.select_unit(q, i, summ, Ksel, s)
                    leaves, sc, mg = u.leaves, u.scores, u.min_margin
                elif kind == "mean":
                    leaves, sc, mg = po.select_unit_mean(q, i, summ, Ksel, s)
                else:
                    leaves, sc, mg = po.select_unit_flat(q, i, summ, Ksel, s)
                idx[b, kv, i, :len(leaves)] = leaves
                score[b, kv, i, :] = -np.inf
                score[b, kv, i, :len(leaves)] = sc
                margin[b, kv, i] = mg
    return dict(idx=idx, score=score, margin=margin)


def _run(B, N, Hq, Hkv, d, Ksel, qs, seed, min_strict):
    dev = torch.device("cuda", 0)
    Qg, Kg, _ = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=seed, needles=True, device=dev)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, Ksel, qtile=4)
    pyr = pisa.build_pyramid(Kg, shape)
    got = {"pyramid": pisa.select(Qg, Kg, pyr, shape), "mean": pisa.select_mean(Qg, Kg, pyr, shape),
           "flat": pisa.select_flat(Qg, Kg, pyr, shape)}
    torch.cuda.synchronize()
    Q, Kt = Qg.cpu(), Kg.cpu()
    stats = {}
    for kind, (gi, gs) in got.items():
        ora = _oracle_units(Q, Kt, Ksel, qs, kind)
        st = check_selection(gi.cpu().numpy(), gs.cpu().numpy(), ora, qs, C, Ksel, N)
        assert st["strict"] + st["exempt"] == st["units"]
        assert st["strict"] >= min_strict * st["units"], (kind, st)
        stats[kind] = st
    print(f"N={N} Hq={Hq} Hkv={Hkv} K={Ksel}: {stats}")
    return stats


@pytest.mark.parametrize("Ksel", [24, 32])
def test_large_k_with_pruning_at_every_level(Ksel):
    # N = 16384: 256 leaves > 2K, so two intermediate levels and the leaf level prune
    B, N, Hq, Hkv, d = 1, 16384, 16, 2, 128
    assert po.level_sizes(N, C)[1] > Ksel and po.level_sizes(N, C)[2] > Ksel // 2
    qs = sorted(set(range(Ksel * C, N, 331)) | {0, 63, 64, 4095, N - 2, N - 1})
    _run(B, N, Hq, Hkv, d, Ksel, qs, seed=2, min_strict=0.9)


@pytest.mark.parametrize("N", [131072, 262144])
def test_sweep_shapes_sampled(N):
    # the selection sweep's configuration at full size: B = 1, Hq = 32, Hkv = 8, d = 128, K = 16
    B, Hq, Hkv, d, Ksel = 1, 32, 8, 128, 16
    step = N // 12 + 1
    qs = sorted(set(range(0, N, step)) | {0, 1, 1023, 1024, N // 2, N - 2, N - 1})
    _run(B, N, Hq, Hkv, d, Ksel, qs, seed=0, min_strict=0.9)
