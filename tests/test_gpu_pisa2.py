"""GPU parity of the PISA-2 ablation selection (every block scored by mean + variance) against
the fp64 oracle on the same seeded bf16 inputs. Needs a GB300 and the built library."""
import pytest
import torch

import pisa_synth as syn
import pyramid_top_selection_gb300 as pisa
from oracle import pisa_oracle as po
from _parity import check_selection
from test_gpu_parity import CASES, C, _inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_pisa2_select_vs_oracle(case):
    _, B, N, Hq, Hkv, d, K, needles = case
    (Q, Kt, _), (Qg, Kg, _) = _inputs(B, N, Hq, Hkv, d, needles)
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=1)
    pyr = pisa.build_pyramid(Kg, shape)
    idx, score = pisa.select_meanvar(Qg, Kg, pyr, shape)
    idx4, score4 = pisa.select_meanvar(Qg, Kg, pyr, pisa.make_shape(B, N, Hq, Hkv, d, C, K, qtile=4))
    torch.cuda.synchronize()
    assert torch.equal(idx, idx4) and torch.equal(score, score4)
    ora = po.select_meanvar(Q, Kt, C, K)
    st = check_selection(idx.cpu().numpy(), score.cpu().numpy(), ora, range(N), C, K, N)
    assert st["strict"] + st["exempt"] == st["units"]
    assert st["strict"] >= 0.9 * st["units"], st


@pytest.mark.parametrize("Ksel", [16, 32])
def test_pisa2_sampled_at_16k(Ksel):
    B, N, Hq, Hkv, d = 1, 16384, 16, 2, 128
    Q, Kt, _ = syn.make_prefill(B, N, Hq, Hkv, d, C=C, seed=1, needles=True)
    Qg, Kg = Q.cuda(), Kt.cuda()
    shape = pisa.make_shape(B, N, Hq, Hkv, d, C, Ksel, qtile=4)
    pyr = pisa.build_pyramid(Kg, shape)
    idx, score = pisa.select_meanvar(Qg, Kg, pyr, shape)
    qs = syn.query_subsample(N, every=97, tail=64).tolist()
    ora = po.select_meanvar(Q, Kt, C, Ksel, queries=qs)
    st = check_selection(idx.cpu().numpy(), score.cpu().numpy(), ora, qs, C, Ksel, N)
    print(f"PISA-2 N={N} K={Ksel}: {st}")
    assert st["strict"] + st["exempt"] == st["units"]
    assert st["strict"] >= 0.9 * st["units"], st
