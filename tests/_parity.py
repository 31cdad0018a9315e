"""Comparison helpers for GPU-vs-oracle parity (the oracle's numbers are the expectation)."""
import numpy as np

# Tolerances: selection scores are fp32 LSE sums (1e-3 absolute); a unit whose oracle
# pruning margin is below 1e-3 at any level is exempt from the index match (a near tie can
# flip a whole subtree); attention outputs are bf16 (atol 2e-2 / rtol 2e-2).
SCORE_ATOL = 1e-3
MARGIN_EXEMPT = 1e-3
OUT_ATOL = 2e-2
OUT_RTOL = 2e-2


def check_selection(gidx, gscore, ora, queries, C, K, N):
    """gidx/gscore: numpy [B,Hkv,N,K] from the GPU; ora: oracle dict. Returns stats."""
    B, Hkv = gidx.shape[:2]
    n = exempt = strict = 0
    for b in range(B):
        for kv in range(Hkv):
            for i in queries:
                n += 1
                g = gidx[b, kv, i]
                nvis = i // C + 1
                want = min(K, nvis)
                valid = g[g >= 0]
                # always: a valid selection (ascending, distinct, causal, right count)
                assert len(valid) == want and np.all(g[want:] == -1), (b, kv, i, g)
                assert np.all(np.diff(valid) > 0) and valid[-1] <= i // C and valid[0] >= 0
                o = ora["idx"][b, kv, i]
                if np.array_equal(g, o):
                    strict += 1
                    np.testing.assert_allclose(gscore[b, kv, i, :want], ora["score"][b, kv, i, :want],
                                               atol=SCORE_ATOL, rtol=0)
                    assert np.all(np.isneginf(gscore[b, kv, i, want:]))
                    continue
                if ora["margin"][b, kv, i] < MARGIN_EXEMPT:
                    exempt += 1
                    continue
                raise AssertionError(f"selection mismatch at b={b} kv={kv} i={i}: gpu={g} oracle={o} "
                                     f"margin={ora['margin'][b, kv, i]}")
    return dict(units=n, strict=strict, exempt=exempt)


def check_close(got, want, atol=OUT_ATOL, rtol=OUT_RTOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    bad = ~(np.abs(got - want) <= atol + rtol * np.abs(want))
    if bad.any():
        k = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tol; first at {tuple(k)}: "
                             f"got {got[tuple(k)]} want {want[tuple(k)]}")
