"""Host-side helpers of the GPU parity tests, checked on the CPU."""
import numpy as np

import _harness as hz


def test_coverage_tokens_hits_every_group_and_tile():
    # the selection rule itself, on a made-up routing (host only)
    rng = np.random.default_rng(5)
    T, E, k = 1000, 6, 2
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    tok = hz.coverage_tokens(T, E, k, 1, idx, bn=96, ct=7, n=200, seed=1)
    assert len(tok) == 200 and len(np.unique(tok)) == 200
    for c0 in range(0, T, 7):
        assert np.any((tok >= c0) & (tok < c0 + 7))
    for g0 in range(0, T, 96):
        assert np.any((tok >= g0) & (tok < g0 + 96))
    counts = np.bincount(idx.ravel(), minlength=E)
    for e in np.argsort(-counts, kind="stable")[:3]:
        rows = np.nonzero((idx == e).any(axis=1))[0]
        for grp in hz.expert_groups(rows, 96):
            assert np.intersect1d(grp, tok).size >= 1
