"""Host-side arithmetic of the benchmark that needs no GPU."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


@pytest.mark.parametrize("N,causal", [(300, True), (300, False), (1000, True), (128, True)])
def test_bench_kept_pairs_matches_brute_force(N, causal):
    """The block-sparse FLOP count of the bench: scores a block mask keeps
    (with the causal rule), against an explicit N x N visibility matrix."""
    import numpy as np
    import bench
    from exact_tiled_attention_22_gb300.inputs import make_block_mask
    m = make_block_mask(2, N, "random", 0.5, seed=N)
    tot = 0
    for h in range(2):
        vis = np.repeat(np.repeat(m[h].numpy().astype(bool), 128, 0), 128, 1)[:N, :N]
        if causal:
            vis &= np.tril(np.ones((N, N), dtype=bool))
        tot += int(vis.sum())
    assert bench.kept_pairs(m, N, causal) == tot
