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


def test_nvml_clock_summary_keeps_the_timed_region_only():
    """The NVML clock sampler's summary, on a fake sample record: only
    samples inside [t0, t1] count, the median is theirs, and the reason bits
    decode to the names the JSON line reports."""
    import threading
    import bench

    class FakeLib:
        def nvmlShutdown(self):
            return 0

    s = object.__new__(bench.NvmlClocks)
    s.lib = FakeLib()
    s.stop_flag = False
    s.thread = threading.Thread(target=lambda: None)
    s.thread.start()
    s.max_mhz = 2070.0
    s.samples = [(0.5, 900.0, 0x1), (1.0, 1900.0, 0x4), (1.1, 1950.0, 0x0), (1.2, 2000.0, 0x4 | 0x20),
                 (3.0, 300.0, 0x8)]
    out = s.stop(1.0, 1.2)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 1950.0
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    s2 = object.__new__(bench.NvmlClocks)
    s2.lib, s2.stop_flag, s2.max_mhz, s2.samples = FakeLib(), False, None, [(5.0, 1.0, 0)]
    s2.thread = threading.Thread(target=lambda: None)
    s2.thread.start()
    assert s2.stop(1.0, 2.0) is None  # no sample inside the region


def test_on_cpus_restores_the_cpu_set():
    """The benchmark's CPU-set guard (used to place pinned host buffers next
    to the GPU) restores the process's CPUs, and is a no-op without a set."""
    import os
    import bench
    before = os.sched_getaffinity(0)
    one = {min(before)}
    with bench.on_cpus(one):
        assert os.sched_getaffinity(0) == one
    assert os.sched_getaffinity(0) == before
    with bench.on_cpus(None):
        assert os.sched_getaffinity(0) == before
    assert bench.gpu_local_cpus("GPU-00000000-0000-0000-0000-000000000000") is None
