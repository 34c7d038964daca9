"""The dropout generator as the kernels run it, on the GPU, against the
published known-answer vectors of Philox4x32-10 (Salmon et al., SC 2011;
the Random123 test file) that also pin the oracle's generator, and against
the oracle's generator on random counters and keys."""
import numpy as np
import pytest
import torch

from golden_io import load_philox_kat

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from exact_tiled_attention_22_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from exact_tiled_attention_22_gb300 import attn
    return attn


def run_gpu(A, rows):
    """rows: list of (counter[4], key[2]) -> list of 4-word outputs."""
    host = np.array([list(c) + list(k) for c, k in rows], dtype=np.uint32)
    inp = torch.from_numpy(host.view(np.int32)).cuda()
    out = torch.full((len(rows), 4), -1, dtype=torch.int32, device="cuda")
    A.check(A.attn_philox4x32_10(inp, out, len(rows)))
    torch.cuda.synchronize()
    return [[int(w) for w in r] for r in out.cpu().numpy().view(np.uint32)]


def test_gpu_philox_known_answers(A):
    kats = load_philox_kat()
    got = run_gpu(A, [(c, k) for c, k, _ in kats])
    for (c, k, ref), g in zip(kats, got):
        assert g == ref, f"ctr {c} key {k}: {[hex(x) for x in g]} != {[hex(x) for x in ref]}"


def test_gpu_philox_matches_oracle(A, oracle):
    g = np.random.default_rng(5)
    rows = [([int(x) for x in g.integers(0, 2**32, 4, dtype=np.uint64)],
             [int(x) for x in g.integers(0, 2**32, 2, dtype=np.uint64)]) for _ in range(1000)]
    got = run_gpu(A, rows)
    for (c, k), gw in zip(rows, got):
        assert gw == list(oracle.philox4x32(c, k)), (c, k)
