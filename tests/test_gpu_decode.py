"""GPU parity of the decoding path (attn_decode) against the fp64 oracle's
decoding routine: Nq query rows that are the last Nq positions, against a
key/value cache of Nk keys, split over key chunks on the GPU and merged.

Every head and element is compared on the small cases; the long caches
(several chunks per head) on sampled heads.  The query rows are the last Nq
rows of the seeded full-sequence inputs, so the result must also equal the
last rows of the GPU forward pass over the whole sequence.
"""
import numpy as np
import pytest
import torch

from exact_tiled_attention_22_gb300.inputs import make_inputs
from parity import TOL_LSE, TOL_O, default_scale, o_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_tiled_attention_22_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from exact_tiled_attention_22_gb300 import attn
    attn.attn_set_wait_limit(0, 0)
    yield
    assert attn.attn_status() == 0


CASES = [
    # (B, H, Nq, Nk, d, dtype, causal)
    (1, 1, 1, 1, 64, "fp16", False),
    (1, 1, 1, 1, 128, "bf16", True),
    (1, 2, 1, 1000, 128, "bf16", True),
    (2, 3, 4, 777, 128, "bf16", True),
    (2, 2, 7, 300, 64, "fp16", False),
    (1, 1, 3, 129, 128, "fp16", True),
    (1, 2, 16, 4096, 128, "bf16", True),
    (1, 2, 64, 5000, 64, "bf16", True),
    (1, 1, 128, 128, 128, "bf16", True),
    (1, 1, 100, 2000, 128, "fp16", False),
    (4, 8, 2, 2048, 128, "bf16", True),
]


def _run(B, H, Nq, Nk, d, dtype, causal, seed):
    from exact_tiled_attention_22_gb300 import attn
    x = make_inputs(B, Nk, H, d, dtype, seed=seed)
    q = x["q"][:, Nk - Nq:].contiguous()
    dev = torch.device("cuda:0")
    scale = default_scale(d)
    o, lse = attn.decode(q.to(dev), x["k"].to(dev), x["v"].to(dev), scale, causal)
    attn.check(attn.attn_status())
    return x, q, scale, o.float().cpu().numpy(), lse.cpu().numpy()


def _check_heads(orc, x, q, scale, causal, dtype, o, lse, heads):
    q64, k64, v64 = (t.double().numpy() for t in (q, x["k"], x["v"]))
    worst_o = worst_l = 0.0
    for (b, h) in heads:
        o_ref, lse_ref = orc.decode_head(q64[b, :, h], k64[b, :, h], v64[b, :, h], scale, causal)
        eo, _ = o_error(o[b, :, h], o_ref, dtype)
        el = float(np.max(np.abs(lse[b, h] - lse_ref)))
        worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    assert worst_o <= TOL_O[dtype], f"O error {worst_o:.3e}"
    assert worst_l <= TOL_LSE, f"LSE error {worst_l:.3e}"


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}q{}k{}d{}{}{}".format(
    *c[:5], c[5], "c" if c[6] else ""))
def test_decode_matches_oracle(oracle, case):
    B, H, Nq, Nk, d, dtype, causal = case
    x, q, scale, o, lse = _run(B, H, Nq, Nk, d, dtype, causal, seed=4242 + Nk)
    heads = [(b, h) for b in range(B) for h in range(H)]
    _check_heads(oracle, x, q, scale, causal, dtype, o, lse, heads)


def test_decode_long_cache_sampled_heads(oracle):
    """A 32K-key cache, 32 heads, 16 query rows: 64 chunks per head."""
    B, H, Nq, Nk, d, dtype, causal = 1, 32, 16, 32768, 128, "bf16", True
    x, q, scale, o, lse = _run(B, H, Nq, Nk, d, dtype, causal, seed=77)
    _check_heads(oracle, x, q, scale, causal, dtype, o, lse, [(0, 0), (0, 13), (0, 31)])


def test_decode_equals_last_rows_of_forward():
    """Decoding the last Nq rows against the whole sequence gives the last Nq
    rows of the forward pass (both on the GPU; each within its own rounding)."""
    from exact_tiled_attention_22_gb300 import attn
    B, H, Nq, Nk, d, dtype = 2, 4, 8, 3000, 128, "bf16"
    x = make_inputs(B, Nk, H, d, dtype, seed=9)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    scale = default_scale(d)
    o_full, lse_full = attn.fwd(q, k, v, scale, True)
    o_dec, lse_dec = attn.decode(q[:, Nk - Nq:].contiguous(), k, v, scale, True)
    attn.check(attn.attn_status())
    diff = (o_dec.float() - o_full[:, Nk - Nq:].float()).abs().max().item()
    assert diff <= 2 * TOL_O[dtype] + 0.0157, diff  # two bf16 roundings of |O| < 4
    assert (lse_dec - lse_full[:, :, Nk - Nq:]).abs().max().item() <= 2 * TOL_LSE
