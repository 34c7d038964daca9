"""GPU parity of the ALiBi variants (attn_fwd_alibi, attn_bwd_alibi,
attn_decode_alibi) against the fp64 oracle with the same per-head slopes:
the scores carry the linear bias -m_h |pos_i - j|.

Shapes cover causal and non-causal masks (so tiles left of, right of and on
the diagonal), both head dims and dtypes, ragged tails, and slopes from the
usual geometric sequence up to a steep one that makes the bias dominate.
"""
import numpy as np
import pytest
import torch

from exact_tiled_attention_22_gb300.inputs import make_inputs
from parity import TOL_GRAD, TOL_LSE, TOL_O, default_scale, o_error, rel_l2

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


def slopes(H, steep=False):
    s = [2.0 ** (-8.0 * (h + 1) / H) for h in range(H)]
    if steep:
        s[-1] = 1.5
    return s


SHAPES = [
    # (B, N, H, d, dtype, causal, steep)
    (1, 257, 3, 128, "bf16", True, False),
    (1, 300, 2, 64, "fp16", False, True),
    (2, 640, 2, 128, "fp16", False, False),
    (1, 1000, 2, 128, "bf16", True, True),
    (1, 129, 2, 64, "bf16", True, False),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}N{}H{}d{}{}{}{}".format(
    *s[:5], "c" if s[5] else "", "s" if s[6] else ""))
def test_alibi_fwd_bwd_match_oracle(oracle, shape):
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d, dtype, causal, steep = shape
    x = make_inputs(B, N, H, d, dtype, seed=3100 + N)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    m = slopes(H, steep)
    al = torch.tensor(m, dtype=torch.float32, device=dev)
    scale = default_scale(d)
    o, lse = attn.fwd(q, k, v, scale, causal, alibi=al)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, do, scale, causal, alibi=al)
    attn.check(attn.attn_status())
    g = {n: t.float().cpu().numpy() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk),
                                                  ("dv", dv))}
    x64 = {n: t.double().numpy() for n, t in x.items()}
    for b in range(B):
        for h in range(H):
            hd = lambda a: np.ascontiguousarray(a[b, :, h, :])  # noqa: E731
            qq, kk, vv, dd = (hd(x64[n]) for n in ("q", "k", "v", "do"))
            o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, causal, alibi=m[h])
            eo, _ = o_error(g["o"][b, :, h, :], o_ref, dtype)
            assert eo <= TOL_O[dtype], f"({b},{h}) O {eo:.3e}"
            assert np.max(np.abs(g["lse"][b, h] - lse_ref)) <= TOL_LSE, f"({b},{h}) LSE"
            dq_r, dk_r, dv_r, _ = oracle.bwd_head(qq, kk, vv, dd, scale, causal, alibi=m[h])
            for name, ref in (("dq", dq_r), ("dk", dk_r), ("dv", dv_r)):
                err = rel_l2(g[name][b, :, h, :], ref)
                assert err <= TOL_GRAD, f"({b},{h}) {name} rel L2 {err:.3e}"


@pytest.mark.parametrize("causal", [True, False])
def test_alibi_decode_matches_oracle(oracle, causal):
    from exact_tiled_attention_22_gb300 import attn
    B, H, Nq, Nk, d, dtype = 1, 4, 5, 3000, 128, "bf16"
    x = make_inputs(B, Nk, H, d, dtype, seed=3200 + int(causal))
    q = x["q"][:, Nk - Nq:].contiguous()
    dev = torch.device("cuda:0")
    m = slopes(H, steep=True)
    al = torch.tensor(m, dtype=torch.float32, device=dev)
    scale = default_scale(d)
    o, lse = attn.decode(q.to(dev), x["k"].to(dev), x["v"].to(dev), scale, causal, alibi=al)
    attn.check(attn.attn_status())
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    q64, k64, v64 = (t.double().numpy() for t in (q, x["k"], x["v"]))
    for h in range(H):
        o_ref, lse_ref = oracle.decode_head(q64[0, :, h], k64[0, :, h], v64[0, :, h], scale, causal,
                                            alibi=m[h])
        eo, _ = o_error(o[0, :, h], o_ref, dtype)
        assert eo <= TOL_O[dtype], f"head {h} O {eo:.3e}"
        assert np.max(np.abs(lse[0, h] - lse_ref)) <= TOL_LSE, f"head {h} LSE"


def test_alibi_zero_slopes_equal_plain():
    """Slopes of zero give exactly the plain forward (same kernel arithmetic
    up to the bias term, which is then 0)."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d = 1, 500, 2, 128
    x = make_inputs(B, N, H, d, "bf16", seed=11)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o1, l1 = attn.fwd(q, k, v, 0.1, True)
    o2, l2 = attn.fwd(q, k, v, 0.1, True, alibi=torch.zeros(H, dtype=torch.float32, device=dev))
    attn.check(attn.attn_status())
    assert (o1.float() - o2.float()).abs().max().item() <= 0.0157
    assert (l1 - l2).abs().max().item() <= 1e-4
