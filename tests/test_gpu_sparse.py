"""GPU parity of the block-sparse variants (attn_fwd_sparse,
attn_bwd_sparse) against the fp64 oracle with the same 128 x 128 block mask.

Masks: random (several densities), banded with global first block row and
column, and masks with a query block that keeps nothing (rows with no key:
O = 0, LSE = -inf, dQ = 0) and a key block that no query keeps (dK = dV = 0).
Shapes cover causal and non-causal, both head dims and dtypes, ragged tails,
query-tile pairs where only one tile keeps a key tile, and ALiBi combined
with a mask.
"""
import numpy as np
import pytest
import torch

from exact_tiled_attention_22_gb300.inputs import make_block_mask, make_inputs
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


def check_head(oracle, x64, g, b, h, scale, causal, dtype, bm, alibi=0.0):
    hd = lambda a: np.ascontiguousarray(a[b, :, h, :])  # noqa: E731
    qq, kk, vv, dd = (hd(x64[n]) for n in ("q", "k", "v", "do"))
    o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, causal, alibi=alibi, block_mask=bm)
    eo, _ = o_error(g["o"][b, :, h, :], o_ref, dtype)
    assert eo <= TOL_O[dtype], f"({b},{h}) O {eo:.3e}"
    lg = g["lse"][b, h]
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty), f"({b},{h}) rows with no key differ"
    assert np.all(g["o"][b, :, h, :][empty] == 0.0), f"({b},{h}) O of an empty row"
    if (~empty).any():
        assert np.max(np.abs(lg[~empty] - lse_ref[~empty])) <= TOL_LSE, f"({b},{h}) LSE"
    if "dq" not in g:
        return
    dq_r, dk_r, dv_r, _ = oracle.bwd_head(qq, kk, vv, dd, scale, causal, alibi=alibi,
                                         block_mask=bm)
    N = qq.shape[0]
    # keys that some query sees (mask and causal rule), from the mask alone
    blk = np.repeat(np.repeat(bm.astype(bool), 128, 0), 128, 1)[:N, :N]
    if causal:
        blk &= np.tril(np.ones((N, N), dtype=bool))
    unseen_key = ~blk.any(axis=0)
    for name, ref, none in (("dq", dq_r, empty), ("dk", dk_r, unseen_key),
                            ("dv", dv_r, unseen_key)):
        got = g[name][b, :, h, :]
        err = rel_l2(got, ref)
        assert err <= TOL_GRAD, f"({b},{h}) {name} rel L2 {err:.3e}"
        assert np.all(ref[none] == 0.0)
        assert np.all(got[none] == 0.0), f"({b},{h}) {name} not zero where no score reaches"


def run(q, k, v, do, scale, causal, mask, alibi=None, bwd=True):
    from exact_tiled_attention_22_gb300 import attn
    o, lse = attn.fwd(q, k, v, scale, causal, alibi=alibi, block_mask=mask)
    out = {"o": o, "lse": lse}
    if bwd:
        dq, dk, dv = attn.bwd(q, k, v, o, lse, do, scale, causal, alibi=alibi, block_mask=mask)
        out.update(dq=dq, dk=dk, dv=dv)
    attn.check(attn.attn_status())
    return {n: t.float().cpu().numpy() for n, t in out.items()}


SHAPES = [
    # (B, N, H, d, dtype, causal, pattern, density)
    (1, 700, 2, 128, "bf16", False, "random", 0.5),
    (1, 1000, 2, 64, "fp16", True, "random", 0.4),
    (2, 520, 2, 128, "fp16", False, "local_global", 0.0),
    (1, 1300, 2, 128, "bf16", True, "local_global", 0.0),
    (1, 900, 3, 64, "bf16", False, "random", 0.2),
    (1, 128, 1, 128, "fp16", True, "random", 0.7),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}N{}H{}d{}{}{}_{}".format(
    *s[:5], "c" if s[5] else "", s[6]))
def test_sparse_fwd_bwd_match_oracle(oracle, shape):
    B, N, H, d, dtype, causal, pattern, density = shape
    x = make_inputs(B, N, H, d, dtype, seed=4100 + N)
    mask = make_block_mask(H, N, pattern, density, seed=4200 + N)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    g = run(q, k, v, do, scale, causal, mask.to(dev))
    x64 = {n: t.double().numpy() for n, t in x.items()}
    for b in range(B):
        for h in range(H):
            check_head(oracle, x64, g, b, h, scale, causal, dtype, mask[h].numpy())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_sparse_empty_rows_and_keys(oracle, causal, d):
    """Query block 1 keeps no key block (its rows see no key); key block 2 is
    kept by no query block (its keys get no gradient); with causal masking,
    query block 0 keeps only key block 3 (above the diagonal), so its rows
    are empty too."""
    B, N, H, dtype = 1, 600, 2, "bf16"
    x = make_inputs(B, N, H, d, dtype, seed=4300 + d + int(causal))
    mask = make_block_mask(H, N, "random", 0.6, seed=4301)
    mask[:, 1, :] = 0
    mask[:, :, 2] = 0
    if causal:
        mask[:, 0, :] = 0
        mask[:, 0, 3] = 1
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    g = run(q, k, v, do, scale, causal, mask.to(dev))
    assert np.all(np.isneginf(g["lse"][:, :, 128:256]))
    assert np.all(g["dk"][:, 256:384] == 0) and np.all(g["dv"][:, 256:384] == 0)
    x64 = {n: t.double().numpy() for n, t in x.items()}
    for h in range(H):
        check_head(oracle, x64, g, 0, h, scale, causal, dtype, mask[h].numpy())


def test_sparse_with_alibi(oracle):
    B, N, H, d, dtype, causal = 1, 1100, 2, 128, "bf16", True
    x = make_inputs(B, N, H, d, dtype, seed=4400)
    mask = make_block_mask(H, N, "random", 0.5, seed=4401)
    slopes = [0.25, 0.0625]
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    g = run(q, k, v, do, scale, causal, mask.to(dev),
            alibi=torch.tensor(slopes, dtype=torch.float32, device=dev))
    x64 = {n: t.double().numpy() for n, t in x.items()}
    for h in range(H):
        check_head(oracle, x64, g, 0, h, scale, causal, dtype, mask[h].numpy(), alibi=slopes[h])


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_equals_dense(causal):
    """A mask that keeps every block visits the same tiles in the same order
    as the dense kernels: O, LSE, dK and dV agree bit for bit (dQ is summed
    by reduce-adds in no fixed order, so only closely)."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d = 1, 777, 2, 128
    x = make_inputs(B, N, H, d, "bf16", seed=4500)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    ones = make_block_mask(H, N, "ones").to(dev)
    o1, l1 = attn.fwd(q, k, v, 0.1, causal)
    o2, l2 = attn.fwd(q, k, v, 0.1, causal, block_mask=ones)
    g1 = attn.bwd(q, k, v, o1, l1, do, 0.1, causal)
    g2 = attn.bwd(q, k, v, o1, l1, do, 0.1, causal, block_mask=ones)
    attn.check(attn.attn_status())
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert (g1[0].float() - g2[0].float()).abs().max().item() <= 0.0157


def test_all_zero_mask():
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d = 2, 400, 2, 64
    x = make_inputs(B, N, H, d, "fp16", seed=4600)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    zeros = torch.zeros(H, 4, 4, dtype=torch.uint8, device=dev)
    o, lse = attn.fwd(q, k, v, 0.125, False, block_mask=zeros)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, do, 0.125, False, block_mask=zeros)
    attn.check(attn.attn_status())
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)


def test_sparse_long_sampled(oracle):
    """N = 8192 with a banded mask (the launch configuration of the long
    workload): rows sampled from every 128-row block region, checked against
    the oracle one by one."""
    B, N, H, d, dtype = 1, 8192, 2, 128, "bf16"
    x = make_inputs(B, N, H, d, dtype, seed=4700)
    mask = make_block_mask(H, N, "local_global", width=2)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    g = run(q, k, v, do, scale, True, mask.to(dev), bwd=False)
    rng = np.random.default_rng(4701)
    rows = np.sort(np.concatenate([[0, 127, 128, N - 1], rng.choice(N, 60, replace=False)]))
    x64 = {n: t.double().numpy() for n, t in x.items()}
    for h in range(H):
        qq, kk, vv = (np.ascontiguousarray(x64[n][0, :, h, :]) for n in ("q", "k", "v"))
        o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, True, rows=rows,
                                         block_mask=mask[h].numpy())
        eo, _ = o_error(g["o"][0, rows, h, :], o_ref, dtype)
        assert eo <= TOL_O[dtype]
        assert np.max(np.abs(g["lse"][0, h, rows] - lse_ref)) <= TOL_LSE


def test_sparse_max_length(oracle):
    """N = 65536, the longest sequence a block mask may describe (512 blocks
    of 128 rows): banded mask with block row and column 0, causal, forward
    and backward, sampled rows and keys against the oracle."""
    B, N, H, d, dtype = 1, 65536, 1, 128, "bf16"
    x = make_inputs(B, N, H, d, dtype, seed=4800)
    mask = make_block_mask(H, N, "local_global", width=1)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    g = run(q, k, v, do, scale, True, mask.to(dev))
    rng = np.random.default_rng(4801)
    rows = np.sort(np.concatenate([[0, 127, 128, 255, N - 129, N - 1],
                                   rng.choice(N, 40, replace=False)]))
    keys = np.sort(np.concatenate([[0, 1, 127, 128, N - 128, N - 1],
                                   rng.choice(N, 40, replace=False)]))
    x64 = {n: t.double().numpy() for n, t in x.items()}
    qq, kk, vv, dd = (np.ascontiguousarray(x64[n][0, :, 0, :]) for n in ("q", "k", "v", "do"))
    bm = mask[0].numpy()
    o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, True, rows=rows, block_mask=bm)
    eo, _ = o_error(g["o"][0, rows, 0, :], o_ref, dtype)
    assert eo <= TOL_O[dtype]
    assert np.max(np.abs(g["lse"][0, 0, rows] - lse_ref)) <= TOL_LSE
    dq_r, dk_r, dv_r, _ = oracle.bwd_head(qq, kk, vv, dd, scale, True, rows=list(rows),
                                         keys=list(keys), block_mask=bm)
    for name, got, ref in (("dq", g["dq"][0, rows, 0, :], dq_r), ("dk", g["dk"][0, keys, 0, :], dk_r),
                           ("dv", g["dv"][0, keys, 0, :], dv_r)):
        err = rel_l2(got, ref)
        assert err <= TOL_GRAD, f"{name} rel L2 {err:.3e}"
