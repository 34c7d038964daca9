"""GPU parity of the dropout variants (attn_fwd_ex, attn_bwd_ex) against the
fp64 oracle with the same Philox4x32-10 decisions.

The decisions are integer work, so they are checked bit for bit: with V
rows one-hot (V_j = e_{j mod d}) and a block mask that keeps one key block
per query block, O_ij = Z_ij P_ij 256/t is zero exactly where the kernel
dropped score (i, j); with dO rows one-hot, dV shows the backward's
decisions the same way.  Values are compared with the usual tolerances on
several shapes (causal and not, both head dims and dtypes, ragged tails),
with ALiBi and a block mask combined, with a block mask that leaves query
rows without keys and keys without queries (outputs start as NaN), and at
N = 8192 on sampled rows and keys.
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


def oracle_keep(oracle, seed, offset, head, rows, keys, t):
    return np.array([[oracle.dropout_keep(seed, offset, head, r, j, t) for j in keys]
                     for r in rows], dtype=bool)


@pytest.mark.parametrize("d,p,causal", [(128, 0.1, False), (128, 0.5, True), (64, 0.3, False)])
def test_dropout_decisions_bit_exact(oracle, d, p, causal):
    """Every forward and backward keep/drop decision of 2 batches x 2 heads x
    512 rows, each query block against one key block, equals the oracle's."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H = 2, 512, 2
    nb = N // 128
    seed, offset = 0x5EED1234ABCD, 17
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(6000 + d)
    q = (0.3 * torch.randn(B, N, H, d, generator=g)).to(torch.bfloat16)
    k = (0.3 * torch.randn(B, N, H, d, generator=g)).to(torch.bfloat16)
    eye = torch.zeros(N, d)
    eye[torch.arange(N), torch.arange(N) % d] = 1.0
    v = eye[None, :, None, :].expand(B, N, H, d).contiguous().to(torch.bfloat16)
    # query block qb keeps key block perm[qb] only (causal: its own block)
    perm = [qb for qb in range(nb)] if causal else [(3 * qb + 1) % nb for qb in range(nb)]
    mask = torch.zeros(H, nb, nb, dtype=torch.uint8)
    for qb in range(nb):
        mask[:, qb, perm[qb]] = 1
    q, k, v, do = q.to(dev), k.to(dev), v.to(dev), v.to(dev)
    bm = mask.to(dev)
    o, lse = attn.fwd(q, k, v, 0.1, causal, block_mask=bm, dropout_p=p, seed=seed, offset=offset)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, do, 0.1, causal, block_mask=bm, dropout_p=p,
                          seed=seed, offset=offset)
    attn.check(attn.attn_status())
    o, dv = o.float().cpu().numpy(), dv.float().cpu().numpy()
    t = oracle.dropout_threshold(p)
    kept_total = 0
    for b in range(B):
        for h in range(H):
            head = b * H + h
            for qb in range(nb):
                rows = range(128 * qb, 128 * qb + 128)
                keys = range(128 * perm[qb], 128 * perm[qb] + 128)
                z = oracle_keep(oracle, seed, offset, head, rows, keys, t)
                vis = np.ones((128, 128), dtype=bool)
                if causal:
                    vis = np.tril(vis)
                # forward: column c of O row i is key 128 perm[qb] + c (c < d;
                # for d = 64 keys c and c + 64 share a column)
                got = o[b, 128 * qb:128 * qb + 128, h, :] != 0
                want = z & vis
                if d == 128:
                    assert np.array_equal(got, want), f"fwd decisions ({b},{h}) block {qb}"
                else:
                    assert np.array_equal(got, want[:, :64] | want[:, 64:]), f"fwd ({b},{h}) {qb}"
                # backward: dV row j = sum_i Z_ij P_ij 256/t dO_i, dO_i = e_(i mod d)
                gotv = dv[b, 128 * perm[qb]:128 * perm[qb] + 128, h, :] != 0
                if d == 128:
                    assert np.array_equal(gotv, want.T), f"bwd decisions ({b},{h}) block {qb}"
                else:
                    assert np.array_equal(gotv, want.T[:, :64] | want.T[:, 64:]), f"bwd ({b},{h}) {qb}"
                kept_total += int(want.sum())
    n_vis = B * H * nb * (128 * 129 // 2 if causal else 128 * 128)
    q_keep = t / 256
    assert abs(kept_total / n_vis - q_keep) < 5 * np.sqrt(q_keep * (1 - q_keep) / n_vis)


SHAPES = [
    # (B, N, H, d, dtype, causal, p)
    (1, 300, 2, 128, "bf16", True, 0.1),
    (2, 257, 2, 64, "fp16", False, 0.25),
    (1, 640, 3, 128, "fp16", False, 0.5),
    (1, 1000, 2, 128, "bf16", True, 0.3),
    (1, 129, 2, 64, "bf16", True, 0.6),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}N{}H{}d{}{}{}p{}".format(
    *s[:5], "c" if s[5] else "", s[6]))
def test_dropout_fwd_bwd_match_oracle(oracle, shape):
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d, dtype, causal, p = shape
    seed, offset = 1234 + N, 5
    x = make_inputs(B, N, H, d, dtype, seed=6100 + N)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o, lse = attn.fwd(q, k, v, scale, causal, dropout_p=p, seed=seed, offset=offset)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, do, scale, causal, dropout_p=p, seed=seed,
                          offset=offset)
    attn.check(attn.attn_status())
    g = {n: t_.float().cpu().numpy() for n, t_ in (("o", o), ("lse", lse), ("dq", dq),
                                                    ("dk", dk), ("dv", dv))}
    x64 = {n: t_.double().numpy() for n, t_ in x.items()}
    for b in range(B):
        for h in range(H):
            hd = lambda a: np.ascontiguousarray(a[b, :, h, :])  # noqa: E731
            qq, kk, vv, dd = (hd(x64[n]) for n in ("q", "k", "v", "do"))
            dr = (p, seed, offset, b * H + h)
            o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, causal, dropout=dr)
            eo, _ = o_error(g["o"][b, :, h, :], o_ref, dtype)
            assert eo <= TOL_O[dtype], f"({b},{h}) O {eo:.3e}"
            assert np.max(np.abs(g["lse"][b, h] - lse_ref)) <= TOL_LSE, f"({b},{h}) LSE"
            dq_r, dk_r, dv_r, _ = oracle.bwd_head(qq, kk, vv, dd, scale, causal, dropout=dr)
            for name, ref in (("dq", dq_r), ("dk", dk_r), ("dv", dv_r)):
                err = rel_l2(g[name][b, :, h, :], ref)
                assert err <= TOL_GRAD, f"({b},{h}) {name} rel L2 {err:.3e}"


def test_dropout_with_alibi_and_mask(oracle):
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d, dtype, causal, p = 1, 700, 2, 128, "bf16", True, 0.2
    x = make_inputs(B, N, H, d, dtype, seed=6200)
    mask = make_block_mask(H, N, "random", 0.6, seed=6201)
    slopes = [0.125, 0.03125]
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    al = torch.tensor(slopes, dtype=torch.float32, device=dev)
    scale = default_scale(d)
    kw = dict(alibi=al, block_mask=mask.to(dev), dropout_p=p, seed=77, offset=3)
    o, lse = attn.fwd(q, k, v, scale, causal, **kw)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, do, scale, causal, **kw)
    attn.check(attn.attn_status())
    x64 = {n: t_.double().numpy() for n, t_ in x.items()}
    for h in range(H):
        qq, kk, vv, dd = (np.ascontiguousarray(x64[n][0, :, h, :]) for n in ("q", "k", "v", "do"))
        ex = dict(alibi=slopes[h], block_mask=mask[h].numpy(), dropout=(p, 77, 3, h))
        o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, causal, **ex)
        empty = np.isneginf(lse_ref)
        eo, _ = o_error(o[0, :, h, :].float().cpu().numpy(), o_ref, dtype)
        assert eo <= TOL_O[dtype]
        lg = lse[0, h].cpu().numpy()
        assert np.array_equal(np.isneginf(lg), empty)
        assert np.max(np.abs(lg[~empty] - lse_ref[~empty])) <= TOL_LSE
        dq_r, dk_r, dv_r, _ = oracle.bwd_head(qq, kk, vv, dd, scale, causal, **ex)
        for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
            err = rel_l2(got[0, :, h, :].float().cpu().numpy(), ref)
            assert err <= TOL_GRAD, f"head {h} {name} rel L2 {err:.3e}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_dropout_empty_rows_and_keys(oracle, causal, d):
    """Dropout with a block mask in which query block 1 keeps no key block and
    key block 2 is kept by no query block: the rows of query block 1 get
    O = 0, LSE = -inf, dQ = 0 and the keys of block 2 dK = dV = 0, written
    over outputs that start as NaN."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, dtype, p = 1, 600, 2, "bf16", 0.3
    x = make_inputs(B, N, H, d, dtype, seed=6500 + d + int(causal))
    mask = make_block_mask(H, N, "random", 0.7, seed=6501)
    mask[:, 1, :] = 0
    mask[:, :, 2] = 0
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    bm = mask.to(dev)
    o, lse = attn.fwd(q, k, v, scale, causal, block_mask=bm, dropout_p=p, seed=31, offset=4)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    ws = attn.workspace(B, H, N, d, dev)
    attn.check(attn.attn_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, None,
                                bm, p, 31, 4, q.dtype, ws, ws.numel(), None))
    attn.check(attn.attn_status())
    lg = lse.cpu().numpy()
    assert np.all(np.isneginf(lg[:, :, 128:256]))
    assert torch.all(o[:, 128:256] == 0) and torch.all(dq[:, 128:256] == 0)
    assert torch.all(dk[:, 256:384] == 0) and torch.all(dv[:, 256:384] == 0)
    x64 = {n: t_.double().numpy() for n, t_ in x.items()}
    for h in range(H):
        qq, kk, vv, dd = (np.ascontiguousarray(x64[n][0, :, h, :]) for n in ("q", "k", "v", "do"))
        ex = dict(block_mask=mask[h].numpy(), dropout=(p, 31, 4, h))
        o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, causal, **ex)
        empty = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lg[0, h]), empty)
        eo, _ = o_error(o[0, :, h, :].float().cpu().numpy(), o_ref, dtype)
        assert eo <= TOL_O[dtype]
        assert np.max(np.abs(lg[0, h][~empty] - lse_ref[~empty])) <= TOL_LSE
        dq_r, dk_r, dv_r, _ = oracle.bwd_head(qq, kk, vv, dd, scale, causal, **ex)
        for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
            g = got[0, :, h, :].float().cpu().numpy()
            assert np.all(np.isfinite(g)), f"head {h} {name} not written everywhere"
            err = rel_l2(g, ref)
            assert err <= TOL_GRAD, f"head {h} {name} rel L2 {err:.3e}"


def test_dropout_deterministic_and_offset_dependent():
    """The same (seed, offset) gives the same output bit for bit, another
    offset another mask; a dropout_p that rounds to t = 256 is the plain
    kernel."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d = 1, 512, 2, 128
    x = make_inputs(B, N, H, d, "bf16", seed=6300)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o1, l1 = attn.fwd(q, k, v, 0.1, True, dropout_p=0.2, seed=9, offset=1)
    o2, l2 = attn.fwd(q, k, v, 0.1, True, dropout_p=0.2, seed=9, offset=1)
    o3, l3 = attn.fwd(q, k, v, 0.1, True, dropout_p=0.2, seed=9, offset=2)
    o4, l4 = attn.fwd(q, k, v, 0.1, True)
    o5, l5 = attn.fwd(q, k, v, 0.1, True, dropout_p=0.001, seed=9, offset=1)
    attn.check(attn.attn_status())
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert not torch.equal(o1, o3) and torch.equal(l1, l3)
    # LSE does not depend on dropout; the dropout kernel adds each row's
    # exponentials in two partial sums (one per column half), so it agrees
    # with the plain kernel's to rounding, not bit for bit
    assert (l1 - l4).abs().max().item() <= 1e-5
    assert torch.equal(o4, o5) and torch.equal(l4, l5)


def test_dropout_long_sampled(oracle):
    """N = 8192, d = 128, causal, p = 0.1, in the launch configuration of the
    long workload: sampled rows (O, LSE, dQ) and keys (dK, dV) against the
    oracle."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d, dtype = 1, 8192, 2, 128, "bf16"
    x = make_inputs(B, N, H, d, dtype, seed=6400)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o_t, lse_t = attn.fwd(q, k, v, scale, True, dropout_p=0.1, seed=2024, offset=8)
    dq, dk, dv = attn.bwd(q, k, v, o_t, lse_t, do, scale, True, dropout_p=0.1, seed=2024,
                          offset=8)
    attn.check(attn.attn_status())
    rng = np.random.default_rng(6401)
    rows = np.sort(np.concatenate([[0, 1, 127, 128, N - 1], rng.choice(N, 40, replace=False)]))
    keys = np.sort(np.unique(np.concatenate([[0, 1, 127, 128, N // 2, N - 129, N - 1],
                                             rng.choice(N, 40, replace=False)])))
    o, lse = o_t.float().cpu().numpy(), lse_t.cpu().numpy()
    grads = {n: t_.float().cpu().numpy() for n, t_ in (("dq", dq), ("dk", dk), ("dv", dv))}
    x64 = {n: t_.double().numpy() for n, t_ in x.items()}
    for h in range(H):
        qq, kk, vv, dd = (np.ascontiguousarray(x64[n][0, :, h, :]) for n in ("q", "k", "v", "do"))
        dr = (0.1, 2024, 8, h)
        o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, True, rows=rows, dropout=dr)
        eo, _ = o_error(o[0, rows, h, :], o_ref, dtype)
        assert eo <= TOL_O[dtype]
        assert np.max(np.abs(lse[0, h, rows] - lse_ref)) <= TOL_LSE
        dq_r, dk_r, dv_r, _ = oracle.bwd_head(qq, kk, vv, dd, scale, True, rows=rows, keys=keys,
                                              dropout=dr)
        for name, sel, ref in (("dq", rows, dq_r), ("dk", keys, dk_r), ("dv", keys, dv_r)):
            err = rel_l2(grads[name][0, sel, h, :], ref)
            assert err <= TOL_GRAD, f"head {h} {name} rel L2 {err:.3e}"
