"""Pins for the fp64 oracle: facts fixed by the definition of attention and
by mathematics, independent of the oracle's own code.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees.  ``tests/test_oracle_pins.py`` runs them on the committed oracle;
``tests/test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake, to show that each plausible mistake fails at least one pin.

Definition followed: page "突破单卡显存极限：FlashAttention-2技术解析与实战指南",
section 1 (S = Q K^T, P = softmax(S), O = P V), with the score scale of page
"Flash Attention V2大模型时代的算力救星", section 4.2; the blockwise recurrence
of the same page "突破单卡显存极限", section 2.1.
"""
import math

import numpy as np

from golden_io import load_cases, load_philox_kat, load_single

RNG = np.random.default_rng(20240707)


def _rand(*shape, rng=None):
    return (rng or RNG).standard_normal(shape)


def _close(a, b, tol, what):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------------------
def pin_golden_closed_form(O):
    """Hand-derived two-key cases (tests/golden/closed_form_two_keys.txt)."""
    for name, c in load_cases("closed_form_two_keys.txt").items():
        scale = float(c["scale"][0, 0])
        causal = bool(c["causal"][0, 0])
        o, lse = O.fwd_head(c["q"], c["k"], c["v"], scale, causal)
        _close(o, c["O"], 1e-13, f"{name} O")
        _close(lse, c["LSE"][:, 0], 1e-13, f"{name} LSE")
        dq, dk, dv, D = O.bwd_head(c["q"], c["k"], c["v"], c["dO"], scale, causal)
        _close(D, c["D"][:, 0], 1e-13, f"{name} D")
        _close(dq, c["dQ"], 1e-13, f"{name} dQ")
        _close(dk, c["dK"], 1e-13, f"{name} dK")
        _close(dv, c["dV"], 1e-13, f"{name} dV")


def pin_identity_v_gives_p(O):
    """With d = N and V = I, O_r is the probability row P_r itself: rows are
    non-negative, sum to 1, and P_rj = exp(s_rj - LSE_r)."""
    N = 8
    for causal in (False, True):
        q, k = _rand(N, N), _rand(N, N)
        scale = 0.37
        P, lse = O.fwd_head(q, k, np.eye(N), scale, causal)
        assert np.all(P >= 0), "negative probability"
        _close(P.sum(axis=1), np.ones(N), 1e-12, "row sums")
        s = scale * q @ k.T
        for r in range(N):
            for j in range(N):
                want = 0.0 if (causal and j > r) else math.exp(s[r, j] - lse[r])
                assert abs(P[r, j] - want) <= 1e-12, f"P[{r},{j}]"


def pin_lse_direct(O):
    """LSE_r = log sum_j exp(s_rj), summed directly with math.fsum on scores of
    moderate size (no shift needed)."""
    N, d = 13, 5
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    for causal in (False, True):
        _, lse = O.fwd_head(q, k, v, 0.5, causal)
        for r in range(N):
            hi = r + 1 if causal else N
            terms = [math.exp(0.5 * float(q[r] @ k[j])) for j in range(hi)]
            assert abs(lse[r] - math.log(math.fsum(terms))) <= 1e-12


def pin_constant_v(O):
    """V_j = v for every key gives O_r = v (rows of P sum to one)."""
    N, d = 11, 6
    q, k = _rand(N, d) * 3, _rand(N, d) * 3
    vrow = _rand(d)
    for causal in (False, True):
        o, _ = O.fwd_head(q, k, np.tile(vrow, (N, 1)), 0.8, causal)
        _close(o, np.tile(vrow, (N, 1)), 1e-12, "constant V")


def pin_causal_row0(O):
    """Causal row 0 sees only key 0: O_0 = V_0, LSE_0 = scale q_0 . k_0."""
    N, d = 9, 7
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    o, lse = O.fwd_head(q, k, v, 0.3, True)
    _close(o[0], v[0], 1e-14, "causal O_0")
    assert abs(lse[0] - 0.3 * float(q[0] @ k[0])) <= 1e-14


def pin_zero_q_uniform(O):
    """Q = 0 makes every score 0: P is uniform over the visible keys, so
    O_r = mean of visible V rows and LSE_r = ln(#visible)."""
    N, d = 10, 4
    k, v = _rand(N, d), _rand(N, d)
    q = np.zeros((N, d))
    o, lse = O.fwd_head(q, k, v, 1.0, False)
    _close(o, np.tile(v.mean(axis=0), (N, 1)), 1e-13, "uniform O")
    _close(lse, np.full(N, math.log(N)), 1e-13, "uniform LSE")
    o, lse = O.fwd_head(q, k, v, 1.0, True)
    want = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None]
    _close(o, want, 1e-13, "causal uniform O")
    _close(lse, np.log(np.arange(1, N + 1)), 1e-13, "causal uniform LSE")


def pin_single_key(O):
    """N = 1: P = 1, so O = V, LSE = scale q.k, dS = 0 -> dQ = dK = 0, dV = dO."""
    d = 6
    q, k, v, dO = _rand(1, d), _rand(1, d), _rand(1, d), _rand(1, d)
    for causal in (False, True):
        o, lse = O.fwd_head(q, k, v, 0.25, causal)
        _close(o, v, 1e-15, "N=1 O")
        assert abs(lse[0] - 0.25 * float(q[0] @ k[0])) <= 1e-15
        dq, dk, dv, _ = O.bwd_head(q, k, v, dO, 0.25, causal)
        _close(dq, np.zeros_like(dq), 1e-15, "N=1 dQ")
        _close(dk, np.zeros_like(dk), 1e-15, "N=1 dK")
        _close(dv, dO, 1e-15, "N=1 dV")


def pin_hardmax_limit(O):
    """Scores far apart (thousands) must not overflow; with a margin of
    hundreds, softmax is one-hot at the row max to fp64 precision."""
    N, d = 6, 3
    k = np.eye(N, d) * 0 + _rand(N, d)
    q = _rand(N, d)
    v = _rand(N, d)
    s = q @ k.T
    scale = 4000.0 / np.max(np.abs(s))
    o, lse = O.fwd_head(q, k, v, scale, False)
    for r in range(N):
        row = scale * s[r]
        top = np.argsort(row)[::-1]
        if row[top[0]] - row[top[1]] > 40:
            _close(o[r], v[top[0]], 1e-12, "hardmax O")
            assert abs(lse[r] - row[top[0]]) <= 1e-9
    assert np.all(np.isfinite(lse))


def pin_key_shift(O):
    """Adding the same vector u to every key adds scale q_r.u to every score of
    row r: P (hence O) is unchanged and LSE_r shifts by scale q_r.u."""
    N, d = 12, 5
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    u = _rand(d) * 2
    for causal in (False, True):
        o1, l1 = O.fwd_head(q, k, v, 0.7, causal)
        o2, l2 = O.fwd_head(q, k + u, v, 0.7, causal)
        _close(o2, o1, 1e-12, "shift O")
        _close(l2, l1 + 0.7 * q @ u, 1e-12, "shift LSE")


def pin_permutation(O):
    """Non-causal attention is invariant to a joint permutation of keys and
    values, and equivariant to a permutation of queries."""
    N, d = 9, 4
    q, k, v, dO = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    pk, pq = RNG.permutation(N), RNG.permutation(N)
    o1, l1 = O.fwd_head(q, k, v, 0.6, False)
    o2, l2 = O.fwd_head(q[pq], k[pk], v[pk], 0.6, False)
    _close(o2, o1[pq], 1e-12, "perm O")
    _close(l2, l1[pq], 1e-12, "perm LSE")
    g1 = O.bwd_head(q, k, v, dO, 0.6, False)
    g2 = O.bwd_head(q[pq], k[pk], v[pk], dO[pq], 0.6, False)
    _close(g2[0], g1[0][pq], 1e-12, "perm dQ")
    _close(g2[1], g1[1][pk], 1e-12, "perm dK")
    _close(g2[2], g1[2][pk], 1e-12, "perm dV")


def pin_finite_differences(O):
    """Gradients equal central finite differences of L = sum(O * dO)."""
    h = 1e-6
    for N, d in ((1, 4), (5, 4), (8, 8), (5, 8)):
        for causal in (False, True):
            q, k, v, dO = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
            scale = 1 / math.sqrt(d)
            dq, dk, dv, _ = O.bwd_head(q, k, v, dO, scale, causal)

            def loss(qq, kk, vv):
                o, _ = O.fwd_head(qq, kk, vv, scale, causal)
                return float(np.sum(o * dO))

            for which, grad in ((0, dq), (1, dk), (2, dv)):
                num = np.zeros((N, d))
                for i in range(N):
                    for c in range(d):
                        args_p = [q.copy(), k.copy(), v.copy()]
                        args_m = [q.copy(), k.copy(), v.copy()]
                        args_p[which][i, c] += h
                        args_m[which][i, c] -= h
                        num[i, c] = (loss(*args_p) - loss(*args_m)) / (2 * h)
                err = np.max(np.abs(num - grad)) / max(1.0, np.max(np.abs(num)))
                assert err <= 1e-6, f"FD N={N} d={d} causal={causal} arg{which}: {err:.2e}"


def pin_d_two_routes(O):
    """D_r from its definition sum_j P_rj dP_rj (oracle backward) equals
    dO_r . O_r with O from the oracle forward."""
    N, d = 33, 8
    q, k, v, dO = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    for causal in (False, True):
        o, _ = O.fwd_head(q, k, v, 0.4, causal)
        _, _, _, D = O.bwd_head(q, k, v, dO, 0.4, causal)
        _close(D, np.sum(dO * o, axis=1), 1e-12, "D two routes")


def pin_row_and_key_subsets(O):
    """Row / key index lists select exactly the corresponding full outputs."""
    N, d = 20, 4
    q, k, v, dO = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    rows, keys = [19, 0, 7, 7], [3, 18, 0]
    for causal in (False, True):
        o, l = O.fwd_head(q, k, v, 0.5, causal)
        os_, ls = O.fwd_head(q, k, v, 0.5, causal, rows=rows)
        _close(os_, o[rows], 0, "row subset O")
        _close(ls, l[rows], 0, "row subset LSE")
        dq, dk, dv, _ = O.bwd_head(q, k, v, dO, 0.5, causal)
        urows = rows[:3]  # the backward takes each row at most once
        sq, sk, sv, _ = O.bwd_head(q, k, v, dO, 0.5, causal, rows=urows, keys=keys)
        _close(sq, dq[urows], 1e-15, "row subset dQ")
        _close(sk, dk[keys], 1e-14, "key subset dK")
        _close(sv, dv[keys], 1e-14, "key subset dV")


def pin_online_golden(O):
    """Hand-worked blockwise statistics (tests/golden/online_softmax_two_blocks.txt)."""
    g = load_single("online_softmax_two_blocks.txt")
    # the worked row is query row 0; the routines take N queries for N keys,
    # so the same query is repeated (non-causal: every row is the worked row)
    q = np.vstack([g["q"].reshape(1, 1)] * 4)
    for tile in (1, 2, 3, 4):
        o, lse = O.online_fwd_head(q, g["k"], g["v"], 1.0, False, tile)
        assert abs(lse[0] - g["LSE"]) <= 1e-13, f"online LSE tile={tile}"
        assert abs(o[0, 0] - g["O"]) <= 1e-12, f"online O tile={tile}"
        of, lf = O.fwd_head(q, g["k"], g["v"], 1.0, False)
        assert abs(lf[0] - g["LSE"]) <= 1e-13 and abs(of[0, 0] - g["O"]) <= 1e-12


def pin_online_equals_full(O):
    """The blockwise recurrence gives the full softmax result for any block
    width (1, 3, 16, 128, N), causal or not, including sharp rows."""
    N, d = 150, 8
    q, k, v = _rand(N, d) * 2, _rand(N, d) * 2, _rand(N, d)
    for causal in (False, True):
        of, lf = O.fwd_head(q, k, v, 0.9, causal)
        for tile in (1, 3, 16, 128, N):
            ot, lt = O.online_fwd_head(q, k, v, 0.9, causal, tile)
            _close(ot, of, 1e-12, f"online O tile={tile}")
            _close(lt, lf, 1e-12, f"online LSE tile={tile}")


def pin_torch_sdpa(O):
    """Special case reducing to a library routine: torch's CPU math attention
    in float64 and its autograd gradients."""
    import torch
    B, N, H, d = 2, 37, 3, 16
    g = np.random.default_rng(5)
    q, k, v, dO = (g.standard_normal((B, N, H, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3), dtype=torch.float64,
                                   requires_grad=True) for x in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, is_causal=causal, scale=scale)
        out.backward(torch.tensor(dO.transpose(0, 2, 1, 3)))
        ref_o = out.detach().numpy().transpose(0, 2, 1, 3)
        ref_g = [t.grad.numpy().transpose(0, 2, 1, 3) for t in (tq, tk, tv)]
        fw = O.fwd(q, k, v, scale, causal)
        bw = O.bwd(q, k, v, dO, scale, causal)
        for (b, h), (o, _) in fw.items():
            _close(o, ref_o[b, :, h, :], 1e-12, "sdpa O")
            for i in range(3):
                _close(bw[(b, h)][i], ref_g[i][b, :, h, :], 1e-11, f"sdpa grad{i}")


def pin_decode_square_equals_fwd(O):
    """Nq = Nk: decoding is the ordinary forward pass, causal or not."""
    N, d = 23, 8
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    for causal in (False, True):
        o, lse = O.decode_head(q, k, v, 0.41, causal)
        o2, lse2 = O.fwd_head(q, k, v, 0.41, causal)
        _close(o, o2, 1e-13, "decode square O")
        _close(lse, lse2, 1e-13, "decode square LSE")


def pin_decode_last_rows(O):
    """The Nq decoded rows are the last Nq rows of the full attention: under
    the causal mask query i of Nq sees keys up to position Nk - Nq + i."""
    Nk, d = 40, 16
    qf, k, v = _rand(Nk, d), _rand(Nk, d), _rand(Nk, d)
    for causal in (False, True):
        full_o, full_lse = O.fwd_head(qf, k, v, 0.3, causal)
        for nq in (1, 3, 7, 16):
            o, lse = O.decode_head(qf[Nk - nq:], k, v, 0.3, causal)
            _close(o, full_o[Nk - nq:], 1e-13, f"decode last rows O nq={nq}")
            _close(lse, full_lse[Nk - nq:], 1e-13, f"decode last rows LSE nq={nq}")


def pin_decode_lse_direct(O):
    """LSE of a decoded row is log of the sum of exp over its visible keys,
    summed directly (math.fsum), and O is the P-weighted mean of those keys'
    values."""
    Nq, Nk, d = 4, 29, 5
    q, k, v = _rand(Nq, d), _rand(Nk, d), _rand(Nk, d)
    scale = 0.7
    o, lse = O.decode_head(q, k, v, scale, True)
    for i in range(Nq):
        vis = Nk - Nq + i + 1
        s = [scale * float(np.dot(q[i], k[j])) for j in range(vis)]
        ref = math.log(math.fsum(math.exp(x) for x in s))
        assert abs(lse[i] - ref) < 1e-12, f"decode LSE row {i}"
        p = np.array([math.exp(x - ref) for x in s])
        _close(o[i], p @ v[:vis], 1e-12, f"decode O row {i}")


def pin_alibi_closed_form(O):
    """ALiBi with all scores zero (q = 0): P_rj is proportional to
    exp(-m |r - j|), a two-sided geometric distribution whose normaliser is a
    sum of powers of exp(-m); with V = I the output row is P_r itself."""
    N = 9
    for m in (0.25, 1.5):
        for causal in (False, True):
            o, lse = O.fwd_head(np.zeros((N, N)), _rand(N, N), np.eye(N), 0.3, causal, alibi=m)
            for r in range(N):
                cols = range(r + 1) if causal else range(N)
                w = {j: math.exp(-m * abs(r - j)) for j in cols}
                z = math.fsum(w.values())
                assert abs(lse[r] - math.log(z)) < 1e-13, f"ALiBi LSE m={m} row {r}"
                ref = np.zeros(N)
                for j, x in w.items():
                    ref[j] = x / z
                _close(o[r], ref, 1e-14, f"ALiBi P m={m} row {r}")


def pin_alibi_torch_sdpa(O):
    """ALiBi reduces to torch's float64 attention with an additive float
    mask -m |i - j| (and -inf above the diagonal when causal), gradients
    included."""
    import torch
    B, N, H, d = 1, 23, 2, 8
    g = np.random.default_rng(8)
    q, k, v, dO = (g.standard_normal((B, N, H, d)) for _ in range(4))
    scale, slopes = 0.4, (0.5, 0.0625)
    idx = np.arange(N)
    for causal in (False, True):
        for h, m in enumerate(slopes):
            bias = -m * np.abs(idx[:, None] - idx[None, :]).astype(np.float64)
            if causal:
                bias = np.where(idx[None, :] > idx[:, None], -np.inf, bias)
            tq, tk, tv = (torch.tensor(x[0, :, h, :], dtype=torch.float64, requires_grad=True)
                          for x in (q, k, v))
            out = torch.nn.functional.scaled_dot_product_attention(
                tq[None], tk[None], tv[None], attn_mask=torch.tensor(bias)[None], scale=scale)[0]
            out.backward(torch.tensor(dO[0, :, h, :]))
            lse_ref = torch.logsumexp(scale * tq.detach() @ tk.detach().T + torch.tensor(bias), dim=1)
            o, lse = O.fwd_head(q[0, :, h], k[0, :, h], v[0, :, h], scale, causal, alibi=m)
            _close(o, out.detach().numpy(), 1e-12, "ALiBi sdpa O")
            _close(lse, lse_ref.numpy(), 1e-12, "ALiBi sdpa LSE")
            grads = O.bwd_head(q[0, :, h], k[0, :, h], v[0, :, h], dO[0, :, h], scale, causal,
                               alibi=m)
            for i, t in enumerate((tq, tk, tv)):
                _close(grads[i], t.grad.numpy(), 1e-11, f"ALiBi sdpa grad{i}")


def pin_alibi_decode_last_rows(O):
    """With ALiBi the decoded rows still equal the last rows of the full
    attention: the bias uses the rows' positions Nk - Nq + i."""
    Nk, d = 31, 8
    qf, k, v = _rand(Nk, d), _rand(Nk, d), _rand(Nk, d)
    for causal in (False, True):
        full_o, full_lse = O.fwd_head(qf, k, v, 0.3, causal, alibi=0.7)
        for nq in (1, 5):
            o, lse = O.decode_head(qf[Nk - nq:], k, v, 0.3, causal, alibi=0.7)
            _close(o, full_o[Nk - nq:], 1e-13, f"ALiBi decode O nq={nq}")
            _close(lse, full_lse[Nk - nq:], 1e-13, f"ALiBi decode LSE nq={nq}")


def _block_bool(mask, N, causal):
    """Element-wise visibility from a block mask over 128 x 128 blocks."""
    idx = np.arange(N)
    vis = mask[idx[:, None] // 128, idx[None, :] // 128].astype(bool)
    if causal:
        vis &= idx[None, :] <= idx[:, None]
    return vis


def pin_block_sparse_torch_sdpa(O):
    """A block mask reduces to torch's float64 attention with the equivalent
    boolean mask (every row keeps its diagonal block, so none is empty),
    gradients included."""
    import torch
    N, d = 300, 8   # 3 blocks, the last one ragged
    g = np.random.default_rng(12)
    q, k, v, dO = (g.standard_normal((N, d)) for _ in range(4))
    mask = np.array([[1, 0, 0], [0, 1, 1], [1, 0, 1]], dtype=np.uint8)
    scale = 0.35
    for causal in (False, True):
        vis = _block_bool(mask, N, causal)
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(
            tq[None], tk[None], tv[None], attn_mask=torch.tensor(vis)[None], scale=scale)[0]
        out.backward(torch.tensor(dO))
        o, lse = O.fwd_head(q, k, v, scale, causal, block_mask=mask)
        _close(o, out.detach().numpy(), 1e-12, "block-sparse sdpa O")
        sc = scale * q @ k.T
        lse_ref = [math.log(math.fsum(math.exp(x) for x in sc[r][vis[r]])) for r in range(N)]
        _close(lse, lse_ref, 1e-11, "block-sparse LSE")
        grads = O.bwd_head(q, k, v, dO, scale, causal, block_mask=mask)
        for i, t in enumerate((tq, tk, tv)):
            _close(grads[i], t.grad.numpy(), 1e-11, f"block-sparse grad{i}")


def pin_block_sparse_key_block_removed(O):
    """Masking key block kb for every query block equals attention over the
    keys with that block deleted."""
    N, d = 384, 6
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    mask = np.ones((3, 3), dtype=np.uint8)
    mask[:, 1] = 0
    keep = np.r_[0:128, 256:384]
    o, lse = O.fwd_head(q, k, v, 0.4, False, block_mask=mask)
    # the reference: each row against the remaining keys, by the definition
    for r in (0, 130, 383):
        s = 0.4 * k[keep] @ q[r]
        w = np.exp(s - s.max())
        _close(o[r], (w / w.sum()) @ v[keep], 1e-12, f"key block removed row {r}")
        ref_lse = math.log(math.fsum(math.exp(x) for x in s))
        assert abs(lse[r] - ref_lse) < 1e-12, f"key block removed LSE row {r}"


def pin_block_sparse_empty_rows(O):
    """A query block whose key blocks are all masked has O = 0, LSE = -inf,
    dQ = 0, and adds nothing to dK and dV: they equal the gradients with its
    rows' dO set to zero."""
    N, d = 256, 4
    q, k, v, dO = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    mask = np.array([[1, 1], [0, 0]], dtype=np.uint8)
    o, lse = O.fwd_head(q, k, v, 0.5, False, block_mask=mask)
    assert np.all(o[128:] == 0) and np.all(np.isneginf(lse[128:])), "empty rows"
    dq, dk, dv, _ = O.bwd_head(q, k, v, dO, 0.5, False, block_mask=mask)
    assert np.all(dq[128:] == 0), "dQ of empty rows"
    dO0 = dO.copy()
    dO0[128:] = 0
    _, dk2, dv2, _ = O.bwd_head(q, k, v, dO0, 0.5, False)
    _close(dk, dk2, 1e-12, "dK without empty rows")
    _close(dv, dv2, 1e-12, "dV without empty rows")


# ---------------------------------------------------------------------------
# Dropout: Philox4x32-10 decisions (Salmon et al., SC 2011), inverted scaling.
def pin_philox4x64_matches_numpy(O):
    """The generator's rounds, instantiated at 64-bit words, are numpy's
    Philox4x64-10 bit generator (numpy increments its 256-bit counter before
    each block of four outputs)."""
    g = np.random.default_rng(77)
    for _ in range(6):
        key = [int(x) for x in g.integers(0, 2**63, size=2, dtype=np.uint64)]
        ctr = [int(x) for x in g.integers(0, 2**62, size=4, dtype=np.uint64)]
        bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                              counter=np.array(ctr, dtype=np.uint64))
        ref = [int(x) for x in bg.random_raw(4)]
        got = O.philox4x64([ctr[0] + 1, ctr[1], ctr[2], ctr[3]], key)
        assert got == ref, f"philox4x64 {ctr} {key}: {got} != {ref}"


def pin_philox4x32_known_answers(O):
    """The 32-bit instance the dropout uses reproduces the published
    known-answer vectors of Philox4x32-10 (Salmon et al., SC 2011; the
    authors' Random123 test file): all-zero, all-ones and digits-of-pi
    counters and keys (tests/golden/philox4x32_10_kat.txt).  This fixes the
    multipliers, the Weyl constants, the round count and the word order."""
    kats = load_philox_kat()
    assert len(kats) == 3
    for ctr, key, ref in kats:
        got = O.philox4x32(ctr, key)
        assert list(got) == ref, f"philox4x32 {ctr} {key}: {[hex(x) for x in got]}"


def pin_philox4x32_statistics(O):
    """The 32-bit instance (the one the dropout uses) is a good generator:
    over consecutive counters every output byte value is about equally
    frequent (chi-square), and one changed counter bit flips about half of
    the 128 output bits."""
    counts = np.zeros(256)
    flips = []
    for c in range(2048):
        x = O.philox4x32([c, 3, 5, 7], [0x12345678, 0x9ABCDEF0])
        for w in x:
            for b in range(4):
                counts[(w >> (8 * b)) & 0xFF] += 1
        y = O.philox4x32([c ^ 1, 3, 5, 7], [0x12345678, 0x9ABCDEF0])
        flips.append(sum(bin(a ^ b).count("1") for a, b in zip(x, y)))
    exp = counts.sum() / 256
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < 255 + 6 * math.sqrt(2 * 255), f"byte chi-square {chi2:.1f}"
    assert abs(np.mean(flips) - 64) < 1.0, f"avalanche {np.mean(flips):.2f} bits"


def pin_dropout_decision_rule(O):
    """Z_rj is byte j % 16 (word (j % 16) / 4, low byte first) of
    Philox4x32-10 at counter (r, j / 16, head, offset), key (seed low, seed
    high), compared with t; t = floor(256 (1 - p) + 1/2)."""
    seed, off, head = 0x0123456789ABCDEF, 7, 3
    assert O.dropout_threshold(0.1) == 230 and O.dropout_threshold(0.5) == 128
    assert O.dropout_threshold(0.7) == 77  # 76.8 rounds up
    assert O.dropout_threshold(0.0) == 256 and O.dropout_threshold(1.0) == -1
    assert O.dropout_threshold(-0.1) == -1 and O.dropout_threshold(0.999) == -1
    for r, j, t in ((0, 0, 230), (5, 17, 128), (1000, 4095, 64), (3, 31, 200)):
        x = O.philox4x32([r, j // 16, head, off], [seed & 0xFFFFFFFF, seed >> 32])
        byte = (x[(j % 16) // 4] >> (8 * (j % 4))) & 0xFF
        assert O.dropout_keep(seed, off, head, r, j, t) == int(byte < t), (r, j)


def pin_dropout_keep_fraction(O):
    """Over many scores the kept fraction is t / 256 (within 5 sigma), and
    the decisions change with the head, the offset and the seed (two
    independent masks agree on a fraction q^2 + (1-q)^2 of the scores)."""
    for p in (0.1, 0.5, 0.8):
        t = O.dropout_threshold(p)
        q = t / 256
        keep = [O.dropout_keep(42, 0, 0, r, j, t) for r in range(64) for j in range(256)]
        n = len(keep)
        assert abs(np.mean(keep) - q) < 5 * math.sqrt(q * (1 - q) / n), (p, np.mean(keep))
    t = 128
    base = np.array([O.dropout_keep(42, 0, 0, r, j, t) for r in range(32) for j in range(64)])
    for other in ((43, 0, 0), (42, 1, 0), (42, 0, 1), (42 + (1 << 32), 0, 0)):
        alt = np.array([O.dropout_keep(*other, r, j, t) for r in range(32) for j in range(64)])
        agree = float(np.mean(base == alt))
        assert abs(agree - 0.5) < 5 * math.sqrt(0.25 / base.size), (other, agree)


def _dropout_weights(O, N, seed, off, head, t, causal):
    """Z / q as an N x N matrix (0 where the causal rule removes a score)."""
    w = np.zeros((N, N))
    for r in range(N):
        for j in range(r + 1 if causal else N):
            w[r, j] = O.dropout_keep(seed, off, head, r, j, t) * 256.0 / t
    return w


def pin_dropout_torch(O):
    """With dropout the forward is (softmax(S) * W) V for the fixed weights
    W = Z / q, and the backward is that function's gradient: torch's float64
    softmax and autograd with W as a constant multiplier.  LSE is the one
    without dropout."""
    import torch
    N, d, scale = 40, 5, 0.45
    g = np.random.default_rng(31)
    q, k, v, dO = (g.standard_normal((N, d)) for _ in range(4))
    for causal, p in ((False, 0.3), (True, 0.6)):
        seed, off, head = 99, 3, 2
        t = O.dropout_threshold(p)
        W = torch.tensor(_dropout_weights(O, N, seed, off, head, t, causal))
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        s = scale * tq @ tk.T
        if causal:
            s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
        out = (torch.softmax(s, dim=1) * W) @ tv
        out.backward(torch.tensor(dO))
        dr = (p, seed, off, head)
        o, lse = O.fwd_head(q, k, v, scale, causal, dropout=dr)
        _close(o, out.detach().numpy(), 1e-12, "dropout O")
        _, lse0 = O.fwd_head(q, k, v, scale, causal)
        assert np.array_equal(lse, lse0), "dropout changed LSE"
        dq, dk, dv, D = O.bwd_head(q, k, v, dO, scale, causal, dropout=dr)
        for i, tt in enumerate((tq, tk, tv)):
            _close((dq, dk, dv)[i], tt.grad.numpy(), 1e-11, f"dropout grad{i}")
        _close(D, np.sum(dO * o, axis=1), 1e-12, "dropout D = rowsum(dO * O)")


def pin_dropout_mean_is_plain(O):
    """E[Z / q] = 1: averaged over many offsets the dropout output tends to
    the output without dropout (within 6 standard errors)."""
    N, d, scale = 6, 3, 0.7
    g = np.random.default_rng(5)
    q, k, v = (g.standard_normal((N, d)) for _ in range(3))
    o0, _ = O.fwd_head(q, k, v, scale, False)
    outs = np.stack([O.fwd_head(q, k, v, scale, False, dropout=(0.4, 1234, off, 0))[0]
                     for off in range(3000)])
    se = outs.std(axis=0) / math.sqrt(len(outs))
    assert np.all(np.abs(outs.mean(axis=0) - o0) <= 6 * se + 1e-12), "dropout mean"


def pin_dropout_p0_is_plain(O):
    """p small enough that t = 256 keeps every score with weight 1."""
    N, d = 50, 4
    q, k, v, dO = _rand(N, d), _rand(N, d), _rand(N, d), _rand(N, d)
    for p in (0.0, 0.001):
        o, lse = O.fwd_head(q, k, v, 0.3, True, dropout=(p, 5, 6, 7))
        o0, lse0 = O.fwd_head(q, k, v, 0.3, True)
        assert np.array_equal(o, o0) and np.array_equal(lse, lse0)
        g = O.bwd_head(q, k, v, dO, 0.3, True, dropout=(p, 5, 6, 7))
        g0 = O.bwd_head(q, k, v, dO, 0.3, True)
        for a, b in zip(g, g0):
            assert np.array_equal(a, b)


PINS = [
    pin_golden_closed_form,
    pin_identity_v_gives_p,
    pin_lse_direct,
    pin_constant_v,
    pin_causal_row0,
    pin_zero_q_uniform,
    pin_single_key,
    pin_hardmax_limit,
    pin_key_shift,
    pin_permutation,
    pin_finite_differences,
    pin_d_two_routes,
    pin_row_and_key_subsets,
    pin_online_golden,
    pin_online_equals_full,
    pin_torch_sdpa,
    pin_decode_square_equals_fwd,
    pin_decode_last_rows,
    pin_decode_lse_direct,
    pin_alibi_closed_form,
    pin_alibi_torch_sdpa,
    pin_alibi_decode_last_rows,
    pin_block_sparse_torch_sdpa,
    pin_block_sparse_key_block_removed,
    pin_block_sparse_empty_rows,
    pin_philox4x64_matches_numpy,
    pin_philox4x32_known_answers,
    pin_philox4x32_statistics,
    pin_dropout_decision_rule,
    pin_dropout_keep_fraction,
    pin_dropout_torch,
    pin_dropout_mean_is_plain,
    pin_dropout_p0_is_plain,
]


def failing_pins(O, first_only=False):
    """Names of the pins the given oracle fails (any exception counts); with
    first_only, stops at the first failing pin."""
    bad = []
    for p in PINS:
        try:
            p(O)
        except Exception:  # noqa: BLE001 - a mutant may crash or return NaN
            bad.append(p.__name__)
            if first_only:
                break
    return bad
