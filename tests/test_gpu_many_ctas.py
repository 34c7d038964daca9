"""GPU parity on shapes with two to three times as many forward work items
(query tile pair, b, h) as the device has SMs, so that the forward's grid
runs in several waves, and three to five backward items (128-key block, b,
h) per CTA of the persistent backward.  Every head is compared with the
fp64 oracle (O and LSE; dQ, dK, dV where the backward runs), for the plain,
ALiBi, dropout and accumulating variants.
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
    yield attn
    assert attn.attn_status() == 0


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _items(B, N, H):
    return ((N + 255) // 256) * B * H


def _check_heads(oracle, x, o, lse, scale, causal, dtype, grads=None, **per_head):
    """O and LSE of every head against the oracle; with grads = (dq, dk, dv),
    the gradients too (relative L2 per head)."""
    g_o, g_l = o.float().cpu().numpy(), lse.float().cpu().numpy()
    g_g = [t.float().cpu().numpy() for t in grads] if grads is not None else None
    x64 = {n: t.double().numpy() for n, t in x.items()}
    B, N, H, d = x64["q"].shape
    for b in range(B):
        for h in range(H):
            hd = lambda a: np.ascontiguousarray(a[b, :, h, :])  # noqa: E731
            kw = {k: f(b, h) for k, f in per_head.items()}
            qq, kk, vv = hd(x64["q"]), hd(x64["k"]), hd(x64["v"])
            o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, scale, causal, **kw)
            eo, _ = o_error(g_o[b, :, h, :], o_ref, dtype)
            assert eo <= TOL_O[dtype], f"({b},{h}) O {eo:.3e}"
            assert np.max(np.abs(g_l[b, h] - lse_ref)) <= TOL_LSE, f"({b},{h}) LSE"
            if g_g is not None:
                refs = oracle.bwd_head(qq, kk, vv, hd(x64["do"]), scale, causal, **kw)[:3]
                for name, g, ref in zip(("dq", "dk", "dv"), g_g, refs):
                    err = rel_l2(g[b, :, h, :], ref)
                    assert err <= TOL_GRAD, f"({b},{h}) {name} rel L2 {err:.3e}"


SHAPES = [
    # (B, N, H, d, dtype, causal): 2 to 3 work items per SM on 152 SMs
    (4, 300, 40, 64, "fp16", True),
    (3, 520, 40, 128, "bf16", False),
    (6, 300, 32, 128, "bf16", True),
    (2, 700, 60, 64, "bf16", True),
]


@pytest.mark.parametrize("B,N,H,d,dtype,causal", SHAPES,
                         ids=[f"B{s[0]}N{s[1]}H{s[2]}d{s[3]}{s[4]}{'c' if s[5] else 'n'}" for s in SHAPES])
def test_plain_many_items(oracle, _lib, B, N, H, d, dtype, causal):
    assert _items(B, N, H) >= 2 * _sms() - 10
    x = make_inputs(B, N, H, d, dtype, seed=8100 + N + H)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o, lse = _lib.fwd(q, k, v, scale, causal)
    grads = _lib.bwd(q, k, v, o, lse, do, scale, causal)
    _lib.check(_lib.attn_status())
    _check_heads(oracle, x, o, lse, scale, causal, dtype, grads=grads)


@pytest.mark.parametrize("causal,d", [(True, 128), (False, 64)])
def test_alibi_many_items(oracle, _lib, causal, d):
    B, N, H, dtype = 4, 300, 40, "bf16"
    x = make_inputs(B, N, H, d, dtype, seed=8200 + d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    m = [2.0 ** (-8.0 * (h + 1) / H) for h in range(H)]
    al = torch.tensor(m, dtype=torch.float32, device="cuda")
    scale = default_scale(d)
    o, lse = _lib.fwd(q, k, v, scale, causal, alibi=al)
    grads = _lib.bwd(q, k, v, o, lse, do, scale, causal, alibi=al)
    _lib.check(_lib.attn_status())
    _check_heads(oracle, x, o, lse, scale, causal, dtype, grads=grads, alibi=lambda b, h: m[h])


@pytest.mark.parametrize("causal,d,dtype", [(False, 64, "fp16"), (True, 128, "bf16")])
def test_dropout_many_items(oracle, _lib, causal, d, dtype):
    B, N, H, p, seed, offset = 4, 260, 40, 0.2, 99, 3
    x = make_inputs(B, N, H, d, dtype, seed=8300 + d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o, lse = _lib.fwd(q, k, v, scale, causal, dropout_p=p, seed=seed, offset=offset)
    grads = _lib.bwd(q, k, v, o, lse, do, scale, causal, dropout_p=p, seed=seed, offset=offset)
    _lib.check(_lib.attn_status())
    _check_heads(oracle, x, o, lse, scale, causal, dtype, grads=grads,
                 dropout=lambda b, h: (p, seed, offset, b * H + h))


def test_accumulating_many_items(oracle, _lib):
    """Two key blocks merged by the accumulating forward (non-causal) give the
    attention of the queries over both blocks' keys."""
    B, N, H, d, dtype = 4, 300, 40, 128, "bf16"
    scale = default_scale(d)
    x1 = make_inputs(B, N, H, d, dtype, seed=8401)
    x2 = make_inputs(B, N, H, d, dtype, seed=8402)
    q = x1["q"].cuda()
    k1, v1, k2, v2 = x1["k"].cuda(), x1["v"].cuda(), x2["k"].cuda(), x2["v"].cuda()
    o_acc = torch.empty((B, N, H, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    o = torch.empty_like(q)
    _lib.check(_lib.attn_fwd_acc(q, k1, v1, o_acc, lse, None, B, H, N, d, scale, False,
                                 _lib.ATTN_ACC_FIRST, dtype))
    _lib.check(_lib.attn_fwd_acc(q, k2, v2, o_acc, lse, o, B, H, N, d, scale, False,
                                 _lib.ATTN_ACC_LAST, dtype))
    _lib.check(_lib.attn_status())
    g_o, g_l = o.float().cpu().numpy(), lse.cpu().numpy()
    q64 = x1["q"].double().numpy()
    kk = np.concatenate([x1["k"].double().numpy(), x2["k"].double().numpy()], axis=1)
    vv = np.concatenate([x1["v"].double().numpy(), x2["v"].double().numpy()], axis=1)
    for b in range(B):
        for h in range(H):
            hd = lambda a: np.ascontiguousarray(a[b, :, h, :])  # noqa: E731
            o_ref, lse_ref = oracle.decode_head(hd(q64), hd(kk), hd(vv), scale, False)
            eo, _ = o_error(g_o[b, :, h, :], o_ref, dtype)
            assert eo <= TOL_O[dtype], f"({b},{h}) O {eo:.3e}"
            assert np.max(np.abs(g_l[b, h] - lse_ref)) <= TOL_LSE, f"({b},{h}) LSE"


def test_accumulating_backward_many_items(_lib):
    """One key block that is both the first and the last (FIRST | LAST) of the
    accumulating backward gives the plain backward's dK and dV bit for bit
    and its dQ within the order of the fp32 sums, on a shape with several
    backward items per CTA."""
    B, N, H, d, dtype = 4, 300, 40, 128, "bf16"
    x = make_inputs(B, N, H, d, dtype, seed=8500)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o, lse = _lib.fwd(q, k, v, scale, True)
    dq_ref, dk_ref, dv_ref = _lib.bwd(q, k, v, o, lse, do, scale, True)
    dq = torch.empty_like(q)
    acc = torch.full((2,) + tuple(q.shape), float("nan"), dtype=torch.float32, device="cuda")
    ws = _lib.workspace(B, H, N, d, q.device)
    _lib.check(_lib.attn_bwd_acc(q, k, v, o, lse, do, dq, acc[0], acc[1], B, H, N, d, scale, True,
                                 _lib.ATTN_ACC_FIRST | _lib.ATTN_ACC_LAST, _lib.ATTN_ACC_FIRST, dtype, ws,
                                 ws.numel()))
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    _lib.check(_lib.attn_cast_acc(acc[0], dk, dk.numel(), 1.0, dtype))
    _lib.check(_lib.attn_cast_acc(acc[1], dv, dv.numel(), 1.0, dtype))
    _lib.check(_lib.attn_status())
    assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)
    assert rel_l2(dq.double().cpu().numpy(), dq_ref.double().cpu().numpy()) < 1e-3
