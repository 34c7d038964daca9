"""GPU parity of the forward kernels on shapes with two to three times as
many (query tile pair, b, h) work items as the device has SMs, so that the
grid runs in several waves and the CTAs of later waves reuse the SMs of
earlier ones.  Every head is compared with the fp64 oracle (O and LSE), for
the plain, ALiBi, dropout and accumulating variants.
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
    yield attn
    assert attn.attn_status() == 0


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _items(B, N, H):
    return ((N + 255) // 256) * B * H


def _check_heads(oracle, x, o, lse, scale, causal, dtype, **per_head):
    g_o, g_l = o.float().cpu().numpy(), lse.float().cpu().numpy()
    x64 = {n: t.double().numpy() for n, t in x.items()}
    B, N, H, d = x64["q"].shape
    for b in range(B):
        for h in range(H):
            hd = lambda a: np.ascontiguousarray(a[b, :, h, :])  # noqa: E731
            kw = {k: f(b, h) for k, f in per_head.items()}
            o_ref, lse_ref = oracle.fwd_head(hd(x64["q"]), hd(x64["k"]), hd(x64["v"]), scale, causal, **kw)
            eo, _ = o_error(g_o[b, :, h, :], o_ref, dtype)
            assert eo <= TOL_O[dtype], f"({b},{h}) O {eo:.3e}"
            assert np.max(np.abs(g_l[b, h] - lse_ref)) <= TOL_LSE, f"({b},{h}) LSE"


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
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    scale = default_scale(d)
    o, lse = _lib.fwd(q, k, v, scale, causal)
    _lib.check(_lib.attn_status())
    _check_heads(oracle, x, o, lse, scale, causal, dtype)


@pytest.mark.parametrize("causal,d", [(True, 128), (False, 64)])
def test_alibi_many_items(oracle, _lib, causal, d):
    B, N, H, dtype = 4, 300, 40, "bf16"
    x = make_inputs(B, N, H, d, dtype, seed=8200 + d)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    m = [2.0 ** (-8.0 * (h + 1) / H) for h in range(H)]
    al = torch.tensor(m, dtype=torch.float32, device="cuda")
    scale = default_scale(d)
    o, lse = _lib.fwd(q, k, v, scale, causal, alibi=al)
    _lib.check(_lib.attn_status())
    _check_heads(oracle, x, o, lse, scale, causal, dtype, alibi=lambda b, h: m[h])


@pytest.mark.parametrize("causal,d,dtype", [(False, 64, "fp16"), (True, 128, "bf16")])
def test_dropout_many_items(oracle, _lib, causal, d, dtype):
    B, N, H, p, seed, offset = 4, 260, 40, 0.2, 99, 3
    x = make_inputs(B, N, H, d, dtype, seed=8300 + d)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    scale = default_scale(d)
    o, lse = _lib.fwd(q, k, v, scale, causal, dropout_p=p, seed=seed, offset=offset)
    _lib.check(_lib.attn_status())
    _check_heads(oracle, x, o, lse, scale, causal, dtype, dropout=lambda b, h: (p, seed, offset, b * H + h))


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
