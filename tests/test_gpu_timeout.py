"""Failure detection on the GPU without a fault: every device-side wait is
bounded.  A debug flag makes the forward's load warp issue no loads, so its
consumers' waits run out; the kernel then gives up cleanly, the status word
reports ATTN_ERR_TIMEOUT, and the context stays usable for the next call."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_22_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_recoverable():
    from exact_tiled_attention_22_gb300 import build
    build.build()
    from exact_tiled_attention_22_gb300 import attn
    dev = torch.device("cuda:0")
    x = make_inputs(1, 256, 1, 64, "fp16", seed=2)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 256), dtype=torch.float32, device=dev)
    assert attn.attn_status() == attn.ATTN_OK
    try:
        attn.attn_set_wait_limit(20_000_000, 1)  # 20 ms, no loads issued
        assert attn.attn_fwd(q, k, v, o, lse, 1, 1, 256, 64, 0.125, 0, "fp16") == attn.ATTN_OK
        assert attn.attn_status() == attn.ATTN_ERR_TIMEOUT
        assert "ran out of time" in attn.last_error()
    finally:
        attn.attn_set_wait_limit(0, 0)
    # the status word was cleared and the context still works
    assert attn.attn_status() == attn.ATTN_OK
    o2, lse2 = attn.fwd(q, k, v, 0.125, False)
    assert attn.attn_status() == attn.ATTN_OK
    assert torch.isfinite(o2.float()).all()
    s = (x["q"][0, :, 0].double() @ x["k"][0, :, 0].double().T) * 0.125
    ref = torch.logsumexp(s, dim=1).numpy()
    assert np.max(np.abs(lse2[0, 0].cpu().numpy() - ref)) < 1e-3


def _recovered(attn):
    assert attn.attn_status() == attn.ATTN_OK


@pytest.fixture(autouse=True)
def _built():
    from exact_tiled_attention_22_gb300 import build
    build.build()


def test_backward_wait_timeout_is_reported_and_recoverable(oracle):
    """Debug bit 1: the backward main kernel's load warp brings K and V but no
    query step, so every role's wait for the first step runs out mid-way
    (after copies have landed and K sits in tensor memory); the kernel drains
    and returns, the timeout is reported, and the next backward is right."""
    from exact_tiled_attention_22_gb300 import attn
    from parity import TOL_GRAD, rel_l2
    dev = torch.device("cuda:0")
    B, N, H, d = 1, 300, 2, 128
    x = make_inputs(B, N, H, d, "bf16", seed=21)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.fwd(q, k, v, 0.1, True)
    _recovered(attn)
    try:
        attn.attn_set_wait_limit(20_000_000, 2)
        attn.bwd(q, k, v, o, lse, do, 0.1, True)
        assert attn.attn_status() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.attn_set_wait_limit(0, 0)
    _recovered(attn)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, do, 0.1, True)
    _recovered(attn)
    hd = lambda t: t[0, :, 1].double().numpy()  # noqa: E731
    ref = oracle.bwd_head(hd(x["q"]), hd(x["k"]), hd(x["v"]), hd(x["do"]), 0.1, True)
    for got, r in zip((dq, dk, dv), ref[:3]):
        assert rel_l2(got[0, :, 1].float().cpu().numpy(), r) <= TOL_GRAD


def test_decode_wait_timeout_is_reported_and_recoverable(oracle):
    """Debug bit 2: the decoding chunk kernel's load warp issues nothing."""
    from exact_tiled_attention_22_gb300 import attn
    from parity import TOL_LSE
    dev = torch.device("cuda:0")
    B, H, Nq, Nk, d = 1, 2, 3, 2000, 64
    x = make_inputs(B, Nk, H, d, "fp16", seed=22)
    q = x["q"][:, Nk - Nq:].contiguous().to(dev)
    k, v = x["k"].to(dev), x["v"].to(dev)
    try:
        attn.attn_set_wait_limit(20_000_000, 4)
        attn.decode(q, k, v, 0.125, True)
        assert attn.attn_status() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.attn_set_wait_limit(0, 0)
    _recovered(attn)
    o, lse = attn.decode(q, k, v, 0.125, True)
    _recovered(attn)
    qh = x["q"][0, Nk - Nq:, 0].double().numpy()
    _, lse_ref = oracle.decode_head(qh, x["k"][0, :, 0].double().numpy(),
                                    x["v"][0, :, 0].double().numpy(), 0.125, True)
    assert np.max(np.abs(lse[0, 0].cpu().numpy() - lse_ref)) <= TOL_LSE
