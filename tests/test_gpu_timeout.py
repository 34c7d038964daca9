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
