"""Capture safety and the autograd wrapper.

The calls allocate nothing and never synchronise, so a forward + backward
can be captured into a CUDA graph and replayed on new input values; the
replay must give the eager results (bit for bit where the kernels are
deterministic: O, LSE, dK, dV; dQ is summed by reduce-adds in no fixed
order).  attn.attention is a torch.autograd.Function over the same calls.
"""
import pytest
import torch

from exact_tiled_attention_22_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def rel(a, b):
    """Relative L2 difference (dQ: the same values summed in another order)."""
    a, b = a.float(), b.float()
    return ((a - b).norm() / b.norm().clamp_min(1e-30)).item()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_tiled_attention_22_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from exact_tiled_attention_22_gb300 import attn
    attn.attn_set_wait_limit(0, 0)
    yield
    assert attn.attn_status() == 0


@pytest.mark.parametrize("dropout_p", [0.0, 0.1])
def test_cuda_graph_replay_matches_eager(dropout_p):
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d = 2, 700, 2, 128
    dev = torch.device("cuda:0")
    xs = [make_inputs(B, N, H, d, "bf16", seed=9000 + i) for i in range(2)]
    q, k, v, do = (xs[0][n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = attn.workspace(B, H, N, d, dev)
    scale = d ** -0.5

    def step(stream):
        attn.check(attn.attn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, True, None, None,
                                    dropout_p, 5, 7, q.dtype, stream))
        attn.check(attn.attn_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, True,
                                    None, None, dropout_p, 5, 7, q.dtype, ws, ws.numel(),
                                    stream))

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step(side)  # eager warm-up on the capture stream
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step(side)
    for x in xs:  # replay on new values copied into the captured buffers
        for n, t in (("q", q), ("k", k), ("v", v), ("do", do)):
            t.copy_(x[n].to(dev))
        g.replay()
        torch.cuda.synchronize(dev)
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        ref_o, ref_lse = attn.fwd(q, k, v, scale, True, dropout_p=dropout_p, seed=5, offset=7)
        ref_dq, ref_dk, ref_dv = attn.bwd(q, k, v, ref_o, ref_lse, do, scale, True,
                                          dropout_p=dropout_p, seed=5, offset=7)
        attn.check(attn.attn_status())
        assert torch.equal(got[0], ref_o) and torch.equal(got[1], ref_lse)
        assert torch.equal(got[3], ref_dk) and torch.equal(got[4], ref_dv)
        assert rel(got[2], ref_dq) <= 1e-3


def test_autograd_function_matches_direct_calls():
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d = 1, 513, 3, 64
    x = make_inputs(B, N, H, d, "fp16", seed=9100)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = attn.attention(qa, ka, va, 0.125, True, dropout_p=0.2, seed=3, offset=4)
    out.backward(do)
    o, lse = attn.fwd(q, k, v, 0.125, True, dropout_p=0.2, seed=3, offset=4)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, do, 0.125, True, dropout_p=0.2, seed=3, offset=4)
    attn.check(attn.attn_status())
    assert torch.equal(out.detach(), o)
    assert torch.equal(ka.grad, dk) and torch.equal(va.grad, dv)
    assert rel(qa.grad, dq) <= 1e-3
