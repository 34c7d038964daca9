"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (code with no CUDA allocator at hand, or loops that must not call
cudaMalloc because it can synchronise the device).  It takes no workspace
and uses a fixed scratch array owned by the library instead.

Checked through the C ABI against attn_bwd (which takes a caller workspace)
on calls made back to back, so the second call runs on the scratch contents
the first one left behind, and against the fp64 oracle on whole heads; a
shape whose workspace fills the scratch exactly is accepted, one a key block
larger is refused.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from parity import TOL_GRAD as TOL_GRAD_ORACLE, rel_l2

from exact_tiled_attention_22_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL_GRAD = 1e-2  # relative L2, the gradient tolerance of the parity tests


@pytest.fixture(scope="module")
def A():
    from exact_tiled_attention_22_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from exact_tiled_attention_22_gb300 import attn
    return attn


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


def _case(A, B, N, H, d, dtype, causal, seed):
    dev = torch.device("cuda:0")
    x = make_inputs(B, N, H, d, dtype, seed=seed)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    o, lse = A.fwd(q, k, v, scale, causal)
    ref = A.bwd(q, k, v, o, lse, do, scale, causal)  # attn_bwd, caller workspace
    return (q, k, v, o, lse, do, scale), ref


def _noalloc(A, args, B, N, H, d, dtype, causal):
    q, k, v, o, lse, do, scale = args
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = A.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, dtype)
    assert rc == A.ATTN_OK, A.last_error()
    return dq, dk, dv


def test_noalloc_matches_attn_bwd_on_consecutive_calls(A):
    shapes = [(2, 333, 3, 128, "bf16", True), (1, 200, 2, 64, "fp16", False)]
    for B, N, H, d, dtype, causal in shapes:
        args, ref = _case(A, B, N, H, d, dtype, causal, seed=N)
        for call in range(2):
            got = _noalloc(A, args, B, N, H, d, dtype, causal)
            assert A.attn_status() == A.ATTN_OK
            for name, g, r in zip(("dq", "dk", "dv"), got, ref):
                err = _rel(g, r)
                assert err <= TOL_GRAD, f"{name} call {call}: rel L2 {err:.2e}"
            # dK and dV do not use atomics: identical to attn_bwd bit for bit
            assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def test_noalloc_rejects_shapes_beyond_its_scratch(A):
    B, H, N, d = 4, 16, 2048, 128
    assert A.attn_bwd_workspace_size(B, H, N, d) > A.NOALLOC_WORKSPACE_BYTES
    dev = torch.device("cuda:0")
    t = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    outs = [torch.zeros(16, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    rc = A.attn_bwd_noalloc(t, t, t, t, t, t, outs[0], outs[1], outs[2], B, H, N, d, 0.1, 1,
                            "bf16")
    assert rc == A.ATTN_ERR_WORKSPACE
    assert "scratch" in A.last_error()


def test_noalloc_matches_oracle(A, oracle):
    """One call per shape, every head of dQ, dK, dV against the fp64 oracle."""
    for B, N, H, d, dtype, causal in [(1, 300, 2, 128, "bf16", True), (2, 129, 1, 64, "fp16", False)]:
        args, _ = _case(A, B, N, H, d, dtype, causal, seed=7 * N)
        got = _noalloc(A, args, B, N, H, d, dtype, causal)
        assert A.attn_status() == A.ATTN_OK
        q, k, v, _, _, do, scale = args
        f64 = [t.double().cpu().numpy() for t in (q, k, v, do)]
        g = [t.double().cpu().numpy() for t in got]
        for b in range(B):
            for h in range(H):
                head = [np.ascontiguousarray(a[b, :, h, :]) for a in f64]
                ref = oracle.bwd_head(*head, scale, causal)[:3]
                for name, gg, rr in zip(("dq", "dk", "dv"), g, ref):
                    err = rel_l2(gg[b, :, h, :], rr)
                    assert err <= TOL_GRAD_ORACLE, f"{name} (b={b}, h={h}): rel L2 {err:.2e}"


def test_noalloc_accepts_the_largest_shape_and_refuses_one_block_more(A):
    """B*H*Npad = 64512 rows at d = 128 fill the scratch (the largest
    multiple of 128 that fits); 64640 rows do not."""
    B, H, N, d = 1, 63, 1024, 128
    assert A.attn_bwd_workspace_size(B, H, N, d) <= A.NOALLOC_WORKSPACE_BYTES
    assert A.attn_bwd_workspace_size(1, 64, 1024, d) > A.NOALLOC_WORKSPACE_BYTES
    args, ref = _case(A, B, N, H, d, "bf16", True, seed=11)
    for call in range(2):
        got = _noalloc(A, args, B, N, H, d, "bf16", True)
        assert A.attn_status() == A.ATTN_OK
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            err = _rel(g, r)
            assert err <= TOL_GRAD, f"{name} call {call}: rel L2 {err:.2e}"
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    Bx, Hx, Nx = 1, 505, 128  # 64640 rows: one 128-row block over
    assert A.attn_bwd_workspace_size(Bx, Hx, Nx, d) > A.NOALLOC_WORKSPACE_BYTES
    dev = torch.device("cuda:0")
    t = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    outs = [torch.zeros(16, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    rc = A.attn_bwd_noalloc(t, t, t, t, t, t, outs[0], outs[1], outs[2], Bx, Hx, Nx, d, 0.1, 1,
                            "bf16")
    assert rc == A.ATTN_ERR_WORKSPACE

