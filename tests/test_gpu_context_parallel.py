"""Sequence (context) parallelism on one GB300: the accumulating kernels
(attn_fwd_acc, attn_bwd_acc, attn_cast_acc) against the plain ones, and
every rank of the zigzag ring (context_parallel.emulate_ring, world sizes
1-4: each rank's K/V blocks, merges and dK/dV accumulators in the ring's
order) against the fp64 oracle over the whole sequence, element by element,
with the library's usual tolerances."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_22_gb300 import context_parallel as cp
from exact_tiled_attention_22_gb300.inputs import make_inputs
from parity import TOL_GRAD, TOL_LSE, TOL_O, half_ulp, o_error, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from exact_tiled_attention_22_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from exact_tiled_attention_22_gb300 import attn
    attn.attn_set_wait_limit(0, 0)
    yield attn
    assert attn.attn_status() == 0


@pytest.mark.parametrize("B,N,H,d,dtype,causal", [
    (2, 333, 3, 128, "bf16", True), (1, 200, 2, 64, "fp16", False), (1, 1000, 2, 64, "bf16", True)])
def test_single_block_equals_plain_calls(A, B, N, H, d, dtype, causal):
    """One block that is both FIRST and LAST is the plain forward bit for
    bit (O and LSE), and its backward the plain backward (dK, dV bit for
    bit; dQ within the tolerance, its fp32 sum is order-dependent)."""
    x = make_inputs(B, N, H, d, dtype, seed=N + d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    o_ref, lse_ref = A.fwd(q, k, v, scale, causal)
    o = torch.empty_like(q)
    lse = torch.empty_like(lse_ref)
    A.check(A.attn_fwd_acc(q, k, v, None, lse, o, B, H, N, d, scale, causal, 3, dtype))
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    dq_ref, dk_ref, dv_ref = A.bwd(q, k, v, o_ref, lse_ref, do, scale, causal)
    dq = torch.empty_like(q)
    acc = torch.full((2,) + tuple(q.shape), float("nan"), dtype=torch.float32, device="cuda")
    ws = A.workspace(B, H, N, d, q.device)
    A.check(A.attn_bwd_acc(q, k, v, o_ref, lse_ref, do, dq, acc[0], acc[1], B, H, N, d, scale, causal,
                           3, 1, dtype, ws, ws.numel()))
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    A.check(A.attn_cast_acc(acc[0], dk, dk.numel(), 1.0, dtype))
    A.check(A.attn_cast_acc(acc[1], dv, dv.numel(), 1.0, dtype))
    A.check(A.attn_status())
    assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)
    assert rel_l2(dq.double().cpu().numpy(), dq_ref.double().cpu().numpy()) < 1e-3


def _oracle_full(oracle, x, scale, causal):
    f64 = {n: x[n].double().numpy() for n in x}
    B, N, H, d = f64["q"].shape
    out = {"o": np.zeros((B, N, H, d)), "lse": np.zeros((B, H, N)), "dq": np.zeros((B, N, H, d)),
           "dk": np.zeros((B, N, H, d)), "dv": np.zeros((B, N, H, d))}
    for b in range(B):
        for h in range(H):
            hd = [np.ascontiguousarray(f64[n][b, :, h]) for n in ("q", "k", "v", "do")]
            out["o"][b, :, h], out["lse"][b, h] = oracle.fwd_head(*hd[:3], scale, causal)
            out["dq"][b, :, h], out["dk"][b, :, h], out["dv"][b, :, h], _ = oracle.bwd_head(*hd, scale, causal)
    return out


@pytest.mark.parametrize("world,B,C,H,d,dtype,causal", [
    (1, 2, 200, 2, 128, "bf16", True),
    (2, 1, 200, 3, 128, "bf16", True),
    (3, 1, 130, 2, 64, "fp16", True),
    (4, 1, 128, 2, 128, "bf16", True),
    (2, 2, 100, 2, 64, "fp16", False),
    (3, 1, 256, 1, 128, "bf16", False),
])
def test_ring_equals_oracle(A, oracle, world, B, C, H, d, dtype, causal):
    N = 2 * world * C
    x = make_inputs(B, N, H, d, dtype, seed=world * 1000 + C)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    got = cp.emulate_ring(q, k, v, do, world, cp.GpuOps(scale), causal)
    A.check(A.attn_status())
    torch.cuda.synchronize()
    g = dict(zip(("o", "lse", "dq", "dk", "dv"), (t.float().cpu().numpy() for t in got)))
    ref = _oracle_full(oracle, x, scale, causal)
    for b in range(B):
        for h in range(H):
            e_o, e_abs = o_error(g["o"][b, :, h], ref["o"][b, :, h], dtype)
            assert e_o <= TOL_O[dtype], f"O (b={b}, h={h}) {e_o:.2e} beyond rounding (max abs {e_abs:.2e})"
            e_l = float(np.max(np.abs(g["lse"][b, h] - ref["lse"][b, h])))
            assert e_l <= TOL_LSE, f"LSE (b={b}, h={h}) {e_l:.2e}"
            for name in ("dq", "dk", "dv"):
                e = rel_l2(g[name][b, :, h], ref[name][b, :, h])
                assert e <= TOL_GRAD, f"{name} (b={b}, h={h}) rel L2 {e:.2e}"


def test_ring_equals_single_device_attention_at_8k(A):
    """A longer sequence over 4 ranks: the ring's results equal the plain
    kernels over the whole sequence (same tolerances, O and LSE against
    attn_fwd, gradients against attn_bwd)."""
    B, N, H, d, world = 1, 8192, 4, 128, 4
    x = make_inputs(B, N, H, d, "bf16", seed=77)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    o_ref, lse_ref = A.fwd(q, k, v, scale, True)
    dq_ref, dk_ref, dv_ref = A.bwd(q, k, v, o_ref, lse_ref, do, scale, True)
    o, lse, dq, dk, dv = cp.emulate_ring(q, k, v, do, world, cp.GpuOps(scale), True)
    A.check(A.attn_status())
    assert float((lse - lse_ref).abs().max()) <= TOL_LSE
    # two rounded outputs of the same exact O: apart by at most both
    # roundings plus both errors
    on, rn = o.double().cpu().numpy(), o_ref.double().cpu().numpy()
    assert float(np.max(np.abs(on - rn) - 2 * half_ulp(rn, "bf16"))) <= 2 * TOL_O["bf16"]
    for name, a, r in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        e = rel_l2(a.double().cpu().numpy(), r.double().cpu().numpy())
        assert e <= TOL_GRAD, f"{name} rel L2 {e:.2e}"
