"""GPU parity: the library (through its C ABI) against the fp64 oracle on
seeded inputs, element by element.

Small shapes are compared on every head and element; they span several
128-row tiles and ragged tails.  The five measured workloads run in the same
launch configuration the benchmark times; the two largest are compared on
sampled heads (and, for the very long one, sampled rows and keys), which the
oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from exact_tiled_attention_22_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from parity import TOL_LSE, TOL_O, assert_within, compare_head, default_scale, o_error, run_gpu

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


def _x64(x):
    return {n: t.double().numpy() for n, t in x.items()}


SHAPES = [
    # (B, N, H, d, dtype, causal)
    (1, 1, 1, 64, "fp16", False),
    (1, 1, 1, 128, "bf16", True),
    (1, 77, 2, 64, "fp16", True),
    (1, 77, 2, 128, "bf16", False),
    (2, 128, 1, 128, "bf16", True),
    (1, 129, 1, 64, "bf16", True),
    (1, 255, 2, 128, "fp16", True),
    (1, 256, 1, 64, "fp16", False),
    (1, 257, 3, 128, "bf16", True),
    (2, 384, 2, 64, "bf16", False),
    (1, 640, 2, 128, "fp16", False),
    (1, 1000, 2, 128, "bf16", True),
    (1, 1000, 2, 64, "fp16", True),
]


@pytest.mark.parametrize("B,N,H,d,dtype,causal", SHAPES,
                         ids=[f"B{s[0]}N{s[1]}H{s[2]}d{s[3]}{s[4]}{'c' if s[5] else 'n'}"
                              for s in SHAPES])
def test_edge_shapes_all_heads(oracle, B, N, H, d, dtype, causal):
    scale = default_scale(d)
    x = make_inputs(B, N, H, d, dtype, seed=31 + N + d)
    g = run_gpu(x, scale, causal, dtype)
    x64 = _x64(x)
    for b in range(B):
        for h in range(H):
            err = compare_head(oracle, x64, g, b, h, scale, causal, dtype)
            assert_within(err, dtype, f"b={b} h={h}")


def test_workload_tiny(oracle):
    w = WORKLOADS["tiny"]
    x = workload_inputs(w)
    g = run_gpu(x, w.scale, w.causal, w.dtype)
    assert_within(compare_head(oracle, _x64(x), g, 0, 0, w.scale, w.causal, w.dtype), w.dtype)


def test_workload_encoder(oracle):
    w = WORKLOADS["encoder"]
    x = workload_inputs(w)
    g = run_gpu(x, w.scale, w.causal, w.dtype)
    x64 = _x64(x)
    for b in range(w.B):
        for h in range(w.H):
            assert_within(compare_head(oracle, x64, g, b, h, w.scale, w.causal, w.dtype),
                          w.dtype, f"b={b} h={h}")


def test_workload_gpt(oracle):
    w = WORKLOADS["gpt"]
    x = workload_inputs(w)
    g = run_gpu(x, w.scale, w.causal, w.dtype)
    x64 = _x64(x)
    for (b, h) in [(0, 0), (1, 7), (2, 11), (3, 15)]:
        assert_within(compare_head(oracle, x64, g, b, h, w.scale, w.causal, w.dtype),
                      w.dtype, f"b={b} h={h}")


def test_workload_long(oracle):
    w = WORKLOADS["long"]
    x = workload_inputs(w)
    g = run_gpu(x, w.scale, w.causal, w.dtype)
    x64 = {n: t[:, :, :, :] for n, t in _x64(x).items()}
    for (b, h) in [(0, 0), (1, 15)]:
        assert_within(compare_head(oracle, x64, g, b, h, w.scale, w.causal, w.dtype),
                      w.dtype, f"b={b} h={h}")


def test_workload_very_long_sampled(oracle):
    w = WORKLOADS["very_long"]
    x = workload_inputs(w)
    g = run_gpu(x, w.scale, w.causal, w.dtype)
    rng = np.random.default_rng(5)
    N = w.N
    rows = sorted(set([0, 1, 127, 128, N - 129, N - 128, N - 1]
                      + list(rng.choice(N, 120, replace=False))))
    keys = sorted(set([0, 1, 127, 128, N // 2, N - 129, N - 1]
                      + list(rng.choice(N, 60, replace=False))))
    for (b, h) in [(0, 0), (0, 31)]:
        x64 = {n: t[b:b + 1, :, h:h + 1, :].double().numpy() for n, t in x.items()}
        gh = {n: (a[b:b + 1, :, h:h + 1, :] if a.ndim == 4 else a[b:b + 1, h:h + 1, :])
              for n, a in g.items()}
        err = compare_head(oracle, x64, gh, 0, 0, w.scale, w.causal, w.dtype, rows=rows,
                           keys=keys, check_bwd=True)
        assert_within(err, w.dtype, f"b={b} h={h}")


def test_forward_is_deterministic():
    x = make_inputs(1, 1000, 2, 128, "bf16", seed=3)
    a = run_gpu(x, 0.1, True, "bf16", bwd=False)
    b = run_gpu(x, 0.1, True, "bf16", bwd=False)
    assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["lse"], b["lse"])


def test_outputs_stay_in_bounds():
    """Canary words around every output: no write lands outside its tensor."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d = 1, 333, 2, 128
    x = make_inputs(B, N, H, d, "bf16", seed=9)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    pad = 4096

    def padded(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), 7, dtype=dtype, device=dev)
        return buf, buf[pad:pad + n].view(*shape)

    ob, o = padded((B, N, H, d), torch.bfloat16)
    lb, lse = padded((B, H, N), torch.float32)
    attn.check(attn.attn_fwd(q, k, v, o, lse, B, H, N, d, 0.09, 1, "bf16"))
    bufs = [padded((B, N, H, d), torch.bfloat16) for _ in range(3)]
    ws = attn.workspace(B, H, N, d, dev)
    attn.check(attn.attn_bwd(q, k, v, o, lse, do, bufs[0][1], bufs[1][1], bufs[2][1], B, H, N, d,
                             0.09, 1, "bf16", ws, ws.numel()))
    attn.check(attn.attn_status())
    for buf, _ in [(ob, o), (lb, lse)] + bufs:
        assert torch.all(buf[:pad] == 7) and torch.all(buf[-pad:] == 7)


def test_side_stream():
    s = torch.cuda.Stream()
    x = make_inputs(1, 300, 1, 64, "fp16", seed=12)
    with torch.cuda.stream(s):
        g = run_gpu(x, 0.125, False, "fp16", stream=s)
    h = run_gpu(x, 0.125, False, "fp16")
    assert np.array_equal(g["o"], h["o"])


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "fp16")])
def test_backward_wide_index_form_equals_narrow(d, dtype):
    """The preprocess and dQ conversion kernels' 64-bit row splits (the form
    they take when B H N reaches 2^31, forced here by debug flag bit 3) give
    the results of the 32-bit form bit for bit: with one key block (N <= 128)
    every dQ tile gets a single contribution, so dQ, dK, dV and the
    workspace's D and -LSE log2 e rows are deterministic."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H = 3, 100, 5
    x = make_inputs(B, N, H, d, dtype, seed=77 + d)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o, lse = attn.fwd(q, k, v, scale, True)
    outs = []
    for flags in (0, 8):
        attn.attn_set_wait_limit(0, flags)
        try:
            ws = attn.workspace(B, H, N, d, dev)
            dq, dk, dv = attn.bwd(q, k, v, o, lse, do, scale, True, ws=ws)
            attn.check(attn.attn_status())
        finally:
            attn.attn_set_wait_limit(0, 0)
        npad = (N + 127) // 128 * 128
        head = ws[: 2 * B * H * npad * 4].clone()  # lse2 and D rows
        outs.append((dq, dk, dv, head))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)


def test_max_length_forward_sampled(oracle):
    """N = 131072 (grid of 512 query-tile pairs for one head, TMA row
    coordinates past 2^16), causal fp16 d=64: sampled rows of O and LSE
    against the oracle."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d, dtype = 1, 131072, 1, 64, "fp16"
    x = make_inputs(B, N, H, d, dtype, seed=77)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = attn.fwd(q, k, v, 0.125, True)
    attn.check(attn.attn_status())
    rows = np.sort(np.concatenate([[0, 1, 65535, 65536, N - 1],
                                   np.random.default_rng(78).choice(N, 25, replace=False)]))
    x64 = {n: t.double().numpy() for n, t in x.items()}
    qq, kk, vv = (np.ascontiguousarray(x64[n][0, :, 0, :]) for n in ("q", "k", "v"))
    o_ref, lse_ref = oracle.fwd_head(qq, kk, vv, 0.125, True, rows=rows)
    eo, _ = o_error(o.float().cpu().numpy()[0, rows, 0, :], o_ref, dtype)
    assert eo <= TOL_O[dtype]
    assert np.max(np.abs(lse.cpu().numpy()[0, 0, rows] - lse_ref)) <= TOL_LSE


def test_tensors_past_2_31_elements(oracle):
    """B=128 H=32 N=4096 d=128 bf16 causal: 2^31 elements per tensor (4 GB),
    element offsets past 2^31 in the last batches.  Inputs are drawn batch
    by batch (seed 9500 + b); two heads of the last batch and one of the
    first are checked against the oracle, forward and backward."""
    from exact_tiled_attention_22_gb300 import attn
    B, N, H, d, dtype = 128, 4096, 32, 128, "bf16"
    dev = torch.device("cuda:0")
    t = {n: torch.empty((B, N, H, d), dtype=torch.bfloat16, device=dev)
         for n in ("q", "k", "v", "do")}
    for b in range(B):
        xb = make_inputs(1, N, H, d, dtype, seed=9500 + b)
        for n in t:
            t[n][b].copy_(xb[n][0])
    scale = default_scale(d)
    o, lse = attn.fwd(t["q"], t["k"], t["v"], scale, True)
    dq, dk, dv = attn.bwd(t["q"], t["k"], t["v"], o, lse, t["do"], scale, True)
    attn.check(attn.attn_status())
    for b, h in ((0, 0), (B - 1, 0), (B - 1, H - 1)):
        xb = make_inputs(1, N, H, d, dtype, seed=9500 + b)
        x64 = {n: xb[n].double().numpy() for n in xb}
        g = {"o": o[b:b + 1, :, h:h + 1].float().cpu().numpy(),
             "lse": lse[b:b + 1, h:h + 1].cpu().numpy(),
             "dq": dq[b:b + 1, :, h:h + 1].float().cpu().numpy(),
             "dk": dk[b:b + 1, :, h:h + 1].float().cpu().numpy(),
             "dv": dv[b:b + 1, :, h:h + 1].float().cpu().numpy()}
        xh = {n: a[:, :, h:h + 1] for n, a in x64.items()}
        assert_within(compare_head(oracle, xh, g, 0, 0, scale, True, dtype), dtype, f"b={b} h={h}")
