"""Shared helpers for the GPU parity tests: run the library through its C ABI
on seeded inputs and compare with the fp64 oracle.

Tolerances (fixed for this library): O max-abs error <= 2e-3 for fp16 and
<= 1e-2 for bf16, counted beyond the output's own rounding: for every element
|O_gpu - O_ref| - ulp(O_ref)/2 <= tol, where ulp is that of the output type
at O_ref.  (O is returned in fp16/bf16; for |O| >= 4 the bf16 half-ulp alone is
0.0156, so a plain max-abs bound of 1e-2 is out of reach for any bf16 output;
the plain max-abs error is reported alongside.)  LSE max-abs error <= 1e-3
(natural-log units); dQ, dK, dV relative L2 error ||g - g_ref|| / ||g_ref||
<= 1e-2 per tensor.
"""
from __future__ import annotations

import math

import numpy as np
import torch

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}
TOL_LSE = 1e-3
TOL_GRAD = 1e-2


MANTISSA_BITS = {"fp16": 10, "bf16": 7}


def half_ulp(x, dtype):
    """Half the spacing of the 16-bit output type at |x| (normal range;
    the fp16 subnormal spacing 2^-24 below 2^-14)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    m = MANTISSA_BITS[dtype]
    e = np.floor(np.log2(np.maximum(a, 1e-300)))
    if dtype == "fp16":
        e = np.maximum(e, -14)
    else:
        e = np.maximum(e, -126)
    return 0.5 * np.exp2(e - m)


def o_error(o_gpu, o_ref, dtype):
    """(error beyond the output rounding, plain max-abs error)."""
    d = np.abs(o_gpu - o_ref)
    return float(np.max(d - half_ulp(o_ref, dtype))), float(np.max(d))


def run_gpu(x, scale, causal, dtype, bwd=True, stream=None):
    from exact_tiled_attention_22_gb300 import attn
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.fwd(q, k, v, scale, causal, stream=stream)
    out = {"o": o, "lse": lse}
    if bwd:
        dq, dk, dv = attn.bwd(q, k, v, o, lse, do, scale, causal, stream=stream)
        out.update(dq=dq, dk=dk, dv=dv)
    attn.check(attn.attn_status(stream))
    torch.cuda.synchronize()
    return {k_: t.float().cpu().numpy() for k_, t in out.items()}


def rel_l2(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def compare_head(orc, x64, g, b, h, scale, causal, dtype, rows=None, keys=None,
                 check_bwd=True):
    """Compares GPU outputs of head (b, h) with the oracle; returns errors."""
    head = lambda a: np.ascontiguousarray(a[b, :, h, :])  # noqa: E731
    q, k, v, do = (head(x64[n]) for n in ("q", "k", "v", "do"))
    N = q.shape[0]
    sel = slice(None) if rows is None else rows
    o_ref, lse_ref = orc.fwd_head(q, k, v, scale, causal, rows=rows)
    o_beyond, o_abs = o_error(g["o"][b, :, h, :][sel], o_ref, dtype)
    err = {
        "o": o_beyond,
        "o_maxabs": o_abs,
        "lse": float(np.max(np.abs(g["lse"][b, h, :][sel] - lse_ref))),
    }
    if check_bwd and "dq" in g:
        urows = None if rows is None else sorted(set(int(r) for r in rows))
        ukeys = None if keys is None else sorted(set(int(r) for r in keys))
        dq_ref, dk_ref, dv_ref, _ = orc.bwd_head(q, k, v, do, scale, causal, rows=urows,
                                                 keys=ukeys)
        rs = slice(None) if urows is None else urows
        ks = slice(None) if ukeys is None else ukeys
        err["dq"] = rel_l2(g["dq"][b, :, h, :][rs], dq_ref)
        err["dk"] = rel_l2(g["dk"][b, :, h, :][ks], dk_ref)
        err["dv"] = rel_l2(g["dv"][b, :, h, :][ks], dv_ref)
    assert N == g["o"].shape[1]
    return err


def assert_within(err, dtype, what=""):
    assert err["o"] <= TOL_O[dtype], (f"{what} O error beyond output rounding {err['o']:.3e} "
                                      f"(max abs {err['o_maxabs']:.3e})")
    assert err["lse"] <= TOL_LSE, f"{what} LSE max abs {err['lse']:.3e}"
    for g in ("dq", "dk", "dv"):
        if g in err:
            assert err[g] <= TOL_GRAD, f"{what} {g} rel L2 {err[g]:.3e}"


def default_scale(d):
    return 1.0 / math.sqrt(d)
