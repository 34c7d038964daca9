"""The C ABI library: it builds, loads, exports every entry point that
include/attn.h declares, and rejects bad arguments on the host before any
device work (these checks need no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def A():
    from exact_tiled_attention_22_gb300 import build
    build.build()
    from exact_tiled_attention_22_gb300 import attn
    return attn


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(attn_[a-z0-9_]+)\s*\(", text):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_status"):
        assert must in names


def test_library_exports_every_declared_symbol(A):
    lib = ctypes.CDLL(A.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_library_is_sm103a_only():
    from exact_tiled_attention_22_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


# Fake, 16-byte aligned addresses: every case below fails validation before
# the library touches the device, so nothing is dereferenced.
P = [0x10000 * (i + 1) for i in range(12)]
BIG = 1 << 40


def fwd(A, **kw):
    args = dict(q=P[0], k=P[1], v=P[2], o=P[3], lse=P[4], B=1, H=1, N=128, d=64,
                scale=0.125, causal=0, dtype=A.ATTN_F16)
    args.update(kw)
    return A.lib.attn_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                          args["H"], args["N"], args["d"], args["scale"], args["causal"],
                          args["dtype"], None)


def bwd(A, ws_bytes=None, **kw):
    args = dict(q=P[0], k=P[1], v=P[2], o=P[3], lse=P[4], dO=P[5], dq=P[6], dk=P[7], dv=P[8],
                B=1, H=1, N=128, d=64, scale=0.125, causal=0, dtype=A.ATTN_F16, ws=BIG)
    args.update(kw)
    need = A.attn_bwd_workspace_size(args["B"], args["H"], args["N"], args["d"])
    return A.lib.attn_bwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["dO"],
                          args["dq"], args["dk"], args["dv"], args["B"], args["H"], args["N"],
                          args["d"], args["scale"], args["causal"], args["dtype"], args["ws"],
                          need if ws_bytes is None else ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(lse=None), -1), (dict(B=0), -1), (dict(H=-1), -1),
    (dict(N=0), -1), (dict(d=96), -2), (dict(d=256), -2), (dict(dtype=7), -2),
    (dict(scale=0.0), -1), (dict(scale=float("nan")), -1), (dict(scale=float("inf")), -1),
    (dict(q=P[0] + 8), -3), (dict(lse=P[4] + 4), -3),
    (dict(o=P[0]), -1),                      # output aliases an input
    (dict(lse=P[3] + 64), -1),               # lse overlaps o
    (dict(B=1 << 15, H=1 << 10, N=1 << 10, d=64), -1),  # size overflow
])
def test_fwd_rejects_bad_arguments(A, kw, code):
    assert fwd(A, **kw) == code
    assert A.last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(dO=None), -1), (dict(dv=None), -1), (dict(d=32), -2), (dict(dk=P[7] + 2), -3),
    (dict(ws=None), -6), (dict(ws=BIG + 128), -3), (dict(dq=P[1]), -1),
    (dict(dk=P[6]), -1), (dict(ws=P[2]), -1),
])
def test_bwd_rejects_bad_arguments(A, kw, code):
    assert bwd(A, **kw) == code


def test_bwd_rejects_small_workspace(A):
    need = A.attn_bwd_workspace_size(1, 1, 128, 64)
    assert bwd(A, ws_bytes=need - 1) == -6


def test_workspace_is_linear_in_n(A):
    """The backward keeps O(N) state per head, never an N x N matrix."""
    for d in (64, 128):
        sizes = [A.attn_bwd_workspace_size(2, 3, n, d) for n in (128, 256, 1024, 8192)]
        per_row = [s / n for s, n in zip(sizes, (128, 256, 1024, 8192))]
        assert max(per_row) - min(per_row) <= 256 * 3 / 128 + 1e-9
        assert per_row[-1] <= 2 * 3 * (d + 2) * 4 + 1
    assert A.attn_bwd_workspace_size(1, 1, 1, 64) > 0
    assert A.attn_bwd_workspace_size(0, 1, 1, 64) == 0
    assert A.attn_bwd_workspace_size(1, 1, 1, 80) == 0


def test_valid_call_without_gpu_fails_cleanly(A):
    """Valid arguments reach the device query; with no usable sm_103 device
    the call returns an error code (never a fallback result)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(A) in (-2, -4)


def dec(A, ws_bytes=None, **kw):
    args = dict(q=P[0], k=P[1], v=P[2], o=P[3], lse=P[4], B=1, H=2, Nq=4, Nk=1000, d=128,
                scale=0.125, causal=1, dtype=A.ATTN_BF16, ws=BIG)
    args.update(kw)
    need = A.attn_decode_workspace_size(args["B"], args["H"], args["Nq"], args["Nk"], args["d"])
    return A.lib.attn_decode(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                             args["H"], args["Nq"], args["Nk"], args["d"], args["scale"],
                             args["causal"], args["dtype"], args["ws"],
                             need if ws_bytes is None else ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(Nq=0), -1), (dict(Nk=0), -1), (dict(Nq=129), -2),
    (dict(Nq=8, Nk=4, causal=1), -1),        # causal needs Nq <= Nk
    (dict(d=80), -2), (dict(dtype=5), -2), (dict(scale=-1.0), -1),
    (dict(k=P[1] + 4), -3), (dict(ws=None), -6), (dict(ws=BIG + 64), -3),
    (dict(o=P[1]), -1),                      # output overlaps the key cache
    (dict(ws=P[0]), -1),                     # workspace overlaps q
])
def test_decode_rejects_bad_arguments(A, kw, code):
    assert dec(A, **kw) == code
    assert A.last_error()


def test_decode_rejects_small_workspace(A):
    need = A.attn_decode_workspace_size(1, 2, 4, 1000, 128)
    assert dec(A, ws_bytes=need - 1) == -6


def test_decode_workspace_is_bounded(A):
    """Chunk partials only: O(Nq) per chunk, at most 64 chunks per head, so the
    workspace does not grow with the cache length once the chunks are long."""
    s1 = A.attn_decode_workspace_size(1, 1, 16, 1 << 16, 128)
    s2 = A.attn_decode_workspace_size(1, 1, 16, 1 << 20, 128)
    assert s1 == s2 and 0 < s1 <= 64 * 16 * (128 + 2) * 4 + 512
    assert A.attn_decode_workspace_size(1, 1, 1, 1, 64) > 0
    assert A.attn_decode_workspace_size(1, 1, 0, 1, 64) == 0
    assert A.attn_decode_workspace_size(1, 1, 1, 1, 96) == 0


def test_alibi_slopes_alignment_checked(A):
    args = (P[0], P[1], P[2], P[3], P[4], 1, 2, 128, 64, 0.125, 1, P[5] + 2, A.ATTN_BF16, None)
    assert A.lib.attn_fwd_alibi(*args) == -3
    assert A.last_error()


def test_block_mask_length_checked(A):
    """The block-sparse kernels take N <= 65536 (512 blocks of 128 rows);
    a longer sequence with a mask is refused on the host."""
    def call(N, mask):
        return A.lib.attn_fwd_sparse(P[0], P[1], P[2], P[3], P[4], 1, 1, N, 64, 0.125, 1, None,
                                     mask, A.ATTN_BF16, None)
    assert call(65537, P[9]) == -1
    assert "block_mask" in A.last_error()
    # at the limit the mask is accepted and the (overlapping) fake buffers are refused next
    assert call(65536, P[9]) == -1
    assert "block_mask" not in A.last_error()
    assert call(65537, None) == -1
    assert "block_mask" not in A.last_error()


@pytest.mark.parametrize("which", ["o", "lse"])
@pytest.mark.parametrize("operand", ["alibi", "mask"])
def test_outputs_must_not_overlap_slopes_or_mask(A, which, operand):
    """An output that overlaps the ALiBi slopes or the block mask (inputs
    the kernels read while they write) is refused, in both passes."""
    al = P[9] if operand == "alibi" else None
    bm = P[9] if operand == "mask" else None
    o, lse = (P[9], P[4]) if which == "o" else (P[3], P[9])
    rc = A.lib.attn_fwd_ex(P[0], P[1], P[2], o, lse, 1, 2, 128, 64, 0.125, 1, al, bm, 0.0, 1, 0,
                           A.ATTN_BF16, None)
    assert rc == -1 and "overlaps" in A.last_error()
    if which == "o":  # dQ over the slopes or the mask
        need = A.attn_bwd_workspace_size(1, 2, 128, 64)
        rc = A.lib.attn_bwd_ex(P[0], P[1], P[2], P[3], P[4], P[5], P[9], P[7], P[8], 1, 2, 128, 64,
                               0.125, 1, al, bm, 0.0, 1, 0, A.ATTN_BF16, BIG, need, None)
        assert rc == -1 and "overlaps" in A.last_error()


@pytest.mark.parametrize("p", [-0.1, 1.0, 0.999, float("nan")])
def test_dropout_probability_checked(A, p):
    """dropout_p outside [0, 1), or so close to 1 that no score would be
    kept, is refused on the host."""
    rc = A.lib.attn_fwd_ex(P[0], P[1], P[2], P[3], P[4], 1, 2, 128, 64, 0.125, 1, None, None, p, 1,
                           0, A.ATTN_BF16, None)
    assert rc == -1 and "dropout_p" in A.last_error()


def test_size_limits(A):
    """Tensors past 2^31 elements are accepted (64-bit offsets in every
    kernel); what must stay below 2^31 is the grid: B*H*ceil(N/128)."""
    assert fwd(A, B=1 << 14, H=1 << 10, N=1 << 14, d=64) == -1   # 2^31 blocks
    assert "blocks" in A.last_error()
    # 2^31 elements exactly: passes the size checks, then the (fake,
    # overlapping) buffers are refused
    assert fwd(A, B=128, H=32, N=4096, d=128) == -1
    assert "too large" not in A.last_error() and "blocks" not in A.last_error()


def fwd_acc(A, **kw):
    args = dict(q=P[0], k=P[1], v=P[2], o_acc=P[3], lse=P[4], o=P[5], B=1, H=1, N=128, d=64,
                scale=0.125, causal=1, flags=0, dtype=A.ATTN_BF16)
    args.update(kw)
    return A.lib.attn_fwd_acc(args["q"], args["k"], args["v"], args["o_acc"], args["lse"], args["o"],
                              args["B"], args["H"], args["N"], args["d"], args["scale"], args["causal"],
                              args["flags"], args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(flags=4), -1), (dict(flags=-1), -1),
    (dict(o_acc=None), -1),                   # needed unless FIRST and LAST
    (dict(o=None, flags=2), -1),              # LAST writes o
    (dict(o_acc=P[0]), -1),                   # accumulator over q
    (dict(lse=P[3] + 16), -1),                # lse inside the fp32 accumulator
    (dict(o_acc=P[3] + 8), -3), (dict(d=80), -2), (dict(N=0), -1),
])
def test_fwd_acc_rejects_bad_arguments(A, kw, code):
    assert fwd_acc(A, **kw) == code
    assert A.last_error()


def test_fwd_acc_optional_pointers(A):
    """o_acc may be omitted when one call is both FIRST and LAST, o when the
    call is not LAST; such calls pass every host check (then fail only for
    want of an sm_103 device, or refuse the fake overlapping buffers)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd_acc(A, o_acc=None, flags=3) in (-2, -4)
    assert fwd_acc(A, o=None, flags=1) in (-2, -4)


def bwd_acc(A, **kw):
    args = dict(q=P[0], k=P[1], v=P[2], o=P[3], lse=P[4], dO=P[5], dq=P[6], dk_acc=P[7],
                dv_acc=P[8], B=1, H=1, N=128, d=64, scale=0.125, causal=1, dq_flags=3, kv_flags=1,
                dtype=A.ATTN_BF16, ws=BIG)
    args.update(kw)
    need = A.attn_bwd_workspace_size(args["B"], args["H"], args["N"], args["d"])
    return A.lib.attn_bwd_acc(args["q"], args["k"], args["v"], args["o"], args["lse"], args["dO"],
                              args["dq"], args["dk_acc"], args["dv_acc"], args["B"], args["H"],
                              args["N"], args["d"], args["scale"], args["causal"], args["dq_flags"],
                              args["kv_flags"], args["dtype"], args["ws"], need, None)


@pytest.mark.parametrize("kw,code", [
    (dict(dq_flags=4), -1), (dict(kv_flags=2), -1), (dict(kv_flags=-1), -1),
    (dict(dq=None), -1),                      # LAST writes dq
    (dict(dk_acc=None), -1), (dict(dv_acc=None), -1),
    (dict(dv_acc=P[7] + 16), -1),             # the two accumulators overlap
    (dict(dk_acc=P[7] + 4), -3), (dict(ws=None), -6),
])
def test_bwd_acc_rejects_bad_arguments(A, kw, code):
    assert bwd_acc(A, **kw) == code
    assert A.last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(n=12), -1), (dict(n=0), -1), (dict(acc=None), -1), (dict(dtype=3), -2),
    (dict(acc=P[0] + 4), -3), (dict(out=P[0] + 32), -1),
])
def test_cast_acc_rejects_bad_arguments(A, kw, code):
    args = dict(acc=P[0], out=P[1], n=1024, mul=1.0, dtype=A.ATTN_BF16)
    args.update(kw)
    assert A.lib.attn_cast_acc(args["acc"], args["out"], args["n"], args["mul"], args["dtype"],
                               None) == code
    assert A.last_error()
