"""ctypes binding of libattn.so (include/attn.h), with the same entry-point
names, plus allocating conveniences ``fwd`` / ``bwd``.

Only argument marshalling happens here: every step of the computation runs
in the library's CUDA kernels.  PyTorch supplies device memory and streams.
Loading fails loudly if the library has not been built; there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn.so")

ATTN_F16, ATTN_BF16 = 0, 1
ATTN_OK = 0
ATTN_ERR_INVALID = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_ALIGN = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_TIMEOUT = -5
ATTN_ERR_WORKSPACE = -6
ERROR_NAMES = {0: "ATTN_OK", -1: "ATTN_ERR_INVALID", -2: "ATTN_ERR_UNSUPPORTED",
               -3: "ATTN_ERR_ALIGN", -4: "ATTN_ERR_CUDA", -5: "ATTN_ERR_TIMEOUT",
               -6: "ATTN_ERR_WORKSPACE"}

# Kernel ids of attn_profile_end.
KERNEL_NAMES = ["attn_fwd", "attn_bwd_pre", "attn_bwd_main", "attn_dq_post",
                "attn_decode_split", "attn_decode_merge"]


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run exact_tiled_attention_22_gb300.build.build() "
            "(needs nvcc).  There is no fallback implementation.")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.attn_fwd.restype = i
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.attn_bwd_workspace_size.restype = sz
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.attn_bwd_noalloc.restype = i
    lib.attn_fwd_alibi.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp]
    lib.attn_fwd_alibi.restype = i
    lib.attn_bwd_alibi.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp, sz, vp]
    lib.attn_bwd_alibi.restype = i
    lib.attn_decode_alibi.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, sz, vp]
    lib.attn_decode_alibi.restype = i
    lib.attn_fwd_sparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i, vp]
    lib.attn_fwd_sparse.restype = i
    lib.attn_bwd_sparse.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i,
                                    vp, sz, vp]
    lib.attn_bwd_sparse.restype = i
    u64, u32 = ctypes.c_uint64, ctypes.c_uint32
    lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, f, u64, u32, i, vp]
    lib.attn_fwd_ex.restype = i
    lib.attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, f, u64,
                                u32, i, vp, sz, vp]
    lib.attn_bwd_ex.restype = i
    lib.attn_decode_workspace_size.argtypes = [i, i, i, i, i]
    lib.attn_decode_workspace_size.restype = sz
    lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    lib.attn_decode.restype = i
    lib.attn_status.argtypes = [vp]
    lib.attn_status.restype = i
    lib.attn_last_error_string.argtypes = []
    lib.attn_last_error_string.restype = ctypes.c_char_p
    lib.attn_set_wait_limit.argtypes = [ctypes.c_ulonglong, i]
    lib.attn_set_wait_limit.restype = i
    lib.attn_profile_begin.argtypes = []
    lib.attn_profile_begin.restype = i
    lib.attn_profile_end.argtypes = [ctypes.POINTER(i), ctypes.POINTER(ctypes.c_double), i]
    lib.attn_profile_end.restype = i
    lib.attn_fwd_acc.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp]
    lib.attn_fwd_acc.restype = i
    lib.attn_bwd_acc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, i, vp,
                                 sz, vp]
    lib.attn_bwd_acc.restype = i
    lib.attn_cast_acc.argtypes = [vp, vp, sz, f, i, vp]
    lib.attn_cast_acc.restype = i
    lib.attn_philox4x32_10.argtypes = [vp, vp, i, vp]
    lib.attn_philox4x32_10.restype = i
    return lib


lib = _load()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(dt) -> int:
    if dt in (torch.bfloat16, "bf16", ATTN_BF16):
        return ATTN_BF16
    if dt in (torch.float16, "fp16", ATTN_F16):
        return ATTN_F16
    raise ValueError(f"unsupported dtype {dt}")


def last_error() -> str:
    return (lib.attn_last_error_string() or b"").decode()


def attn_philox4x32_10(inp, out, n: int, stream=None) -> int:
    """Device uint32 [n, 6] (counter words, key words) -> [n, 4] outputs."""
    return lib.attn_philox4x32_10(_ptr(inp), _ptr(out), n, _stream(stream))


def check(rc: int) -> int:
    if rc != ATTN_OK:
        raise AttnError(rc, last_error())
    return rc


# ---- raw entry points (same names and argument order as include/attn.h) ----
def attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream=None) -> int:
    return lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                        float(scale), int(bool(causal)), dtype_code(dtype), _stream(stream))


def attn_bwd_workspace_size(B, H, N, d) -> int:
    return int(lib.attn_bwd_workspace_size(B, H, N, d))


def attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, dtype,
             workspace, workspace_bytes, stream=None) -> int:
    return lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                        _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                        dtype_code(dtype), _ptr(workspace), int(workspace_bytes),
                        _stream(stream))


# Bytes of the library-owned scratch array used by attn_bwd_noalloc.
NOALLOC_WORKSPACE_BYTES = 32 * 1024 * 1024


def attn_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, dtype,
                     stream=None) -> int:
    """attn_bwd without a caller workspace (library-owned scratch array);
    for callers that cannot allocate device memory."""
    return lib.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                int(bool(causal)), dtype_code(dtype), _stream(stream))


def attn_fwd_alibi(q, k, v, o, lse, B, H, N, d, scale, causal, alibi_slopes, dtype,
                   stream=None) -> int:
    return lib.attn_fwd_alibi(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                              float(scale), int(bool(causal)), _ptr(alibi_slopes),
                              dtype_code(dtype), _stream(stream))


def attn_bwd_alibi(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, alibi_slopes,
                   dtype, workspace, workspace_bytes, stream=None) -> int:
    return lib.attn_bwd_alibi(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                              _ptr(alibi_slopes), dtype_code(dtype), _ptr(workspace),
                              int(workspace_bytes), _stream(stream))


def attn_fwd_sparse(q, k, v, o, lse, B, H, N, d, scale, causal, alibi_slopes, block_mask, dtype,
                    stream=None) -> int:
    return lib.attn_fwd_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                               float(scale), int(bool(causal)), _ptr(alibi_slopes),
                               _ptr(block_mask), dtype_code(dtype), _stream(stream))


def attn_bwd_sparse(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, alibi_slopes,
                    block_mask, dtype, workspace, workspace_bytes, stream=None) -> int:
    return lib.attn_bwd_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                               _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                               _ptr(alibi_slopes), _ptr(block_mask), dtype_code(dtype),
                               _ptr(workspace), int(workspace_bytes), _stream(stream))


def attn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, alibi_slopes, block_mask, dropout_p,
                seed, offset, dtype, stream=None) -> int:
    return lib.attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                           float(scale), int(bool(causal)), _ptr(alibi_slopes), _ptr(block_mask),
                           float(dropout_p), int(seed), int(offset), dtype_code(dtype),
                           _stream(stream))


def attn_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, alibi_slopes,
                block_mask, dropout_p, seed, offset, dtype, workspace, workspace_bytes,
                stream=None) -> int:
    return lib.attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                           _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                           _ptr(alibi_slopes), _ptr(block_mask), float(dropout_p), int(seed),
                           int(offset), dtype_code(dtype), _ptr(workspace), int(workspace_bytes),
                           _stream(stream))


ATTN_ACC_FIRST, ATTN_ACC_LAST = 1, 2


def attn_fwd_acc(q, k, v, o_acc, lse, o, B, H, N, d, scale, causal, flags, dtype,
                 stream=None) -> int:
    return lib.attn_fwd_acc(_ptr(q), _ptr(k), _ptr(v), _ptr(o_acc), _ptr(lse), _ptr(o), B, H, N, d,
                            float(scale), int(bool(causal)), int(flags), dtype_code(dtype),
                            _stream(stream))


def attn_bwd_acc(q, k, v, o, lse, dO, dq, dk_acc, dv_acc, B, H, N, d, scale, causal, dq_flags,
                 kv_flags, dtype, workspace, workspace_bytes, stream=None) -> int:
    return lib.attn_bwd_acc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                            _ptr(dk_acc), _ptr(dv_acc), B, H, N, d, float(scale),
                            int(bool(causal)), int(dq_flags), int(kv_flags), dtype_code(dtype),
                            _ptr(workspace), int(workspace_bytes), _stream(stream))


def attn_cast_acc(acc, out, n, mul, dtype, stream=None) -> int:
    return lib.attn_cast_acc(_ptr(acc), _ptr(out), int(n), float(mul), dtype_code(dtype),
                             _stream(stream))


def attn_decode_alibi(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, alibi_slopes, dtype,
                      workspace, workspace_bytes, stream=None) -> int:
    return lib.attn_decode_alibi(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                 float(scale), int(bool(causal)), _ptr(alibi_slopes),
                                 dtype_code(dtype), _ptr(workspace), int(workspace_bytes),
                                 _stream(stream))


def attn_decode_workspace_size(B, H, Nq, Nk, d) -> int:
    return int(lib.attn_decode_workspace_size(B, H, Nq, Nk, d))


def attn_decode(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, workspace,
                workspace_bytes, stream=None) -> int:
    return lib.attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                           float(scale), int(bool(causal)), dtype_code(dtype), _ptr(workspace),
                           int(workspace_bytes), _stream(stream))


def attn_status(stream=None) -> int:
    return lib.attn_status(_stream(stream))


def attn_set_wait_limit(limit_ns: int, debug_flags: int = 0) -> int:
    return lib.attn_set_wait_limit(int(limit_ns), int(debug_flags))


def attn_profile_begin() -> int:
    return lib.attn_profile_begin()


def attn_profile_end():
    """Returns {kernel name: (launches, total ms)}."""
    n = len(KERNEL_NAMES)
    launches = (ctypes.c_int * n)()
    ms = (ctypes.c_double * n)()
    check(min(0, lib.attn_profile_end(launches, ms, n)))
    return {KERNEL_NAMES[i]: (launches[i], ms[i]) for i in range(n)}


# ---- allocating conveniences --------------------------------------------
def _shape(q):
    if q.dim() != 4 or not q.is_contiguous():
        raise ValueError("tensors must be contiguous [B, N, H, d]")
    B, N, H, d = q.shape
    return B, N, H, d


def _block_mask(block_mask, H, N):
    """None, or a contiguous uint8 CUDA tensor [H, nb, nb], nb = ceil(N / 128)."""
    if block_mask is None:
        return None
    nb = (N + 127) // 128
    if (block_mask.dtype != torch.uint8 or tuple(block_mask.shape) != (H, nb, nb)
            or not block_mask.is_contiguous() or not block_mask.is_cuda):
        raise ValueError(f"block_mask must be a contiguous uint8 CUDA tensor [{H}, {nb}, {nb}]")
    return block_mask


def fwd(q, k, v, scale=None, causal=False, stream=None, alibi=None, block_mask=None,
        dropout_p=0.0, seed=0, offset=0):
    """(o, lse) for contiguous [B, N, H, d] fp16/bf16 CUDA tensors.
    alibi: optional fp32 CUDA tensor [H] of ALiBi slopes.
    block_mask: optional uint8 CUDA tensor [H, nb, nb] over 128 x 128 blocks
    (0 removes a block).
    dropout_p, seed, offset: dropout of the probabilities (attn_fwd_ex)."""
    B, N, H, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    bm = _block_mask(block_mask, H, N)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    check(attn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, alibi, bm, dropout_p, seed,
                      offset, q.dtype, stream))
    return o, lse


def workspace(B, H, N, d, device) -> torch.Tensor:
    n = attn_bwd_workspace_size(B, H, N, d)
    return torch.empty(n, dtype=torch.uint8, device=device)


def bwd(q, k, v, o, lse, do, scale=None, causal=False, ws=None, stream=None, alibi=None,
        block_mask=None, dropout_p=0.0, seed=0, offset=0):
    """(dq, dk, dv) for the forward that produced (o, lse) (same alibi,
    block_mask and dropout)."""
    B, N, H, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    bm = _block_mask(block_mask, H, N)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if ws is None:
        ws = workspace(B, H, N, d, q.device)
    check(attn_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, alibi, bm,
                      dropout_p, seed, offset, q.dtype, ws, ws.numel(), stream))
    return dq, dk, dv


def decode(q, k, v, scale=None, causal=False, ws=None, stream=None, alibi=None):
    """(o, lse) of q [B, Nq, H, d] (the last Nq positions) against the cache
    k, v [B, Nk, H, d]."""
    B, Nq, H, d = _shape(q)
    Nk = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = torch.empty(attn_decode_workspace_size(B, H, Nq, Nk, d), dtype=torch.uint8,
                         device=q.device)
    check(attn_decode_alibi(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, alibi, q.dtype, ws,
                            ws.numel(), stream))
    return o, lse


# ---- autograd -------------------------------------------------------------
class AttentionFunction(torch.autograd.Function):
    """O = attention(q, k, v) with the backward of the library (attn_bwd_ex):
    saves q, k, v, O and LSE (O(N) extra state), never P."""

    @staticmethod
    def forward(ctx, q, k, v, scale, causal, alibi, block_mask, dropout_p, seed, offset):
        o, lse = fwd(q, k, v, scale, causal, alibi=alibi, block_mask=block_mask,
                     dropout_p=dropout_p, seed=seed, offset=offset)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.opts = (scale, causal, alibi, block_mask, dropout_p, seed, offset)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        scale, causal, alibi, block_mask, dropout_p, seed, offset = ctx.opts
        dq, dk, dv = bwd(q, k, v, o, lse, do.contiguous(), scale, causal, alibi=alibi,
                         block_mask=block_mask, dropout_p=dropout_p, seed=seed, offset=offset)
        return dq, dk, dv, None, None, None, None, None, None, None


def attention(q, k, v, scale=None, causal=False, alibi=None, block_mask=None, dropout_p=0.0,
              seed=0, offset=0):
    """Differentiable attention on contiguous [B, N, H, d] fp16/bf16 CUDA
    tensors (forward and backward in the library's kernels)."""
    return AttentionFunction.apply(q, k, v, scale, causal, alibi, block_mask, dropout_p, seed,
                                   offset)
