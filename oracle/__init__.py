"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The GPU library never imports, links or calls it, and it
imports nothing from the library: the two share no code.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, one head at a time;
its header comment cites the passages it follows).  This module only compiles
that file with gcc, loads it with ctypes, and slices heads out of
``[B, N, H, d]`` tensors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(src_path: str = SRC, out_path: str = LIB, force: bool = False) -> str:
    """Compile the oracle into a shared library with gcc -O2 (no tuning)."""
    if (not force and os.path.exists(out_path)
            and os.path.getmtime(out_path) >= os.path.getmtime(src_path)):
        return out_path
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
           src_path, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build_from_text(c_source: str, workdir: str | None = None) -> str:
    """Compile an edited copy of the oracle source (used by the tests that
    plant a mistake in the oracle to check that the pins catch it)."""
    d = workdir or tempfile.mkdtemp(prefix="oracle_mut_")
    src = os.path.join(d, "attn_oracle_edit.c")
    with open(src, "w") as f:
        f.write(c_source)
    return build(src, os.path.join(d, "liboracle_edit.so"), force=True)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str | None = None):
        self.path = path or build()
        lib = ctypes.CDLL(self.path)
        _bp = ctypes.c_void_p  # block mask: uint8 [nb][nb] or NULL
        # dropout: threshold t (256 = none), seed, offset, head index
        _dr = [ctypes.c_int, ctypes.c_ulonglong, ctypes.c_uint, ctypes.c_uint]
        lib.oracle_fwd.argtypes = ([_dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_double,
                                    ctypes.c_int, _bp] + _dr +
                                   [_ip, ctypes.c_int, _dp, _dp, ctypes.c_int])
        lib.oracle_bwd.argtypes = ([_dp, _dp, _dp, _dp, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_double,
                                    ctypes.c_double, ctypes.c_int, _bp] + _dr +
                                   [_ip, ctypes.c_int, _ip, ctypes.c_int, _dp,
                                    _dp, _dp, _dp, ctypes.c_int])
        _u32p = ctypes.POINTER(ctypes.c_uint)
        _u64p = ctypes.POINTER(ctypes.c_ulonglong)
        lib.oracle_philox4x32.argtypes = [_u32p, _u32p, _u32p]
        lib.oracle_philox4x32.restype = None
        lib.oracle_philox4x64.argtypes = [_u64p, _u64p, _u64p]
        lib.oracle_philox4x64.restype = None
        lib.oracle_dropout_threshold.argtypes = [ctypes.c_double]
        lib.oracle_dropout_threshold.restype = ctypes.c_int
        lib.oracle_dropout_keep.argtypes = [ctypes.c_ulonglong, ctypes.c_uint,
                                            ctypes.c_uint, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int]
        lib.oracle_dropout_keep.restype = ctypes.c_int
        lib.oracle_online_fwd.argtypes = [_dp, _dp, _dp, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_double,
                                          ctypes.c_int, ctypes.c_int, _dp, _dp,
                                          ctypes.c_int]
        lib.oracle_decode_fwd.argtypes = [_dp, _dp, _dp, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int,
                                          ctypes.c_double, ctypes.c_double,
                                          ctypes.c_int, _dp, _dp, ctypes.c_int]
        for f in (lib.oracle_fwd, lib.oracle_bwd, lib.oracle_online_fwd,
                  lib.oracle_decode_fwd):
            f.restype = ctypes.c_int
        lib.oracle_default_threads.restype = ctypes.c_int
        self.lib = lib

    @staticmethod
    def _f64(a) -> np.ndarray:
        return np.ascontiguousarray(a, dtype=np.float64)

    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data_as(_dp)

    @staticmethod
    def _idx(lst):
        if lst is None:
            return None, None
        arr = np.ascontiguousarray(lst, dtype=np.int32)
        return arr, arr.ctypes.data_as(_ip)

    def threads(self) -> int:
        return int(self.lib.oracle_default_threads())

    # ---- dropout generator ---------------------------------------------
    def philox4x32(self, ctr, key):
        c = (ctypes.c_uint * 4)(*[int(x) for x in ctr])
        k = (ctypes.c_uint * 2)(*[int(x) for x in key])
        out = (ctypes.c_uint * 4)()
        self.lib.oracle_philox4x32(c, k, out)
        return [int(x) for x in out]

    def philox4x64(self, ctr, key):
        c = (ctypes.c_ulonglong * 4)(*[int(x) for x in ctr])
        k = (ctypes.c_ulonglong * 2)(*[int(x) for x in key])
        out = (ctypes.c_ulonglong * 4)()
        self.lib.oracle_philox4x64(c, k, out)
        return [int(x) for x in out]

    def dropout_threshold(self, p) -> int:
        """Keep threshold t for dropout probability p (given as fp32, the
        precision of the library's argument); -1 if p is not allowed."""
        return int(self.lib.oracle_dropout_threshold(float(np.float32(p))))

    def dropout_keep(self, seed, offset, head, r, j, t) -> int:
        return int(self.lib.oracle_dropout_keep(int(seed), int(offset), int(head),
                                                int(r), int(j), int(t)))

    def _dropout(self, dropout):
        """(t, seed, offset, head) for dropout = None or (p, seed, offset, head)."""
        if dropout is None:
            return 256, 0, 0, 0
        p, seed, offset, head = dropout
        t = self.dropout_threshold(p)
        if t < 1:
            raise ValueError(f"dropout probability {p} not allowed")
        return t, int(seed), int(offset), int(head)

    # ---- one head ------------------------------------------------------
    @staticmethod
    def _bmask(block_mask, N):
        """uint8 [nb, nb] mask over 128 x 128 blocks (nb = ceil(N/128)), or None."""
        if block_mask is None:
            return None, None
        nb = (N + 127) // 128
        m = np.ascontiguousarray(block_mask, dtype=np.uint8)
        if m.shape != (nb, nb):
            raise ValueError(f"block mask must be [{nb}, {nb}]")
        return m, m.ctypes.data

    def fwd_head(self, q, k, v, scale, causal, rows=None, nthreads=0, alibi=0.0,
                 block_mask=None, dropout=None):
        """q, k, v: [N, d].  Returns (O [nrows, d], LSE [nrows]).
        alibi: the head's ALiBi slope (bias -alibi*|i - j| on the scores).
        block_mask: uint8 [nb, nb] over 128 x 128 blocks; 0 removes a block.
        dropout: None or (p, seed, offset, head index b*H + h)."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        N, d = q.shape
        rows_arr, rows_p = self._idx(rows)
        nrows = N if rows is None else len(rows_arr)
        bm, bm_p = self._bmask(block_mask, N)
        o = np.zeros((nrows, d))
        lse = np.zeros(nrows)
        rc = self.lib.oracle_fwd(self._ptr(q), self._ptr(k), self._ptr(v), N, d,
                                 float(scale), float(alibi), int(bool(causal)), bm_p,
                                 *self._dropout(dropout), rows_p, nrows,
                                 self._ptr(o), self._ptr(lse), int(nthreads))
        if rc != 0:
            raise RuntimeError(f"oracle_fwd failed: {rc}")
        return o, lse

    def bwd_head(self, q, k, v, dO, scale, causal, rows=None, keys=None,
                 nthreads=0, alibi=0.0, block_mask=None, dropout=None):
        """Returns (dQ [nrows, d], dK [nkeys, d], dV [nkeys, d], D [N])."""
        q, k, v, dO = (self._f64(x) for x in (q, k, v, dO))
        N, d = q.shape
        rows_arr, rows_p = self._idx(rows)
        keys_arr, keys_p = self._idx(keys)
        nrows = N if rows is None else len(rows_arr)
        nkeys = N if keys is None else len(keys_arr)
        bm, bm_p = self._bmask(block_mask, N)
        dq = np.zeros((nrows, d))
        dk = np.zeros((nkeys, d))
        dv = np.zeros((nkeys, d))
        D = np.zeros(N)
        rc = self.lib.oracle_bwd(self._ptr(q), self._ptr(k), self._ptr(v),
                                 self._ptr(dO), N, d, float(scale), float(alibi),
                                 int(bool(causal)), bm_p, *self._dropout(dropout),
                                 rows_p, nrows, keys_p,
                                 nkeys, self._ptr(dq), self._ptr(dk),
                                 self._ptr(dv), self._ptr(D), int(nthreads))
        if rc != 0:
            raise RuntimeError(f"oracle_bwd failed: {rc}")
        return dq, dk, dv, D

    def online_fwd_head(self, q, k, v, scale, causal, tile, nthreads=0):
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        N, d = q.shape
        o = np.zeros((N, d))
        lse = np.zeros(N)
        rc = self.lib.oracle_online_fwd(self._ptr(q), self._ptr(k),
                                        self._ptr(v), N, d, float(scale),
                                        int(bool(causal)), int(tile),
                                        self._ptr(o), self._ptr(lse),
                                        int(nthreads))
        if rc != 0:
            raise RuntimeError(f"oracle_online_fwd failed: {rc}")
        return o, lse

    def decode_head(self, q, k, v, scale, causal, nthreads=0, alibi=0.0):
        """q: [Nq, d], the last Nq positions; k, v: [Nk, d].
        Returns (O [Nq, d], LSE [Nq])."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        Nq, d = q.shape
        Nk = k.shape[0]
        o = np.zeros((Nq, d))
        lse = np.zeros(Nq)
        rc = self.lib.oracle_decode_fwd(self._ptr(q), self._ptr(k), self._ptr(v),
                                        Nq, Nk, d, float(scale), float(alibi),
                                        int(bool(causal)), self._ptr(o),
                                        self._ptr(lse), int(nthreads))
        if rc != 0:
            raise RuntimeError(f"oracle_decode_fwd failed: {rc}")
        return o, lse

    # ---- [B, N, H, d] tensors ------------------------------------------
    @staticmethod
    def head(x, b, h) -> np.ndarray:
        """Head (b, h) of a [B, N, H, d] array as a contiguous fp64 [N, d]."""
        return np.ascontiguousarray(np.asarray(x)[b, :, h, :], dtype=np.float64)

    def fwd(self, q, k, v, scale, causal, heads=None, nthreads=0):
        """Forward over the listed (b, h) heads (default: all).
        Returns {(b, h): (O [N, d], LSE [N])}."""
        B, N, H, d = np.asarray(q).shape
        heads = heads if heads is not None else [(b, h) for b in range(B)
                                                 for h in range(H)]
        return {(b, h): self.fwd_head(self.head(q, b, h), self.head(k, b, h),
                                      self.head(v, b, h), scale, causal,
                                      nthreads=nthreads)
                for (b, h) in heads}

    def bwd(self, q, k, v, dO, scale, causal, heads=None, nthreads=0):
        """Backward over the listed heads.  Returns {(b, h): (dQ, dK, dV, D)}."""
        B, N, H, d = np.asarray(q).shape
        heads = heads if heads is not None else [(b, h) for b in range(B)
                                                 for h in range(H)]
        return {(b, h): self.bwd_head(self.head(q, b, h), self.head(k, b, h),
                                      self.head(v, b, h), self.head(dO, b, h),
                                      scale, causal, nthreads=nthreads)
                for (b, h) in heads}


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from the committed source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
