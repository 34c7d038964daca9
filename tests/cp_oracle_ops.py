"""CPU stand-in for the library's block kernels, for the context-parallel
tests that run without a GPU (the ring driver on gloo ranks).  fp64 numpy on
CPU tensors, the same flag semantics as attn_fwd_acc / attn_bwd_acc /
attn_cast_acc.  The block forward is the fp64 oracle; the block backward
with a given final LSE is the plain calculus written out here (the oracle's
backward takes no external LSE); the totals are checked against the oracle.
"""
import numpy as np

ACC_FIRST, ACC_LAST = 1, 2


class OracleOps:
    def __init__(self, orc, scale):
        import torch
        self.orc = orc
        self.scale = scale
        self.acc_dtype = torch.float64

    def fwd_block(self, q, k, v, o_acc, lse, o, causal, flags):
        B, C, H, d = q.shape
        qn, kn, vn = q.numpy(), k.numpy(), v.numpy()
        la, oa, on = lse.numpy(), o_acc.numpy(), o.numpy()
        for b in range(B):
            for h in range(H):
                ob, lb = self.orc.fwd_head(np.ascontiguousarray(qn[b, :, h]), np.ascontiguousarray(kn[b, :, h]),
                                           np.ascontiguousarray(vn[b, :, h]), self.scale, causal)
                if flags & ACC_FIRST:
                    lo, oo = np.full(C, -np.inf), np.zeros((C, d))
                else:
                    lo, oo = la[b, h].copy(), oa[b, :, h].copy()
                m = np.maximum(lo, lb)
                wo, wb = np.exp(lo - m), np.exp(lb - m)
                merged = (wo[:, None] * oo + wb[:, None] * ob) / (wo + wb)[:, None]
                la[b, h] = m + np.log(wo + wb)
                if flags & ACC_LAST:
                    on[b, :, h] = merged
                else:
                    oa[b, :, h] = merged

    def bwd_block(self, q, k, v, o, lse, do, dq, dk_acc, dv_acc, causal, q_flags, kv_flags, ws):
        B, C, H, d = q.shape
        qn, kn, vn, onp, ln, don = (t.numpy() for t in (q, k, v, o, lse, do))
        if q_flags & ACC_FIRST:
            ws["dq"] = np.zeros((B, C, H, d))
        dka, dva = dk_acc.numpy(), dv_acc.numpy()
        if kv_flags & ACC_FIRST:
            dka[...] = 0.0
            dva[...] = 0.0
        for b in range(B):
            for h in range(H):
                qh, kh, vh, oh, dh = (a[b, :, h] for a in (qn, kn, vn, onp, don))
                s = self.scale * qh @ kh.T
                if causal:
                    s = np.where(np.tril(np.ones((C, C), dtype=bool)), s, -np.inf)
                p = np.exp(s - ln[b, h][:, None])
                dp = dh @ vh.T
                dvec = (dh * oh).sum(axis=1)
                ds = p * (dp - dvec[:, None])
                ws["dq"][b, :, h] += self.scale * ds @ kh
                dka[b, :, h] += self.scale * ds.T @ qh
                dva[b, :, h] += p.T @ dh
        if q_flags & ACC_LAST:
            dq.numpy()[...] = ws["dq"]

    def cast(self, acc, out):
        out.numpy()[...] = acc.numpy()

    def workspace(self, q):
        return {}
