"""Sequence (context) parallelism: exact attention over a sequence split
across R ranks (page "Flash Attention V2大模型时代的算力救星", section 6: long
sequences split over devices).

Layout.  The sequence of N positions is cut into 2R chunks of C = N / (2R)
positions; rank r holds chunks r and 2R - 1 - r ("zigzag"), so that under the
causal mask every rank has the same amount of work (a low chunk sees few keys,
its partner high chunk many).  A rank's shard of Q, K, V, dO, O, dQ, dK, dV
is a chunk-major [2, B, C, H, d] tensor (its two chunks in that order) and of
LSE a [2, B, H, C] tensor.

Forward.  K and V travel around the ring: at step s rank r holds the shard
of rank (r - s) mod R, sends it on to rank r + 1 and receives the next one
from rank r - 1 while it computes.  Each of its query chunks a meets each
held key chunk b: b < a is a full block, b = a the causal diagonal block,
b > a is skipped.  attn_fwd_acc merges every block into an fp32 (O, LSE)
accumulator per query chunk, which is exact whatever the order of blocks;
the last block writes the 16-bit O.

Backward.  K and V travel again, now with fp32 accumulators of their dK and
dV.  Every block (a, b) adds its dQ to query chunk a's sum (kept in that
chunk's workspace from its first block to its last) and its dK, dV to the
travelling accumulators (attn_bwd_acc, given the final O and LSE of chunk
a).  After R steps the accumulators have visited every rank; one more hop
brings them home, where attn_cast_acc turns them into 16-bit dK, dV.

Every exchange moves whole shards between ranks' own buffers through
torch.distributed point-to-point calls (NCCL between GPUs, gloo on CPUs); no
kernel reads another device's memory.  The compute goes through an `ops`
object: `GpuOps` calls the library's kernels; tests on CPU pass their own.
"""
from __future__ import annotations

from dataclasses import dataclass, field

ACC_FIRST, ACC_LAST = 1, 2


def zigzag_chunks(world: int, rank: int) -> tuple[int, int]:
    """Global chunk indices held by `rank` (its local chunks 0 and 1)."""
    return rank, 2 * world - 1 - rank


def block_kind(q_chunk: int, kv_chunk: int, causal: bool) -> str | None:
    """'full', 'diag' (causal mask inside the block) or None (no visible key)."""
    if not causal:
        return "full"
    if kv_chunk < q_chunk:
        return "full"
    if kv_chunk == q_chunk:
        return "diag"
    return None


@dataclass
class Block:
    """One (query chunk, key chunk) block computed at a step."""
    q_local: int       # local index (0/1) of the query chunk on this rank
    kv_local: int      # local index (0/1) of the key chunk within the held shard
    q_chunk: int       # global chunk indices
    kv_chunk: int
    causal: bool       # True for the diagonal block
    q_flags: int = 0   # ACC_FIRST / ACC_LAST for the query chunk's accumulators
    kv_flags: int = 0  # ACC_FIRST for the key chunk's dK/dV accumulators (backward)


@dataclass
class Step:
    src: int                     # rank whose K/V shard is held at this step
    send_to: int
    recv_from: int
    blocks: list = field(default_factory=list)


def ring_plan(world: int, rank: int, causal: bool = True) -> list[Step]:
    """The ring schedule of `rank`: per step, the shard held and the blocks
    computed on it, with the accumulation flags of every block.

    Query chunk flags: FIRST on the chunk's first block on this rank, LAST on
    its last.  Key chunk flags: FIRST on the first block of the chunk's whole
    journey around the ring (always at step 0 on its owner: the diagonal
    block, or the first full block when not causal), else 0."""
    mine = zigzag_chunks(world, rank)
    steps = []
    for s in range(world):
        src = (rank - s) % world
        st = Step(src=src, send_to=(rank + 1) % world, recv_from=(rank - 1) % world)
        held = zigzag_chunks(world, src)
        for qi, qc in enumerate(mine):
            for ki, kc in enumerate(held):
                kind = block_kind(qc, kc, causal)
                if kind is not None:
                    st.blocks.append(Block(qi, ki, qc, kc, kind == "diag"))
        steps.append(st)
    # query-chunk flags, in the order the blocks run on this rank
    seen = {}
    last = {}
    for s, st in enumerate(steps):
        for bi, blk in enumerate(st.blocks):
            if blk.q_local not in seen:
                seen[blk.q_local] = (s, bi)
            last[blk.q_local] = (s, bi)
    for qi, (s, bi) in seen.items():
        steps[s].blocks[bi].q_flags |= ACC_FIRST
    for qi, (s, bi) in last.items():
        steps[s].blocks[bi].q_flags |= ACC_LAST
    # key-chunk flags: the journey of each key chunk starts at step 0 on its
    # owner, which always has a block with it (its diagonal block, or any
    # block when not causal); the first such block starts the accumulators
    started = set()
    for blk in steps[0].blocks:
        if blk.kv_local not in started:
            blk.kv_flags = ACC_FIRST
            started.add(blk.kv_local)
    return steps


def kv_journey_first(world: int, kv_chunk: int, causal: bool = True) -> tuple[int, int]:
    """(rank, step) of the first block of key chunk `kv_chunk` on its way
    around the ring (a check of ring_plan's key flags)."""
    owner = kv_chunk if kv_chunk < world else 2 * world - 1 - kv_chunk
    for s in range(world):
        r = (owner + s) % world
        if any(block_kind(qc, kv_chunk, causal) for qc in zigzag_chunks(world, r)):
            return r, s
    raise ValueError("key chunk with no visible query")


# ------------------------------------------------------------------ compute
class GpuOps:
    """The library's kernels on chunk views [B, C, H, d] (contiguous) of the
    shards; accumulators are fp32 tensors of the same layout."""

    def __init__(self, scale: float):
        import torch
        from exact_tiled_attention_22_gb300 import attn
        self.A = attn
        self.scale = scale
        self.acc_dtype = torch.float32  # O, LSE, dK and dV accumulators

    def fwd_block(self, q, k, v, o_acc, lse, o, causal, flags):
        B, C, H, d = q.shape
        self.A.check(self.A.attn_fwd_acc(q, k, v, o_acc, lse, o, B, H, C, d, self.scale, causal, flags,
                                         q.dtype))

    def bwd_block(self, q, k, v, o, lse, do, dq, dk_acc, dv_acc, causal, q_flags, kv_flags, ws):
        B, C, H, d = q.shape
        self.A.check(self.A.attn_bwd_acc(q, k, v, o, lse, do, dq, dk_acc, dv_acc, B, H, C, d,
                                         self.scale, causal, q_flags, kv_flags, q.dtype, ws,
                                         ws.numel()))

    def cast(self, acc, out):
        self.A.check(self.A.attn_cast_acc(acc, out, acc.numel(), 1.0, out.dtype))

    def workspace(self, q):
        B, C, H, d = q.shape
        return self.A.workspace(B, H, C, d, q.device)


# ------------------------------------------------------------------ exchange
def _start_exchange(dist, group, send_buf, recv_buf, to, frm):
    ops = [dist.P2POp(dist.isend, send_buf, to, group), dist.P2POp(dist.irecv, recv_buf, frm, group)]
    return dist.batch_isend_irecv(ops)


def _wait(reqs):
    for r in reqs:
        r.wait()


def _group_rank(dist, group, world_rank):
    """Global rank of a rank of `group` (P2P calls take global ranks)."""
    return dist.get_global_rank(group, world_rank) if group is not None else world_rank


def ring_forward(q, k, v, ops, causal=True, group=None):
    """O [2, B, C, H, d] and LSE [2, B, H, C] of this rank's query chunks over
    the whole sequence.  q, k, v: this rank's chunk-major shards."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    plan = ring_plan(world, rank, causal)
    _, B, C, H, d = q.shape
    o = torch.empty_like(q)
    o_acc = torch.empty(q.shape, dtype=ops.acc_dtype, device=q.device)
    lse = torch.empty((2, B, H, C), dtype=ops.acc_dtype, device=q.device)
    cur = torch.stack([k, v]).contiguous()  # [2 (K, V), 2 chunks, B, C, H, d]
    nxt = torch.empty_like(cur)
    for s, st in enumerate(plan):
        reqs = []
        if s + 1 < world:
            reqs = _start_exchange(dist, group, cur, nxt, _group_rank(dist, group, st.send_to),
                                   _group_rank(dist, group, st.recv_from))
        for blk in st.blocks:
            ops.fwd_block(q[blk.q_local], cur[0, blk.kv_local], cur[1, blk.kv_local],
                          o_acc[blk.q_local], lse[blk.q_local], o[blk.q_local], blk.causal,
                          blk.q_flags)
        _wait(reqs)
        if s + 1 < world:
            cur, nxt = nxt, cur
    return o, lse


def ring_backward(q, k, v, o, lse, do, ops, causal=True, group=None):
    """dQ, dK, dV [2, B, C, H, d] of this rank's chunks.  o, lse: the
    forward's results for this rank's query chunks (ring_forward)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    plan = ring_plan(world, rank, causal)
    dq = torch.empty_like(q)
    ws = [ops.workspace(q[0]), ops.workspace(q[1])]
    cur = torch.stack([k, v]).contiguous()
    nxt = torch.empty_like(cur)
    acc = torch.zeros((2,) + tuple(k.shape), dtype=ops.acc_dtype, device=k.device)  # [dK, dV]
    acc_nxt = torch.empty_like(acc)
    for s, st in enumerate(plan):
        to = _group_rank(dist, group, st.send_to)
        frm = _group_rank(dist, group, st.recv_from)
        reqs = _start_exchange(dist, group, cur, nxt, to, frm) if s + 1 < world else []
        for blk in st.blocks:
            qi, ki = blk.q_local, blk.kv_local
            ops.bwd_block(q[qi], cur[0, ki], cur[1, ki], o[qi], lse[qi], do[qi], dq[qi],
                          acc[0, ki], acc[1, ki], blk.causal, blk.q_flags, blk.kv_flags, ws[qi])
        _wait(reqs)
        # the accumulators follow their K/V (after this step's blocks added to
        # them); after the last step one more hop takes them home
        if world > 1:
            _wait(_start_exchange(dist, group, acc, acc_nxt, to, frm))
            acc, acc_nxt = acc_nxt, acc
        if s + 1 < world:
            cur, nxt = nxt, cur
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    for c in range(2):
        ops.cast(acc[0, c], dk[c])
        ops.cast(acc[1, c], dv[c])
    return dq, dk, dv


# ------------------------------------------------------------- one device
def shard(x, world: int, rank: int, seq_dim: int = 1):
    """Rank `rank`'s chunk-major shard [2, ...] of a full [B, N, H, d] (or
    [B, H, N] with seq_dim=2) tensor."""
    import torch
    n = x.shape[seq_dim]
    c = n // (2 * world)
    parts = [x.narrow(seq_dim, i * c, c) for i in zigzag_chunks(world, rank)]
    return torch.stack(parts).contiguous()


def unshard(shards, seq_dim: int = 1):
    """Inverse of shard over all ranks: the full tensor from the ranks' shards."""
    import torch
    world = len(shards)
    chunks = [None] * (2 * world)
    for r, sh in enumerate(shards):
        a, b = zigzag_chunks(world, r)
        chunks[a], chunks[b] = sh[0], sh[1]
    return torch.cat(chunks, dim=seq_dim)


def emulate_ring(q, k, v, do, world: int, ops, causal=True):
    """Runs every rank's ring schedule in one process on one device (the
    shards are all local, so an exchange is just reading another rank's
    shard): the forward and backward of the full [B, N, H, d] inputs, as the
    ring over `world` ranks computes them.  Returns full-sequence
    (o, lse, dq, dk, dv)."""
    import torch
    B, N, H, d = q.shape
    if N % (2 * world):
        raise ValueError(f"N = {N} must be a multiple of 2 x world = {2 * world}")
    qs = [shard(q, world, r) for r in range(world)]
    ks = [shard(k, world, r) for r in range(world)]
    vs = [shard(v, world, r) for r in range(world)]
    dos = [shard(do, world, r) for r in range(world)]
    plans = [ring_plan(world, r, causal) for r in range(world)]
    # forward
    os_, lses = [], []
    for r in range(world):
        o = torch.empty_like(qs[r])
        o_acc = torch.empty(qs[r].shape, dtype=ops.acc_dtype, device=q.device)
        lse = torch.empty((2, B, H, N // (2 * world)), dtype=ops.acc_dtype, device=q.device)
        for st in plans[r]:
            for blk in st.blocks:
                ops.fwd_block(qs[r][blk.q_local], ks[st.src][blk.kv_local], vs[st.src][blk.kv_local],
                              o_acc[blk.q_local], lse[blk.q_local], o[blk.q_local], blk.causal,
                              blk.q_flags)
        os_.append(o)
        lses.append(lse)
    # backward: ranks in lockstep, step by step, so that the key chunks'
    # accumulators see their blocks in the ring's order
    dqs = [torch.empty_like(x) for x in qs]
    wss = [[ops.workspace(x[0]), ops.workspace(x[1])] for x in qs]
    accs = [torch.zeros((2,) + tuple(x.shape), dtype=ops.acc_dtype, device=q.device) for x in ks]
    for s in range(world):
        for r in range(world):
            st = plans[r][s]
            for blk in st.blocks:
                qi, ki = blk.q_local, blk.kv_local
                ops.bwd_block(qs[r][qi], ks[st.src][ki], vs[st.src][ki], os_[r][qi], lses[r][qi],
                              dos[r][qi], dqs[r][qi], accs[st.src][0, ki], accs[st.src][1, ki],
                              blk.causal, blk.q_flags, blk.kv_flags, wss[r][qi])
    dks, dvs = [], []
    for r in range(world):
        dk, dv = torch.empty_like(ks[r]), torch.empty_like(vs[r])
        for c in range(2):
            ops.cast(accs[r][0, c], dk[c])
            ops.cast(accs[r][1, c], dv[c])
        dks.append(dk)
        dvs.append(dv)
    return (unshard(os_), unshard(lses, seq_dim=2), unshard(dqs), unshard(dks), unshard(dvs))
