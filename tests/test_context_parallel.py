"""Sequence (context) parallelism, host side, on CPU: the ring schedule's
properties, the one-process emulation of every rank, and the ring itself on
gloo ranks (world size 2 and 3) with an fp64 CPU stand-in for the block
kernels; the unsharded results equal the fp64 oracle over the whole
sequence."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from exact_tiled_attention_22_gb300 import context_parallel as cp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("world", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("causal", [True, False])
def test_plan_covers_every_block_once(world, causal):
    done = []
    for r in range(world):
        for s, st in enumerate(cp.ring_plan(world, r, causal)):
            assert st.src == (r - s) % world
            assert st.send_to == (r + 1) % world and st.recv_from == (r - 1) % world
            for blk in st.blocks:
                assert blk.q_chunk == cp.zigzag_chunks(world, r)[blk.q_local]
                assert blk.kv_chunk == cp.zigzag_chunks(world, st.src)[blk.kv_local]
                assert blk.causal == (causal and blk.q_chunk == blk.kv_chunk)
                done.append((blk.q_chunk, blk.kv_chunk))
    want = [(a, b) for a in range(2 * world) for b in range(2 * world) if (b <= a or not causal)]
    assert sorted(done) == sorted(want)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("causal", [True, False])
def test_plan_flags(world, causal):
    kv_first = {}
    for r in range(world):
        plan = cp.ring_plan(world, r, causal)
        for qi in range(2):
            flags = [b.q_flags for st in plan for b in st.blocks if b.q_local == qi]
            assert flags[0] & cp.ACC_FIRST and flags[-1] & cp.ACC_LAST
            assert sum(1 for f in flags if f & cp.ACC_FIRST) == 1
            assert sum(1 for f in flags if f & cp.ACC_LAST) == 1
        for s, st in enumerate(plan):
            for b in st.blocks:
                if b.kv_flags & cp.ACC_FIRST:
                    assert b.kv_chunk not in kv_first
                    kv_first[b.kv_chunk] = (r, s)
    assert sorted(kv_first) == list(range(2 * world))
    for c, where in kv_first.items():
        assert where == cp.kv_journey_first(world, c, causal)


@pytest.mark.parametrize("world", [2, 3, 4])
def test_zigzag_balances_causal_work(world):
    # a full block costs two diagonal blocks
    work = [sum(2 - b.causal for st in cp.ring_plan(world, r, True) for b in st.blocks)
            for r in range(world)]
    assert len(set(work)) == 1


def test_shard_unshard_roundtrip():
    x = torch.arange(2 * 24 * 3 * 4, dtype=torch.float64).reshape(2, 24, 3, 4)
    for world in (1, 2, 3):
        parts = [cp.shard(x, world, r) for r in range(world)]
        assert parts[0].shape == (2, 2, 24 // (2 * world), 3, 4)
        assert torch.equal(cp.unshard(parts), x)
    y = torch.arange(2 * 3 * 24, dtype=torch.float64).reshape(2, 3, 24)
    parts = [cp.shard(y, 3, r, seq_dim=2) for r in range(3)]
    assert torch.equal(cp.unshard(parts, seq_dim=2), y)


def _inputs(B, N, H, d, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((B, N, H, d), generator=g, dtype=torch.float64) for _ in range(4)]


def _reference(orc, q, k, v, do, scale, causal):
    B, N, H, d = q.shape
    o = np.zeros((B, N, H, d)); lse = np.zeros((B, H, N))
    dq, dk, dv = (np.zeros((B, N, H, d)) for _ in range(3))
    for b in range(B):
        for h in range(H):
            hq, hk, hv, hd = (np.ascontiguousarray(t[b, :, h].numpy()) for t in (q, k, v, do))
            o[b, :, h], lse[b, h] = orc.fwd_head(hq, hk, hv, scale, causal)
            dq[b, :, h], dk[b, :, h], dv[b, :, h], _ = orc.bwd_head(hq, hk, hv, hd, scale, causal)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("world,causal", [(1, True), (2, True), (3, True), (4, False), (3, False)])
def test_emulated_ring_equals_oracle(oracle, world, causal):
    from cp_oracle_ops import OracleOps
    B, H, d = 2, 2, 8
    N = 2 * world * 5
    q, k, v, do = _inputs(B, N, H, d, seed=world)
    scale = 0.4
    got = cp.emulate_ring(q, k, v, do, world, OracleOps(oracle, scale), causal)
    ref = _reference(oracle, q, k, v, do, scale, causal)
    for name, g, r in zip(("o", "lse", "dq", "dk", "dv"), got, ref):
        np.testing.assert_allclose(g.numpy(), r, rtol=1e-9, atol=1e-11, err_msg=name)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ring_worker(rank, world, port, causal, out_q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    import oracle as oracle_pkg
    from cp_oracle_ops import OracleOps
    from exact_tiled_attention_22_gb300 import context_parallel as cpm
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, H, d, N = 2, 2, 8, 2 * world * 6
    q, k, v, do = _inputs(B, N, H, d, seed=100 + world)
    sh = [cpm.shard(t, world, rank) for t in (q, k, v, do)]
    ops = OracleOps(oracle_pkg.get(), 0.3)
    o, lse = cpm.ring_forward(sh[0], sh[1], sh[2], ops, causal)
    dq, dk, dv = cpm.ring_backward(sh[0], sh[1], sh[2], o, lse, sh[3], ops, causal)
    dist.barrier()
    dist.destroy_process_group()
    out_q.put((rank, [t.numpy().copy() for t in (o, lse, dq, dk, dv)]))


@pytest.mark.parametrize("world,causal", [(2, True), (3, True), (2, False)])
def test_ring_on_gloo_ranks_equals_oracle(oracle, world, causal):
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ring_worker, args=(r, world, port, causal, out_q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(out_q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    B, H, d, N = 2, 2, 8, 2 * world * 6
    q, k, v, do = _inputs(B, N, H, d, seed=100 + world)
    ref = _reference(oracle, q, k, v, do, 0.3, causal)
    for i, name in enumerate(("o", "lse", "dq", "dk", "dv")):
        seq_dim = 2 if name == "lse" else 1
        got = cp.unshard([torch.from_numpy(res[r][i]) for r in range(world)], seq_dim=seq_dim)
        np.testing.assert_allclose(got.numpy(), ref[i], rtol=1e-9, atol=1e-11, err_msg=name)
