"""The cross-rank exchange steps of sequence parallelism on CPU gloo ranks
(world size 2 and 4): the reduce-scatter's exchange half, the norm-weight
gradient all-reduce and the all-gather of the partials' gradient, checked
against the oracle's simulated collectives (MiniMind-tron ch.3, §3.2.1,
§3.2.3, §3.3.3.1, §3.4.2.1)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _partial(t, S, B, H):
    g = torch.Generator().manual_seed(100 + t)
    return torch.randint(-8, 9, (S, B, H), generator=g).to(torch.float64) / 4


def _rank(rank, world, port, q, S, B, H):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from residual_sp_rs_gb300 import sp_exchange as ex
    blocks = ex.exchange_partials(_partial(rank, S, B, H))
    dg = torch.arange(H, dtype=torch.float64) * (rank + 1)
    db = torch.ones(H, dtype=torch.float64) * (rank + 1)
    ex.allreduce_norm_grads(dg, db)
    d_sum = torch.full(((S // world) * B, H), float(rank), dtype=torch.float64)
    grads = ex.gather_partial_grads(d_sum)
    q.put((rank, blocks.numpy(), dg.numpy(), db.numpy(), grads.numpy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_exchange_allreduce_and_gather_on_gloo_ranks(world):
    import oracle
    S, B, H = 4 * world, 2, 8
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q, S, B, H)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted([q.get(timeout=180) for _ in range(world)], key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    P = [_partial(t, S, B, H).numpy() for t in range(world)]
    R = (S // world) * B
    for j, blocks, dg, db, grads in got:
        # block t = rank t's rows of shard j; their rank-order sum is the
        # reduce-scatter's shard j (the oracle's simulated collective)
        for t in range(world):
            assert np.array_equal(blocks[t], P[t].reshape(-1, H)[j * R:(j + 1) * R])
        rs = oracle.reduce_scatter([p.ravel() for p in P], j)
        assert np.array_equal(blocks.sum(axis=0).ravel(), rs)
        # every rank holds the sum over ranks of the per-shard partials
        exp_g = oracle.all_reduce([np.arange(H) * (r + 1.0) for r in range(world)])
        exp_b = oracle.all_reduce([np.ones(H) * (r + 1.0) for r in range(world)])
        assert np.array_equal(dg, exp_g) and np.array_equal(db, exp_b)
        # the gradient of every partial: the ranks' d_sum shards in rank order
        assert np.array_equal(grads, np.repeat(np.arange(world, dtype=np.float64), R)[:, None] * np.ones(H))
    # the exchange moves (T-1)/T of a partial per rank, as the ring reduce-scatter
    _, sent = oracle.ring_reduce_scatter([p.ravel() for p in P])
    per_rank = (world - 1) * R * H
    assert all(int(s) == per_rank for s in sent)


def test_shard_row_addressing_rejects_mismatched_blocks():
    sys.path.insert(0, ROOT)
    from residual_sp_rs_gb300 import ops, sp_exchange as ex
    d = ops.make_desc(2, 1, 8, 2, 16, "bf16", "rms", 0.1, 1e-6, 0)
    with pytest.raises(ValueError):
        ex.forward_from_shard_rows(d, torch.zeros(2, 4, 16, dtype=torch.bfloat16), None, None, None,
                                   None, None, None, None, None)
    # right shape, but a strided view: the blocks' base addresses would not hold its rows
    strided = torch.zeros(8, 2, 16, dtype=torch.bfloat16).transpose(0, 1)
    assert strided.shape == (2, 8, 16) and not strided.is_contiguous()
    with pytest.raises(ValueError):
        ex.forward_from_shard_rows(d, strided, None, None, None, None, None, None, None, None)


def _pipelined_rank(rank, world, port, q, S, B, H, chunks):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from residual_sp_rs_gb300 import sp_exchange as ex
    R = (S // world) * B
    own = _partial(rank, S, B, H).to(torch.float32).view(-1, H)
    res, gam, bet = _norm_inputs(S, B, H)
    pr = oracle.problem(world, rank, S, B, H, "f32", "ln", 0.25, 1e-5, 7)
    bounds = ex.chunk_bounds(R, H, chunks)
    recv, works = ex.pull_chunks(own, bounds)
    outs = []
    for (b, e), buf, ws in zip(bounds, recv, works):
        for w in ws:
            w.wait()
        # the chunk's rows of every partial: this rank's own in place, the rest as received
        rows = [own[rank * R + b:rank * R + e] if t == rank else buf[t] for t in range(world)]
        grows = rank * R + b + np.arange(e - b)
        outs.append(oracle.fwd_rows(pr, grows, [r.numpy() for r in rows], res[rank * R + b:rank * R + e].numpy(),
                                    gam.numpy(), bet.numpy(), "f32"))
    cat = {k: np.concatenate([o[k] for o in outs]) for k in ("h", "y", "mask", "rstd", "mean")}
    q.put((rank, bounds, cat))
    dist.barrier()
    dist.destroy_process_group()


def _norm_inputs(S, B, H):
    g = torch.Generator().manual_seed(5)
    res = torch.randn(S * B, H, generator=g, dtype=torch.float32)
    gam = 1 + 0.1 * torch.randn(H, generator=g, dtype=torch.float32)
    bet = 0.1 * torch.randn(H, generator=g, dtype=torch.float32)
    return res, gam, bet


@pytest.mark.parametrize("world,chunks", [(2, 3), (4, 4)])
def test_pipelined_exchange_feeds_each_chunk_its_rows(world, chunks):
    """The exchange in pipeline chunks ("Sequence Parallel" notes,
    communication-computation overlap: the reduce-scatter in chunks): each
    chunk's forward, run on just the rows that chunk brought in, reproduces
    the whole shard's forward (MiniMind-tron ch.3, §3.2.3)."""
    import oracle
    oracle.build()
    S, B, H = 8 * world, 2, 24
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_pipelined_rank, args=(r, world, port, q, S, B, H, chunks))
             for r in range(world)]
    for p in procs:
        p.start()
    got = sorted([q.get(timeout=180) for _ in range(world)], key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    P = [_partial(t, S, B, H).to(torch.float32).numpy() for t in range(world)]
    res, gam, bet = _norm_inputs(S, B, H)
    R = (S // world) * B
    for j, bounds, cat in got:
        assert len(bounds) == chunks and bounds[0][0] == 0 and bounds[-1][1] == R
        assert all(e0 == b1 for (_, e0), (b1, _) in zip(bounds[:-1], bounds[1:]))
        pr = oracle.problem(world, j, S, B, H, "f32", "ln", 0.25, 1e-5, 7)
        full = oracle.fwd(pr, P, res[j * R:(j + 1) * R].numpy(), gam.numpy(), bet.numpy(), "f32")
        for k in ("h", "y", "mask", "rstd", "mean"):
            assert np.array_equal(cat[k], full[k]), (j, k)


def test_chunk_bounds_keep_mask_rows_aligned():
    sys.path.insert(0, ROOT)
    from residual_sp_rs_gb300 import sp_exchange as ex
    for R in (0, 1, 3, 16, 17, 2048, 4097):
        for H in (8, 24, 768, 4104):
            for chunks in (1, 2, 4, 7):
                b = ex.chunk_bounds(R, H, chunks)
                assert len(b) <= chunks
                assert [x for x, _ in b][:1] in ([], [0]) and (not b or b[-1][1] == R)
                assert all(e0 == b1 for (_, e0), (b1, _) in zip(b[:-1], b[1:]))
                assert all(e > s and (s * H) % 16 == 0 for s, e in b)
    with pytest.raises(ValueError):
        ex.chunk_bounds(4, 8, 0)


def _gather_rank(rank, world, port, q, R, H, chunks):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from residual_sp_rs_gb300 import sp_exchange as ex
    d_sum = (1000.0 * rank + torch.arange(R, dtype=torch.float64)[:, None]) * torch.ones(R, H, dtype=torch.float64)
    grad = torch.full((world * R, H), float("nan"), dtype=torch.float64)
    works = [ex.post_chunk_gather(d_sum, grad, R, b, e) for b, e in ex.chunk_bounds(R, H, chunks)]
    for w in works:
        w.wait()
    whole = ex.gather_partial_grads(d_sum)
    q.put((rank, grad.numpy(), whole.numpy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,chunks", [(2, 3), (4, 4)])
def test_chunked_gather_assembles_the_partials_gradient(world, chunks):
    """The backward of the reduce-scatter gathered chunk by chunk, as the
    pipelined backward posts it, equals the whole shard's all-gather."""
    R, H = 10, 8
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gather_rank, args=(r, world, port, q, R, H, chunks)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = np.repeat(1000.0 * np.arange(world), R)[:, None] + np.tile(np.arange(R, dtype=np.float64), world)[:, None]
    for _, grad, whole in got:
        assert np.array_equal(grad, whole)
        assert np.array_equal(grad, expect * np.ones(H))
