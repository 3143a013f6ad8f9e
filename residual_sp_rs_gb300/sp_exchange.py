"""The exchange steps of sequence parallelism across ranks (torch.distributed).

On one GPU the fused forward reads all T row-parallel partials from local
memory.  Across T ranks, rank t holds only its own partial P_t (a full
[S,B,H] tensor) and owns sequence shard j = t.  These helpers are the
communication around the fused kernels; all arithmetic stays in libspfuse:

* ``exchange_partials``: the exchange half of the reduce-scatter.  Rank j
  receives block j (its sequence shard's rows) of every rank's partial, and
  sends block t of its own partial to rank t -- (T-1)/T of the partial per
  rank, the volume of the ring reduce-scatter (MiniMind-tron ch.3, §3.2.3).
  The reduce half is the fused forward, which sums the received blocks in
  rank order.
* ``forward_from_shard_rows``: calls the fused forward with the received
  blocks.  The call addresses every partial by global row (shard j starts at
  row j*R), so each block is passed as the address its row 0 would have.
* ``forward_pipelined``: the same exchange split into pipeline chunks of the
  shard's rows ("Sequence Parallel" notes, communication-computation
  overlap: the reduce-scatter in chunks, 4 by default).  Every chunk is
  pulled from the peers by grouped point-to-point transfers posted at once;
  the fused forward of a chunk's rows (``sp_rs_dropout_residual_norm_fwd_rows``)
  runs as soon as that chunk has landed, while the later chunks are still in
  flight.  A rank's own partial is read in place: only (T-1)/T of the shard's
  rows travel.
* ``backward_pipelined``: the backward in the same chunks, each chunk's
  d_sum all-gathered (``post_chunk_gather``) while the next chunk computes
  (``sp_rs_dropout_residual_norm_bwd_rows``, dgamma/dbeta accumulated over
  the chunks in order).
* ``allreduce_norm_grads``: dgamma/dbeta are per-shard partial sums; the
  replicated norm weights need their sum over ranks (MiniMind-tron ch.3,
  §3.4.2.1).
* ``gather_partial_grads``: the backward of the reduce-scatter is an
  all-gather: every row-parallel partial's gradient is the concatenation of
  the ranks' d_sum shards (MiniMind-tron ch.3, §3.3.3.1).

The collectives run on the process group's backend (NCCL for CUDA tensors,
gloo for CPU tensors in the tests).
"""
from __future__ import annotations

import math

import torch
import torch.distributed as dist

from . import ops


def exchange_partials(partial: torch.Tensor, group=None) -> torch.Tensor:
    """partial: this rank's full partial [S, B, H] (or [S*B, H]).  Returns
    [T, R, H]: block t = rows [j*R, (j+1)*R) of rank t's partial, j = this
    rank, R = S*B/T."""
    T = dist.get_world_size(group)
    H = partial.shape[-1]
    flat = partial.contiguous().view(-1, H)
    if flat.shape[0] % T:
        raise ValueError("S*B must split evenly into T sequence shards")
    R = flat.shape[0] // T
    out = torch.empty((T, R, H), dtype=partial.dtype, device=partial.device)
    # chunk t of the input goes to rank t; chunk t of the output comes from rank t
    dist.all_to_all_single(out.view(-1, H), flat, group=group)
    return out


def forward_from_shard_rows(desc, blocks: torch.Tensor, residual, gamma, beta, h_out, y_out,
                            mask_out, rstd_out, mean_out, stream=None) -> None:
    """The fused forward of shard desc.j from its rows of each partial:
    blocks [T, R, H] as returned by exchange_partials (contiguous, each
    block 16-byte aligned)."""
    T, R, H = blocks.shape
    if desc.T != T or desc.H != H or desc.R != R or max(1, desc.nshards) != 1:
        raise ValueError("blocks do not match the descriptor's single shard")
    if not blocks.is_contiguous():
        raise ValueError("blocks must be contiguous: each block is passed by its base address")
    row_bytes = H * blocks.element_size()
    base = [blocks[t].data_ptr() - desc.j * R * row_bytes for t in range(T)]
    ops.sp_rs_dropout_residual_norm_fwd(desc, base, residual, gamma, beta, h_out, y_out, mask_out,
                                        rstd_out, mean_out, stream)


def allreduce_norm_grads(dgamma: torch.Tensor, dbeta: torch.Tensor | None = None, group=None) -> None:
    """Sum the per-shard dgamma (and dbeta) over the ranks, in place."""
    dist.all_reduce(dgamma, op=dist.ReduceOp.SUM, group=group)
    if dbeta is not None:
        dist.all_reduce(dbeta, op=dist.ReduceOp.SUM, group=group)


def gather_partial_grads(d_sum: torch.Tensor, group=None) -> torch.Tensor:
    """d_sum: this rank's [R, H] gradient of its shard's reduced sum.
    Returns the [T*R, H] gradient of every row-parallel partial."""
    T = dist.get_world_size(group)
    R, H = d_sum.shape
    out = torch.empty((T * R, H), dtype=d_sum.dtype, device=d_sum.device)
    dist.all_gather_into_tensor(out, d_sum.contiguous(), group=group)
    return out


def chunk_bounds(R: int, H: int, chunks: int = 4) -> list[tuple[int, int]]:
    """Row ranges [b, e) that split a shard's R rows into at most `chunks`
    non-empty pipeline chunks of near-equal size, each start a multiple of
    16 / gcd(H, 16) rows so that it keeps the 16-byte alignment of the mask
    bytes (H per row)."""
    if R < 0 or H <= 0 or chunks < 1:
        raise ValueError("need R >= 0, H > 0 and at least one chunk")
    unit = 16 // math.gcd(H, 16)
    cuts = sorted({min(R, -(-(c * R // chunks) // unit) * unit) for c in range(chunks)} | {R})
    return [(b, e) for b, e in zip(cuts[:-1], cuts[1:]) if e > b]


def pull_chunks(partial: torch.Tensor, bounds, group=None):
    """Post the exchange of every chunk at once.  partial: this rank's full
    partial [S, B, H] (or [S*B, H]); bounds: row ranges of the shard as from
    chunk_bounds.  Returns (recv, works): recv[c] is a [T, e-b, H] buffer
    whose block t (t != this rank) receives rows [j*R + b, j*R + e) of rank
    t's partial, j = this rank; block j is left unused (the rank's own rows
    stay in `partial`).  works[c] are the chunk's transfer handles: wait on
    them before using recv[c]."""
    T = dist.get_world_size(group)
    j = dist.get_rank(group)
    H = partial.shape[-1]
    flat = partial.contiguous().view(-1, H)
    if flat.shape[0] % T:
        raise ValueError("S*B must split evenly into T sequence shards")
    R = flat.shape[0] // T
    recv, works = [], []
    for b, e in bounds:
        if not 0 <= b < e <= R:
            raise ValueError("chunk bounds must be non-empty ranges inside the shard")
        buf = torch.empty((T, e - b, H), dtype=partial.dtype, device=partial.device)
        p2p = []
        for t in range(T):
            if t == j:
                continue
            # to rank t: my partial's rows of shard t; from rank t: its rows of shard j
            p2p.append(dist.P2POp(dist.isend, flat[t * R + b:t * R + e], t, group=group))
            p2p.append(dist.P2POp(dist.irecv, buf[t], t, group=group))
        works.append(dist.batch_isend_irecv(p2p) if p2p else [])
        recv.append(buf)
    return recv, works


def chunk_partial_bases(own: torch.Tensor, recv_chunk: torch.Tensor, j: int, R: int, b: int) -> list:
    """The partial addresses of one chunk's fused forward: the call addresses
    partial t by global row, so this rank's own partial `own` ([S*B, H],
    contiguous) is passed as is, and the chunk buffer block recv_chunk[t],
    which holds rows [j*R + b, j*R + e) of partial t, as the address its
    global row 0 would have."""
    T, _, H = recv_chunk.shape
    if not (own.is_contiguous() and recv_chunk.is_contiguous()):
        raise ValueError("the partial and the chunk buffer must be contiguous")
    row_bytes = H * recv_chunk.element_size()
    return [own.data_ptr() if t == j else recv_chunk[t].data_ptr() - (j * R + b) * row_bytes
            for t in range(T)]


def forward_pipelined(desc, partial: torch.Tensor, residual, gamma, beta, h_out, y_out, mask_out,
                      rstd_out, mean_out, chunks: int = 4, group=None):
    """The fused forward of this rank's shard (desc.j = rank, desc.T = world
    size, one shard) from every rank's full partial, the exchange pipelined
    in chunks.  The kernels go to the current stream, which each chunk's
    transfers are ordered with.  Returns the chunk receive buffers: keep them
    alive until the forward has run."""
    T = dist.get_world_size(group)
    j = dist.get_rank(group)
    H = partial.shape[-1]
    own = partial.contiguous().view(-1, H)
    R = own.shape[0] // T
    if desc.T != T or desc.j != j or desc.H != H or desc.R != R or max(1, desc.nshards) != 1:
        raise ValueError("the descriptor must describe this rank's single shard")
    bounds = chunk_bounds(R, H, chunks)
    recv, works = pull_chunks(own, bounds, group)
    for (b, e), buf, ws in zip(bounds, recv, works):
        for w in ws:
            w.wait()
        ops.sp_rs_dropout_residual_norm_fwd_rows(desc, b, e - b, chunk_partial_bases(own, buf, j, R, b),
                                                 residual, gamma, beta, h_out, y_out, mask_out, rstd_out,
                                                 mean_out)
    return recv


def post_chunk_gather(d_sum: torch.Tensor, grad: torch.Tensor, R: int, b: int, e: int, group=None):
    """Post the all-gather of rows [b, e) of this rank's d_sum shard ([R, H])
    into rows [t*R + b, t*R + e) of grad ([T*R, H], the gradient of every
    row-parallel partial) for every rank t.  Returns the work handle."""
    T = dist.get_world_size(group)
    outs = [grad[t * R + b:t * R + e] for t in range(T)]
    return dist.all_gather(outs, d_sum[b:e], group=group, async_op=True)


def backward_pipelined(desc, dy, dh_out, h_saved, gamma, mask, rstd, mean, d_residual, d_sum, dgamma,
                       dbeta, workspace, chunks: int = 4, group=None):
    """The fused backward of this rank's shard (desc.j = rank, desc.T = world
    size, one shard) in pipeline chunks of its rows: as soon as a chunk's
    d_sum rows are computed, their all-gather -- the backward of the
    reduce-scatter (MiniMind-tron ch.3, §3.3.3.1) -- is posted, and it runs
    while the next chunk is computed.  The chunks accumulate dgamma/dbeta in
    order (this shard's sums; allreduce_norm_grads adds them over ranks).
    The kernels go to the current stream.  Returns (grad, works): grad is the
    [T*R, H] gradient of every row-parallel partial, complete once every work
    handle has been waited on."""
    T = dist.get_world_size(group)
    j = dist.get_rank(group)
    R, H = desc.R, desc.H
    if desc.T != T or desc.j != j or max(1, desc.nshards) != 1:
        raise ValueError("the descriptor must describe this rank's single shard")
    bounds = chunk_bounds(R, H, chunks)
    grad = torch.empty((T * R, H), dtype=d_sum.dtype, device=d_sum.device)
    works = []
    if not bounds:  # no rows: dgamma/dbeta are zeros
        ops.sp_rs_dropout_residual_norm_bwd_rows(desc, 0, 0, False, dy, dh_out, h_saved, gamma, mask, rstd,
                                                 mean, d_residual, d_sum, dgamma, dbeta, workspace)
    for c, (b, e) in enumerate(bounds):
        ops.sp_rs_dropout_residual_norm_bwd_rows(desc, b, e - b, c > 0, dy, dh_out, h_saved, gamma, mask, rstd,
                                                 mean, d_residual, d_sum, dgamma, dbeta, workspace)
        works.append(post_chunk_gather(d_sum, grad, R, b, e, group))
    return grad, works
