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
