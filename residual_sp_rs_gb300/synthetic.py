"""Seeded synthetic inputs for the SP-region workloads.

This module draws inputs and nothing else: it holds none of the arithmetic
of the method (no reduction, mask, dropout, residual add or norm), so both
the CUDA path and the CPU oracle can take their inputs from it.

Shapes and value distributions follow the workloads the SP pages measure
(MiniMind-tron ch.4 "Sequence Parallelism: memory bounds, async communication
and recompute", §4.1: S=2048, micro-batch B=2, H=768, TP=2, bf16) plus a tiny
fp32 case, a GPT-style LayerNorm case, a large-hidden stress case and the
sp2hp/hp2sp layout case.  Row-parallel partial outputs are small
(N(0, 0.02^2)), the residual stream is N(0, 1), gamma is near 1.

Every tensor is drawn in fp32 from a seeded ``torch.Generator`` on the
requested device and cast to the activation dtype with round-to-nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tensor/sequence parallel group size
    S: int            # full sequence length
    B: int            # micro-batch
    H: int            # hidden size
    dtype: str        # "bf16" or "f32"
    norm: str         # "rms" or "ln"
    p: float          # dropout probability
    eps: float
    seed: int         # Philox key of the dropout mask
    p_std: float      # std of the row-parallel partials P_t
    res_std: float    # std of the residual stream
    gamma_lo: float   # gamma ~ U(gamma_lo, gamma_hi)
    gamma_hi: float
    beta_std: float   # beta ~ N(0, beta_std^2) (LayerNorm only)
    input_seed: int   # torch.Generator seed of the inputs

    @property
    def R(self) -> int:
        """Token rows per sequence shard, (S/T)*B."""
        return (self.S // self.T) * self.B

    @property
    def tokens(self) -> int:
        return self.S * self.B

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # tiny RMSNorm forward, fp32: 8 tokens x 2 batch per shard
    "tiny_rms_f32": Workload("tiny_rms_f32", 2, 16, 2, 64, "f32", "rms", 0.1, 1e-6, 0,
                             1.0, 1.0, 0.5, 1.5, 0.0, 1000),
    # the pages' benchmark shape
    "pages_rms_bf16": Workload("pages_rms_bf16", 2, 2048, 2, 768, "bf16", "rms", 0.1, 1e-6, 0,
                               0.02, 1.0, 0.9, 1.1, 0.0, 1001),
    # GPT-style LayerNorm, 512 tokens per shard
    "gpt_ln_bf16": Workload("gpt_ln_bf16", 8, 4096, 1, 4096, "bf16", "ln", 0.1, 1e-5, 0,
                            0.02, 1.0, 0.9, 1.1, 0.01, 1002),
    # large-hidden stress, RMSNorm (run at p = 0.1 and p = 0.0)
    "large_rms_bf16": Workload("large_rms_bf16", 8, 8192, 2, 8192, "bf16", "rms", 0.1, 1e-6, 0,
                               0.02, 1.0, 0.9, 1.1, 0.0, 1003),
}


@dataclass(frozen=True)
class LayoutWorkload:
    name: str
    T: int
    N: int       # num_tokens
    H: int
    dtype: str
    std: float
    input_seed: int


LAYOUT = LayoutWorkload("layout_bf16", 4, 16384, 4096, "bf16", 1.0, 1004)


def torch_dtype(dtype: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device, dtype):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch_dtype(dtype))


def fwd_inputs(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """partials: T tensors [S,B,H]; residual: [S,B,H] (the residual stream of
    the whole sequence; shard j is rows [j*R, (j+1)*R) of its [S*B, H] view);
    gamma, beta: [H] in the activation dtype (beta None for RMSNorm)."""
    g = _gen(device, w.input_seed if seed is None else seed)
    shape = (w.S, w.B, w.H)
    partials = [_normal(shape, w.p_std, g, device, w.dtype) for _ in range(w.T)]
    residual = _normal(shape, w.res_std, g, device, w.dtype)
    u = torch.rand((w.H,), generator=g, device=device, dtype=torch.float32)
    gamma = (u * (w.gamma_hi - w.gamma_lo) + w.gamma_lo).to(torch_dtype(w.dtype))
    beta = _normal((w.H,), w.beta_std, g, device, w.dtype) if w.norm == "ln" else None
    return dict(partials=partials, residual=residual, gamma=gamma, beta=beta)


def upstream_grads(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """dy (gradient of the norm output) and dh_out (gradient arriving along
    the residual stream), both N(0,1) [S,B,H]."""
    g = _gen(device, (w.input_seed if seed is None else seed) + 7919)
    shape = (w.S, w.B, w.H)
    return dict(dy=_normal(shape, 1.0, g, device, w.dtype),
                dh_out=_normal(shape, 1.0, g, device, w.dtype))


def saved_activations(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """Stand-ins for what a forward saves, for backward tests at full size:
    h ~ N(0,1) [S,B,H] in the activation dtype and a 0/1 byte mask with keep
    probability 1-p.  (Row statistics are not drawn here: they are a function
    of h that the caller computes.)"""
    g = _gen(device, (w.input_seed if seed is None else seed) + 104729)
    shape = (w.S, w.B, w.H)
    h = _normal(shape, 1.0, g, device, w.dtype)
    mask = (torch.rand(shape, generator=g, device=device) >= w.p).to(torch.uint8)
    return dict(h=h, mask=mask)


def layout_input(lw: LayoutWorkload = LAYOUT, device="cpu", seed: int | None = None,
                 N: int | None = None, H: int | None = None) -> torch.Tensor:
    g = _gen(device, lw.input_seed if seed is None else seed)
    return _normal((N or lw.N, H or lw.H), lw.std, g, device, lw.dtype)


def to_storage(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy with the exact bytes: bf16 -> uint16 bit patterns."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def from_storage(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Inverse of to_storage (CPU tensor)."""
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    if dtype == "f32":
        return torch.from_numpy(a.astype(np.float32, copy=True))
    raise ValueError(dtype)
