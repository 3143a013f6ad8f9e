"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Inputs come from residual_sp_rs_gb300.synthetic (seeded, shared by both
sides); expected values come only from the oracle.  Small and mid-size
workloads are compared element by element; the large-hidden workload is
compared on sampled rows (all outputs), with the dropout mask checked over
every element.
"""
import numpy as np
import pytest
import torch

import oracle
from residual_sp_rs_gb300 import ops, synthetic as syn
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from residual_sp_rs_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _np(t):
    return syn.to_storage(t)


def _desc(w, j, nshards=1, p=None, seed=None):
    return ops.make_desc(w.T, j, w.S, w.B, w.H, w.dtype, w.norm, w.p if p is None else p, w.eps,
                         w.seed if seed is None else seed, nshards)


def _oracle_problem(w, j, nshards=1, p=None, seed=None):
    pf = float(np.float32(w.p if p is None else p))
    return oracle.problem(w.T, j, w.S, w.B, w.H, w.dtype, w.norm, pf, float(np.float32(w.eps)),
                          w.seed if seed is None else seed, nshards)


def _gpu_fwd(w, inp, j, nshards=1, p=None, seed=None, with_mask=True):
    d = _desc(w, j, nshards, p, seed)
    R = w.R
    res = inp["residual"].view(w.S * w.B, w.H)[j * R:(j + nshards) * R]
    out = ops.forward(d, inp["partials"], res, inp["gamma"], inp["beta"])
    if not with_mask and d.p == 0:
        assert out["mask"] is None
    return out


def _host(out):
    return {k: (None if v is None else _np(v)) for k, v in out.items()}


def _full_fwd_check(w, inp, j, nshards=1, p=None, seed=None):
    out = _gpu_fwd(w, inp, j, nshards, p, seed)
    torch.cuda.synchronize()
    pr = _oracle_problem(w, j, nshards, p, seed)
    R = w.R
    res = _np(inp["residual"]).reshape(w.S * w.B, w.H)[j * R:(j + nshards) * R]
    parts = [_np(t) for t in inp["partials"]]
    orc = oracle.fwd(pr, parts, res, _np(inp["gamma"]),
                     None if inp["beta"] is None else _np(inp["beta"]), w.dtype)
    g = _host(out)
    if g["mask"] is None:
        g["mask"] = np.ones_like(orc["mask"])
    if g["mean"] is None:
        g["mean"] = np.zeros(len(orc["rstd"]))
    parity.compare_fwd(w.dtype, w.norm, g, orc, pr, _np(inp["gamma"]),
                       None if inp["beta"] is None else _np(inp["beta"]))
    return out, orc


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("j", [0, 1])
def test_fwd_tiny_rms_f32(j):
    w = syn.WORKLOADS["tiny_rms_f32"]
    inp = syn.fwd_inputs(w, DEV)
    _full_fwd_check(w, inp, j)


def test_fwd_pages_shape_bf16_all_shards_and_single():
    w = syn.WORKLOADS["pages_rms_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    both, _ = _full_fwd_check(w, inp, 0, nshards=2)
    for j in range(2):
        one, _ = _full_fwd_check(w, inp, j)
        R = w.R
        for k in ["h", "y", "mask", "rstd"]:   # one launch over both shards == two launches
            assert torch.equal(one[k], both[k][j * R:(j + 1) * R] if k != "rstd"
                               else both[k][j * R:(j + 1) * R])


def test_fwd_gpt_layernorm_every_shard():
    w = syn.WORKLOADS["gpt_ln_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    for j in range(w.T):
        _full_fwd_check(w, inp, j)


def _sample_rows(R, n, seed):
    rng = np.random.default_rng(seed)
    rows = set([0, 1, R - 2, R - 1]) | set(int(x) for x in rng.integers(0, R, n))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("p", [0.1, 0.0])
def test_fwd_large_hidden_every_shard_sampled(p):
    w = syn.WORKLOADS["large_rms_bf16"].with_(p=p)
    inp = syn.fwd_inputs(w, DEV)
    R, H = w.R, w.H
    gam = _np(inp["gamma"])
    flat_parts = [t.view(w.S * w.B, H) for t in inp["partials"]]
    flat_res = inp["residual"].view(w.S * w.B, H)
    for j in range(w.T):
        out = _gpu_fwd(w, inp, j)
        torch.cuda.synchronize()
        if p > 0:   # the whole mask, bit-exact
            ref = oracle.mask_range(w.seed, float(np.float32(p)), j * R * H, R * H)
            assert np.array_equal(_np(out["mask"]).ravel(), ref), f"mask shard {j}"
        rows = _sample_rows(R, 40, 100 + j)
        grows = j * R + rows
        idx = torch.from_numpy(grows).to(DEV)
        prows = [_np(fp.index_select(0, idx)) for fp in flat_parts]
        pr = _oracle_problem(w, j)
        orc = oracle.fwd_rows(pr, grows, prows, _np(flat_res.index_select(0, idx)), gam, None, w.dtype)
        ridx = torch.from_numpy(rows).to(DEV)
        g = dict(h=_np(out["h"].index_select(0, ridx)), y=_np(out["y"].index_select(0, ridx)),
                 mask=(_np(out["mask"].index_select(0, ridx)) if out["mask"] is not None
                       else np.ones((len(rows), H), np.uint8)),
                 rstd=_np(out["rstd"][ridx]), mean=np.zeros(len(rows)))
        parity.compare_fwd(w.dtype, w.norm, g, orc, pr, gam)
        del out


@pytest.mark.parametrize("case", [
    # (T, S, B, H, dtype, norm, p): ragged tails, minimum/maximum widths, T = 1, odd T
    (3, 21, 1, 776, "bf16", "rms", 0.1),
    (3, 21, 1, 776, "bf16", "ln", 0.3),
    (1, 5, 3, 8, "bf16", "rms", 0.5),
    (8, 16, 3, 64, "bf16", "ln", 0.1),
    (2, 6, 1, 16384, "bf16", "rms", 0.1),
    (5, 10, 2, 4104, "bf16", "ln", 0.2),
    (2, 4, 5, 8192, "f32", "ln", 0.1),
    (4, 8, 3, 12, "f32", "rms", 0.7),
    (7, 14, 1, 1032, "f32", "ln", 0.0),
    # rows too long for a whole-row ring stage: column-chunk stages, one ragged
    (8, 16, 1, 8200, "bf16", "rms", 0.1),
    (8, 8, 2, 8192, "bf16", "ln", 0.1),
    (4, 8, 2, 12288, "bf16", "rms", 0.5),
])
def test_fwd_edge_shapes(case):
    T, S, B, H, dt, nm, p = case
    w = syn.Workload("edge", T, S, B, H, dt, nm, p, 1e-5, 0x0123456789ABCDEF, 0.5, 1.0, 0.5, 1.5, 0.1,
                     4242 + H)
    inp = syn.fwd_inputs(w, DEV)
    for j in sorted({0, T - 1}):
        _full_fwd_check(w, inp, j)
    _full_fwd_check(w, inp, 0, nshards=T)
    if T >= 3:   # a run of shards from the middle of the group
        _full_fwd_check(w, inp, 1, nshards=T - 2)


def test_fwd_p0_without_mask_is_exact_residual_add():
    w = syn.WORKLOADS["pages_rms_bf16"].with_(p=0.0)
    inp = syn.fwd_inputs(w, DEV)
    d = _desc(w, 1)
    R = w.R
    res = inp["residual"].view(-1, w.H)[R:2 * R]
    out = ops.forward(d, inp["partials"], res, inp["gamma"])
    assert out["mask"] is None
    torch.cuda.synchronize()
    pr = _oracle_problem(w, 1)
    orc = oracle.fwd(pr, [_np(t) for t in inp["partials"]], _np(res), _np(inp["gamma"]), None, "bf16")
    g = _host(out)
    g["mask"] = np.ones_like(orc["mask"])
    g["mean"] = np.zeros(R)
    parity.compare_fwd("bf16", "rms", g, orc, pr, _np(inp["gamma"]))


@pytest.mark.parametrize("name,j,nshards", [("gpt_ln_bf16", 2, 3), ("gpt_ln_bf16", 5, 3)])
def test_fwd_run_of_middle_shards(name, j, nshards):
    """Shards j .. j+nshards-1 from the middle of the group in one call: the
    global row offset j*R keys the partial rows and the mask."""
    w = syn.WORKLOADS[name]
    inp = syn.fwd_inputs(w, DEV)
    _full_fwd_check(w, inp, j, nshards)


def test_fwd_from_shard_rows_equals_full_tensor_call():
    """A rank that holds only its shard's rows of each partial (after the
    reduce-scatter's exchange) gets the same forward, bit for bit, as the
    call that reads them out of the full tensors."""
    from residual_sp_rs_gb300 import sp_exchange as ex
    w = syn.WORKLOADS["pages_rms_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    R, H = w.R, w.H
    for j in range(w.T):
        d = _desc(w, j)
        ref = _gpu_fwd(w, inp, j)
        blocks = torch.stack([p.view(-1, H)[j * R:(j + 1) * R] for p in inp["partials"]]).contiguous()
        res = inp["residual"].view(-1, H)[j * R:(j + 1) * R]
        out = {k: torch.empty_like(v) for k, v in ref.items() if v is not None}
        ex.forward_from_shard_rows(d, blocks, res, inp["gamma"], None, out["h"], out["y"], out["mask"],
                                   out["rstd"], None)
        torch.cuda.synchronize()
        for k in out:
            assert torch.equal(out[k], ref[k]), (j, k)


def _sentinel_like(ref):
    """Outputs shaped like `ref`, filled with values no forward writes (-3.0; mask byte 7)."""
    return {k: torch.full_like(v, 7 if v.dtype == torch.uint8 else -3.0) for k, v in ref.items()
            if v is not None}


def _fwd_rows_call(w, inp, d, j, b, count, out, partials=None):
    R = w.R
    res = inp["residual"].view(w.S * w.B, w.H)[j * R:]
    ops.sp_rs_dropout_residual_norm_fwd_rows(d, b, count, inp["partials"] if partials is None else partials,
                                             res, inp["gamma"], inp["beta"], out["h"], out["y"],
                                             out["mask"], out["rstd"], out.get("mean"))


@pytest.mark.parametrize("name,j,nshards,cuts", [
    ("pages_rms_bf16", 0, 2, [0, 1, 1000, 2049, 4096]),   # crosses the shard boundary at 2048
    ("gpt_ln_bf16", 3, 1, [0, 129, 130, 512]),
    ("tiny_rms_f32", 1, 1, [0, 3, 11, 16]),
])
def test_fwd_rows_chunks_equal_the_full_call(name, j, nshards, cuts):
    """The forward run chunk by chunk over row ranges (the receiving side of
    a reduce-scatter in pipeline chunks) writes, bit for bit, what one call
    over all the rows writes: the mask is keyed by the global element index."""
    w = syn.WORKLOADS[name]
    inp = syn.fwd_inputs(w, DEV)
    ref = _gpu_fwd(w, inp, j, nshards)
    d = _desc(w, j, nshards)
    out = _sentinel_like(ref)
    for b, e in zip(cuts[:-1], cuts[1:]):
        _fwd_rows_call(w, inp, d, j, b, e - b, out)
    torch.cuda.synchronize()
    for k in out:
        assert torch.equal(out[k], ref[k]), k


def test_fwd_rows_chunks_without_mask_equal_the_full_call():
    """Row ranges with no stored mask: the keep decisions come from the
    global element index, so h and y match the full call's bit for bit."""
    w = syn.WORKLOADS["pages_rms_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    d = _desc(w, 0, 2)
    ref = _gpu_fwd(w, inp, 0, 2)
    out = _sentinel_like(ref)
    out["mask"] = None
    for b, e in zip([0, 777, 2048], [777, 2048, 4096]):
        _fwd_rows_call(w, inp, d, 0, b, e - b, out)
    torch.cuda.synchronize()
    for k in ("h", "y", "rstd"):
        assert torch.equal(out[k], ref[k]), k


def test_fwd_rows_writes_only_its_range():
    w = syn.WORKLOADS["pages_rms_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    ref = _gpu_fwd(w, inp, 1)
    d = _desc(w, 1)
    out = _sentinel_like(ref)
    b, e = 700, 1301
    _fwd_rows_call(w, inp, d, 1, b, e - b, out)
    _fwd_rows_call(w, inp, d, 1, 5, 0, out)   # an empty range launches nothing
    torch.cuda.synchronize()
    blank = _sentinel_like(ref)
    for k in out:
        assert torch.equal(out[k][b:e], ref[k][b:e]), k
        assert torch.equal(out[k][:b], blank[k][:b]) and torch.equal(out[k][e:], blank[k][e:]), k


def test_pipelined_chunks_from_received_rows_equal_the_full_call():
    """Rank j of the pipelined exchange, emulated on one GPU: its own partial
    in place and each chunk's rows of the other partials in a chunk buffer,
    passed by the addresses chunk_partial_bases derives."""
    from residual_sp_rs_gb300 import sp_exchange as ex
    w = syn.WORKLOADS["pages_rms_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    R, H, T = w.R, w.H, w.T
    for j in range(T):
        ref = _gpu_fwd(w, inp, j)
        d = _desc(w, j)
        own = inp["partials"][j].view(-1, H)
        out = _sentinel_like(ref)
        bufs = []
        for b, e in ex.chunk_bounds(R, H, 4):
            buf = torch.empty((T, e - b, H), device=DEV, dtype=own.dtype)
            for t in range(T):
                if t != j:
                    buf[t].copy_(inp["partials"][t].view(-1, H)[j * R + b:j * R + e])
            bufs.append(buf)
            _fwd_rows_call(w, inp, d, j, b, e - b, out, ex.chunk_partial_bases(own, buf, j, R, b))
        torch.cuda.synchronize()
        for k in out:
            assert torch.equal(out[k], ref[k]), (j, k)


def _near_midpoint_inputs(R2, H, p, seed=11):
    """Seeded forward inputs for T = 2 whose kept elements put
    E = residual + (P0 + P1)/(1 - p) within 40 fp32 ulps of a bf16 rounding
    midpoint (P1 = 0, so the sum is P0 exactly): random bf16 candidates,
    kept by the distance of fp32(E) to the midpoint of its bf16 interval.
    Every 8th row instead nearly cancels against the residual
    (|E| < 2^-12 |residual|)."""
    rng = np.random.default_rng(seed)
    n = R2 * H

    def bf16(x):  # round float64 -> bf16 bits (to nearest even via fp32) and back
        b = np.asarray(x, np.float32).view(np.uint32)
        b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
        return b, (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    s = 1.0 / (1.0 - np.float64(np.float32(p)))
    p0s, ress = [], []
    need = n
    while need > 0:
        m = 1 << 20
        b0, v0 = bf16(rng.standard_normal(m) * 2.0 ** rng.integers(-4, 5, m))
        br, vr = bf16(rng.standard_normal(m) * 2.0 ** rng.integers(-4, 5, m))
        e32 = (vr + v0 * s).astype(np.float32)
        low = (e32.view(np.uint32) & 0xFFFF).astype(np.int64)
        hit = (np.abs(low - 0x8000) <= 40) & (v0 != 0)
        p0s.append(b0[hit][:need])
        ress.append(br[hit][:need])
        need -= int(hit.sum())
    P0 = np.concatenate(p0s)[:n].reshape(R2, H)
    RES = np.concatenate(ress)[:n].reshape(R2, H)
    # cancellation rows: residual = -bf16(P0*s) (+ one bf16 step), so E is tiny
    v0 = (P0[::8].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bc, _ = bf16(-v0 * s)
    bc = bc + (rng.integers(0, 2, bc.shape)).astype(np.uint16)
    RES[::8] = bc
    return P0, np.zeros_like(P0), RES


def test_fwd_h_rounding_near_bf16_midpoints():
    """h = residual + sum/(1-p) rounded once to bf16 must be the correctly
    rounded value also where it lies within a few fp32 ulps of a bf16
    rounding midpoint, and where the residual add cancels."""
    T, S, B, H, p = 2, 32, 2, 768, 0.1
    w = syn.WORKLOADS["pages_rms_bf16"].with_(S=S, B=B)
    R2 = S * B
    P0, P1, RES = _near_midpoint_inputs(R2, H, p)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)
    gamma = torch.ones(H, device=DEV, dtype=torch.bfloat16)
    inp = {"partials": [to_dev(P0), to_dev(P1)], "residual": to_dev(RES), "gamma": gamma, "beta": None}
    d = _desc(w, 0, 2)
    out = ops.forward(d, inp["partials"], inp["residual"], gamma, None)
    torch.cuda.synchronize()
    pr = _oracle_problem(w, 0, 2)
    orc = oracle.fwd(pr, [P0, P1], RES, _np(gamma), None, "bf16")
    g = _np(out["h"])
    kept = orc["mask"] == 1
    assert kept.mean() > 0.8
    assert np.array_equal(g, orc["h"]), int((g != orc["h"]).sum())
    assert np.array_equal(_np(out["mask"]), orc["mask"])


@pytest.mark.parametrize("T,H", [(2, 768), (4, 12288), (2, 16384)])   # whole-row ring, column chunks, registers
def test_fwd_exact_ties_round_half_to_even(T, H):
    """Every kept element an exact bf16 midpoint (p = 0.5): h must be the
    neighbour with the even mantissa in each forward kernel, as in the oracle."""
    S, B = 4 * T, 2
    w = syn.WORKLOADS["pages_rms_bf16"].with_(T=T, S=S, B=B, H=H, p=0.5, seed=5)
    P0, R, tie = parity.tie_inputs(S * B, H, seed=H)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)
    gamma = torch.ones(H, device=DEV, dtype=torch.bfloat16)
    parts = [P0] + [np.zeros_like(P0)] * (T - 1)
    out = ops.forward(_desc(w, 0, T), [to_dev(p) for p in parts], to_dev(R), gamma, None)
    torch.cuda.synchronize()
    orc = oracle.fwd(_oracle_problem(w, 0, T), parts, R, _np(gamma), None, "bf16")
    kept = orc["mask"] == 1
    assert np.array_equal(_np(out["mask"]), orc["mask"])
    assert np.array_equal(orc["h"], np.where(kept, tie, R))
    assert np.array_equal(_np(out["h"]), orc["h"]), int((_np(out["h"]) != orc["h"]).sum())


def test_fwd_empty_rows_is_a_no_op():
    w = syn.WORKLOADS["pages_rms_bf16"].with_(S=0)
    d = _desc(w, 0)
    z = torch.empty((0, w.H), device=DEV, dtype=torch.bfloat16)
    g = torch.ones(w.H, device=DEV, dtype=torch.bfloat16)
    ops.sp_rs_dropout_residual_norm_fwd(d, [z, z], z, g, None, z, z,
                                        torch.empty((0, w.H), device=DEV, dtype=torch.uint8),
                                        torch.empty(0, device=DEV), None)
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------

def _bwd_inputs_from_oracle_fwd(w, j, nshards, inp, grads):
    """Saved activations for the backward = the ORACLE forward's outputs."""
    pr = _oracle_problem(w, j, nshards)
    R = w.R
    res = _np(inp["residual"]).reshape(-1, w.H)[j * R:(j + nshards) * R]
    orc = oracle.fwd(pr, [_np(t) for t in inp["partials"]], res, _np(inp["gamma"]),
                     None if inp["beta"] is None else _np(inp["beta"]), w.dtype)
    tdt = syn.torch_dtype(w.dtype)
    dev = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a)).to(DEV) if dt is None else \
        syn.from_storage(a, dt).to(DEV)
    saved = dict(h=dev(orc["h"], w.dtype), mask=dev(orc["mask"]),
                 rstd=dev(orc["rstd"].astype(np.float32)), mean=dev(orc["mean"].astype(np.float32)))
    dy = grads["dy"].view(-1, w.H)[j * R:(j + nshards) * R]
    dh = grads["dh_out"].view(-1, w.H)[j * R:(j + nshards) * R]
    return pr, orc, saved, dy, dh


def _check_bwd(w, pr, saved_np, dy_np, dh_np, gamma_np, mask_np, gout):
    orc = oracle.bwd(pr, dy_np, dh_np, saved_np, gamma_np, mask_np, w.dtype)
    g = _host(gout)
    parity.check_act("d_residual", w.dtype, g["d_res"], orc["dres_exact"])
    parity.check_act("d_sum", w.dtype, g["d_sum"], orc["dsum_exact"])
    parity.check_reduction("dgamma", g["dgamma"], orc["dgamma"])
    if w.norm == "ln":
        parity.check_reduction("dbeta", g["dbeta"], orc["dbeta"])


@pytest.mark.parametrize("name,j,nshards", [("tiny_rms_f32", 0, 1), ("tiny_rms_f32", 1, 1),
                                            ("pages_rms_bf16", 0, 1), ("pages_rms_bf16", 0, 2),
                                            ("gpt_ln_bf16", 3, 1), ("gpt_ln_bf16", 0, 8),
                                            ("gpt_ln_bf16", 2, 3)])   # a run of shards from the middle
@pytest.mark.parametrize("with_dh", [True, False])
def test_bwd_parity(name, j, nshards, with_dh):
    w = syn.WORKLOADS[name]
    inp = syn.fwd_inputs(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    pr, orc_f, saved, dy, dh = _bwd_inputs_from_oracle_fwd(w, j, nshards, inp, grads)
    d = _desc(w, j, nshards)
    out = ops.backward(d, dy, dh if with_dh else None, saved["h"], inp["gamma"], saved["mask"],
                       saved["rstd"], saved["mean"] if w.norm == "ln" else None)
    torch.cuda.synchronize()
    _check_bwd(w, pr, orc_f["h"], _np(dy), _np(dh) if with_dh else None, _np(inp["gamma"]),
               orc_f["mask"], out)


def _bwd_rows_chunks(w, d, cuts, dy, dh, saved, gamma, ws):
    """The backward run chunk by chunk over row ranges, dgamma/dbeta
    accumulated: sentinel-filled outputs, garbage in dgamma/dbeta before the
    first chunk (which must replace it)."""
    rows, H = dy.shape
    out = dict(d_res=torch.full_like(dy, -3.0), d_sum=torch.full_like(dy, -3.0),
               dgamma=torch.full((H,), 1e30, device=DEV), dbeta=torch.full((H,), 1e30, device=DEV)
               if w.norm == "ln" else None)
    for c, (b, e) in enumerate(zip(cuts[:-1], cuts[1:])):
        ops.sp_rs_dropout_residual_norm_bwd_rows(d, b, e - b, c > 0, dy, dh, saved["h"], gamma, saved["mask"],
                                                 saved["rstd"], saved["mean"] if w.norm == "ln" else None,
                                                 out["d_res"], out["d_sum"], out["dgamma"], out["dbeta"], ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,j,nshards,cuts", [
    ("pages_rms_bf16", 0, 2, [0, 1, 1000, 2049, 4096]),
    ("gpt_ln_bf16", 3, 1, [0, 129, 130, 512]),
    ("tiny_rms_f32", 1, 1, [0, 3, 11, 16]),
])
def test_bwd_rows_chunks_accumulate_to_the_full_call(name, j, nshards, cuts):
    """The backward chunk by chunk over row ranges (each chunk's d_sum ready
    for its all-gather while the next one computes): d_residual and d_sum bit
    for bit the full call's; dgamma/dbeta, accumulated over the chunks in
    order, equal the full call's up to the grouping of the sum, and the same
    from run to run."""
    w = syn.WORKLOADS[name]
    inp = syn.fwd_inputs(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    pr, orc_f, saved, dy, dh = _bwd_inputs_from_oracle_fwd(w, j, nshards, inp, grads)
    d = _desc(w, j, nshards)
    ws = ops.workspace_for(d, DEV)
    ref = ops.backward(d, dy, dh, saved["h"], inp["gamma"], saved["mask"], saved["rstd"],
                       saved["mean"] if w.norm == "ln" else None, ws)
    torch.cuda.synchronize()
    one = _bwd_rows_chunks(w, d, cuts, dy, dh, saved, inp["gamma"], ws)
    two = _bwd_rows_chunks(w, d, cuts, dy, dh, saved, inp["gamma"], ws)
    for k in ("d_res", "d_sum"):
        assert torch.equal(one[k], ref[k]), k
    for k in ("dgamma", "dbeta"):
        if ref[k] is None:
            continue
        assert torch.equal(one[k], two[k]), k
        scale = ref[k].abs().max().item()
        assert (one[k] - ref[k]).abs().max().item() <= 1e-5 * scale, k
    _check_bwd(w, pr, orc_f["h"], _np(dy), _np(dh), _np(inp["gamma"]), orc_f["mask"], one)


def test_bwd_rows_chunks_regenerate_the_mask_of_their_rows():
    """Row ranges of the mask-free backward: each range draws the keep bits of
    its own global rows, so d_residual and d_sum match the full call's (which
    reads the stored mask) bit for bit."""
    w = syn.WORKLOADS["pages_rms_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    pr, orc_f, saved, dy, dh = _bwd_inputs_from_oracle_fwd(w, 0, 2, inp, grads)
    d = _desc(w, 0, 2)
    ws = ops.workspace_for(d, DEV)
    ref = ops.backward(d, dy, dh, saved["h"], inp["gamma"], saved["mask"], saved["rstd"], None, ws)
    torch.cuda.synchronize()
    free = dict(saved, mask=None)
    one = _bwd_rows_chunks(w, d, [0, 333, 2049, 4096], dy, dh, free, inp["gamma"], ws)
    for k in ("d_res", "d_sum"):
        assert torch.equal(one[k], ref[k]), k
    assert (one["dgamma"] - ref["dgamma"]).abs().max().item() <= 1e-5 * ref["dgamma"].abs().max().item()


def test_pipelined_exchange_on_one_nccl_rank():
    """forward_pipelined and backward_pipelined through NCCL on a one-rank
    group (T = 1): the chunked kernels are ordered with the collectives on the
    current stream and reproduce the whole-shard calls."""
    import socket
    import torch.distributed as dist
    from residual_sp_rs_gb300 import sp_exchange as ex
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        w = syn.WORKLOADS["pages_rms_bf16"].with_(T=1, S=1024, B=2)
        inp = syn.fwd_inputs(w, DEV)
        grads = syn.upstream_grads(w, DEV)
        d = _desc(w, 0)
        ref = _gpu_fwd(w, inp, 0)
        out = _sentinel_like(ref)
        ex.forward_pipelined(d, inp["partials"][0], inp["residual"].view(-1, w.H), inp["gamma"], None,
                             out["h"], out["y"], out["mask"], out["rstd"], None, chunks=4)
        torch.cuda.synchronize()
        for k in out:
            assert torch.equal(out[k], ref[k]), k
        ws = ops.workspace_for(d, DEV)
        dy, dh = grads["dy"].view(-1, w.H), grads["dh_out"].view(-1, w.H)
        bref = ops.backward(d, dy, dh, ref["h"], inp["gamma"], ref["mask"], ref["rstd"], None, ws)
        d_res, d_sum = torch.empty_like(dy), torch.empty_like(dy)
        dgamma = torch.empty(w.H, device=DEV)
        grad, works = ex.backward_pipelined(d, dy, dh, ref["h"], inp["gamma"], ref["mask"], ref["rstd"], None,
                                            d_res, d_sum, dgamma, None, ws, chunks=4)
        for wk in works:
            wk.wait()
        torch.cuda.synchronize()
        assert torch.equal(d_res, bref["d_res"]) and torch.equal(d_sum, bref["d_sum"])
        assert torch.equal(grad, bref["d_sum"])       # one rank: the gather is its own shard
        assert (dgamma - bref["dgamma"]).abs().max().item() <= 1e-5 * bref["dgamma"].abs().max().item()
    finally:
        dist.destroy_process_group()


def test_bwd_gpt_layernorm_every_shard():
    """GPT-style LayerNorm (T=8, 512 token rows per shard): the backward of
    each single shard j = 0..7, with dgamma/dbeta over that shard's rows."""
    w = syn.WORKLOADS["gpt_ln_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    for j in range(w.T):
        pr, orc_f, saved, dy, dh = _bwd_inputs_from_oracle_fwd(w, j, 1, inp, grads)
        out = ops.backward(_desc(w, j), dy, dh, saved["h"], inp["gamma"], saved["mask"], saved["rstd"],
                           saved["mean"])
        torch.cuda.synchronize()
        _check_bwd(w, pr, orc_f["h"], _np(dy), _np(dh), _np(inp["gamma"]), orc_f["mask"], out)


@pytest.mark.parametrize("p", [0.1, 0.0])
def test_bwd_large_hidden_sampled(p):
    w = syn.WORKLOADS["large_rms_bf16"].with_(p=p)
    saved = syn.saved_activations(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    gam = syn.fwd_inputs(w.with_(T=1, S=1, B=1), DEV)["gamma"]   # gamma only
    R, H = w.R, w.H
    for j in range(w.T):   # every shard, in sequence
        sl = slice(j * R, (j + 1) * R)
        h = saved["h"].view(-1, H)[sl]
        pr = _oracle_problem(w, j, p=p)
        h_np = _np(h)
        rstd, mean = oracle.norm_stats(pr, h_np, w.dtype)     # row statistics from the oracle
        rstd_t = torch.from_numpy(rstd.astype(np.float32)).to(DEV)
        dy = grads["dy"].view(-1, H)[sl]
        dh = grads["dh_out"].view(-1, H)[sl]
        mask = saved["mask"].view(-1, H)[sl] if p > 0 else None
        d = _desc(w, j, p=p)
        out = ops.backward(d, dy, dh, h, gam, mask, rstd_t)
        torch.cuda.synchronize()
        # dgamma needs every row: full oracle backward for this shard
        full = oracle.bwd(pr, _np(dy), _np(dh), h_np, _np(gam), None if mask is None else _np(mask))
        parity.check_reduction("dgamma", _np(out["dgamma"]), full["dgamma"])
        rows = _sample_rows(R, 40, 300 + j)
        ridx = torch.from_numpy(rows).to(DEV)
        for key, ex in [("d_res", "dres_exact"), ("d_sum", "dsum_exact")]:
            parity.check_bf16(key, _np(out[key].index_select(0, ridx)), full[ex][rows])
        del out, full


@pytest.mark.parametrize("case", [
    (3, 21, 1, 776, "bf16", "ln", 0.3), (1, 5, 3, 8, "bf16", "rms", 0.5),
    (2, 6, 1, 16384, "bf16", "ln", 0.1), (5, 10, 2, 4104, "bf16", "rms", 0.2),
    (2, 4, 5, 8192, "f32", "ln", 0.1), (4, 8, 3, 12, "f32", "rms", 0.7), (7, 14, 1, 1032, "f32", "ln", 0.0),
    (2, 2000, 1, 768, "bf16", "rms", 0.1),
    # each shared-memory-ring variant: 1, 2, 4 vectors a thread; LayerNorm 1
    # and 2; ragged last vector slot in the 16-warp and the 544-thread block
    (4, 24, 2, 256, "bf16", "rms", 0.1), (2, 16, 3, 512, "bf16", "rms", 0.25),
    (3, 12, 2, 1024, "bf16", "rms", 0.1), (4, 16, 2, 256, "bf16", "ln", 0.1),
    (2, 10, 3, 512, "bf16", "ln", 0.5), (3, 9, 2, 2064, "bf16", "rms", 0.1),
    (2, 8, 3, 2064, "bf16", "ln", 0.1),
    # two 8-warp LayerNorm row groups in the 544-thread block, several rows
    # per CTA: ragged last slot, and no dropout
    (2, 128, 3, 2064, "bf16", "ln", 0.1), (2, 160, 2, 4096, "bf16", "ln", 0.0),
    # RMSNorm rows of 256 threads and 3 vectors in the 544-thread block, an
    # odd number of rows per CTA
    (2, 400, 1, 5120, "bf16", "rms", 0.1), (3, 306, 1, 5120, "bf16", "rms", 0.2),
])
def test_bwd_edge_shapes(case):
    T, S, B, H, dt, nm, p = case
    w = syn.Workload("edge", T, S, B, H, dt, nm, p, 1e-5, 7, 0.5, 1.0, 0.5, 1.5, 0.1, 999 + H)
    inp = syn.fwd_inputs(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    for j, nsh in sorted({(0, 1), (T - 1, 1), (0, T)}):
        pr, orc_f, saved, dy, dh = _bwd_inputs_from_oracle_fwd(w, j, nsh, inp, grads)
        d = _desc(w, j, nsh)
        out = ops.backward(d, dy, dh, saved["h"], inp["gamma"], saved["mask"] if p > 0 else None,
                           saved["rstd"], saved["mean"] if nm == "ln" else None)
        torch.cuda.synchronize()
        _check_bwd(w, pr, orc_f["h"], _np(dy), _np(dh), _np(inp["gamma"]),
                   orc_f["mask"] if p > 0 else None, out)


def test_bwd_empty_rows_zeroes_dgamma():
    w = syn.WORKLOADS["gpt_ln_bf16"].with_(S=0)
    d = _desc(w, 0)
    z = torch.empty((0, w.H), device=DEV, dtype=torch.bfloat16)
    g = torch.ones(w.H, device=DEV, dtype=torch.bfloat16)
    dg = torch.full((w.H,), 7.0, device=DEV)
    dbt = torch.full((w.H,), 7.0, device=DEV)
    ws = ops.workspace_for(d, DEV)
    ops.sp_rs_dropout_residual_norm_bwd(d, z, None, z, g, torch.empty((0, w.H), device=DEV,
                                        dtype=torch.uint8), torch.empty(0, device=DEV),
                                        torch.empty(0, device=DEV), z, z, dg, dbt, ws)
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(dbt == 0)


def test_bwd_workspace_too_small_is_rejected():
    w = syn.WORKLOADS["pages_rms_bf16"]
    d = _desc(w, 0)
    need = ops.sp_rs_bwd_workspace_bytes(d)
    assert need > 0
    t = torch.zeros((w.R, w.H), device=DEV, dtype=torch.bfloat16)
    m = torch.zeros((w.R, w.H), device=DEV, dtype=torch.uint8)
    r = torch.ones(w.R, device=DEV)
    g = torch.ones(w.H, device=DEV, dtype=torch.bfloat16)
    dg = torch.empty(w.H, device=DEV)
    ws = torch.empty(need - 16, device=DEV, dtype=torch.uint8)
    with pytest.raises(RuntimeError, match="WORKSPACE"):
        ops.sp_rs_dropout_residual_norm_bwd(d, t, None, t, g, m, r, None, t.clone(), t.clone(), dg,
                                            None, ws)


# ---------------------------------------------------------------------------
# mask-free mode: the forward stores no mask, the backward regenerates it
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["pages_rms_bf16", "gpt_ln_bf16", "tiny_rms_f32"])
def test_mask_free_forward_and_regenerated_backward(name):
    w = syn.WORKLOADS[name]
    inp = syn.fwd_inputs(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    d = _desc(w, 0, w.T)
    rows = d.rows
    res = inp["residual"].view(rows, w.H)
    stored = ops.forward(d, inp["partials"], res, inp["gamma"], inp["beta"])
    free = ops.forward(d, inp["partials"], res, inp["gamma"], inp["beta"], store_mask=False)
    assert free["mask"] is None
    for k in ("h", "y", "rstd"):
        assert torch.equal(stored[k], free[k]), k
    dy, dh = grads["dy"].view(rows, w.H), grads["dh_out"].view(rows, w.H)
    with_mask = ops.backward(d, dy, dh, stored["h"], inp["gamma"], stored["mask"], stored["rstd"],
                             stored["mean"])
    regen = ops.backward(d, dy, dh, stored["h"], inp["gamma"], None, stored["rstd"], stored["mean"])
    torch.cuda.synchronize()
    for k in ("d_res", "d_sum", "dgamma"):   # identical keep decisions: bit-identical results
        assert torch.equal(with_mask[k], regen[k]), k
    # and against the oracle (given the oracle's own mask)
    pr, orc_f, saved, dy_o, dh_o = _bwd_inputs_from_oracle_fwd(w, 0, w.T, inp, grads)
    out = ops.backward(d, dy_o, dh_o, saved["h"], inp["gamma"], None, saved["rstd"],
                       saved["mean"] if w.norm == "ln" else None)
    torch.cuda.synchronize()
    _check_bwd(w, pr, orc_f["h"], _np(dy_o), _np(dh_o), _np(inp["gamma"]), orc_f["mask"], out)


@pytest.mark.parametrize("case", [(3, 21, 1, 776, "bf16", "ln", 0.3), (2, 6, 1, 16384, "bf16", "ln", 0.1)])
def test_regenerated_mask_register_backward(case):
    """Shapes that take the register backward (H % 16 != 0; LayerNorm rows too
    long for the TMA ring)."""
    T, S, B, H, dt, nm, p = case
    w = syn.Workload("edge", T, S, B, H, dt, nm, p, 1e-5, 0x0123456789ABCDEF, 0.5, 1.0, 0.5, 1.5, 0.1,
                     77 + H)
    inp = syn.fwd_inputs(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    for j in sorted({0, T - 1}):
        pr, orc_f, saved, dy, dh = _bwd_inputs_from_oracle_fwd(w, j, 1, inp, grads)
        d = _desc(w, j)
        out = ops.backward(d, dy, dh, saved["h"], inp["gamma"], None, saved["rstd"], saved["mean"])
        torch.cuda.synchronize()
        _check_bwd(w, pr, orc_f["h"], _np(dy), _np(dh), _np(inp["gamma"]), orc_f["mask"], out)


# ---------------------------------------------------------------------------
# layout transforms
# ---------------------------------------------------------------------------

def test_layout_full_size_bit_exact_and_roundtrip():
    lw = syn.LAYOUT
    x = syn.layout_input(lw, DEV)
    hp = ops.sp2hp_out(x, lw.T)
    back = ops.hp2sp_out(hp)
    torch.cuda.synchronize()
    xn = _np(x)
    assert np.array_equal(_np(hp), oracle.sp2hp(xn, lw.T))
    assert torch.equal(back, x)
    y = syn.layout_input(lw, DEV, seed=5).view(lw.T, lw.N, lw.H // lw.T)
    assert np.array_equal(_np(ops.hp2sp_out(y)), oracle.hp2sp(_np(y)))


@pytest.mark.parametrize("T,N,H,dt", [(1, 4, 8, "bf16"), (3, 9, 24, "bf16"), (8, 64, 512, "bf16"),
                                      (2, 6, 8, "f32"), (4, 12, 48, "f32"), (3, 300, 2064, "bf16")])
def test_layout_edge_shapes(T, N, H, dt):
    lw = syn.LayoutWorkload("edge", T, N, H, dt, 1.0, 77)
    x = syn.layout_input(lw, DEV)
    hp = ops.sp2hp_out(x, T)
    torch.cuda.synchronize()
    assert np.array_equal(_np(hp), oracle.sp2hp_all_to_all(_np(x), T))
    assert torch.equal(ops.hp2sp_out(hp), x)


# ---------------------------------------------------------------------------
# determinism, guard zones, streams
# ---------------------------------------------------------------------------

def test_bitwise_deterministic_runs():
    w = syn.WORKLOADS["gpt_ln_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    grads = syn.upstream_grads(w, DEV)
    d = _desc(w, 0, w.T)
    outs = []
    for _ in range(2):
        f = ops.forward(d, inp["partials"], inp["residual"].view(-1, w.H), inp["gamma"], inp["beta"])
        b = ops.backward(d, grads["dy"].view(-1, w.H), grads["dh_out"].view(-1, w.H), f["h"],
                         inp["gamma"], f["mask"], f["rstd"], f["mean"])
        outs.append({**f, **b})
    torch.cuda.synchronize()
    for k, v in outs[0].items():
        if v is not None:
            assert torch.equal(v, outs[1][k]), k


@pytest.mark.parametrize("name", ["gpt_ln_bf16", "pages_rms_bf16"])
def test_back_to_back_launches_match_a_single_launch(name):
    """Many forward and backward launches back to back on one stream (the
    next kernel's CTAs start while the previous one drains, and the ring
    slots of every CTA are reused many times) give, bit for bit, the results
    of the same call made alone."""
    w = syn.WORKLOADS[name]
    d = _desc(w, 0, w.T)
    rows, H = d.rows, w.H
    ins = [syn.fwd_inputs(w, DEV, seed=w.input_seed + 31 * k) for k in range(2)]
    grs = [syn.upstream_grads(w, DEV, seed=w.input_seed + 31 * k) for k in range(2)]

    def run(k):
        f = ops.forward(d, ins[k]["partials"], ins[k]["residual"].view(rows, H), ins[k]["gamma"],
                        ins[k]["beta"])
        b = ops.backward(d, grs[k]["dy"].view(rows, H), grs[k]["dh_out"].view(rows, H), f["h"],
                         ins[k]["gamma"], f["mask"], f["rstd"], f["mean"])
        return {**f, **b}

    ref = []
    for k in range(2):
        ref.append(run(k))
        torch.cuda.synchronize()
    outs = [run(i % 2) for i in range(24)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        for key, v in o.items():
            if v is not None:
                assert torch.equal(v, ref[i % 2][key]), (i, key)


def test_outputs_stay_inside_their_buffers():
    w = syn.WORKLOADS["pages_rms_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    R, H, PAD = w.R, w.H, 4096
    d = _desc(w, 1)

    def guarded(n, dtype):
        buf = torch.full((n + 2 * PAD,), 0x5A if dtype == torch.uint8 else 3.0, device=DEV, dtype=dtype)
        return buf, buf[PAD:PAD + n]

    hb, h = guarded(R * H, torch.bfloat16)
    yb, y = guarded(R * H, torch.bfloat16)
    mb, m = guarded(R * H, torch.uint8)
    rb, r = guarded(R, torch.float32)
    ops.sp_rs_dropout_residual_norm_fwd(d, inp["partials"], inp["residual"].view(-1, H)[R:2 * R],
                                        inp["gamma"], None, h, y, m, r, None)
    grads = syn.upstream_grads(w, DEV)
    drb, dres = guarded(R * H, torch.bfloat16)
    dsb, dsum = guarded(R * H, torch.bfloat16)
    dgb, dg = guarded(H, torch.float32)
    ops.sp_rs_dropout_residual_norm_bwd(d, grads["dy"].view(-1, H)[R:2 * R], None, h, inp["gamma"], m,
                                        r, None, dres, dsum, dg, None, ops.workspace_for(d, DEV))
    torch.cuda.synchronize()
    for buf in [hb, yb, mb, rb, drb, dsb, dgb]:
        fill = 0x5A if buf.dtype == torch.uint8 else 3.0
        assert torch.all(buf[:PAD] == fill) and torch.all(buf[-PAD:] == fill)


def test_side_stream_matches_default_stream():
    w = syn.WORKLOADS["pages_rms_bf16"]
    inp = syn.fwd_inputs(w, DEV)
    d = _desc(w, 0, 2)
    ref = ops.forward(d, inp["partials"], inp["residual"].view(-1, w.H), inp["gamma"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        got = ops.forward(d, inp["partials"], inp["residual"].view(-1, w.H), inp["gamma"])
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for k in ["h", "y", "mask", "rstd"]:
        assert torch.equal(ref[k], got[k])
