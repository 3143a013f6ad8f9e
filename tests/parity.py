"""Comparison rules for the CUDA path against the fp64 oracle.

Tolerances (stated for the SP-region hot path, derived from its arithmetic):
  * mask, layout transforms: bit-exact.
  * bf16 outputs: |gpu - exact| <= 1 bf16 ulp of the oracle's unrounded value
    (the kernel rounds its fp32 value once, <= 1/2 ulp, and its fp32 error is
    far below the other 1/2 ulp), with an absolute floor of 2^-16 * max|row|
    for elements that cancel to near zero (where fp32 rounding of the terms,
    not the final rounding, dominates).
  * the stored residual stream h is rounded once from (almost) the exact
    value on both sides, so the two agree bit for bit except in vanishingly
    rare cases (at most 1e-5 of the elements, checked; each within 1 ulp).
    Wherever a row's stored h differs, that row's norm outputs (y, rstd,
    mean) are checked against the oracle's norm of the GPU's stored row.
  * fp32 outputs: |gpu - exact| <= 1e-5 * max(|exact|, rms(row)).
  * rstd: relative 1e-5; mean: 1e-5 * max(|mean|, 1/rstd).
  * dgamma / dbeta: |gpu - exact| <= 1e-3 * max(|exact|, mean|exact|).
"""
from __future__ import annotations

import numpy as np

import oracle


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def row_floor(exact: np.ndarray) -> np.ndarray:
    ex = np.asarray(exact, dtype=np.float64)
    m = np.max(np.abs(ex), axis=-1, keepdims=True)
    return np.ldexp(m, -16)


def check_bf16(name: str, gpu_bits: np.ndarray, exact: np.ndarray, extra=None):
    g = oracle.f64_from_bf16(gpu_bits).reshape(exact.shape)
    err = np.abs(g - exact)
    tol = np.maximum(bf16_ulp(exact), row_floor(exact))
    if extra is not None:
        tol = tol + extra
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = "; ".join(f"{tuple(i)}: gpu={g[tuple(i)]!r} exact={exact[tuple(i)]!r} tol={tol[tuple(i)]!r}"
                        for i in idx)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} bf16 elements out of tolerance: {msg}")


def check_f32(name: str, gpu: np.ndarray, exact: np.ndarray, rtol=1e-5):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(exact.shape)
    rms = np.sqrt(np.mean(exact * exact, axis=-1, keepdims=True))
    tol = rtol * np.maximum(np.abs(exact), rms)
    bad = np.abs(gpu - exact) > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = "; ".join(f"{tuple(i)}: gpu={gpu[tuple(i)]!r} exact={exact[tuple(i)]!r}" for i in idx)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} f32 elements out of tolerance: {msg}")


def check_act(name, dtype, gpu, exact, extra=None):
    if dtype == "bf16":
        check_bf16(name, gpu, exact, extra)
    else:
        if extra is not None:
            gpu64 = np.asarray(gpu, dtype=np.float64).reshape(exact.shape)
            rms = np.sqrt(np.mean(exact * exact, axis=-1, keepdims=True))
            tol = 1e-5 * np.maximum(np.abs(exact), rms) + extra
            bad = np.abs(gpu64 - exact) > tol
            assert not bad.any(), f"{name}: {bad.sum()} f32 elements out of tolerance"
        else:
            check_f32(name, gpu, exact)


def check_reduction(name: str, gpu: np.ndarray, exact: np.ndarray, rtol=1e-3):
    gpu = np.asarray(gpu, dtype=np.float64)
    scale = np.maximum(np.abs(exact), np.mean(np.abs(exact)))
    bad = np.abs(gpu - exact) > rtol * scale
    if bad.any():
        i = np.argwhere(bad)[:5].ravel()
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} out of tolerance, e.g. "
                             f"{[(int(k), float(gpu[k]), float(exact[k])) for k in i]}")


def norm_of_stored_rows(pr, h_rows, gamma, beta, dtype: str) -> dict:
    """The oracle's norm step evaluated on the given stored h rows.

    This is the oracle's own row forward with every partial zero and p = 0:
    the reduced sum is 0, the mask keeps everything, so the residual stream
    it forms and stores is exactly the given (already representable) row and
    the norm reads that row.  Returns y_exact, rstd and mean per row."""
    h_rows = np.ascontiguousarray(h_rows).reshape(-1, pr.H)
    n = h_rows.shape[0]
    pz = oracle.Problem(**{f: getattr(pr, f) for f, _ in oracle.Problem._fields_})
    pz.p = 0.0
    zeros = np.zeros_like(h_rows)
    return oracle.fwd_rows(pz, np.arange(n), [zeros] * pr.T, h_rows, gamma, beta, dtype)


def compare_fwd(dtype: str, norm: str, gpu: dict, orc: dict, pr, gamma, beta=None):
    """gpu: host numpy arrays (storage form) h, y, mask, rstd, mean;
    orc: oracle outputs for the same rows; pr, gamma, beta: the oracle
    problem and the norm weights (storage form) those outputs came from.

    The mask must match bit for bit and h must lie within 1 ulp of the
    oracle's exact residual stream; a bf16 h must moreover be the oracle's
    bit for bit (both round the exact value once).  The norm is compared
    against the oracle evaluated on the GPU's own stored h: on any row where
    that h differs from the oracle's (possible only for fp32 h), y, rstd and
    mean are checked against the oracle's norm of the GPU's row, not against
    the oracle's forward of the inputs."""
    assert np.array_equal(gpu["mask"], orc["mask"]), "mask differs"
    check_act("h", dtype, gpu["h"], orc["h_exact"])
    shape = orc["h_exact"].shape
    h_gpu = np.asarray(gpu["h"]).reshape(shape)
    h_or = np.asarray(orc["h"]).reshape(shape)
    differ = h_gpu != h_or
    if dtype == "bf16":
        # the kernel rounds h once from the exact value, as the oracle does:
        # the stored residual stream must be the oracle's, bit for bit
        flips = int(differ.sum())
        assert flips == 0, f"h: {flips} rounding flips"
    y_ref = np.array(orc["y_exact"], dtype=np.float64, copy=True).reshape(shape)
    rstd_ref = np.array(orc["rstd"], dtype=np.float64, copy=True)
    mean_ref = np.array(orc["mean"], dtype=np.float64, copy=True)
    rows = np.flatnonzero(differ.any(axis=-1))
    if rows.size:
        rn = norm_of_stored_rows(pr, h_gpu[rows], gamma, beta, dtype)
        y_ref[rows] = rn["y_exact"]
        rstd_ref[rows] = rn["rstd"]
        mean_ref[rows] = rn["mean"]
    check_act("y", dtype, gpu["y"], y_ref)
    r_gpu = np.asarray(gpu["rstd"], dtype=np.float64)
    bad = np.abs(r_gpu - rstd_ref) > 1e-5 * rstd_ref
    assert not bad.any(), f"rstd: {bad.sum()} rows out of tolerance"
    if norm == "ln":
        m_gpu = np.asarray(gpu["mean"], dtype=np.float64)
        tolm = 1e-5 * np.maximum(np.abs(mean_ref), 1.0 / rstd_ref)
        bad = np.abs(m_gpu - mean_ref) > tolm
        assert not bad.any(), f"mean: {bad.sum()} rows out of tolerance"


def tie_inputs(rows: int, H: int, seed: int = 3):
    """Seeded bf16 forward inputs (for p = 0.5, so 1/(1-p) = 2) whose every
    kept element lands EXACTLY on a bf16 rounding midpoint: residual r with a
    7-bit mantissa m in 1..126 (both neighbours in r's binade), P0 =
    +-ulp(r)/4 and every other partial 0, so E = r +- ulp(r)/2.  Returns
    (P0, R, tie) as uint16 bf16 bit patterns; tie is the round-half-to-even result (of the
    neighbours m and m +- 1 of |r|, the even mantissa), the expected h of a
    kept element (a dropped one keeps r)."""
    rng = np.random.default_rng(seed)
    shape = (rows, H)
    neg = rng.integers(0, 2, shape).astype(np.uint32)
    exp = rng.integers(-6, 7, shape).astype(np.int64)
    mant = rng.integers(1, 127, shape).astype(np.uint32)
    away = rng.integers(0, 2, shape).astype(np.uint32)       # does P0 move |E| up?
    r = (neg << 15) | ((exp + 127).astype(np.uint32) << 7) | mant
    p0_neg = neg ^ (1 - away)                                 # same sign as r: |E| grows
    p0 = (p0_neg << 15) | ((exp - 9 + 127).astype(np.uint32) << 7)
    k = np.where(away == 1, 1, -1)
    m_out = np.where(mant % 2 == 0, mant.astype(np.int64), mant.astype(np.int64) + k).astype(np.uint32)
    tie = (neg << 15) | ((exp + 127).astype(np.uint32) << 7) | m_out
    u16 = lambda a: a.astype(np.uint16)
    return u16(p0), u16(r), u16(tie)
