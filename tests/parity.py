"""Comparison rules for the CUDA path against the fp64 oracle.

Tolerances (stated for the SP-region hot path, derived from its arithmetic):
  * mask, layout transforms: bit-exact.
  * bf16 outputs: |gpu - exact| <= 1 bf16 ulp of the oracle's unrounded value
    (the kernel rounds its fp32 value once, <= 1/2 ulp, and its fp32 error is
    far below the other 1/2 ulp), with an absolute floor of 2^-16 * max|row|
    for elements that cancel to near zero (where fp32 rounding of the terms,
    not the final rounding, dominates).
  * y additionally allows |gamma * rstd| * |h_gpu - h_oracle| where the two
    stored residual-stream values differ: an fp32-vs-f64 rounding flip of the
    stored h (at most 1 ulp, checked separately) is read by the norm.
  * fp32 outputs: |gpu - exact| <= 1e-5 * max(|exact|, rms(row)).
  * rstd: relative 1e-5 plus the first-order effect of h flips on the row's
    second moment.
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


def compare_fwd(dtype: str, norm: str, gpu: dict, orc: dict, gamma_f64: np.ndarray):
    """gpu: host numpy arrays (storage form) h, y, mask, rstd, mean;
    orc: oracle outputs for the same rows."""
    assert np.array_equal(gpu["mask"], orc["mask"]), "mask differs"
    check_act("h", dtype, gpu["h"], orc["h_exact"])
    h_gpu = oracle.to_f64(gpu["h"], dtype).reshape(orc["h_exact"].shape)
    h_or = oracle.to_f64(orc["h"], dtype).reshape(orc["h_exact"].shape)
    dh = np.abs(h_gpu - h_or)
    rstd = orc["rstd"][:, None]
    extra = np.abs(gamma_f64)[None, :] * rstd * dh if dtype == "bf16" else None
    check_act("y", dtype, gpu["y"], orc["y_exact"], extra)
    # rstd: first-order effect of flipped h on the row's second moment
    if norm == "ln":
        cen = np.abs(h_or - orc["mean"][:, None])
    else:
        cen = np.abs(h_or)
    H = h_or.shape[-1]
    second = (1.0 / orc["rstd"]) ** 2
    flip_rel = (cen * dh).sum(-1) / (H * second)
    r_gpu = np.asarray(gpu["rstd"], dtype=np.float64)
    bad = np.abs(r_gpu - orc["rstd"]) > (1e-5 + 2 * flip_rel) * orc["rstd"]
    assert not bad.any(), f"rstd: {bad.sum()} rows out of tolerance"
    if norm == "ln":
        m_gpu = np.asarray(gpu["mean"], dtype=np.float64)
        rms = np.sqrt(second)
        tolm = 1e-5 * np.maximum(np.abs(orc["mean"]), rms) + dh.sum(-1) / H
        bad = np.abs(m_gpu - orc["mean"]) > tolm
        assert not bad.any(), f"mean: {bad.sum()} rows out of tolerance"
