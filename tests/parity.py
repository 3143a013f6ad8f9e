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
    rare cases (at most 1e-5 of the elements, checked); where they differ,
    y additionally allows the first-order effect of that difference on the
    element and on its row's mean and rstd.
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
    shape = orc["h_exact"].shape
    H = shape[-1]
    h_gpu = oracle.to_f64(gpu["h"], dtype).reshape(shape)
    h_or = oracle.to_f64(orc["h"], dtype).reshape(shape)
    dh = np.abs(h_gpu - h_or)
    if dtype == "bf16":
        # the kernel rounds h once from (almost) the exact value: flips of the
        # stored residual stream must be vanishingly rare
        flips = int((dh > 0).sum())
        assert flips <= max(2, int(1e-5 * dh.size)), f"h: {flips} rounding flips"
    r = orc["rstd"][:, None]
    mu = orc["mean"][:, None] if norm == "ln" else 0.0
    xhat = (h_or - mu) * r
    second = (1.0 / orc["rstd"]) ** 2
    # first-order effect of any flipped h on the row statistics
    flip_rel = (np.abs(h_or - mu) * dh).sum(-1) / (H * second)
    dmu = dh.sum(-1) / H if norm == "ln" else np.zeros(len(second))
    extra = None
    if dtype == "bf16":
        g = np.abs(gamma_f64)[None, :]
        extra = g * r * (dh + dmu[:, None]) + 2 * g * np.abs(xhat) * flip_rel[:, None]
    check_act("y", dtype, gpu["y"], orc["y_exact"], extra)
    r_gpu = np.asarray(gpu["rstd"], dtype=np.float64)
    bad = np.abs(r_gpu - orc["rstd"]) > (1e-5 + 2 * flip_rel) * orc["rstd"]
    assert not bad.any(), f"rstd: {bad.sum()} rows out of tolerance"
    if norm == "ln":
        m_gpu = np.asarray(gpu["mean"], dtype=np.float64)
        tolm = 1e-5 * np.maximum(np.abs(orc["mean"]), np.sqrt(second)) + dmu
        bad = np.abs(m_gpu - orc["mean"]) > tolm
        assert not bad.any(), f"mean: {bad.sum()} rows out of tolerance"
