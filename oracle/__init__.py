"""ctypes binding of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference leg are the only callers.  The product
library never imports this package and shares no code with it.

Arrays cross the boundary as contiguous numpy arrays: bf16 as ``np.uint16``
bit patterns, fp32 as ``np.float32``, f64 as ``np.float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SOURCES = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]

DTYPES = {"f32": 0, "bf16": 1, "f64": 2}
NORMS = {"rms": 0, "ln": 1}
NP_STORAGE = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C11, no FMA contraction)."""
    newest = max(os.path.getmtime(s) for s in _SOURCES)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SOURCES[0], "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("j", ctypes.c_int32), ("nshards", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("norm", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("S", ctypes.c_int64), ("B", ctypes.c_int64), ("H", ctypes.c_int64),
                ("p", ctypes.c_double), ("eps", ctypes.c_double), ("seed", ctypes.c_uint64)]


def problem(T, j, S, B, H, dtype="bf16", norm="rms", p=0.0, eps=1e-6, seed=0, nshards=1):
    """Problem descriptor; p and eps are taken as given (pass the float32
    values the GPU path receives to compare like with like)."""
    return Problem(T=T, j=j, nshards=nshards, dtype=DTYPES[dtype], norm=NORMS[norm], pad=0,
                   S=S, B=B, H=H, p=float(p), eps=float(eps), seed=int(seed) & (2**64 - 1))


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, u64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        P = ctypes.POINTER(Problem)
        sig = {
            "orc_f64_from_bf16": (dbl, [ctypes.c_uint16]),
            "orc_bf16_from_f64": (ctypes.c_uint16, [dbl]),
            "orc_philox4x32_10": (None, [vp, vp, vp]),
            "orc_mask_word": (ctypes.c_uint32, [u64, u64]),
            "orc_keep_threshold": (ctypes.c_uint32, [dbl]),
            "orc_fwd_row": (None, [P, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "orc_fwd": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "orc_bwd_row": (None, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "orc_bwd": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "orc_norm_stats_row": (None, [P, vp, vp, vp]),
            "orc_bf16_from_f64_array": (None, [vp, vp, i64]),
            "orc_f64_from_bf16_array": (None, [vp, vp, i64]),
            "orc_mask_range": (None, [u64, dbl, u64, i64, vp]),
            "orc_reduce_scatter": (ctypes.c_int, [i32, i64, vp, i32, vp]),
            "orc_all_gather": (ctypes.c_int, [i32, i64, vp, vp]),
            "orc_all_reduce": (ctypes.c_int, [i32, i64, vp, vp]),
            "orc_ring_reduce_scatter": (ctypes.c_int, [i32, i64, vp, vp]),
            "orc_ring_reduce_scatter_symbolic": (ctypes.c_int, [i32, i32, vp, vp]),
            "orc_sp2hp": (ctypes.c_int, [vp, vp, i64, i64, i32, i32]),
            "orc_hp2sp": (ctypes.c_int, [vp, vp, i64, i64, i32, i32]),
            "orc_sp2hp_all_to_all": (ctypes.c_int, [vp, vp, i64, i64, i32, i32]),
            "orc_hp2sp_all_to_all": (ctypes.c_int, [vp, vp, i64, i64, i32, i32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dt=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a if dt is None else a.astype(dt, copy=False))
    return a


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


# ---- conversions / RNG --------------------------------------------------------

def bf16_from_f64(x) -> np.ndarray:
    x = _c(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_from_f64_array(_p(x), _p(out), x.size)
    return out


def f64_from_bf16(b) -> np.ndarray:
    b = _c(np.asarray(b, dtype=np.uint16))
    out = np.empty(b.shape, np.float64)
    lib().orc_f64_from_bf16_array(_p(b), _p(out), b.size)
    return out


def to_f64(arr, dtype: str) -> np.ndarray:
    """Widen stored activations to f64 (exact)."""
    return f64_from_bf16(arr) if dtype == "bf16" else np.asarray(arr, dtype=np.float64)


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.empty(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def mask_word(seed: int, g: int) -> int:
    return int(lib().orc_mask_word(seed & (2**64 - 1), g))


def keep_threshold(p: float) -> int:
    return int(lib().orc_keep_threshold(float(p)))


def mask_range(seed: int, p: float, g0: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint8)
    lib().orc_mask_range(seed & (2**64 - 1), float(p), g0, n, _p(out))
    return out


# ---- forward / backward ---------------------------------------------------------

def fwd(pr: Problem, partials, residual, gamma, beta=None, dtype="bf16"):
    """Full forward over the problem's shards.  Returns a dict of numpy arrays."""
    st = NP_STORAGE[dtype]
    parts = [_c(p, st) for p in partials]
    res, gam = _c(residual, st), _c(gamma, st)
    bet = _c(beta, st) if beta is not None else None
    R = (pr.S // pr.T) * pr.B
    rows = R * pr.nshards
    H = pr.H
    out = dict(h=np.empty((rows, H), st), y=np.empty((rows, H), st),
               mask=np.empty((rows, H), np.uint8), rstd=np.empty(rows), mean=np.empty(rows),
               h_exact=np.empty((rows, H)), y_exact=np.empty((rows, H)))
    err = lib().orc_fwd(ctypes.byref(pr), _ptr_array(parts), _p(res), _p(gam), _p(bet),
                        _p(out["h"]), _p(out["y"]), _p(out["mask"]), _p(out["rstd"]),
                        _p(out["mean"]), _p(out["h_exact"]), _p(out["y_exact"]))
    if err:
        raise ValueError(f"oracle fwd rejected the problem ({err})")
    return out


def fwd_rows(pr: Problem, grows, prows, res_rows, gamma, beta=None, dtype="bf16"):
    """Forward of selected rows.  grows: global row indices; prows: T arrays
    [n, H] holding those rows of each partial; res_rows: [n, H]."""
    st = NP_STORAGE[dtype]
    grows = np.asarray(grows, dtype=np.int64)
    n, H = len(grows), pr.H
    prows = [_c(p, st).reshape(n, H) for p in prows]
    res_rows = _c(res_rows, st).reshape(n, H)
    gam = _c(gamma, st)
    bet = _c(beta, st) if beta is not None else None
    out = dict(h=np.empty((n, H), st), y=np.empty((n, H), st), mask=np.empty((n, H), np.uint8),
               rstd=np.empty(n), mean=np.empty(n), h_exact=np.empty((n, H)), y_exact=np.empty((n, H)))
    L = lib()
    for i in range(n):
        ptrs = (ctypes.c_void_p * pr.T)(*[p[i].ctypes.data for p in prows])
        L.orc_fwd_row(ctypes.byref(pr), int(grows[i]), ptrs, res_rows[i].ctypes.data, _p(gam), _p(bet),
                      out["h"][i].ctypes.data, out["y"][i].ctypes.data, out["mask"][i].ctypes.data,
                      out["rstd"][i:].ctypes.data, out["mean"][i:].ctypes.data,
                      out["h_exact"][i].ctypes.data, out["y_exact"][i].ctypes.data)
    return out


def bwd(pr: Problem, dy, dh_out, h_saved, gamma, mask, dtype="bf16"):
    st = NP_STORAGE[dtype]
    R = (pr.S // pr.T) * pr.B
    rows, H = R * pr.nshards, pr.H
    dy_, dh_, h_, gam = _c(dy, st), _c(dh_out, st), _c(h_saved, st), _c(gamma, st)
    m_ = _c(mask, np.uint8) if mask is not None else None
    out = dict(d_res=np.empty((rows, H), st), d_sum=np.empty((rows, H), st),
               dres_exact=np.empty((rows, H)), dsum_exact=np.empty((rows, H)),
               dgamma=np.empty(H), dbeta=np.empty(H))
    err = lib().orc_bwd(ctypes.byref(pr), _p(dy_), _p(dh_), _p(h_), _p(gam), _p(m_),
                        _p(out["d_res"]), _p(out["d_sum"]), _p(out["dres_exact"]),
                        _p(out["dsum_exact"]), _p(out["dgamma"]), _p(out["dbeta"]))
    if err:
        raise ValueError(f"oracle bwd rejected the problem ({err})")
    return out


def bwd_rows(pr: Problem, dy_rows, dh_rows, h_rows, gamma, mask_rows, dtype="bf16"):
    """Backward of selected rows; dgamma/dbeta are those rows' contributions."""
    st = NP_STORAGE[dtype]
    H = pr.H
    h_rows = _c(h_rows, st).reshape(-1, H)
    n = h_rows.shape[0]
    dy_rows = _c(dy_rows, st).reshape(n, H)
    dh_rows = _c(dh_rows, st).reshape(n, H) if dh_rows is not None else None
    mask_rows = _c(mask_rows, np.uint8).reshape(n, H) if mask_rows is not None else None
    gam = _c(gamma, st)
    out = dict(d_res=np.empty((n, H), st), d_sum=np.empty((n, H), st),
               dres_exact=np.empty((n, H)), dsum_exact=np.empty((n, H)),
               dgamma=np.zeros(H), dbeta=np.zeros(H))
    L = lib()
    for i in range(n):
        L.orc_bwd_row(ctypes.byref(pr), dy_rows[i].ctypes.data,
                      None if dh_rows is None else dh_rows[i].ctypes.data,
                      h_rows[i].ctypes.data, _p(gam),
                      None if mask_rows is None else mask_rows[i].ctypes.data,
                      out["d_res"][i].ctypes.data, out["d_sum"][i].ctypes.data,
                      out["dres_exact"][i].ctypes.data, out["dsum_exact"][i].ctypes.data,
                      _p(out["dgamma"]), _p(out["dbeta"]))
    return out


def norm_stats(pr: Problem, h_rows, dtype="bf16"):
    """f64 (rstd, mean) of each stored row."""
    st = NP_STORAGE[dtype]
    h_rows = _c(h_rows, st).reshape(-1, pr.H)
    n = h_rows.shape[0]
    rstd, mean = np.empty(n), np.empty(n)
    L = lib()
    for i in range(n):
        L.orc_norm_stats_row(ctypes.byref(pr), h_rows[i].ctypes.data, rstd[i:].ctypes.data,
                             mean[i:].ctypes.data)
    return rstd, mean


# ---- simulated collectives --------------------------------------------------------

def reduce_scatter(P, j):
    P = [_c(p, np.float64) for p in P]
    n = P[0].size
    out = np.empty(n // len(P))
    if lib().orc_reduce_scatter(len(P), n, _ptr_array(P), j, _p(out)):
        raise ValueError("reduce_scatter: bad arguments")
    return out


def all_gather(blocks):
    blocks = [_c(b, np.float64) for b in blocks]
    m = blocks[0].size
    out = np.empty(m * len(blocks))
    if lib().orc_all_gather(len(blocks), m, _ptr_array(blocks), _p(out)):
        raise ValueError("all_gather: bad arguments")
    return out


def all_reduce(P):
    P = [_c(p, np.float64) for p in P]
    out = np.empty(P[0].size)
    if lib().orc_all_reduce(len(P), P[0].size, _ptr_array(P), _p(out)):
        raise ValueError("all_reduce: bad arguments")
    return out


def ring_reduce_scatter(P):
    """Runs the ring schedule on copies of P; returns (work buffers, sent)."""
    work = [np.array(p, dtype=np.float64, copy=True).ravel() for p in P]
    sent = np.zeros(len(P), np.int64)
    if lib().orc_ring_reduce_scatter(len(P), work[0].size, _ptr_array(work), _p(sent)):
        raise ValueError("ring_reduce_scatter: bad arguments")
    return work, sent


def ring_reduce_scatter_symbolic(T, steps):
    contrib = np.zeros((T, T), np.uint64)
    used = np.zeros((T, T), np.uint8)
    if lib().orc_ring_reduce_scatter_symbolic(T, steps, _p(contrib), _p(used)):
        raise ValueError("ring_reduce_scatter_symbolic: bad arguments")
    return contrib, used


# ---- layout --------------------------------------------------------------------------

def _layout(fn, x, N, H, T, out_shape):
    x = np.ascontiguousarray(x)
    out = np.empty(out_shape, x.dtype)
    if getattr(lib(), fn)(_p(x), _p(out), N, H, T, x.itemsize):
        raise ValueError(f"{fn}: bad arguments")
    return out


def sp2hp(x, T):
    N, H = x.shape
    return _layout("orc_sp2hp", x, N, H, T, (T, N, H // T))


def hp2sp(x):
    T, N, Hc = x.shape
    return _layout("orc_hp2sp", x, N, Hc * T, T, (N, Hc * T))


def sp2hp_all_to_all(x, T):
    N, H = x.shape
    return _layout("orc_sp2hp_all_to_all", x, N, H, T, (T, N, H // T))


def hp2sp_all_to_all(x):
    T, N, Hc = x.shape
    return _layout("orc_hp2sp_all_to_all", x, N, Hc * T, T, (N, Hc * T))
