"""Python binding of libspfuse: argument marshalling only.

Every function named like a C entry point (``sp_rs_dropout_residual_norm_fwd``,
``sp_rs_bwd_workspace_bytes``, ``sp_rs_dropout_residual_norm_bwd``, ``sp2hp``,
``hp2sp``) passes tensor pointers, sizes and the current CUDA stream to the
function of the same name in ``libspfuse.so`` and raises ``RuntimeError`` with
the library's status string when it reports an error.  All arithmetic runs in
the library's CUDA kernels; there is no other implementation to fall back to:
if the library is missing, the first call raises.

``forward`` / ``backward`` / ``sp2hp_out`` / ``hp2sp_out`` are conveniences
that allocate the outputs with torch (device memory only) and call the above.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH, source_hash

SP_F32, SP_BF16 = 0, 1
SP_RMSNORM, SP_LAYERNORM = 0, 1
DTYPE_CODE = {torch.float32: SP_F32, torch.bfloat16: SP_BF16}
NAME_CODE = {"f32": SP_F32, "bf16": SP_BF16}
NORM_CODE = {"rms": SP_RMSNORM, "ln": SP_LAYERNORM}


class SpRsDesc(ctypes.Structure):
    """Mirror of sp_rs_desc_t (include/spfuse.h)."""
    _fields_ = [("T", ctypes.c_int32), ("j", ctypes.c_int32), ("S", ctypes.c_int64),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("norm", ctypes.c_int32), ("p", ctypes.c_float), ("eps", ctypes.c_float),
                ("seed", ctypes.c_uint64), ("nshards", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("status", ctypes.c_void_p)]

    @property
    def R(self) -> int:
        return (self.S // self.T) * self.B

    @property
    def rows(self) -> int:
        return self.R * max(1, self.nshards)


class SpKernelPlan(ctypes.Structure):
    """Mirror of sp_kernel_plan_t (include/spfuse.h)."""
    _fields_ = [(n, ctypes.c_int32) for n in ("tma", "block", "nthr", "tpr", "vpt", "row_groups",
                                              "rows_per_stage", "stages", "chunked", "noalloc_fits")] + \
               [(n, ctypes.c_int64) for n in ("stage_bytes", "smem_bytes", "rows_per_cta", "ctas",
                                              "workspace_bytes")]


class SpPlanInfo(ctypes.Structure):
    """Mirror of sp_plan_info_t (include/spfuse.h)."""
    _fields_ = [("fwd", SpKernelPlan), ("bwd", SpKernelPlan)]


def make_desc(T, j, S, B, H, dtype="bf16", norm="rms", p=0.0, eps=1e-6, seed=0, nshards=1,
              status=None):
    """status: an int32/uint32 CUDA tensor of one element (the device status
    word, see include/spfuse.h) or None."""
    return SpRsDesc(T=T, j=j, S=S, B=B, H=H, dtype=NAME_CODE.get(dtype, dtype),
                    norm=NORM_CODE.get(norm, norm), p=p, eps=eps, seed=int(seed) & (2**64 - 1),
                    nshards=nshards, reserved=0, status=_ptr(status))


_lib = None


def lib() -> ctypes.CDLL:
    """Load libspfuse.so (built by ``residual_sp_rs_gb300.build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libspfuse.so is not built ({LIB_PATH}); run residual_sp_rs_gb300.build.build() "
                "with the CUDA toolkit installed. There is no fallback implementation.")
        L = ctypes.CDLL(LIB_PATH)
        L.sp_build_hash.restype = ctypes.c_char_p
        L.sp_build_hash.argtypes = []
        _verify_hash(L, source_hash())
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        D = ctypes.POINTER(SpRsDesc)
        L.sp_rs_dropout_residual_norm_fwd.restype = ctypes.c_int
        L.sp_rs_dropout_residual_norm_fwd.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.sp_rs_dropout_residual_norm_fwd_rows.restype = ctypes.c_int
        L.sp_rs_dropout_residual_norm_fwd_rows.argtypes = [D, i64, i64, vp, vp, vp, vp, vp, vp, vp,
                                                           vp, vp, vp]
        L.sp_rs_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.sp_rs_bwd_workspace_bytes.argtypes = [D]
        L.sp_rs_dropout_residual_norm_bwd.restype = ctypes.c_int
        L.sp_rs_dropout_residual_norm_bwd.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                      vp, vp, ctypes.c_size_t, vp]
        L.sp_rs_dropout_residual_norm_bwd_rows.restype = ctypes.c_int
        L.sp_rs_dropout_residual_norm_bwd_rows.argtypes = [D, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp,
                                                           vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        for name in ("sp2hp", "hp2sp"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [vp, vp, i64, i64, i32, i32, vp]
        L.sp_status_string.restype = ctypes.c_char_p
        L.sp_status_string.argtypes = [ctypes.c_int]
        L.sp_version.restype = ctypes.c_int32
        L.sp_version.argtypes = []
        L.sp_last_cuda_error.restype = ctypes.c_char_p
        L.sp_last_cuda_error.argtypes = []
        L.sp_plan_describe.restype = ctypes.c_int
        L.sp_plan_describe.argtypes = [D, i32, i32, i32, i32, ctypes.POINTER(SpPlanInfo)]
        _lib = L
    return _lib


def _verify_hash(L: ctypes.CDLL, expected: str) -> None:
    """Refuse a library built from other sources than these."""
    got = L.sp_build_hash().decode()
    if got != expected:
        raise RuntimeError(f"libspfuse.so is stale: built from sources {got[:12]}, the tree is "
                           f"{expected[:12]}; rebuild it with residual_sp_rs_gb300.build.build()")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("libspfuse takes dense row-major tensors")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(code: int):
    if code != 0:
        msg = lib().sp_status_string(code).decode()
        if code == 6:  # SP_ERR_CUDA
            msg += f" ({lib().sp_last_cuda_error().decode()})"
        raise RuntimeError(msg)


def sp_plan_describe(desc: SpRsDesc, sms: int, smem_optin: int, has_dh: bool = True,
                     has_mask: bool = True) -> dict:
    """The launch configurations the forward and backward would use on a device
    with `sms` multiprocessors and `smem_optin` bytes of opt-in shared memory
    per block; host arithmetic only (no GPU needed).  Returns
    {"fwd": {...}, "bwd": {...}} with the fields of sp_kernel_plan_t."""
    info = SpPlanInfo()
    _check(lib().sp_plan_describe(ctypes.byref(desc), int(sms), int(smem_optin), int(bool(has_dh)),
                                  int(bool(has_mask)), ctypes.byref(info)))
    out = {}
    for k in ("fwd", "bwd"):
        kp = getattr(info, k)
        out[k] = {n: getattr(kp, n) for n, _ in SpKernelPlan._fields_}
    return out


def status_string(code: int) -> str:
    return lib().sp_status_string(code).decode()


# ---- C entry points, same names ---------------------------------------------------

def sp_rs_dropout_residual_norm_fwd(desc: SpRsDesc, partials, residual, gamma, beta, h_out, y_out,
                                    mask_out, rstd_out, mean_out, stream=None) -> None:
    arr = (ctypes.c_void_p * max(1, len(partials)))(*[_ptr(p) for p in partials])
    _check(lib().sp_rs_dropout_residual_norm_fwd(
        ctypes.byref(desc), arr, _ptr(residual), _ptr(gamma), _ptr(beta), _ptr(h_out),
        _ptr(y_out), _ptr(mask_out), _ptr(rstd_out), _ptr(mean_out), _stream(stream)))


def sp_rs_dropout_residual_norm_fwd_rows(desc: SpRsDesc, row_begin: int, row_count: int, partials,
                                         residual, gamma, beta, h_out, y_out, mask_out, rstd_out,
                                         mean_out, stream=None) -> None:
    arr = (ctypes.c_void_p * max(1, len(partials)))(*[_ptr(p) for p in partials])
    _check(lib().sp_rs_dropout_residual_norm_fwd_rows(
        ctypes.byref(desc), int(row_begin), int(row_count), arr, _ptr(residual), _ptr(gamma),
        _ptr(beta), _ptr(h_out), _ptr(y_out), _ptr(mask_out), _ptr(rstd_out), _ptr(mean_out),
        _stream(stream)))


def sp_rs_bwd_workspace_bytes(desc: SpRsDesc) -> int:
    return int(lib().sp_rs_bwd_workspace_bytes(ctypes.byref(desc)))


def sp_rs_dropout_residual_norm_bwd(desc: SpRsDesc, dy, dh_out, h_saved, gamma, mask, rstd, mean,
                                    d_residual, d_sum, dgamma, dbeta, workspace,
                                    workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sp_rs_dropout_residual_norm_bwd(
        ctypes.byref(desc), _ptr(dy), _ptr(dh_out), _ptr(h_saved), _ptr(gamma), _ptr(mask),
        _ptr(rstd), _ptr(mean), _ptr(d_residual), _ptr(d_sum), _ptr(dgamma), _ptr(dbeta),
        _ptr(workspace), workspace_bytes, _stream(stream)))


def sp_rs_dropout_residual_norm_bwd_rows(desc: SpRsDesc, row_begin: int, row_count: int, accumulate: bool,
                                         dy, dh_out, h_saved, gamma, mask, rstd, mean, d_residual, d_sum,
                                         dgamma, dbeta, workspace, stream=None) -> None:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sp_rs_dropout_residual_norm_bwd_rows(
        ctypes.byref(desc), int(row_begin), int(row_count), int(bool(accumulate)), _ptr(dy), _ptr(dh_out),
        _ptr(h_saved), _ptr(gamma), _ptr(mask), _ptr(rstd), _ptr(mean), _ptr(d_residual), _ptr(d_sum),
        _ptr(dgamma), _ptr(dbeta), _ptr(workspace), nbytes, _stream(stream)))


def sp2hp(inp, out, N, H, T, dtype, stream=None) -> None:
    _check(lib().sp2hp(_ptr(inp), _ptr(out), N, H, T, NAME_CODE.get(dtype, dtype), _stream(stream)))


def hp2sp(inp, out, N, H, T, dtype, stream=None) -> None:
    _check(lib().hp2sp(_ptr(inp), _ptr(out), N, H, T, NAME_CODE.get(dtype, dtype), _stream(stream)))


# ---- conveniences that allocate outputs ------------------------------------------

def forward(desc: SpRsDesc, partials, residual, gamma, beta=None, stream=None,
            store_mask: bool = True) -> dict:
    """store_mask=False: the mask is not stored (the backward regenerates it)."""
    rows, H = desc.rows, desc.H
    dev, dt = residual.device, residual.dtype
    out = dict(h=torch.empty((rows, H), device=dev, dtype=dt),
               y=torch.empty((rows, H), device=dev, dtype=dt),
               mask=torch.empty((rows, H), device=dev, dtype=torch.uint8)
               if desc.p > 0 and store_mask else None,
               rstd=torch.empty(rows, device=dev, dtype=torch.float32),
               mean=torch.empty(rows, device=dev, dtype=torch.float32)
               if desc.norm == SP_LAYERNORM else None)
    sp_rs_dropout_residual_norm_fwd(desc, partials, residual, gamma, beta, out["h"], out["y"],
                                    out["mask"], out["rstd"], out["mean"], stream)
    return out


def workspace_for(desc: SpRsDesc, device) -> torch.Tensor:
    n = sp_rs_bwd_workspace_bytes(desc)
    return torch.empty(max(16, n), device=device, dtype=torch.uint8)


def backward(desc: SpRsDesc, dy, dh_out, h_saved, gamma, mask, rstd, mean=None, workspace=None,
             stream=None) -> dict:
    rows, H = desc.rows, desc.H
    dev, dt = dy.device, dy.dtype
    if workspace is None:
        workspace = workspace_for(desc, dev)
    out = dict(d_res=torch.empty((rows, H), device=dev, dtype=dt),
               d_sum=torch.empty((rows, H), device=dev, dtype=dt),
               dgamma=torch.empty(H, device=dev, dtype=torch.float32),
               dbeta=torch.empty(H, device=dev, dtype=torch.float32)
               if desc.norm == SP_LAYERNORM else None)
    sp_rs_dropout_residual_norm_bwd(desc, dy, dh_out, h_saved, gamma, mask, rstd, mean,
                                    out["d_res"], out["d_sum"], out["dgamma"], out["dbeta"],
                                    workspace, stream=stream)
    return out


def sp2hp_out(x: torch.Tensor, T: int, stream=None) -> torch.Tensor:
    N, H = x.shape
    out = torch.empty((T, N, H // T), device=x.device, dtype=x.dtype)
    sp2hp(x, out, N, H, T, DTYPE_CODE[x.dtype], stream)
    return out


def hp2sp_out(x: torch.Tensor, stream=None) -> torch.Tensor:
    T, N, Hc = x.shape
    out = torch.empty((N, Hc * T), device=x.device, dtype=x.dtype)
    hp2sp(x, out, N, Hc * T, T, DTYPE_CODE[x.dtype], stream)
    return out
