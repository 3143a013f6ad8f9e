"""The allocation-free backward entry point, called through the C ABI.

sp_rs_dropout_residual_norm_bwd_noalloc serves callers that cannot allocate
device memory where they run the backward (allocator callbacks, frameworks
whose caching allocator owns the device memory, paths that must not risk the
device synchronisation of cudaMalloc/cudaFree).  It keeps its partial rows in
a fixed array inside the library instead of a caller workspace.  This test
checks that its outputs are bit-identical to the workspace entry point's
(the same kernels on the same inputs) on two calls in a row, with different
inputs, so leftovers of the first call in the shared array cannot leak into
the second.  Its refusal of problems larger than the array is host
arithmetic, checked on the CPU (tests/test_plan_host.py): no problem on a
152-SM device needs more than 5 MB.  The file name sorts last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from residual_sp_rs_gb300 import ops, synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from residual_sp_rs_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = ops.lib()
    f = L.sp_rs_dropout_residual_norm_bwd_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ops.SpRsDesc)] + [ctypes.c_void_p] * 12
    return L


def _p(t):
    return None if t is None else t.data_ptr()


@pytest.mark.parametrize("name", ["pages_rms_bf16", "gpt_ln_bf16"])
def test_noalloc_backward_matches_workspace_backward(lib, name):
    w = syn.WORKLOADS[name]
    dev = "cuda"
    desc = ops.make_desc(w.T, 0, w.S, w.B, w.H, w.dtype, w.norm, w.p, w.eps, w.seed, w.T)
    assert ops.sp_rs_bwd_workspace_bytes(desc) <= (8 << 20)
    rows, H = desc.rows, w.H
    for call in range(2):   # two calls in a row, different inputs each time
        inp = syn.fwd_inputs(w, dev, seed=w.input_seed + 31 * call)
        gr = syn.upstream_grads(w, dev, seed=w.input_seed + 31 * call)
        f = ops.forward(desc, inp["partials"], inp["residual"].view(rows, H), inp["gamma"], inp["beta"])
        dy, dh = gr["dy"].view(rows, H), gr["dh_out"].view(rows, H)
        ref = ops.backward(desc, dy, dh, f["h"], inp["gamma"], f["mask"], f["rstd"], f["mean"])
        out = dict(d_res=torch.empty_like(ref["d_res"]), d_sum=torch.empty_like(ref["d_sum"]),
                   dgamma=torch.empty_like(ref["dgamma"]),
                   dbeta=None if ref["dbeta"] is None else torch.empty_like(ref["dbeta"]))
        code = lib.sp_rs_dropout_residual_norm_bwd_noalloc(
            ctypes.byref(desc), _p(dy), _p(dh), _p(f["h"]), _p(inp["gamma"]), _p(f["mask"]),
            _p(f["rstd"]), _p(f["mean"]), _p(out["d_res"]), _p(out["d_sum"]), _p(out["dgamma"]),
            _p(out["dbeta"]), torch.cuda.current_stream().cuda_stream)
        assert code == 0, ops.status_string(code)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bit-identical results
        for k in ("d_res", "d_sum", "dgamma", "dbeta"):
            if ref[k] is not None:
                assert torch.equal(out[k], ref[k]), (call, k)
