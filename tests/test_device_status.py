"""The device status word and the bounded waits of the TMA-fed kernels.

Every wait of the TMA-fed kernels on data in flight has a time limit; a
kernel whose wait runs out marks the results it could not compute (NaN) and
ORs a bit into the caller's status word instead of hanging the GPU.  The
timeout is provoked without any fault: in a child process the library's test
hooks shorten the limit to 2 ms and make CTA 0's producer skip one ring
stage, so the waits on that stage run out.  The parent then checks that only
the rows of that stage are marked, that every other output equals a normal
run, and that the status word carries the right bit.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from residual_sp_rs_gb300 import ops, synthetic as syn

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FWD_BIT, BWD_BIT = 0x1, 0x2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from residual_sp_rs_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(status):
    """Forward and backward of both shards of the pages' shape."""
    w = syn.WORKLOADS["pages_rms_bf16"]
    d = ops.make_desc(w.T, 0, w.S, w.B, w.H, w.dtype, w.norm, w.p, w.eps, w.seed, w.T, status=status)
    inp = syn.fwd_inputs(w, "cuda")
    gr = syn.upstream_grads(w, "cuda")
    rows = d.rows
    f = ops.forward(d, inp["partials"], inp["residual"].view(rows, w.H), inp["gamma"])
    torch.cuda.synchronize()
    fwd_status = int(status.item())
    status.zero_()
    b = ops.backward(d, gr["dy"].view(rows, w.H), gr["dh_out"].view(rows, w.H), f["h"], inp["gamma"],
                     f["mask"], f["rstd"])
    torch.cuda.synchronize()
    return f, b, fwd_status, int(status.item())


def _child(out_path):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    f, b, fs, bs = _run(status)
    torch.save({"fwd": {k: v.cpu() for k, v in f.items() if v is not None},
                "bwd": {k: v.cpu() for k, v in b.items() if v is not None},
                "fwd_status": fs, "bwd_status": bs}, out_path)


def test_clean_run_leaves_the_status_word_alone():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    f, b, fs, bs = _run(status)
    assert fs == 0 and bs == 0
    assert torch.isfinite(f["rstd"]).all() and torch.isfinite(b["dgamma"]).all()


def test_timed_out_waits_mark_results_and_set_the_status_word(tmp_path):
    out = str(tmp_path / "child.pt")
    env = dict(os.environ, SPFUSE_TEST_WAIT_NS="2000000", SPFUSE_TEST_DROP_STAGE="1")
    code = f"import sys; sys.path.insert(0, {ROOT!r}); from tests.test_device_status import _child; _child({out!r})"
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    got = torch.load(out)
    assert got["fwd_status"] == FWD_BIT
    assert got["bwd_status"] == BWD_BIT
    ref_f, ref_b, _, _ = _run(torch.zeros(1, dtype=torch.int32, device="cuda"))

    # forward: the plan of this shape (checked on the host by the plan tests)
    # gives CTA 0 rows 0..26 in stages of 6 rows, so stage 1 is rows 6..11;
    # exactly those rows are marked and every other output is the normal one
    d = ops.make_desc(2, 0, 2048, 2, 768, "bf16", "rms", 0.1, 1e-6, 0, 2)
    props = torch.cuda.get_device_properties(0)
    plan = ops.sp_plan_describe(d, props.multi_processor_count,
                                getattr(props, "shared_memory_per_block_optin", 232448))
    rb = plan["fwd"]["rows_per_stage"]
    dropped = np.arange(rb, 2 * rb)
    rstd = got["fwd"]["rstd"].numpy()
    assert np.isnan(rstd[dropped]).all()
    keep = np.setdiff1d(np.arange(len(rstd)), dropped)
    assert np.array_equal(rstd[keep], ref_f["rstd"].cpu().numpy()[keep])
    for k in ("h", "y", "mask"):
        assert torch.equal(got["fwd"][k][keep], ref_f[k].cpu()[keep]), k
    # backward: CTA 0 could not finish its rows, so its dgamma partial (and
    # with it every dgamma element) is NaN; the rows of every other CTA are
    # the normal ones
    assert torch.isnan(got["bwd"]["dgamma"]).all()
    rpc = plan["bwd"]["rows_per_cta"]
    for k in ("d_res", "d_sum"):
        assert torch.equal(got["bwd"][k][rpc:], ref_b[k].cpu()[rpc:]), k

