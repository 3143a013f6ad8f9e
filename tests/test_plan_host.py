"""The kernels' launch plans, through sp_plan_describe (host arithmetic, no
GPU): invariants that the TMA-fed kernels rely on, checked over a grid of
shapes, and the configurations the three benchmark workloads run with."""
import itertools
import math

import pytest

from residual_sp_rs_gb300 import ops

SMS, OPTIN = 152, 232448  # GB300: multiprocessors, opt-in shared memory per block
STATIC_SMEM = 1024        # the kernels' static shared arrays, rounded up
MAX_SMEM = OPTIN - STATIC_SMEM


@pytest.fixture(scope="module")
def spf():
    try:
        ops.lib()
    except (RuntimeError, OSError) as e:
        pytest.skip(f"libspfuse not built: {e}")
    return ops


NOALLOC_SCRATCH = 8 << 20  # SP_NOALLOC_SCRATCH_BYTES


def _plans(spf, T, S, B, H, norm, nshards=1, has_dh=True, has_mask=True, sms=SMS, optin=OPTIN, p=0.1):
    d = spf.make_desc(T, 0, S, B, H, "bf16", norm, p, 1e-5, 0, nshards)
    return spf.sp_plan_describe(d, sms, optin, has_dh, has_mask)


def _check_fwd(f, T, H, rows, sms=SMS, max_smem=MAX_SMEM):
    nvec = H // 8
    assert f["nthr"] == (896 if T <= 4 else 544)
    assert f["block"] == f["row_groups"] * f["tpr"] + 32 <= f["nthr"]
    assert f["tpr"] % 32 == 0 and f["vpt"] == -(-nvec // f["tpr"]) <= 3
    # the narrowest row group with at most 3 vectors a thread
    assert f["tpr"] == 32 or -(-nvec // (f["tpr"] // 2)) > 3
    if f["tpr"] > 32:
        assert f["row_groups"] <= 15  # one named barrier per group, ids 1..15
    assert 1 <= f["row_groups"] <= f["rows_per_cta"]
    assert f["stages"] >= 2
    assert f["smem_bytes"] <= max_smem
    assert f["smem_bytes"] >= f["stages"] * f["stage_bytes"]
    if f["chunked"]:
        assert f["rows_per_stage"] == 1 and f["stage_bytes"] == f["tpr"] * 16 * (T + 1)
        assert f["vpt"] >= 2
    else:
        assert 1 <= f["rows_per_stage"] <= f["row_groups"]
        assert f["stage_bytes"] == f["rows_per_stage"] * 2 * H * (T + 1)
    assert f["ctas"] <= sms and f["ctas"] * f["rows_per_cta"] >= rows
    assert (f["ctas"] - 1) * f["rows_per_cta"] < rows
    # when ring slots are reused, a slot always returns to the row group that
    # consumed its previous stage (rows go to the groups round robin)
    per_row = f["vpt"] if f["chunked"] else 1
    nstage = -(-f["rows_per_cta"] // f["rows_per_stage"]) * per_row
    if nstage > f["stages"] and f["row_groups"] > 1:
        g = f["row_groups"]
        lanes = g * per_row if f["chunked"] else g // math.gcd(g, f["rows_per_stage"])
        assert f["stages"] % lanes == 0


def _check_bwd(b, H, ln, rows, has_dh, has_mask, sms=SMS, max_smem=MAX_SMEM):
    nvec = H // 8
    assert H % 16 == 0
    assert b["nthr"] in (512, 544)
    assert b["block"] == b["row_groups"] * b["tpr"] + 32 <= b["nthr"]
    assert b["vpt"] == -(-nvec // b["tpr"]) <= (2 if ln else 4)
    if b["nthr"] == 544:
        # two 8-warp row groups, where the 16-warp block would hold one
        assert b["tpr"] == 256 and b["row_groups"] == 2 and b["vpt"] <= 3
    # rows go to the row groups round robin: the groups of a stage recur
    # every `lanes` stages
    lanes = b["row_groups"] // math.gcd(b["row_groups"], b["rows_per_stage"])
    # when ring slots are reused, a slot always returns to the group(s) that
    # consumed its previous stage, so a wait by barrier parity cannot match
    # a phase two behind
    if -(-b["rows_per_cta"] // b["rows_per_stage"]) > b["stages"]:
        assert b["stages"] % lanes == 0
    if b["nthr"] == 512:
        # the 16-warp block walks the ring stage by stage: rows per stage
        # divide the row groups
        assert b["row_groups"] % b["rows_per_stage"] == 0
    assert 1 <= b["row_groups"] <= b["rows_per_cta"]
    rb = b["rows_per_stage"]
    per_row = 2 * H * (3 if has_dh else 2) + (H if has_mask else 0)
    assert b["stage_bytes"] == -(-rb * per_row // 16) * 16
    assert b["stages"] >= 2 and b["smem_bytes"] <= max_smem
    # at the end the ring holds every row group's column sums
    ns = 2 if ln else 1
    assert b["stages"] * b["stage_bytes"] >= b["row_groups"] * ns * 8 * (nvec + 4) * 4
    assert b["ctas"] <= sms and b["ctas"] * b["rows_per_cta"] >= rows
    # one fp32 partial row per CTA (and statistic)
    assert b["workspace_bytes"] == min(max(rows, 1), sms) * H * 4 * ns
    assert b["noalloc_fits"] == (1 if b["workspace_bytes"] <= NOALLOC_SCRATCH else 0)


SHAPES = list(itertools.product(
    [1, 2, 3, 4, 8],                                  # T
    [(24, 2), (2040, 2), (96, 3), (4104, 1)],          # (S, B); S a multiple of every T
    [64, 256, 768, 1024, 2064, 4096, 6144, 8192, 12288, 16384],  # H
    ["rms", "ln"]))


@pytest.mark.parametrize("T,SB,H,norm", SHAPES)
def test_plan_invariants(spf, T, SB, H, norm):
    S, B = SB
    for nshards in (1, T):
        rows = (S // T) * B * nshards
        for has_dh, has_mask in ((True, True), (False, True), (True, False)):
            pl = _plans(spf, T, S, B, H, norm, nshards, has_dh, has_mask)
            f, b = pl["fwd"], pl["bwd"]
            if f["tma"]:
                _check_fwd(f, T, H, rows)
            if b["tma"]:
                _check_bwd(b, H, norm == "ln", rows, has_dh, has_mask)
            else:
                assert all(v == 0 for v in b.values())


def test_smaller_device_limits_are_respected(spf):
    # a device with fewer SMs and less shared memory gets plans that fit it
    for H in (768, 4096, 8192):
        pl = _plans(spf, 2, 2048, 2, H, "rms", 2, sms=40, optin=101376)
        if pl["fwd"]["tma"]:
            _check_fwd(pl["fwd"], 2, H, 4096, sms=40, max_smem=101376 - STATIC_SMEM)
        if pl["bwd"]["tma"]:
            _check_bwd(pl["bwd"], H, False, 4096, True, True, sms=40, max_smem=101376 - STATIC_SMEM)


def test_pages_shape_configuration(spf):
    # T=2, S=2048, B=2, H=768, both shards in one launch: 27 rows per SM,
    # every one in flight at once in the forward
    pl = _plans(spf, 2, 2048, 2, 768, "rms", 2)
    f, b = pl["fwd"], pl["bwd"]
    assert (f["nthr"], f["block"], f["row_groups"], f["tpr"], f["vpt"]) == (896, 896, 27, 32, 3)
    assert f["rows_per_stage"] == 6 and not f["chunked"]  # 9 KB copies per input
    assert f["rows_per_cta"] == 27 and f["ctas"] == 152
    assert f["rows_per_stage"] * f["stages"] >= f["rows_per_cta"]
    assert (b["nthr"], b["block"], b["row_groups"], b["rows_per_stage"]) == (512, 512, 15, 15)
    assert b["rows_per_cta"] == 27


def test_gpt_layernorm_configuration(spf):
    # T=8, S=4096, B=1, H=4096, LayerNorm: rows of 256 threads; the backward
    # takes the 544-thread block with two 8-warp row groups
    pl = _plans(spf, 8, 4096, 1, 4096, "ln", 8)
    f, b = pl["fwd"], pl["bwd"]
    assert (f["nthr"], f["tpr"], f["vpt"], f["row_groups"]) == (544, 256, 2, 2)
    assert (b["nthr"], b["block"], b["tpr"], b["vpt"], b["row_groups"]) == (544, 544, 256, 2, 2)


def test_large_hidden_configuration(spf):
    # T=8, S=8192, B=2, H=8192: a whole row of the 9 forward inputs does not
    # fit twice, so the forward streams column-chunk stages
    pl = _plans(spf, 8, 8192, 2, 8192, "rms", 8)
    assert pl["fwd"]["chunked"] == 1 and pl["fwd"]["tpr"] == 512
    assert pl["bwd"]["nthr"] == 512 and pl["bwd"]["vpt"] == 4


def test_f32_runs_the_register_kernels(spf):
    d = spf.make_desc(2, 0, 16, 2, 64, "f32", "rms", 0.1, 1e-6, 0, 1)
    pl = spf.sp_plan_describe(d, SMS, OPTIN)
    assert pl["fwd"]["tma"] == 0 and pl["bwd"]["tma"] == 0


def test_noalloc_scratch_covers_this_device_and_refuses_larger_ones(spf):
    """The allocation-free backward refuses a problem whose partial rows do
    not fit its fixed 8 MiB array.  On a 152-SM device no TMA-fed backward
    gets there (at most 152 rows of H = 4096 x 2 statistics, or H = 8192 x 1:
    5 MB); a device with twice the SMs would be refused the GPT LayerNorm
    backward."""
    most = 0
    for T, SB, H, norm in SHAPES:
        S, B = SB
        b = _plans(spf, T, S, B, H, norm, T)["bwd"]
        if b["tma"]:
            assert b["noalloc_fits"] == 1
            most = max(most, b["workspace_bytes"])
    assert most == 152 * 4096 * 4 * 2
    b = _plans(spf, 8, 4096, 1, 4096, "ln", 8, sms=304)["bwd"]
    assert b["tma"] and b["workspace_bytes"] == 304 * 4096 * 8 > NOALLOC_SCRATCH
    assert b["noalloc_fits"] == 0
    b = _plans(spf, 8, 4096, 1, 4096, "rms", 8, sms=304)["bwd"]
    assert b["workspace_bytes"] == 304 * 4096 * 4 and b["noalloc_fits"] == 1


def test_describe_matches_what_the_calls_launch(spf):
    # no rows: the forward launches nothing
    pl = _plans(spf, 2, 0, 2, 768, "rms", 2)
    assert all(v == 0 for v in pl["fwd"].values())
    # p = 0: the backward reads no mask even when one is passed
    with_p0 = _plans(spf, 2, 2048, 2, 768, "rms", 2, has_mask=True, p=0.0)["bwd"]
    no_mask = _plans(spf, 2, 2048, 2, 768, "rms", 2, has_mask=False)["bwd"]
    assert with_p0["stage_bytes"] == no_mask["stage_bytes"] == -(-no_mask["rows_per_stage"] * 3 * 2 * 768 // 16) * 16
    # an opt-in limit below the kernels' static shared memory leaves no room
    # for a ring: no TMA-fed plan (and no wrapped-around size)
    for optin in (1, 512, STATIC_SMEM):
        pl = _plans(spf, 2, 2048, 2, 768, "rms", 2, optin=optin)
        assert pl["fwd"]["tma"] == 0 and pl["bwd"]["tma"] == 0


def test_bad_limits_are_rejected(spf):
    d = spf.make_desc(2, 0, 16, 2, 64, "bf16", "rms", 0.1, 1e-6, 0, 1)
    with pytest.raises(RuntimeError, match="INVALID"):
        spf.sp_plan_describe(d, 0, OPTIN)
    bad = spf.make_desc(3, 0, 16, 2, 64, "bf16", "rms", 0.1, 1e-6, 0, 1)  # S % T != 0
    with pytest.raises(RuntimeError):
        spf.sp_plan_describe(bad, SMS, OPTIN)
