"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (ring reduce-scatter tables, the two-rank block example),
published known-answer vectors and an independent implementation of the
generator, closed forms, library routines (torch f64 LayerNorm / RMSNorm and
autograd, numpy sums), invariants and brute force on tiny inputs.
"""
import os
import shutil
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Philox4x32-10 and the dropout mask
# ---------------------------------------------------------------------------

def _read_kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w = [int(x, 16) for x in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answer_vectors():
    kat = _read_kat()
    assert len(kat) == 3
    for ctr, key, expect in kat:
        got = oracle.philox4x32_10(ctr, key)
        assert [int(x) for x in got] == expect


def _torch_probe_binary(tmpdir):
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    if not os.path.exists(os.path.join(inc, "ATen", "core", "PhiloxRNGEngine.h")):
        pytest.skip("torch headers not installed")
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = os.path.join(tmpdir, "probe")
    src = os.path.join(os.path.dirname(__file__), "philox_torch_probe.cpp")
    subprocess.run([cxx, "-std=c++17", "-O1", f"-I{inc}", src, "-o", exe], check=True)
    return exe


def test_philox_matches_torch_header_engine():
    """Independent implementation: PyTorch's header-only philox_engine with
    key = seed and offset g>>2 gives the same word g&3 as the oracle."""
    rng = np.random.default_rng(7)
    seeds = [0, 0x0123456789ABCDEF, 2**64 - 1] + [int(x) for x in rng.integers(0, 2**63, 5)]
    pairs = []
    for s in seeds:
        gs = [0, 1, 2, 3, 4, 5, 7, 2**32 - 1, 2**32, 2**34 + 3, 2**62 + 1]
        gs += [int(x) for x in rng.integers(0, 2**40, 20)]
        pairs += [(s, g) for g in gs]
    with tempfile.TemporaryDirectory() as d:
        exe = _torch_probe_binary(d)
        inp = "".join(f"{s} {g}\n" for s, g in pairs)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
    ref = [int(x) for x in out.split()]
    got = [oracle.mask_word(s, g) for s, g in pairs]
    assert got == ref


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_mask_density_binomial(p):
    p32 = float(np.float32(p))
    n = 400_000
    m = oracle.mask_range(0, p32, 12345, n)
    assert set(np.unique(m)) <= {0, 1}
    keep = 1.0 - p32
    sigma = np.sqrt(n * keep * (1 - keep))
    assert abs(m.sum() - n * keep) < 5 * sigma


def test_mask_p0_keeps_everything():
    assert oracle.mask_range(0x0123456789ABCDEF, 0.0, 0, 50_000).min() == 1
    assert oracle.keep_threshold(0.0) == 0


def test_keep_threshold_is_floor_of_p_times_2_32():
    # p = 0.5 -> exactly 2^31; p = 0.25 -> 2^30; the largest float below 1
    assert oracle.keep_threshold(0.5) == 2**31
    assert oracle.keep_threshold(0.25) == 2**30
    p = float(np.nextafter(np.float32(1.0), np.float32(0.0)))
    assert oracle.keep_threshold(p) == 2**32 - 2**8


# ---------------------------------------------------------------------------
# bf16 conversion (round once, to nearest even)
# ---------------------------------------------------------------------------

def test_bf16_widen_narrow_roundtrip_all_patterns():
    pats = np.arange(65536, dtype=np.uint16)
    x = oracle.f64_from_bf16(pats)
    finite = ~np.isnan(x)
    back = oracle.bf16_from_f64(x[finite])
    assert np.array_equal(back, pats[finite])
    # widening agrees with torch's bf16 -> f64
    t = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(t[finite], x[finite])


def test_bf16_rounding_matches_torch_for_binary32_inputs():
    """For values exactly representable in binary32 a single RNE to bf16 is
    torch's float32 -> bfloat16 cast (a library routine)."""
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2**32, 200_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # add exact ties and near-overflow/subnormal values
    extra = np.array([1.00390625, -1.01171875, 3.3895313892515355e38, 3.39e38, 1e-40, -2e-39,
                      9.18354961579912115600575419705e-41, 0.0, -0.0], dtype=np.float32)
    f = np.concatenate([f, extra])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_f64(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rounding_is_single_step_from_f64():
    # 1 + 2^-8 is the midpoint between bf16 1.0 (0x3F80) and 1.0078125 (0x3F81)
    mid = 1.0 + 2.0**-8
    assert oracle.bf16_from_f64([mid])[0] == 0x3F80               # tie -> even
    assert oracle.bf16_from_f64([mid + 2.0**-40])[0] == 0x3F81    # just above: up
    assert oracle.bf16_from_f64([mid - 2.0**-40])[0] == 0x3F80    # just below: down
    mid2 = 1.0078125 + 2.0**-8                                   # between 0x3F81 and 0x3F82
    assert oracle.bf16_from_f64([mid2])[0] == 0x3F82
    # rounding through binary32 first would give the even neighbour here
    via32 = torch.tensor([mid + 2.0**-40], dtype=torch.float64).float().to(torch.bfloat16)
    assert via32.view(torch.int16).item() == 0x3F80


# ---------------------------------------------------------------------------
# a1: reduce-scatter, all-gather, all-reduce (MiniMind-tron ch.3 §3.2.1, §3.2.3)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 3, 4, 8])
def test_allreduce_is_allgather_of_reducescatter(T):
    rng = np.random.default_rng(T)
    S, B, H = 4 * T, 3, 5
    # integer-valued so every sum is exact in f64
    P = [rng.integers(-1000, 1000, (S, B, H)).astype(np.float64) for _ in range(T)]
    blocks = [oracle.reduce_scatter(P, j) for j in range(T)]
    ag = oracle.all_gather(blocks)
    ar = oracle.all_reduce(P)
    assert np.array_equal(ag, ar)
    assert np.array_equal(ar, np.sum(np.stack(P), axis=0).ravel())
    # block j is the contiguous sequence range [j*S/T, (j+1)*S/T) of dim 0
    for j in range(T):
        ref = np.sum(np.stack([p[j * S // T:(j + 1) * S // T] for p in P]), axis=0).ravel()
        assert np.array_equal(blocks[j], ref)


def test_two_rank_block_example():
    """The T=2 example: with P_t^(b) = 2^(2t+b) the sum's bits name its
    contributors, which must be exactly the pairs the page lists."""
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "block_reduce_scatter_T2.txt"))
             if l.strip() and not l.startswith("#")]
    P = [np.array([2.0 ** (2 * t + 0), 2.0 ** (2 * t + 1)]) for t in range(2)]
    for line in lines:
        head, tail = line.split(":")
        names = tail.split()
        if head.startswith("reduce_scatter"):
            j = int(head.split()[1])
            val = int(oracle.reduce_scatter(P, j)[0])
            expect = sum(2 ** (2 * int(n[1]) + int(n[3])) for n in names)
            assert val == expect
        else:
            ys = [oracle.reduce_scatter(P, j) for j in range(2)]
            assert np.array_equal(oracle.all_gather(ys), P[0] + P[1])


def _parse_ring_tables():
    tables, cur, vol = {}, None, {}
    for line in open(os.path.join(GOLDEN, "ring_reduce_scatter_T4.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line == "init":
            cur = tables.setdefault(0, [])
        elif line.startswith("step"):
            cur = tables.setdefault(int(line.split()[1]), [])
        elif line.startswith("volume"):
            k, v = line.split()
            vol[k] = int(v)
        else:
            cur.append(line.split()[1:])
    return tables, vol


def test_ring_reduce_scatter_reproduces_page_tables():
    tables, vol = _parse_ring_tables()
    T = 4
    letters = "abcd"
    for step, rows in tables.items():
        contrib, used = oracle.ring_reduce_scatter_symbolic(T, step)
        for r in range(T):
            for b in range(T):
                cell = rows[r][b]
                if cell == "-":
                    assert used[r, b] == 1, (step, r, b)
                    continue
                assert used[r, b] == 0, (step, r, b)
                terms = cell.split("+")
                assert all(t[0] == letters[b] for t in terms)
                ranks = {int(t[1:]) for t in terms}
                assert int(contrib[r, b]) == sum(1 << k for k in ranks), (step, r, b)
    # per-rank volume (T-1)/T * N
    P = [np.arange(16.0) + 100 * t for t in range(T)]
    _, sent = oracle.ring_reduce_scatter(P)
    assert all(s * vol["volume_per_rank_denominator"] == vol["volume_per_rank_numerator"] * 16
               for s in sent)


@pytest.mark.parametrize("T", [2, 3, 5, 8])
def test_ring_reduce_scatter_matches_direct_and_volume(T):
    rng = np.random.default_rng(10 + T)
    n = T * 6
    P = [rng.integers(-50, 50, n).astype(np.float64) for _ in range(T)]
    work, sent = oracle.ring_reduce_scatter(P)
    m = n // T
    for j in range(T):
        assert np.array_equal(work[j][j * m:(j + 1) * m], oracle.reduce_scatter(P, j))
    assert np.all(sent == (T - 1) * n // T)
    contrib, _ = oracle.ring_reduce_scatter_symbolic(T, T - 1)
    for r in range(T):
        assert int(contrib[r, r]) == (1 << T) - 1


# ---------------------------------------------------------------------------
# forward: per-token independence, mask, dropout scaling, norms
# ---------------------------------------------------------------------------

def _int_partials(T, S, B, H, rng):
    return [rng.integers(-8, 9, (S, B, H)).astype(np.float32) / 4 for _ in range(T)]


@pytest.mark.parametrize("norm", ["rms", "ln"])
@pytest.mark.parametrize("T", [2, 4])
def test_sharded_forward_equals_forward_of_allreduce(norm, T):
    """Per-token work: running f on every reduce-scatter shard and gathering
    gives f of the all-reduced tensor (with the mask keyed by global index)."""
    rng = np.random.default_rng(5)
    S, B, H = 4 * T, 2, 16
    P = _int_partials(T, S, B, H, rng)
    res = rng.standard_normal((S, B, H)).astype(np.float32)
    gam = rng.uniform(0.5, 1.5, H).astype(np.float32)
    bet = rng.standard_normal(H).astype(np.float32) if norm == "ln" else None
    p = float(np.float32(0.3))
    R = (S // T) * B
    outs = []
    for j in range(T):
        pr = oracle.problem(T, j, S, B, H, "f32", norm, p, 1e-5, 42)
        outs.append(oracle.fwd(pr, P, res.reshape(S * B, H)[j * R:(j + 1) * R], gam, bet, "f32"))
    ar = np.sum(np.stack(P).astype(np.float64), axis=0).astype(np.float32)  # exact
    full = oracle.fwd(oracle.problem(1, 0, S, B, H, "f32", norm, p, 1e-5, 42), [ar],
                      res.reshape(S * B, H), gam, bet, "f32")
    for key in ["h", "y", "mask", "rstd", "mean", "h_exact", "y_exact"]:
        cat = np.concatenate([o[key] for o in outs])
        assert np.array_equal(cat, full[key]), key
    # multi-shard call = concatenation of single-shard calls
    pr = oracle.problem(T, 0, S, B, H, "f32", norm, p, 1e-5, 42, nshards=T)
    allj = oracle.fwd(pr, P, res.reshape(S * B, H), gam, bet, "f32")
    assert np.array_equal(allj["y"], full["y"]) and np.array_equal(allj["mask"], full["mask"])


def test_forward_mask_is_generator_at_global_index():
    rng = np.random.default_rng(9)
    T, S, B, H = 2, 8, 2, 32
    P = _int_partials(T, S, B, H, rng)
    res = rng.standard_normal((S * B, H)).astype(np.float32)
    gam = np.ones(H, np.float32)
    p = float(np.float32(0.25))
    R = (S // T) * B
    for j in range(T):
        pr = oracle.problem(T, j, S, B, H, "f32", "rms", p, 1e-6, 0x0123456789ABCDEF)
        out = oracle.fwd(pr, P, res[j * R:(j + 1) * R], gam, None, "f32")
        ref = oracle.mask_range(0x0123456789ABCDEF, p, j * R * H, R * H).reshape(R, H)
        assert np.array_equal(out["mask"], ref)


def test_dropout_scaling_and_p0_residual_add():
    """Kept elements carry Y/(1-p), dropped ones nothing; at p = 0 the
    residual stream is exactly residual + sum of partials (numpy f64 sum)."""
    rng = np.random.default_rng(11)
    T, S, B, H = 3, 6, 1, 24
    P = [rng.standard_normal((S, B, H)) for _ in range(T)]
    res = rng.standard_normal((S * B, H))
    gam = np.ones(H)
    Y = np.sum(np.stack(P), axis=0).reshape(S * B, H)
    for p in [0.0, float(np.float32(0.4))]:
        pr = oracle.problem(T, 0, S, B, H, "f64", "rms", p, 1e-6, 3, nshards=T)
        out = oracle.fwd(pr, P, res, gam, None, "f64")
        z = out["h_exact"] - res
        keep = out["mask"] == 1
        np.testing.assert_allclose(z[keep], Y[keep] / (1 - p), rtol=1e-13, atol=1e-13)
        assert np.all(z[~keep] == 0)
        if p == 0.0:
            assert keep.all()
            np.testing.assert_array_equal(out["h_exact"], res + Y)


def test_forward_bf16_stores_round_once():
    rng = np.random.default_rng(12)
    T, S, B, H = 2, 4, 2, 40
    P = [oracle.bf16_from_f64(rng.standard_normal((S, B, H)) * 0.02) for _ in range(T)]
    res = oracle.bf16_from_f64(rng.standard_normal((S * B, H)))
    gam = oracle.bf16_from_f64(rng.uniform(0.9, 1.1, H))
    pr = oracle.problem(T, 0, S, B, H, "bf16", "rms", float(np.float32(0.1)), 1e-6, 0, nshards=T)
    out = oracle.fwd(pr, P, res, gam, None, "bf16")
    assert np.array_equal(out["h"], oracle.bf16_from_f64(out["h_exact"]))
    assert np.array_equal(out["y"], oracle.bf16_from_f64(out["y_exact"]))
    # y is computed from the stored (rounded) h
    h = oracle.f64_from_bf16(out["h"])
    g = oracle.f64_from_bf16(gam)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h), (H,), torch.from_numpy(g), eps=1e-6)
    np.testing.assert_allclose(out["y_exact"], ref.numpy(), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("norm", ["rms", "ln"])
def test_norm_matches_torch_f64(norm):
    rng = np.random.default_rng(13)
    T, S, B, H = 2, 8, 2, 48
    P = [rng.standard_normal((S, B, H)) for _ in range(T)]
    res = rng.standard_normal((S * B, H))
    gam = rng.uniform(0.5, 1.5, H)
    bet = rng.standard_normal(H) if norm == "ln" else None
    eps = 1e-5
    pr = oracle.problem(T, 0, S, B, H, "f64", norm, 0.2, eps, 1, nshards=T)
    out = oracle.fwd(pr, P, res, gam, bet, "f64")
    h = torch.from_numpy(out["h"])
    if norm == "ln":
        ref = torch.nn.functional.layer_norm(h, (H,), torch.from_numpy(gam), torch.from_numpy(bet), eps)
        np.testing.assert_allclose(out["mean"], h.mean(-1).numpy(), rtol=1e-13, atol=1e-15)
        var = h.var(-1, unbiased=False).numpy()
    else:
        ref = torch.nn.functional.rms_norm(h, (H,), torch.from_numpy(gam), eps)
        var = (h * h).mean(-1).numpy()
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out["rstd"], 1 / np.sqrt(var + eps), rtol=1e-13)


def test_rmsnorm_unit_rms_closed_form():
    """gamma = 1: mean(y^2) = ms / (ms + eps) exactly; unit rms as eps -> 0."""
    rng = np.random.default_rng(14)
    T, S, B, H = 2, 4, 4, 64
    P = [rng.standard_normal((S, B, H)) for _ in range(T)]
    res = rng.standard_normal((S * B, H))
    for eps in [1e-6, 1e-2, 1e-300]:
        pr = oracle.problem(T, 0, S, B, H, "f64", "rms", 0.1, eps, 2, nshards=T)
        out = oracle.fwd(pr, P, res, np.ones(H), None, "f64")
        ms = (out["h"] ** 2).mean(-1)
        np.testing.assert_allclose((out["y"] ** 2).mean(-1), ms / (ms + eps), rtol=1e-13)
        if eps == 1e-300:
            np.testing.assert_allclose(np.sqrt((out["y"] ** 2).mean(-1)), 1.0, rtol=1e-14)


def test_layernorm_moments_and_constant_rows():
    rng = np.random.default_rng(15)
    T, S, B, H = 1, 6, 1, 32
    P = [rng.standard_normal((S, B, H))]
    res = rng.standard_normal((S * B, H))
    res[2] = 3.25 - P[0][2, 0]          # residual + partial is constant on row 2 (p = 0)
    eps = 1e-5
    bet = rng.standard_normal(H)
    pr = oracle.problem(T, 0, S, B, H, "f64", "ln", 0.0, eps, 0)
    out = oracle.fwd(pr, P, res, np.ones(H), np.zeros(H), "f64")
    var = out["h"].var(-1)
    np.testing.assert_allclose(out["y"].mean(-1), 0.0, atol=1e-14)
    np.testing.assert_allclose(out["y"].var(-1), var / (var + eps), rtol=1e-12, atol=1e-15)
    out2 = oracle.fwd(pr, P, res, np.ones(H), bet, "f64")
    np.testing.assert_allclose(out2["y"][2], bet, rtol=0, atol=1e-12)  # constant row -> beta


def test_norm_scale_invariance():
    rng = np.random.default_rng(16)
    T, S, B, H = 1, 4, 1, 32
    P = [rng.standard_normal((S, B, H))]
    res = rng.standard_normal((S * B, H))
    for norm in ["rms", "ln"]:
        pr = oracle.problem(T, 0, S, B, H, "f64", norm, 0.0, 1e-300, 0)
        a = oracle.fwd(pr, P, res, np.ones(H), np.zeros(H), "f64")["y"]
        b = oracle.fwd(pr, [P[0] * 7.5], res * 7.5, np.ones(H), np.zeros(H), "f64")["y"]
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# backward: finite differences, autograd, the dropout-backward identity
# ---------------------------------------------------------------------------

def _loss(pr, P, res, gam, bet, dy, dh):
    out = oracle.fwd(pr, P, res, gam, bet, "f64")
    return float(np.sum(dy * out["y"]) + (0.0 if dh is None else np.sum(dh * out["h"])))


@pytest.mark.parametrize("norm", ["rms", "ln"])
@pytest.mark.parametrize("with_dh", [True, False])
def test_backward_matches_central_differences(norm, with_dh):
    rng = np.random.default_rng(17)
    T, S, B, H = 2, 4, 1, 12
    P = [rng.standard_normal((S, B, H)) for _ in range(T)]
    res = rng.standard_normal((S * B, H))
    gam = rng.uniform(0.5, 1.5, H)
    bet = rng.standard_normal(H) if norm == "ln" else None
    dy = rng.standard_normal((S * B, H))
    dh = rng.standard_normal((S * B, H)) if with_dh else None
    pr = oracle.problem(T, 0, S, B, H, "f64", norm, 0.3, 1e-3, 99, nshards=T)
    fw = oracle.fwd(pr, P, res, gam, bet, "f64")
    bw = oracle.bwd(pr, dy, dh, fw["h"], gam, fw["mask"], "f64")
    step = 1e-6

    def fd(perturb):
        plus, minus = perturb(step), perturb(-step)
        return (plus - minus) / (2 * step)

    for (r, c) in [(0, 0), (1, 5), (3, 11), (2, 7)]:
        def pres(d):
            rr = res.copy(); rr[r, c] += d
            return _loss(pr, P, rr, gam, bet, dy, dh)
        np.testing.assert_allclose(fd(pres), bw["dres_exact"][r, c], rtol=1e-6, atol=1e-8)
        s, b = divmod(r, B)
        for t in range(T):   # every partial gets the same gradient d_sum
            def ppart(d, t=t):
                PP = [p.copy() for p in P]; PP[t][s, b, c] += d
                return _loss(pr, PP, res, gam, bet, dy, dh)
            np.testing.assert_allclose(fd(ppart), bw["dsum_exact"][r, c], rtol=1e-6, atol=1e-8)
    for c in [0, 4, 11]:
        def pgam(d):
            gg = gam.copy(); gg[c] += d
            return _loss(pr, P, res, gg, bet, dy, dh)
        np.testing.assert_allclose(fd(pgam), bw["dgamma"][c], rtol=1e-6, atol=1e-8)
        if norm == "ln":
            def pbet(d):
                bb = bet.copy(); bb[c] += d
                return _loss(pr, P, res, gam, bb, dy, dh)
            np.testing.assert_allclose(fd(pbet), bw["dbeta"][c], rtol=1e-6, atol=1e-8)
    # dbeta is the column sum of dy (closed form)
    np.testing.assert_allclose(bw["dbeta"], dy.sum(0), rtol=1e-13)


@pytest.mark.parametrize("norm", ["rms", "ln"])
def test_backward_matches_torch_autograd(norm):
    rng = np.random.default_rng(18)
    T, S, B, H = 3, 6, 2, 40
    P = [rng.standard_normal((S, B, H)) for _ in range(T)]
    res = rng.standard_normal((S * B, H))
    gam = rng.uniform(0.5, 1.5, H)
    bet = rng.standard_normal(H)
    dy = rng.standard_normal((S * B, H))
    dh = rng.standard_normal((S * B, H))
    p, eps = 0.25, 1e-5
    pr = oracle.problem(T, 0, S, B, H, "f64", norm, p, eps, 5, nshards=T)
    fw = oracle.fwd(pr, P, res, gam, bet if norm == "ln" else None, "f64")
    bw = oracle.bwd(pr, dy, dh, fw["h"], gam, fw["mask"], "f64")

    tP = [torch.tensor(x.reshape(S * B, H), requires_grad=True) for x in P]
    tres = torch.tensor(res, requires_grad=True)
    tg = torch.tensor(gam, requires_grad=True)
    tb = torch.tensor(bet, requires_grad=True)
    M = torch.from_numpy(fw["mask"].astype(np.float64))
    h = tres + sum(tP) * M / (1 - p)
    y = (torch.nn.functional.layer_norm(h, (H,), tg, tb, eps) if norm == "ln"
         else torch.nn.functional.rms_norm(h, (H,), tg, eps))
    L = (y * torch.from_numpy(dy)).sum() + (h * torch.from_numpy(dh)).sum()
    L.backward()
    np.testing.assert_allclose(bw["dres_exact"], tres.grad.numpy(), rtol=1e-10, atol=1e-12)
    for t in range(T):
        np.testing.assert_allclose(bw["dsum_exact"], tP[t].grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bw["dgamma"], tg.grad.numpy(), rtol=1e-10, atol=1e-12)
    if norm == "ln":
        np.testing.assert_allclose(bw["dbeta"], tb.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_dropout_backward_identity_needs_no_saved_input():
    """"Sequence Parallel" notes, MLP activation size: with Z' = Y B and
    Z = Z' (.) M, dL/dB = Y^T (dL/dZ (.) M) (times the inverted-dropout
    scale), so the pre-dropout Z' is never needed.  The oracle backward takes
    no Z' at all; Y^T d_sum must equal the finite-difference dL/dB."""
    rng = np.random.default_rng(19)
    m, k, n = 8, 5, 16       # tokens, inner dim, hidden
    Yin = rng.standard_normal((m, k))
    Bw = rng.standard_normal((k, n))
    res = rng.standard_normal((m, n))
    gam = rng.uniform(0.5, 1.5, n)
    dy = rng.standard_normal((m, n))
    p = 0.3
    pr = oracle.problem(1, 0, m, 1, n, "f64", "rms", p, 1e-5, 77)

    def loss(Bmat):
        return _loss(pr, [(Yin @ Bmat).reshape(m, 1, n)], res, gam, None, dy, None)

    fw = oracle.fwd(pr, [(Yin @ Bw).reshape(m, 1, n)], res, gam, None, "f64")
    bw = oracle.bwd(pr, dy, None, fw["h"], gam, fw["mask"], "f64")
    dB = Yin.T @ bw["dsum_exact"]
    # the same as Y^T (dL/dZ (.) M) / (1-p) with dL/dZ = d_residual
    np.testing.assert_allclose(dB, Yin.T @ (bw["dres_exact"] * fw["mask"]) / (1 - p), rtol=1e-13)
    for (a, b) in [(0, 0), (2, 7), (4, 15)]:
        e = np.zeros_like(Bw); e[a, b] = 1e-6
        fd = (loss(Bw + e) - loss(Bw - e)) / 2e-6
        np.testing.assert_allclose(fd, dB[a, b], rtol=1e-6, atol=1e-8)


def test_backward_p0_needs_no_mask_and_no_dh():
    rng = np.random.default_rng(20)
    T, S, B, H = 2, 4, 1, 16
    h = rng.standard_normal((S * B, H))
    dy = rng.standard_normal((S * B, H))
    gam = rng.uniform(0.5, 1.5, H)
    pr = oracle.problem(T, 0, S, B, H, "f64", "rms", 0.0, 1e-6, 0, nshards=T)
    a = oracle.bwd(pr, dy, None, h, gam, None, "f64")
    b = oracle.bwd(pr, dy, np.zeros_like(dy), h, gam, np.ones((S * B, H), np.uint8), "f64")
    for k in ["dres_exact", "dsum_exact", "dgamma"]:
        assert np.array_equal(a[k], b[k])
    assert np.array_equal(a["dres_exact"], a["dsum_exact"])
    # with gamma = 1 and eps -> 0 the RMS input gradient is orthogonal to h
    pr0 = oracle.problem(T, 0, S, B, H, "f64", "rms", 0.0, 1e-300, 0, nshards=T)
    c = oracle.bwd(pr0, dy, None, h, np.ones(H), None, "f64")
    np.testing.assert_allclose((c["dres_exact"] * h).sum(-1), 0.0, atol=1e-12)
    prl = oracle.problem(T, 0, S, B, H, "f64", "ln", 0.0, 1e-300, 0, nshards=T)
    d = oracle.bwd(prl, dy, None, h, np.ones(H), None, "f64")
    np.testing.assert_allclose(d["dres_exact"].sum(-1), 0.0, atol=1e-12)


def test_backward_rows_match_full_backward():
    rng = np.random.default_rng(21)
    T, S, B, H = 2, 8, 1, 24
    h = oracle.bf16_from_f64(rng.standard_normal((S * B // T, H)))
    dy = oracle.bf16_from_f64(rng.standard_normal((S * B // T, H)))
    dh = oracle.bf16_from_f64(rng.standard_normal((S * B // T, H)))
    gam = oracle.bf16_from_f64(rng.uniform(0.9, 1.1, H))
    mask = (rng.random((S * B // T, H)) > 0.1).astype(np.uint8)
    pr = oracle.problem(T, 1, S, B, H, "bf16", "ln", float(np.float32(0.1)), 1e-5, 0)
    full = oracle.bwd(pr, dy, dh, h, gam, mask)
    rows = oracle.bwd_rows(pr, dy, dh, h, gam, mask)
    for k in ["d_res", "d_sum", "dres_exact", "dsum_exact", "dgamma", "dbeta"]:
        assert np.array_equal(full[k], rows[k]), k


def _fwd_case(dtype, norm, seed):
    """Shard-sized inputs in storage form: T=4, S=16, B=3, H=40 (12 rows per
    shard), p = 0.25, LayerNorm beta when asked."""
    rng = np.random.default_rng(seed)
    T, S, B, H = 4, 16, 3, 40
    st = np.float32 if dtype == "f32" else None

    def draw(a):
        return a.astype(np.float32) if st else oracle.bf16_from_f64(a)

    parts = [draw(rng.standard_normal((S * B, H)) * 0.5) for _ in range(T)]
    res = draw(rng.standard_normal((S * B, H)))
    gam = draw(rng.uniform(0.5, 1.5, H))
    bet = draw(rng.standard_normal(H) * 0.1) if norm == "ln" else None
    return T, S, B, H, parts, res, gam, bet


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("norm", ["rms", "ln"])
def test_forward_rows_match_full_forward(dtype, norm):
    """The row-sampling forward (caller-given global row indices) equals the
    matching rows of the full forward over every shard: contiguous, scattered
    and reversed row sets inside each shard and across shards."""
    T, S, B, H, parts, res, gam, bet = _fwd_case(dtype, norm, 31)
    R = (S // T) * B
    p = float(np.float32(0.25))
    full = oracle.fwd(oracle.problem(T, 0, S, B, H, dtype, norm, p, 1e-5, 0x0123456789ABCDEF, nshards=T),
                      parts, res, gam, bet, dtype)
    sets = [np.arange(R), np.array([0, 5, 2, R - 1]), np.arange(R)[::-1]]
    for j in range(T):
        pr = oracle.problem(T, j, S, B, H, dtype, norm, p, 1e-5, 0x0123456789ABCDEF)
        for local in sets:
            grows = j * R + local
            got = oracle.fwd_rows(pr, grows, [q[grows] for q in parts], res[grows], gam, bet, dtype)
            for k in ["h", "y", "mask", "rstd", "mean", "h_exact", "y_exact"]:
                assert np.array_equal(got[k], full[k][grows]), (j, k)
    across = np.array([S * B - 1, 0, R, 3 * R + 1, R - 1])
    pr = oracle.problem(T, 0, S, B, H, dtype, norm, p, 1e-5, 0x0123456789ABCDEF)
    got = oracle.fwd_rows(pr, across, [q[across] for q in parts], res[across], gam, bet, dtype)
    for k in ["h", "y", "mask", "rstd", "mean"]:
        assert np.array_equal(got[k], full[k][across]), k
    # a slip of the row index moves the mask to another row's generator words
    slipped = oracle.fwd_rows(pr, across + 1, [q[across] for q in parts], res[across], gam, bet, dtype)
    assert not np.array_equal(slipped["mask"], full["mask"][across])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("norm", ["rms", "ln"])
def test_norm_stats_match_forward_and_library_moments(dtype, norm):
    """Row statistics of stored rows equal the forward's own rstd/mean on the
    same stored h, and torch's f64 moments: population variance (LayerNorm)
    or mean square (RMSNorm, as the squared 2-norm over H)."""
    T, S, B, H, parts, res, gam, bet = _fwd_case(dtype, norm, 32)
    eps = 1e-5
    pr = oracle.problem(T, 0, S, B, H, dtype, norm, float(np.float32(0.25)), eps, 7, nshards=T)
    full = oracle.fwd(pr, parts, res, gam, bet, dtype)
    rstd, mean = oracle.norm_stats(pr, full["h"], dtype)
    assert np.array_equal(rstd, full["rstd"])
    h = torch.from_numpy(oracle.to_f64(full["h"], dtype))
    if norm == "ln":
        assert np.array_equal(mean, full["mean"])
        var, mu = torch.var_mean(h, dim=-1, correction=0)
        np.testing.assert_allclose(mean, mu.numpy(), rtol=1e-13, atol=1e-15)
    else:
        assert np.all(mean == 0.0)
        var = torch.linalg.vector_norm(h, dim=-1) ** 2 / H
    np.testing.assert_allclose(rstd, 1.0 / np.sqrt(var.numpy() + eps), rtol=1e-13)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("norm", ["rms", "ln"])
def test_norm_of_stored_rows_is_the_norm_of_the_given_rows(dtype, norm):
    """The parity rule's re-evaluation of the norm on another stored h: on the
    forward's own h it reproduces the forward bit for bit; on a row with one
    element moved by one unit in the last place it equals torch's f64 norm of
    that row, and only that row changes."""
    from tests import parity

    T, S, B, H, parts, res, gam, bet = _fwd_case(dtype, norm, 33)
    eps = 1e-5
    pr = oracle.problem(T, 0, S, B, H, dtype, norm, float(np.float32(0.25)), eps, 7, nshards=T)
    full = oracle.fwd(pr, parts, res, gam, bet, dtype)
    same = parity.norm_of_stored_rows(pr, full["h"], gam, bet, dtype)
    for k in ["y", "y_exact", "rstd", "mean"]:
        assert np.array_equal(same[k], full[k]), k
    h2 = full["h"].copy()
    if dtype == "bf16":
        h2[3, 5] = h2[3, 5] + np.uint16(1)
    else:
        h2[3, 5] = np.nextafter(h2[3, 5], np.float32(np.inf))
    moved = parity.norm_of_stored_rows(pr, h2, gam, bet, dtype)
    changed = np.flatnonzero((moved["y_exact"] != full["y_exact"]).any(-1))
    assert list(changed) == [3]
    x = torch.from_numpy(oracle.to_f64(h2[3:4], dtype))
    g = torch.from_numpy(oracle.to_f64(gam, dtype))
    if norm == "ln":
        ref = torch.nn.functional.layer_norm(x, (H,), g, torch.from_numpy(oracle.to_f64(bet, dtype)), eps)
    else:
        ref = torch.nn.functional.rms_norm(x, (H,), g, eps)
    np.testing.assert_allclose(moved["y_exact"][3:4], ref.numpy(), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# a8/a9: sp2hp / hp2sp (LLM Infra Atlas "03 · Sequence Parallelism", §5)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,N,H", [(1, 4, 8), (2, 6, 8), (4, 16, 32), (3, 9, 24), (8, 16, 64)])
@pytest.mark.parametrize("dt", [np.uint16, np.float32])
def test_layout_roundtrip_and_all_to_all(T, N, H, dt):
    rng = np.random.default_rng(T * 100 + N)
    x = rng.integers(0, 2**16, (N, H)).astype(dt)
    hp = oracle.sp2hp(x, T)
    assert hp.shape == (T, N, H // T)
    assert np.array_equal(hp, oracle.sp2hp_all_to_all(x, T))
    back = oracle.hp2sp(hp)
    assert np.array_equal(back, x)
    assert np.array_equal(back, oracle.hp2sp_all_to_all(hp))
    y = rng.integers(0, 2**16, (T, N, H // T)).astype(dt)
    assert np.array_equal(oracle.sp2hp(oracle.hp2sp(y), T), y)
    # torch.split + cat restatement of the same map (library routines)
    ref = np.stack(np.split(x, T, axis=1))
    assert np.array_equal(hp, ref)
    if T == 1:
        assert np.array_equal(hp[0], x)


def test_oracle_rejects_invalid_problems():
    z = np.zeros((4, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.fwd(oracle.problem(3, 0, 4, 1, 8, "f32"), [z] * 3, z, np.ones(8, np.float32))
    with pytest.raises(ValueError):
        oracle.fwd(oracle.problem(2, 2, 4, 1, 8, "f32"), [z] * 2, z, np.ones(8, np.float32))
    with pytest.raises(ValueError):
        oracle.fwd(oracle.problem(2, 0, 4, 1, 8, "f32", p=1.0), [z] * 2, z, np.ones(8, np.float32))
    with pytest.raises(ValueError):
        oracle.bwd(oracle.problem(2, 0, 4, 1, 8, "f32", p=0.5), z, None, z, np.ones(8, np.float32),
                   None, "f32")
    with pytest.raises(ValueError):
        oracle.sp2hp(np.zeros((5, 8), np.float32), 2)


def test_forward_ties_round_half_to_even():
    """With p = 0.5 (1/(1-p) = 2) every kept element of these inputs sums to
    an exact bf16 midpoint: the stored h is the neighbour with the even
    mantissa (IEEE round-half-to-even), and a dropped element keeps its
    residual."""
    from tests import parity
    T, S, B, H = 2, 6, 1, 64
    P0, R, tie = parity.tie_inputs(S * B, H)
    pr = oracle.problem(T, 0, S, B, H, "bf16", "rms", 0.5, 1e-6, 5, nshards=T)
    gamma = np.full(H, 0x3F80, np.uint16)                    # 1.0
    out = oracle.fwd(pr, [P0, np.zeros_like(P0)], R, gamma, None, "bf16")
    kept = out["mask"] == 1
    assert 0.3 < kept.mean() < 0.7
    assert np.array_equal(out["h"], np.where(kept, tie, R))
