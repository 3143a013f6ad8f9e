"""Host-side helpers of bench.py: the rotation count that keeps every kernel's
working set out of the L2, the algorithmic byte counts, and the packed
host/device blocks the end-to-end pipeline copies once each way."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from residual_sp_rs_gb300 import synthetic as syn  # noqa: E402


def test_rotation_exceeds_twice_l2_for_every_kernel():
    l2 = 132 * 2**20
    for name in ("pages_rms_bf16", "gpt_ln_bf16", "large_rms_bf16"):
        w = syn.WORKLOADS[name]
        rows = w.S * w.B
        kb = (bench.fwd_bytes(w, rows), bench.bwd_bytes(w, rows), bench.layout_bytes(w, rows))
        per_set = sum(kb) * 2  # any set is larger than each kernel's own bytes
        n = bench.rotation_sets(l2, per_set, *kb)
        assert n >= 2
        for b in kb:
            assert n * b > 2 * l2, (name, n, b)
        # one set fewer would leave the smallest kernel's rotation within 2x L2
        if n > 2:
            assert (n - 2) * min(kb) <= 2 * l2


def test_rotation_at_least_two_sets():
    assert bench.rotation_sets(1024, 10**12, 10**12) == 2


def test_pages_shape_byte_counts():
    # the pages' shape: 11 bytes per element each way (2T+7 at T=2, and
    # dy, dh_out, h, d_residual, d_sum + mask), 2e per element for the layout
    w = syn.WORKLOADS["pages_rms_bf16"]
    rows = w.S * w.B
    elems = rows * w.H
    assert bench.fwd_bytes(w, rows) == 11 * elems + 4 * rows + 2 * w.H
    assert bench.bwd_bytes(w, rows) == 11 * elems + 4 * rows + w.H * (2 + 4)
    assert bench.layout_bytes(w, rows) == 4 * elems


def test_packed_block_views_share_one_aligned_buffer():
    named = [("a", torch.zeros(3, 5, dtype=torch.bfloat16)),
             ("b", torch.zeros(7, dtype=torch.float32)),
             ("c", torch.zeros(2, 3, dtype=torch.uint8))]
    flat, views = bench.packed_block(named, "cpu")
    assert flat.dtype == torch.uint8
    base = flat.data_ptr()
    ends = []
    for (_, t), v in zip(named, views):
        assert v.shape == t.shape and v.dtype == t.dtype
        off = v.data_ptr() - base
        assert off % 256 == 0
        ends.append((off, off + t.numel() * t.element_size()))
    # in order, not overlapping, inside the buffer
    for (s0, e0), (s1, _) in zip(ends, ends[1:]):
        assert e0 <= s1
    assert ends[-1][1] <= flat.numel()
    # writing a view writes the one buffer that is copied
    views[1].fill_(1.5)
    assert torch.equal(flat[ends[1][0]:ends[1][1]].view(torch.float32), torch.full((7,), 1.5))


def test_graph_steps_cover_the_timed_run_exactly():
    for k in (1, 20, 97, 200, 512):
        assert bench.graph_steps(k) == k
    for k in (1000, 50000, 4096):
        g = bench.graph_steps(k)
        assert k % g == 0 and 16 <= g <= bench.MAX_GRAPH_STEPS


def test_graph_rotation_continues_across_replays():
    """Replaying the graph variants in turn walks the sets in order, so every
    set is reused only after all the others (the L2 rule holds across the
    replay boundaries), and there are at least the sets the rule needs."""
    for g, need in ((20, 23), (200, 23), (256, 23), (5, 2), (97, 23), (512, 3)):
        n, variants = bench.graph_rotation(g, need)
        assert n >= need
        seq = []
        for rep in range(3 * variants):
            v = rep % variants
            seq += [((v * g) % n + i) % n for i in range(g)]
        assert seq == [i % n for i in range(len(seq))], (g, need)


def test_timed_runs_reach_the_minimum_span():
    durations = iter([10.0] * 100)
    runs = bench.timed_runs(lambda: next(durations), min_ms=50.0, min_runs=3)
    assert len(runs) == 5 and sum(runs) >= 50.0
    runs = bench.timed_runs(lambda: 100.0, min_ms=50.0, min_runs=3)
    assert len(runs) == 3


def test_ranks_own_their_sequence_shard():
    # one GPU plays the whole tensor-parallel group
    assert bench.tp_dp_rank(0, 1, 2) == (0, 2, 0)
    # N ranks: rank r is tensor-parallel rank r % T of replica r // T
    got = [bench.tp_dp_rank(r, 8, 2) for r in range(8)]
    assert got == [(r % 2, 1, r // 2) for r in range(8)]
    shards = {(dp, j) for j, _, dp in got}
    assert len(shards) == 8   # every (replica, shard) pair exactly once
