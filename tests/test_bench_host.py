"""Host logic of bench.py, on CPU: the graph plan replays exactly the timed steps in order, the
algorithmic byte counts the roofline divides by agree with the oracle's packed layouts, the
weight rotation keeps the timed copies out of L2, and a stored DRAM-traffic figure is void once
any CUDA source it was taken with changes."""
import itertools
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402
from oracle import binplane as obp  # noqa: E402
from oracle import int4 as oint4  # noqa: E402
from oracle import nvfp4 as onv  # noqa: E402
from oracle import q8 as oq8  # noqa: E402
from oracle import sa as osa  # noqa: E402


class _PlanOnly(bench.Replay):
    """A replayer whose graphs are (first step, length) records instead of CUDA graphs."""

    def __init__(self, n, short):
        super().__init__(torch=None, step=None, n=n, short=short)
        self.captured = set()

    def _graph(self, start, length):
        self.captured.add((start % self.n, length))
        return (start % self.n, length)


def _replayed(plan):
    """Weight-copy indices in the order the plan's graphs run them."""
    return [(s + i) for s, length in plan for i in range(length)]


@pytest.mark.parametrize("n,short", [(2, 4), (3, 1), (11, 512), (11, 5), (7, 7)])
def test_graph_plan_replays_exactly_the_requested_steps_in_rotation_order(n, short):
    rep = _PlanOnly(n, short)
    for steps, start in itertools.product((0, 1, 2, 5, 6, 7, 11, 20, 23, 200, 2000), (0, 1, 6, 13)):
        got = _replayed(rep.plan(steps, start))
        # step i of a run reads weight copy i mod n; a graph starting at copy c replays
        # c, c+1, ... so its records must continue the rotation exactly
        assert [c % n for c in got] == [(start + i) % n for i in range(steps)], (steps, start)
        assert all(s + length <= n or length <= short for s, length in rep.plan(steps, start)), \
            "a long graph must not wrap past the last copy"


def test_graph_plan_reuses_whole_rotation_graphs_for_long_runs():
    rep = _PlanOnly(11, 16)
    plan = rep.plan(20000, 200)
    assert len(plan) <= 20000 // 11 + 2
    assert len(set(plan)) <= 3  # a head to the rotation boundary, the rotation, a tail
    assert sum(length for _, length in plan) == 20000


def test_algorithmic_bytes_equal_the_oracle_payload_on_aligned_shapes():
    for N, K in ((128, 128), (4096, 2560), (2560, 9728), (32768, 4096)):
        assert bench.algorithmic_int4_bytes(N, K) == oint4.packed_sizes(N, K)[2]
        assert bench.algorithmic_q8_bytes(N, K) == oq8.packed_sizes(N, K)[2]
        assert bench.algorithmic_nvfp4_bytes(N, K) == onv.packed_sizes(N, K)[2]
    for (K, N), P in itertools.product(synth.BINPLANE_SHAPES + ((256, 128),), (1, 3, 4, 8)):
        assert bench.algorithmic_binplane_bytes(P, N, K) == obp.packed_sizes(P, N, K)[2]
        for G in osa.GROUPS:
            assert bench.algorithmic_sa_bytes(P, G, N, K) == osa.packed_sizes(P, G, N, K)[2]


def test_headline_step_bytes_are_the_seven_projections_of_the_layer():
    total = sum(bench.algorithmic_int4_bytes(N, K) for _, K, N in synth.LAYER_4B)
    assert total == bench.LAYER_BYTES == 50_012_160


@pytest.mark.parametrize("copy_bytes", [1, 12_503_040, bench.LAYER_BYTES, 524_000_000, 10**10])
def test_weight_rotation_exceeds_l2(copy_bytes):
    l2 = 129 * 2**20
    n = bench.copies_for(copy_bytes, l2)
    assert n >= 2
    assert n * copy_bytes >= 4 * l2 or n == 2


def test_traffic_record_is_void_once_a_source_changes(tmp_path, monkeypatch):
    csrc = tmp_path / "bit_weight_gemv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("kernel a\n")
    (csrc / "b.cuh").write_text("helpers\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench._src_sha(("a.cu", "b.cuh"))
    assert h is not None and h == bench._src_sha(("b.cuh", "a.cu"))  # order-free
    (csrc / "b.cuh").write_text("helpers, edited\n")
    assert bench._src_sha(("a.cu", "b.cuh")) != h
    assert bench._src_sha(("a.cu", "missing.cu")) is None
    assert bench._src_sha(()) is None
