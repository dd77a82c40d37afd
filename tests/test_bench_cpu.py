"""bench.py's host-side choices, on the CPU: how many weight copies a timed
loop rotates through (enough to beat the L2, a divisor of both graph
lengths) and which workload --workload selects."""
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402
import synthetic  # noqa: E402


def test_weight_copies_beat_the_l2_and_divide_the_graphs():
    for wl in (synthetic.HEADLINE, synthetic.GRAPH_8192, synthetic.CHAIN_4096):
        c = bench.weight_copies(wl.weight_bytes)
        assert bench.GRAPH_STEPS % c == 0 and bench.E2E_GRAPH_STEPS % c == 0
        assert c * wl.weight_bytes > 2 * bench.L2_BYTES, (wl.name, c)
    assert bench.weight_copies(synthetic.HEADLINE.weight_bytes) == 3
    # A weight too small to outgrow the L2 gets the largest rotation.
    assert bench.weight_copies(synthetic.TINY.weight_bytes) == 30


def test_workload_selection():
    try:
        for name, attr in bench.WORKLOAD_CHOICES.items():
            bench._WORKLOAD = name
            assert bench.workload() is getattr(synthetic, attr)
        assert bench.parse_args([]).workload == "headline"
    finally:
        bench._WORKLOAD = "headline"
