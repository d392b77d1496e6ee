"""Host-side helpers of bench.py that need no GPU."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_cpulist_parser_reads_the_sysfs_format():
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("5") == {5}
    assert bench.parse_cpulist("72-143") == set(range(72, 144))
    assert bench.parse_cpulist("\n") == set()


def test_launch_count_per_step_follows_the_rounds():
    # each k-means round launches the assignment, the update and the three argsort kernels
    assert bench.launches_per_step({"iters": 4}) == bench.launches_per_step({"iters": 3}) + 5
