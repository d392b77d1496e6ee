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


def test_cpu_baseline_heads_spread_over_the_batch():
    # the CPU-baseline sample covers heads across the whole range, head 0 first, never past the last
    assert bench.spread_heads(40, 8) == [0, 5, 10, 15, 20, 25, 30, 35]
    assert bench.spread_heads(48, 8) == [0, 6, 12, 18, 24, 30, 36, 42]
    assert bench.spread_heads(3, 8) == [0, 1, 2]
    assert bench.spread_heads(1, 8) == [0]
    assert bench.spread_heads(16, 1) == [0]


def test_kernel_hash_ignores_comments_only():
    # the ncu figures in profiles/ stay attached to the kernel while only its comments change
    a = "int x = 1;  // one\n/* block\n comment */\n\n  int y = x + 2;\n"
    b = "// header\nint x = 1;\nint y = x + 2;  /* two */\n"
    assert bench.code_only(a) == bench.code_only(b) == "int x = 1;\nint y = x + 2;"
    assert bench.code_only("int x = 2;") != bench.code_only("int x = 1;")
