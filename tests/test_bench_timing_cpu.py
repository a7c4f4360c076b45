"""bench.py's timing consistency rule, on the CPU: the logits kernel is one part of a
step, so a kernel time above the step time means the two were not measured on the same
work, and bench.py refuses to print such a line."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_kernel_time_within_step_passes():
    bench.check_kernel_within_step(2.70, 2.79)
    bench.check_kernel_within_step(0.1830, 0.1830)


def test_kernel_time_above_step_is_refused():
    with pytest.raises(SystemExit) as e:
        bench.check_kernel_within_step(2.9742, 2.7908)
    assert "inconsistent timing" in str(e.value)
