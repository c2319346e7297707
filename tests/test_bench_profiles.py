"""The ncu summaries bench.py reads its roofline traffic from.

Each (operand kind, workload) that bench.py maps to a profile must find the
file, a DRAM figure in it, and the kernel-source key of the current GEMM
sources; otherwise the bench would report traffic null without saying why.
A kernel change that is not comment-only changes the key, and this test then
asks for the capture to be taken again.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("quant,workload", sorted(bench.TRAFFIC_PROFILES,
                                                  key=lambda q: (str(q[0]), q[1])))
def test_profile_traffic_is_current(quant, workload):
    assert workload in bench.WORKLOADS
    path = os.path.join(ROOT, "profiles", bench.TRAFFIC_PROFILES[(quant, workload)])
    assert os.path.exists(path), path
    traffic = bench.recorded_traffic(quant, workload)
    assert traffic is not None, (
        f"{path}: no gate/up DRAM figure for the current kernel sources "
        f"(kernel_source_key {bench.kernel_source_key()})")
    assert traffic > 0


def test_source_key_format():
    """The key is the first 16 hex digits of a sha256."""
    key = bench.kernel_source_key()
    assert key is not None and len(key) == 16
    int(key, 16)
