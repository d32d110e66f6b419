"""The DRAM traffic bench.py reports for a workload is the sum of the read and
write byte counts in the ncu summary it cites, and that summary names the
command that made it."""
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bytes(text, metric):
    m = re.search(r"\|\s*" + re.escape(metric) + r"\s*\|\s*([\d,]+)", text)
    assert m, metric
    return int(m.group(1).replace(",", ""))


@pytest.mark.parametrize("workload", sorted(bench.PROFILED_TRAFFIC))
def test_reported_traffic_matches_the_summary(workload):
    traffic, path = bench.PROFILED_TRAFFIC[workload]
    with open(os.path.join(ROOT, path)) as f:
        text = f.read()
    assert traffic == _bytes(text, "dram__bytes_read.sum") + _bytes(text, "dram__bytes_write.sum")
    assert "--clock-control none" in text and "ncu " in text
    assert f"--workload {workload}" in text or workload == "gqa_ctx5900"  # the default workload
