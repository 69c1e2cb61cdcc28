"""The ncu summaries under profiles/ from which bench.py reads each timed
kernel's DRAM traffic record the sha256 of the kernel sources they were
captured on, and bench.py reports the traffic only while those sources are
unchanged.  These tests check that every such summary is current (a kernel
edit without a new capture fails here instead of turning the bench's traffic
field into null) and that each figure is plausible against the kernel's
algorithmic bytes: DRAM traffic can exceed them (re-reads, the fp32 dq
accumulator) but not fall far below them."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_for_tests", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

B, H, T, D = 1, 32, 8192, 128  # the headline workload the forward and backward summaries cover


@pytest.mark.parametrize(
    "path, key, sources, algorithmic",
    [
        # q, k, v read and o written in bf16, lse in fp32: per launch
        (bench.PROFILE_SUMMARY, "traffic_bytes_per_launch", bench.KERNEL_SOURCES,
         4 * B * H * T * D * 2 + B * H * T * 4),
        # q, k, v, o, dout, lse read; dq, dk, dv written (bf16): per head
        (bench.BACKWARD_PROFILE, "traffic_bytes_per_head", bench.BACKWARD_SOURCES,
         (8 * T * D * 2 + T * 4)),
        # one cached key and value (bf16, d = 128): per position
        (bench.DECODE_PROFILE, "traffic_bytes_per_position", bench.DECODE_SOURCES, 2 * D * 2),
    ],
    ids=["forward", "backward", "decode"],
)
def test_recorded_traffic_is_current_and_plausible(path, key, sources, algorithmic):
    value = bench.recorded_figure(path, key, sources)
    assert value is not None, f"{os.path.basename(path)}: source hash differs or {key} missing"
    assert 0.9 * algorithmic <= value <= 3.0 * algorithmic, (value, algorithmic)
