"""Host-side paths of bench.py that run without a GPU: the CPU baseline
(the oracle on a bounded sample) for every workload, and the command line."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

WORKLOADS = ["ffn_up", "dgrad", "decode", "fp8_256", "mxfp4_1024", "mxfp8_ffn_up", "ffn_up_q8out",
             "nvfp4_ffn_up", "bs16_ffn_up"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_cpu_baseline_runs_for_every_workload(name):
    cb = bench.cpu_baseline(name, None)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["unit"] == ("GB/s" if name == "decode" else "TFLOP/s")
    assert name in cb["sample"] or name == "decode"


def test_command_line_accepts_every_workload(monkeypatch):
    for name in WORKLOADS:
        monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", name, "--steps", "3", "--warmup", "3"])
        a = bench.parse()
        assert a.workload == name and a.gpus == 1 and a.impl == "ours"
