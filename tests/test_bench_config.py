"""bench.py names every override of a preset workload in its config object, so a line
measured with --layout, --P, --seed or --head-dim cannot pass for the preset."""
import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from online_softmax_merge_gb300.inputs import WORKLOADS  # noqa: E402


def _args():
    return argparse.Namespace(out_dtype="fp32", gpus=1)


def test_preset_has_no_override_note():
    c = bench.config_obj(WORKLOADS["c4"], _args())
    assert "overridden" not in c["workload"]
    assert c["head_dim"] == 128 and c["P"] == 16


def test_overrides_are_named():
    w = WORKLOADS["c4"].with_(head_dim=64, layout="zigzag")
    c = bench.config_obj(w, _args())
    assert "overridden: layout=zigzag, head_dim=64" in c["workload"]
    assert c["head_dim"] == 64 and c["layout"] == "zigzag"
    assert w != WORKLOADS["c4"]          # the stored DRAM counters are then not reported
