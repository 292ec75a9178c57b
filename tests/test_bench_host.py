"""Host logic of bench.py that needs no GPU: the key that ties the committed in_proj DRAM
traffic to the code it was captured from, and the per-workload step defaults."""
import os
import sys

import pytest

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "flow_matching_image_flux3_b300", "csrc")


def test_launch_path_functions_are_found_whole():
    src = open(os.path.join(CSRC, "flux3.cu")).read()
    for head in bench.IN_PROJ_LAUNCH_PATH:
        text = bench._function_text(src, head)
        assert text.startswith(head) and text.rstrip().endswith("}")
        assert text.count("{") == text.count("}")
        assert src.count("\n" + head) == 1, head   # one definition, so the key is unambiguous


def test_key_follows_the_launch_path_only():
    src = open(os.path.join(CSRC, "flux3.cu")).read()
    text = bench._function_text(src, "flux3_status run_in_proj(")
    assert "launch_gemm<256, EPI_QKV_SWIGLU, 2>" in text   # the captured launch is in the keyed text
    assert "flux3_block_bwd" not in "".join(bench._function_text(src, h) for h in bench.IN_PROJ_LAUNCH_PATH)


@pytest.mark.parametrize("workload,steps", [("joint", 1000), ("loop", 2), ("joint_bwd", 50)])
def test_default_steps_per_workload(monkeypatch, workload, steps):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", workload])
    a = bench.parse()
    assert a.steps == steps and a.warmup >= 1
