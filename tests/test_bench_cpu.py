"""Host-side accounting of bench.py (no GPU): the algorithmic bytes the roofline divides by."""
import importlib.util
import os
import sys

import torch

import moe_inputs as mi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_expert_weight_bytes():
    b = load_bench()
    wl = mi.WORKLOADS["dsv3"]
    H, I = wl.H, wl.I
    w13, both = b.expert_weight_bytes(wl)
    assert w13 == 2 * I * H + (2 * I // 128) * (H // 128) * 4
    assert both == 3 * H * I + ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128)) * 4
    f13, fboth = b.expert_weight_bytes(wl, nvfp4=True)
    # 4-bit codes and one e4m3 scale per 16 weights (9/16 byte per weight) plus a global scale
    assert f13 == 2 * I * H * 9 // 16 + 4
    assert fboth == 3 * H * I * 9 // 16 + 8
    # the packed layout has exactly these bytes (16 x 64 code + 16 x 8 scale bytes per 16 x 128)
    assert (2 * I // 16) * (H // 128) * 1152 == f13 - 4


def test_touched_experts_per_pass():
    b = load_bench()
    ids = torch.tensor([[0, 1], [1, 2], [3, 0], [2, 2], [5, 6]])
    assert b.touched_per_pass(ids, 8) == 6
    assert b.touched_per_pass(ids, 2) == 3 + 3 + 2
    assert b.touched_per_pass(ids, 1) == 2 + 2 + 2 + 1 + 2
