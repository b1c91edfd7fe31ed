"""The seeded synthetic inputs both sides read (moe_inputs): deterministic, every tensor and
every expert regenerable on its own, the shapes and distributions each workload states, and
the Zipf router offsets of the skewed workload."""
import math

import numpy as np
import pytest
import torch

import moe_inputs as mi


def test_workload_shapes():
    want = {"tiny": (16, 256, 256, 4, 2), "mixtral": (512, 4096, 14336, 8, 2),
            "dsv3": (4096, 7168, 2048, 256, 8), "qwen3_skew": (16384, 2048, 768, 128, 8)}
    for name, (T, H, I, E, k) in want.items():
        wl = mi.WORKLOADS[name]
        assert (wl.T, wl.H, wl.I, wl.E, wl.topk) == (T, H, I, E, k)
    d = mi.WORKLOADS["dsv3_decode"]
    assert (d.H, d.I, d.E, d.topk) == (7168, 2048, 256, 8)
    assert mi.WORKLOADS["dsv3"].n_group == 8 and mi.WORKLOADS["dsv3"].topk_group == 4


def test_generators_are_deterministic_and_per_tensor():
    wl = mi.WORKLOADS["tiny"]
    assert torch.equal(mi.hidden(wl), mi.hidden(wl))
    assert torch.equal(mi.router_logits(wl), mi.router_logits(wl))
    assert torch.equal(mi.w13_bf16(wl), mi.w13_bf16(wl))
    assert mi.hidden(wl).dtype == torch.bfloat16 and mi.hidden(wl).shape == (wl.T, wl.H)
    assert mi.router_logits(wl).dtype == torch.float32 and mi.router_logits(wl).shape == (wl.T, wl.E)
    # another seed (a replica's batch) gives other tokens, the same shapes
    other = wl.with_(number=wl.number + 100)
    assert not torch.equal(mi.hidden(wl), mi.hidden(other))
    assert mi.hidden(other).shape == mi.hidden(wl).shape


def test_any_expert_subset_regenerates_the_same_weights():
    """The oracle quantises the experts it needs one at a time; the GPU side generates them in
    batches: both must see the same bytes."""
    wl = mi.WORKLOADS["tiny"]
    full13, full2 = mi.w13_bf16(wl), mi.w2_bf16(wl)
    assert full13.shape == (wl.E, 2 * wl.I, wl.H) and full2.shape == (wl.E, wl.H, wl.I)
    for ex in ([3], [1, 2], [0, 3]):
        assert torch.equal(mi.w13_bf16(wl, experts=ex), full13[ex])
        assert torch.equal(mi.w2_bf16(wl, experts=ex), full2[ex])
    assert not torch.equal(full13[0], full13[1])


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode"])
def test_distributions(name):
    wl = mi.WORKLOADS[name].with_tokens(64) if name == "dsv3_decode" else mi.WORKLOADS[name]
    h = mi.hidden(wl).float()
    assert abs(h.mean().item()) < 0.05 and abs(h.std().item() - 1.0) < 0.05
    lg = mi.router_logits(wl)
    assert abs(lg.mean().item()) < 0.1 and abs(lg.std().item() - 1.0) < 0.1
    w = mi.w13_bf16(wl, experts=[0]).float()
    assert abs(w.std().item() - 0.02) < 0.001 and abs(w.mean().item()) < 0.001
    bias = mi.expert_bias(wl)
    if name == "dsv3_decode":
        assert bias is not None and bias.shape == (wl.E,) and abs(bias.std().item() - 0.01) < 0.003
    else:
        assert bias is None


def test_zipf_offsets_of_the_skewed_workload():
    wl = mi.WORKLOADS["qwen3_skew"].with_tokens(8)
    plain = wl.with_(zipf_s=0.0)
    d = (mi.router_logits(wl) - mi.router_logits(plain)).numpy()
    want = np.array([-1.2 * math.log(e + 1.0) for e in range(wl.E)], dtype=np.float32)
    assert np.allclose(d, want[None, :], atol=1e-5)
