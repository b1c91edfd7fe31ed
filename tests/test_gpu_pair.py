"""The block-scaled w2 GEMM on the CTA-pair kernel.

With packed UE8M0 or MXFP8 scales, a batch whose routed rows average at least 512 per expert (and
whose hidden size is a multiple of 256) runs the w2 grouped GEMM on the two-SM MMA: a cluster of two
CTAs computes two consecutive 128-row tiles of one expert, each CTA holding its own rows of A and
one of the item's two weight bands (tcgen05.mma.cta_group::2).  The shapes below give experts an
odd number of tiles (the second CTA of the last pair then has no rows of the expert), single-tile
experts under Zipf-skewed routing, both weight layouts and both block-scaled formats; every token is
compared with the oracle's UE8M0 or MXFP8 mode.  A profiler trace checks which GEMM kernel ran.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import block_fp8_mixture_topk_gb300 as moe
from moe_testutil import assert_output_close, routing_of
from test_gpu_block_scaled import PackedLayer, run_packed_layer
from test_gpu_mxfp8 import run_mx_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"

# name, number, T, H, I, E, top-k, Zipf s.  Tiles per expert: [5, 5]; [9, 8, 9, 9];
# [21, 13, 7, 4, 2, 2, 1, 1].
PAIR_SHAPES = [
    ("pair_odd", 191, 1200, 256, 256, 2, 1, 0.0),
    ("pair_wide", 192, 2100, 512, 384, 4, 2, 0.0),
    ("pair_zipf", 193, 3000, 256, 256, 8, 2, 1.5),
]


@pytest.fixture(autouse=True)
def device_status_stays_clean():
    moe.moe_get_device_status(clear=True)
    yield
    assert moe.moe_get_device_status(clear=True) == 0


def workload(shape):
    name, number, T, H, I, E, topk, zipf_s = shape
    wl = mi.Workload(name, number, T, H, I, E, topk, zipf_s=zipf_s)
    assert wl.P >= 512 * E and H % 256 == 0    # the forward's condition for the pair kernel
    return wl


def tiles_per_expert(wl):
    _, okw = routing_of(wl)
    oids, _ = oracle.route(mi.router_logits(wl).numpy(), wl.topk, wl.renormalize, **okw)
    return (np.bincount(oids.reshape(-1), minlength=wl.E) + 127) // 128


@pytest.mark.parametrize("fmt", ["ue8m0_packed", "mxfp8"])
@pytest.mark.parametrize("shape", PAIR_SHAPES, ids=[s[0] for s in PAIR_SHAPES])
def test_pair_layer_all_tokens(shape, fmt):
    wl = workload(shape)
    assert np.any(tiles_per_expert(wl) % 2 == 1)
    out, ref = (run_packed_layer if fmt == "ue8m0_packed" else run_mx_layer)(wl)
    assert_output_close(out, ref["out"])


def gemm_kernels_of(fn):
    """Names of the grouped-GEMM kernels that one call of fn launches (profiler trace), or None if
    the profiler records no kernels of this library (its launches go through a statically linked
    CUDA runtime, which the profiler may not trace)."""
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = {e.key for e in prof.key_averages() if "grouped_gemm" in e.key}
    return names or None


def test_forward_takes_the_pair_kernel_for_many_rows_per_expert():
    """The w2 GEMM runs on the pair kernel exactly when moe_fp8_block_pair_path says so (the w13
    GEMM on the one-CTA block-scaled kernel in both cases)."""
    many = workload(PAIR_SHAPES[0])
    few = mi.Workload("pair_few", 195, 300, 256, 256, 2, 1)   # 150 rows per expert
    for wl, want_pair in ((many, True), (few, False)):
        clusters = moe.moe_fp8_block_pair_path(wl.T, wl.H, wl.E, wl.topk, "ue8m0_packed")
        assert (clusters > 0) == want_pair
        layer = PackedLayer(wl)
        rp, _ = routing_of(wl)
        h, l = mi.hidden(wl).to(DEV), mi.router_logits(wl).to(DEV)
        out_first = layer.forward(h, l, rp)
        names = gemm_kernels_of(lambda: layer.forward(h, l, rp))
        torch.cuda.synchronize()
        assert torch.isfinite(out_first.float()).all()
        if names is None:
            continue
        pair = [n for n in names if "grouped_gemm_pair_kernel" in n]
        one = [n for n in names if "grouped_gemm_bs_kernel" in n]
        if want_pair:
            assert len(pair) == 1 and len(one) == 1, names
        else:
            assert len(one) == 2 and not pair, names
