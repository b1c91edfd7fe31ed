"""The decode path (steps of up to 8 tokens: a prologue kernel, one kernel that routes, sorts
and runs both GEMMs, then the weighted sum): the whole layer against the oracle on every
token, the same steps through the tile GEMMs, both weight layouts, both scale formats, the
in-kernel routing against the routing kernel bit for bit, the routing kernel's ids where the
in-kernel selection does not apply, and repeated calls on one workspace (the counters start
from zero on every call)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import block_fp8_mixture_topk_gb300 as moe
from moe_testutil import Layer, assert_output_close, routing_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def workload(name, T):
    return mi.WORKLOADS[name].with_tokens(T)


def forward(layer, hidden, logits, rp, decode, packed=False, workspace=None):
    wl = layer.wl
    w13, w2 = layer.w13q, layer.w2q
    if packed:
        w13, w2 = moe.moe_fp8_block_pack_weights(w13), moe.moe_fp8_block_pack_weights(w2)
    return moe.moe_fp8_block_forward(hidden, logits, w13, layer.w13s, w2, layer.w2s, wl.topk, wl.renormalize, rp,
                                     scale_fmt=layer.scale_fmt, decode=decode, workspace=workspace)


def oracle_out(layer, hidden, logits, okw):
    wl = layer.wl
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    w13q, w13s, w2q, w2s = layer.oracle_weights(set(oids.reshape(-1).tolist()))
    fmt = oracle.SCALE_UE8M0 if layer.scale_fmt == "ue8m0" else oracle.SCALE_F32
    return oracle.moe_forward(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, wl.renormalize,
                              scale_fmt=fmt, **okw)["out"]


CASES = [
    ("dsv3_decode", 1), ("dsv3_decode", 2), ("dsv3_decode", 3), ("dsv3_decode", 8),
    ("mixtral", 1), ("mixtral", 8),      # 8 experts, top-2: up to 8 rows on one expert
    ("tiny", 5), ("tiny", 8),            # 4 experts, top-2: experts with several rows
]


@pytest.mark.parametrize("name,T", CASES)
def test_decode_path_matches_oracle_and_tile_path(name, T):
    wl = workload(name, T)
    assert moe.moe_fp8_block_decode_path(T, wl.H, wl.I, wl.topk, "on")
    layer = Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    h, l = hidden.to(DEV), logits.to(DEV)
    dec = forward(layer, h, l, rp, "on")
    dec_packed = forward(layer, h, l, rp, "on", packed=True)
    tile = forward(layer, h, l, rp, "off")
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(clear=True) == 0
    # the two weight layouts read the same bytes in the same order
    assert torch.equal(dec, dec_packed)
    ref = oracle_out(layer, hidden, logits, okw)
    assert_output_close(dec, ref)
    assert_output_close(tile, ref)
    # decode and tile paths differ only in the fp32 summation order
    assert_output_close(dec, tile.float().cpu().double().numpy())


@pytest.mark.parametrize("T,H,I,E,topk", [(1, 128, 128, 1, 1), (8, 128, 256, 1, 1), (6, 256, 128, 3, 3),
                                          (4, 384, 384, 32, 32)])
def test_decode_path_edge_shapes(T, H, I, E, topk):
    """One expert and top-1 (a dense block-FP8 MLP), every token on the single expert (8 rows),
    top-k equal to the number of experts, and K smaller than the eight warps' K blocks."""
    wl = mi.Workload("dec_edge", 90 + T + E, T, H, I, E, topk)
    layer = Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = forward(layer, hidden.to(DEV), logits.to(DEV), rp, "on")
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(clear=True) == 0
    assert_output_close(out, oracle_out(layer, hidden, logits, okw))


def test_decode_path_ue8m0_scales():
    wl = workload("dsv3_decode", 4)
    layer = Layer(wl, scale_fmt="ue8m0")
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = forward(layer, hidden.to(DEV), logits.to(DEV), rp, "on")
    assert_output_close(out, oracle_out(layer, hidden, logits, okw))


def test_decode_path_repeated_calls_on_one_workspace():
    """Ten calls on one workspace, on changing inputs: each equals a call on a fresh workspace
    (the counters and the ticket are zeroed by every call's decode prologue)."""
    wl = workload("dsv3_decode", 2)
    layer = Layer(wl)
    rp, _ = routing_of(wl)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.topk), dtype=torch.uint8,
                     device=DEV)
    ws.fill_(0x7F)   # garbage in every counter before the first call
    for seed in range(10):
        wl_s = wl.with_(number=wl.number + 700 + seed)
        h, l = mi.hidden(wl_s).to(DEV), mi.router_logits(wl_s).to(DEV)
        got = forward(layer, h, l, rp, "on", workspace=ws)
        fresh = torch.empty_like(ws)
        want = forward(layer, h, l, rp, "on", workspace=fresh)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    assert moe.moe_get_device_status(clear=True) == 0


@pytest.mark.parametrize("T", [1, 8])
def test_decode_path_replays_from_a_cuda_graph(T):
    """The decode path captured once in a CUDA graph and replayed on new inputs: the counters
    and the ticket are zeroed inside every replay, and each replay equals an eager call."""
    wl = workload("dsv3_decode", T)
    layer = Layer(wl)
    rp, _ = routing_of(wl)
    w13p, w2p = moe.moe_fp8_block_pack_weights(layer.w13q), moe.moe_fp8_block_pack_weights(layer.w2q)
    hid = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    log = torch.empty(wl.T, wl.E, dtype=torch.float32, device=DEV)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.topk), dtype=torch.uint8,
                     device=DEV)
    hid.copy_(mi.hidden(wl).to(DEV))
    log.copy_(mi.router_logits(wl).to(DEV))

    def step():
        moe.moe_fp8_block_forward(hid, log, w13p, layer.w13s, w2p, layer.w2s, wl.topk, wl.renormalize, rp,
                                  out=out, workspace=ws, decode="on")

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in range(3):
        wl_s = wl.with_(number=wl.number + 900 + seed)
        h, l = mi.hidden(wl_s).to(DEV), mi.router_logits(wl_s).to(DEV)
        hid.copy_(h)
        log.copy_(l)
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        want = moe.moe_fp8_block_forward(h, l, w13p, layer.w13s, w2p, layer.w2s, wl.topk, wl.renormalize, rp,
                                         decode="on")
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    assert moe.moe_get_device_status(clear=True) == 0


def routing_in_workspace(ws, T, topk):
    """The decode kernel's CTA 0 writes the step's chosen experts and router weights at the start
    of the forward workspace: ids [T*topk] int32, then the weights [T*topk] fp32 at the next
    256-byte boundary (the layout's first two regions)."""
    P = T * topk
    off = (P * 4 + 255) // 256 * 256
    return ws[:P * 4].view(torch.int32).view(T, topk), ws[off:off + P * 4].view(torch.float32).view(T, topk)


ROUTE_CASES = [
    ("dsv3_decode", 1, True), ("dsv3_decode", 2, True), ("dsv3_decode", 8, True),   # sigmoid, 8 groups, bias
    ("mixtral", 1, True), ("mixtral", 8, True), ("mixtral", 4, False),               # softmax, 1 expert per lane
    ("qwen3_skew", 4, True), ("qwen3_skew", 3, False),                               # 4 experts per lane
    ("tiny", 8, True),
]


@pytest.mark.parametrize("name,T,renorm", ROUTE_CASES)
def test_decode_kernel_routes_like_the_routing_kernel(name, T, renorm):
    """Every CTA of the decode kernel routes the step's tokens itself with the routing kernel's
    selection: the ids and weights it writes are bit-identical to moe_route_topk's, and the
    layer equals the oracle."""
    wl = workload(name, T).with_(renormalize=renorm)
    layer = Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    h, l = hidden.to(DEV), logits.to(DEV)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(T, wl.H, wl.I, wl.E, wl.topk), dtype=torch.uint8, device=DEV)
    out = forward(layer, h, l, rp, "on", workspace=ws)
    ids, wts = moe.moe_route_topk(l, wl.topk, wl.renormalize, rp)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(clear=True) == 0
    got_ids, got_wts = routing_in_workspace(ws, T, wl.topk)
    assert torch.equal(got_ids, ids)
    assert torch.equal(got_wts.view(torch.int32), wts.view(torch.int32))
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    assert np.array_equal(ids.cpu().numpy(), oids)
    assert_output_close(out, oracle_out(layer, hidden, logits, okw))


def test_decode_kernel_routing_on_tied_scores():
    """Logits on a coarse grid: many equal scores, so the fp32 fast path hands the token to the
    exact fp64 scores and equal values go to the lower expert index -- in the decode kernel as in
    the routing kernel and the oracle."""
    wl = workload("dsv3_decode", 8)
    layer = Layer(wl)
    hidden = mi.hidden(wl)
    logits = torch.round(mi.router_logits(wl) * 2.0) / 2.0
    rp, okw = routing_of(wl)
    h, l = hidden.to(DEV), logits.to(DEV)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.topk), dtype=torch.uint8,
                     device=DEV)
    out = forward(layer, h, l, rp, "on", workspace=ws)
    ids, wts = moe.moe_route_topk(l, wl.topk, wl.renormalize, rp)
    torch.cuda.synchronize()
    got_ids, got_wts = routing_in_workspace(ws, wl.T, wl.topk)
    assert torch.equal(got_ids, ids) and torch.equal(got_wts, wts)
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    assert np.array_equal(ids.cpu().numpy(), oids)
    assert_output_close(out, oracle_out(layer, hidden, logits, okw))


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
def test_decode_path_with_the_routing_kernel(scoring):
    """512 experts (16 per lane): the decode kernel takes the routing kernel's ids and weights
    instead of routing in every CTA; the layer still equals the oracle and the tile path."""
    wl = mi.Workload("dec_e512", 77, 2, 256, 256, 512, 8)
    if scoring == "sigmoid":
        wl = wl.with_(scoring=mi.SIGMOID, n_group=8, topk_group=4, routed_scaling=2.5, bias_std=0.01)
    assert moe.moe_fp8_block_forward_kernel_count(wl.T, wl.H, wl.I, wl.E, wl.topk, decode="on") == 4
    layer = Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    h, l = hidden.to(DEV), logits.to(DEV)
    out = forward(layer, h, l, rp, "on")
    tile = forward(layer, h, l, rp, "off")
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(clear=True) == 0
    ref = oracle_out(layer, hidden, logits, okw)
    assert_output_close(out, ref)
    assert_output_close(tile, ref)
