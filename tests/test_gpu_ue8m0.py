"""GPU parity of the FLOAT32_CEIL_UE8M0 scale format (every scale rounded up to a power of
two) against the oracle in the same format, through the C ABI: quantised bytes and scales
bit-exact, the SiLU requantisation within one code, the whole layer (routed and masked) within
the layer tolerance."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import block_fp8_mixture_topk_gb300 as moe
from moe_testutil import Layer, assert_output_close, routing_of, unpadded_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
UE8M0 = oracle.SCALE_UE8M0


@pytest.fixture(autouse=True)
def device_status_stays_clean():
    moe.moe_get_device_status(clear=True)
    yield
    assert moe.moe_get_device_status(clear=True) == 0


@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 384), (4096, 7168)])
def test_group_quant_ue8m0_bit_exact(rows, cols):
    g = torch.Generator().manual_seed(rows)
    x = torch.randn(rows, cols, generator=g) * torch.exp2(torch.randint(-40, 40, (rows, 1), generator=g).float())
    x[0, :128] = 0.0
    if rows > 2:
        x[1, :128] = 448.0 * 2.0 ** 3            # a power-of-two scale stays
        x[2, 5] = -1e30
    x = x.to(torch.bfloat16)
    q, s = moe.fp8_group_quant(x.to(DEV), "ue8m0")
    oq, os_ = oracle.quant_1x128_bf16(mi.bf16_bits(x), UE8M0)
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.all(np.frexp(s.cpu().numpy())[0] == 0.5)


@pytest.mark.parametrize("name,experts", [("tiny", None), ("dsv3", [3, 200])])
def test_block_quant_weight_ue8m0_bit_exact(name, experts):
    wl = mi.WORKLOADS[name]
    for w in (mi.w13_bf16(wl, DEV, experts), mi.w2_bf16(wl, DEV, experts)):
        q, s = moe.fp8_block_quant_weight(w, "ue8m0")
        oq, os_ = oracle.quant_128x128_bf16(mi.bf16_bits(w), UE8M0)
        assert np.array_equal(s.cpu().numpy(), os_)
        assert np.array_equal(q.cpu().numpy(), oq)


def test_silu_requant_ue8m0_within_one_code():
    wl = mi.Workload("ue8m0stage", 55, 200, 512, 256, 16, 4)
    layer = Layer(wl, scale_fmt="ue8m0")
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    oids, ow = oracle.route(logits.numpy(), wl.topk, True)
    perm = moe.moe_align_permute(torch.from_numpy(oids).to(DEV), wl.E)
    q, s = moe.fp8_group_quant(hidden.to(DEV), "ue8m0")
    used = int(perm["padded_offsets"][-1].item())
    sp = perm["sorted_pair_ids"].cpu().numpy()[:used].astype(np.int64)
    valid = np.nonzero(sp >= 0)[0]
    rows = perm["max_rows"]
    A = torch.zeros(rows, wl.H, dtype=torch.uint8)
    As = torch.ones(rows, wl.H // 128, dtype=torch.float32)
    A[torch.from_numpy(valid)] = q.cpu()[torch.from_numpy(sp[valid] // wl.topk)]
    As[torch.from_numpy(valid)] = s.cpu()[torch.from_numpy(sp[valid] // wl.topk)]
    oq = torch.empty(rows, wl.I, dtype=torch.uint8, device=DEV)
    osc = torch.empty(rows, wl.I // 128, dtype=torch.float32, device=DEV)
    moe.fp8_block_grouped_gemm(A.to(DEV), As.to(DEV), (wl.H // 128, 1), layer.w13q, layer.w13s, perm["tile_expert"],
                               perm["tile_row0"], perm["num_tiles"], "silu_mul_quant", out_q=oq, out_scale=osc,
                               out_scale_strides=(wl.I // 128, 1), scale_fmt="ue8m0")
    w13q, w13s, w2q, w2s = layer.oracle_weights(range(wl.E))
    ref = oracle.moe_forward(mi.bf16_bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, scale_fmt=UE8M0)
    m = unpadded_rows(perm["padded_offsets"].cpu().numpy(), ref["offsets"])
    gs = osc.cpu().numpy()[m]
    assert np.all(np.frexp(gs)[0] == 0.5)
    # a scale may differ by one power of two where the fp32 amax sits on a boundary
    ratio = gs / ref["a2s"]
    assert np.all((ratio == 1.0) | (ratio == 2.0) | (ratio == 0.5)) and (ratio == 1.0).mean() > 0.99
    gq = oq.cpu().numpy()[m].astype(np.int32)
    same_rows = np.all(ratio == 1.0, axis=1)
    rq = ref["a2q"].astype(np.int32)
    same = gq[same_rows] == rq[same_rows]
    assert same.mean() >= 0.99
    d = ~same
    assert np.all(np.abs((gq[same_rows][d] & 0x7F) - (rq[same_rows][d] & 0x7F)) <= 1)


@pytest.mark.parametrize("name,tokens", [("tiny", None), ("dsv3", [0, 1, 2047, 4095]),
                                         ("qwen3_skew", [0, 9000, 16383])])
def test_forward_ue8m0_matches_oracle(name, tokens):
    wl = mi.WORKLOADS[name]
    layer = Layer(wl, scale_fmt="ue8m0")
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = layer.forward(hidden.to(DEV), logits.to(DEV), rp)
    torch.cuda.synchronize()
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    toks = range(wl.T) if tokens is None else tokens
    w13q, w13s, w2q, w2s = layer.oracle_weights(set(oids[list(toks)].reshape(-1).tolist()))
    ref = oracle.moe_forward(mi.bf16_bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, wl.renormalize,
                             tokens=tokens, scale_fmt=UE8M0, **okw)
    assert_output_close(out, ref["out"], rows=tokens)


def test_masked_ue8m0_matches_oracle():
    E, M, H, I = 3, 50, 256, 256
    counts = [50, 0, 13]
    wl = mi.Workload("masked_ue8m0", 66, E * M, H, I, E, 1)
    layer = Layer(wl, scale_fmt="ue8m0")
    g = torch.Generator().manual_seed(66)
    hidden = torch.randn(E, M, H, generator=g).to(torch.bfloat16)
    out = moe.moe_fp8_block_forward_masked(hidden.to(DEV), torch.tensor(counts, dtype=torch.int32, device=DEV),
                                           layer.w13q, layer.w13s, layer.w2q, layer.w2s, scale_fmt="ue8m0")
    torch.cuda.synchronize()
    w13q, w13s, w2q, w2s = layer.oracle_weights(range(E))
    ref, _ = oracle.moe_forward_masked(mi.bf16_bits(hidden), counts, w13q, w13s, w2q, w2s, UE8M0)
    for e, c in enumerate(counts):
        if c:
            assert_output_close(out[e, :c], ref[e, :c])
