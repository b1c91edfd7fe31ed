"""GPU parity: every kernel of the layer against the CPU oracle, through the C ABI.

Bit-exact: routing ids, the expert sort, quantised activation / weight bytes
and scales.  Floating point: the layer's output within relative Frobenius
1e-2 and per-element 5e-2 * rms(reference); the GEMM stages in isolation
within 1e-5 (fp32 accumulation against fp64); requantised intermediate bytes
within one e4m3 code (>= 99% identical), since fp32 rounding order decides them.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import block_fp8_mixture_topk_gb300 as moe
from moe_testutil import Layer, assert_output_close, check_sort, routing_of, tile_sample_tokens, unpadded_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def device_status_stays_clean():
    moe.moe_get_device_status(clear=True)
    yield
    assert moe.moe_get_device_status(clear=True) == 0


def bits(t):
    return mi.bf16_bits(t)


# ----------------------------------------------------------------------------- quantisation

def special_rows(rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp2(torch.randint(-12, 12, (rows, 1), generator=g).float())
    if rows > 3:
        x[0] = 0.0                                   # zero groups -> floor scale, zero codes
        x[1] = 1e-12                                 # below the 1e-8 amax floor
        x[2, :128] = 3e38                            # near the bf16 maximum
        x[3, 5] = -x[3].abs().max() * 1.5            # negative group maximum
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 384), (300, 2048), (4096, 7168)])
def test_group_quant_bit_exact(rows, cols):
    x = special_rows(rows, cols, rows + cols)
    q, s = moe.fp8_group_quant(x.to(DEV))
    oq, os_ = oracle.quant_1x128_bf16(bits(x))
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(q.cpu().numpy(), oq)


def test_group_quant_bit_exact_wide_range():
    """8M values, per-group magnitudes from 2^-60 to 2^60, and groups whose scale is an exact power
    of two holding e4m3 tie midpoints (ties to even) -- the quotient x/scale must round exactly as
    IEEE division does."""
    g = torch.Generator().manual_seed(77)
    rows, cols = 2048, 4096
    x = torch.randn(rows, cols, generator=g)
    x = x * torch.exp2(torch.randint(-60, 60, (rows, cols // 128), generator=g).float()).repeat_interleave(128, 1)
    vals = oracle.e4m3_values()
    mids = torch.from_numpy(((vals[1:126] + vals[2:127]) / 2).astype(np.float32))
    for r in range(0, rows, 64):                       # tie rows: amax 448 * 2^k, the rest midpoints * 2^k
        k = float(r % 17 - 8)
        row = mids[torch.randint(0, mids.numel(), (cols,), generator=g)] * (2.0 ** k)
        row[::128] = 448.0 * 2.0 ** k
        x[r] = row * torch.where(torch.rand(cols, generator=g) < 0.5, -1.0, 1.0)
    x = x.to(torch.bfloat16)
    q, s = moe.fp8_group_quant(x.to(DEV))
    oq, os_ = oracle.quant_1x128_bf16(bits(x))
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(q.cpu().numpy(), oq)


@pytest.mark.parametrize("name,experts", [("tiny", None), ("dsv3", [0, 255])])
def test_block_quant_weight_bit_exact(name, experts):
    wl = mi.WORKLOADS[name]
    for w in (mi.w13_bf16(wl, DEV, experts), mi.w2_bf16(wl, DEV, experts)):
        q, s = moe.fp8_block_quant_weight(w)
        oq, os_ = oracle.quant_128x128_bf16(bits(w))
        assert np.array_equal(s.cpu().numpy(), os_)
        assert np.array_equal(q.cpu().numpy(), oq)


# ----------------------------------------------------------------------------- routing / sort

ROUTE_CASES = [
    ("tiny", None), ("mixtral", None), ("dsv3", None), ("dsv3_decode", 1), ("dsv3_decode", 128),
    ("qwen3_skew", None),
]


def workload(name, T=None):
    wl = mi.WORKLOADS[name]
    return wl.with_tokens(T) if T else wl


@pytest.mark.parametrize("name,T", ROUTE_CASES)
def test_route_bit_exact_ids(name, T):
    wl = workload(name, T)
    logits = mi.router_logits(wl)
    rp, okw = routing_of(wl)
    ids, w = moe.moe_route_topk(logits.to(DEV), wl.topk, wl.renormalize, rp)
    oids, ow = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    assert np.array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("E,topk,scoring", [(1024, 32, "softmax"), (1024, 32, "sigmoid"), (1, 1, "softmax"),
                                            (8, 8, "softmax"), (96, 7, "sigmoid")])
def test_route_limits(E, topk, scoring):
    g = torch.Generator().manual_seed(E + topk)
    logits = torch.randn(33, E, generator=g)
    logits[0] = 0.5                                   # all ties -> lowest indices
    sc = 1 if scoring == "sigmoid" else 0
    ids, w = moe.moe_route_topk(logits.to(DEV), topk, True, moe.RoutingParams(scoring, 1, 1, 1.0))
    oids, ow = oracle.route(logits.numpy(), topk, True, scoring=sc)
    assert np.array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=1e-6, atol=1e-7)
    assert ids.cpu()[0].tolist() == list(range(topk))


@pytest.mark.parametrize("T", [300, 40])
@pytest.mark.parametrize("E,n_group,topk_group,topk", [
    (96, 4, 2, 6),      # 24-expert groups over 6 lanes: the shared-memory kernel
    (72, 6, 3, 5),      # 12-expert groups over 3 lanes: the shared-memory kernel
    (48, 3, 2, 5),      # 16-expert groups over 8 lanes: the register kernel
    (160, 5, 3, 8),     # 32-expert groups over 4 lanes, 20 of 32 lanes used: the register kernel
    (512, 16, 5, 12),   # 32-expert groups over 2 lanes: the register kernel
    (1024, 32, 7, 32),  # the most experts, groups and choices
])
def test_route_grouped_shapes_bit_exact(E, n_group, topk_group, topk, T):
    g = torch.Generator().manual_seed(E + n_group)
    logits = torch.randn(T, E, generator=g)
    logits[0] = 0.25                                  # all ties: lowest groups, lowest indices
    bias = torch.randn(E, generator=g) * 0.01
    rp = moe.RoutingParams("sigmoid", n_group, topk_group, 2.5, bias.to(DEV))
    ids, w = moe.moe_route_topk(logits.to(DEV), topk, True, rp)
    oids, ow = oracle.route(logits.numpy(), topk, True, scoring=oracle.SIGMOID, bias=bias.numpy(),
                            n_group=n_group, topk_group=topk_group, routed_scaling=2.5)
    assert np.array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("T", [512, 64])
@pytest.mark.parametrize("n_group,topk_group,with_bias", [(1, 1, False), (8, 4, True), (4, 2, False)])
def test_route_near_ties_fall_back_to_exact_scores(n_group, topk_group, with_bias, T):
    """Logits a few fp32 ulps apart make the fp32 sigmoids too close to decide: the kernel must
    repeat those tokens on the exact (fp64-evaluated) scores and still match the oracle bit-exactly."""
    g = torch.Generator().manual_seed(n_group * 10 + topk_group)
    E, k = 64, 6
    logits = (0.5 + torch.randint(0, 6, (T, E), generator=g).float() * 2.0 ** -22).float()
    logits[T // 2:] = torch.randn(T - T // 2, E, generator=g)       # ordinary rows take the fast path
    bias = (torch.randint(0, 3, (E,), generator=g).float() * 2.0 ** -24) if with_bias else None
    rp = moe.RoutingParams("sigmoid", n_group, topk_group, 1.0, None if bias is None else bias.to(DEV))
    ids, w = moe.moe_route_topk(logits.to(DEV), k, True, rp)
    oids, ow = oracle.route(logits.numpy(), k, True, scoring=oracle.SIGMOID,
                            bias=None if bias is None else bias.numpy(), n_group=n_group, topk_group=topk_group)
    assert np.array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=1e-6, atol=1e-7)


def test_route_without_renormalize():
    g = torch.Generator().manual_seed(2)
    logits = torch.randn(50, 64, generator=g)
    for scoring, sc in (("softmax", 0), ("sigmoid", 1)):
        ids, w = moe.moe_route_topk(logits.to(DEV), 6, False, moe.RoutingParams(scoring, 1, 1, 1.5))
        oids, ow = oracle.route(logits.numpy(), 6, False, scoring=sc, routed_scaling=1.5)
        assert np.array_equal(ids.cpu().numpy(), oids)
        np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("name,T", ROUTE_CASES)
def test_align_permute_exact(name, T):
    wl = workload(name, T)
    rp, okw = routing_of(wl)
    oids, _ = oracle.route(mi.router_logits(wl).numpy(), wl.topk, wl.renormalize, **okw)
    perm = moe.moe_align_permute(torch.from_numpy(oids).to(DEV), wl.E)
    check_sort(perm, oids, wl.E)


@pytest.mark.parametrize("T,k,E,block_m", [(3000, 4, 16, 128), (1, 1, 1, 128), (700, 3, 1024, 64), (5, 2, 4, 1)])
def test_align_permute_shapes(T, k, E, block_m):
    g = torch.Generator().manual_seed(T)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    ids[: T // 2, 0] = 0                              # skew towards expert 0
    perm = moe.moe_align_permute(ids.to(DEV), E, block_m)
    check_sort(perm, ids.numpy(), E, block_m)


def test_align_permute_drops_invalid_ids_and_reports():
    ids = torch.tensor([[0, 1], [5, 1], [-1, 0]], dtype=torch.int32)
    perm = moe.moe_align_permute(ids.to(DEV), 4)
    assert moe.moe_get_device_status(clear=True) & 2
    pos = perm["pos"].cpu().numpy()[:6]
    assert pos[2] == -1 and pos[4] == -1
    assert perm["expert_offsets"].cpu().tolist() == [0, 2, 4, 4, 4]


# ----------------------------------------------------------------------------- grouped GEMM stages

GEMM_CASES = [
    dict(T=24, H=384, I=256, E=4, topk=2),
    dict(T=300, H=256, I=384, E=2, topk=1),           # several tiles per expert
    dict(T=200, H=512, I=128, E=16, topk=4),          # many small experts, some empty
]


def stage_inputs(c, seed):
    wl = mi.Workload("stage", seed, c["T"], c["H"], c["I"], c["E"], c["topk"])
    layer = Layer(wl)
    hidden = mi.hidden(wl)
    logits = mi.router_logits(wl)
    oids, ow = oracle.route(logits.numpy(), wl.topk, True)
    ids = torch.from_numpy(oids).to(DEV)
    perm = moe.moe_align_permute(ids, wl.E)
    q, s = moe.fp8_group_quant(hidden.to(DEV))
    # gather the sorted activation rows on the host, from indices checked against their bounds
    used = int(perm["padded_offsets"][-1].item())
    sp = perm["sorted_pair_ids"].cpu().numpy()[:used].astype(np.int64)
    assert used <= perm["max_rows"] and np.all(sp < wl.T * wl.topk) and np.all(sp >= -1)
    valid = np.nonzero(sp >= 0)[0]
    tok = sp[valid] // wl.topk
    rows = perm["max_rows"]
    A = torch.zeros(rows, wl.H, dtype=torch.uint8)
    As = torch.ones(rows, wl.H // 128, dtype=torch.float32)
    A[torch.from_numpy(valid)] = q.cpu()[torch.from_numpy(tok)]
    As[torch.from_numpy(valid)] = s.cpu()[torch.from_numpy(tok)]
    A, As = A.to(DEV), As.to(DEV)
    w13q, w13s, w2q, w2s = layer.oracle_weights(range(wl.E))
    ref = oracle.moe_forward(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, want_c1=True)
    m = unpadded_rows(perm["padded_offsets"].cpu().numpy(), ref["offsets"])
    return wl, layer, perm, A, As, ref, m, torch.from_numpy(ow).to(DEV)


@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_store_matches_oracle(ci):
    wl, layer, perm, A, As, ref, m, _ = stage_inputs(GEMM_CASES[ci], 40 + ci)
    out = torch.full((A.shape[0], 2 * wl.I), float("nan"), dtype=torch.float32, device=DEV)
    moe.fp8_block_grouped_gemm(A, As, (wl.H // 128, 1), layer.w13q, layer.w13s, perm["tile_expert"],
                               perm["tile_row0"], perm["num_tiles"], "store", out_f32=out)
    got = out.cpu().double().numpy()[m]
    want = ref["c1"]
    err = np.abs(got - want)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-5
    assert err.max() <= 1e-4 * np.sqrt(np.mean(want ** 2))


def test_gemm_store_ragged_n():
    """N = 384: the last 256-wide tile is half empty (128-column MMA)."""
    g = torch.Generator().manual_seed(3)
    E, N, K, M = 2, 384, 256, 256
    B = torch.randint(0, 256, (E, N, K), generator=g, dtype=torch.uint8)
    B[(B & 0x7F) == 0x7F] = 0x3E
    A = torch.randint(0, 256, (M, K), generator=g, dtype=torch.uint8)
    A[(A & 0x7F) == 0x7F] = 0x3E
    bs = torch.rand(E, N // 128, K // 128, generator=g) + 0.5
    as_ = torch.rand(M, K // 128, generator=g) + 0.5
    te = torch.tensor([1, 0], dtype=torch.int32)
    tr = torch.tensor([0, 128], dtype=torch.int32)
    nt = torch.tensor([2], dtype=torch.int32)
    out = torch.full((M, N), float("nan"), device=DEV)
    moe.fp8_block_grouped_gemm(A.to(DEV), as_.to(DEV), (K // 128, 1), B.to(DEV), bs.to(DEV), te.to(DEV), tr.to(DEV),
                               nt.to(DEV), "store", out_f32=out)
    Ad = A.view(torch.float8_e4m3fn).double() * as_.double().repeat_interleave(128, 1)
    Bd = B.view(torch.float8_e4m3fn).double() * bs.double().repeat_interleave(128, 1).repeat_interleave(128, 2)
    want = torch.cat([Ad[:128] @ Bd[1].T, Ad[128:] @ Bd[0].T]).numpy()
    got = out.cpu().double().numpy()
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-5


@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_silu_requant_matches_oracle(ci):
    wl, layer, perm, A, As, ref, m, _ = stage_inputs(GEMM_CASES[ci], 40 + ci)
    rows = A.shape[0]
    oq = torch.empty(rows, wl.I, dtype=torch.uint8, device=DEV)
    osc = torch.empty(rows, wl.I // 128, dtype=torch.float32, device=DEV)
    moe.fp8_block_grouped_gemm(A, As, (wl.H // 128, 1), layer.w13q, layer.w13s, perm["tile_expert"],
                               perm["tile_row0"], perm["num_tiles"], "silu_mul_quant", out_q=oq, out_scale=osc,
                               out_scale_strides=(wl.I // 128, 1))
    gs = osc.cpu().numpy()[m]
    np.testing.assert_allclose(gs, ref["a2s"], rtol=2e-5)
    gq = oq.cpu().numpy()[m].astype(np.int32)
    rq = ref["a2q"].astype(np.int32)
    same = gq == rq
    assert same.mean() >= 0.99, same.mean()
    # where they differ: same sign, adjacent codes (or +-0 around zero)
    diff = ~same
    mag_g, mag_r = gq[diff] & 0x7F, rq[diff] & 0x7F
    sign_ok = ((gq[diff] ^ rq[diff]) & 0x80 == 0) | ((mag_g <= 1) & (mag_r <= 1))
    assert np.all(sign_ok) and np.all(np.abs(mag_g - mag_r) <= 1)


@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_weighted_scatter_matches_oracle(ci):
    """GEMM2 on the oracle's own intermediate codes, so only GEMM2 + scatter are compared."""
    wl, layer, perm, A, As, ref, m, w = stage_inputs(GEMM_CASES[ci], 40 + ci)
    rows = A.shape[0]
    A2 = torch.zeros(rows, wl.I, dtype=torch.uint8)
    A2s = torch.ones(rows, wl.I // 128, dtype=torch.float32)
    A2[torch.from_numpy(m)] = torch.from_numpy(ref["a2q"])
    A2s[torch.from_numpy(m)] = torch.from_numpy(ref["a2s"])
    out = torch.zeros(wl.T, wl.H, dtype=torch.float32, device=DEV)
    moe.fp8_block_grouped_gemm(A2.to(DEV), A2s.to(DEV), (wl.I // 128, 1), layer.w2q, layer.w2s, perm["tile_expert"],
                               perm["tile_row0"], perm["num_tiles"], "weighted_scatter", out_f32=out,
                               sorted_pair_ids=perm["sorted_pair_ids"], topk_weights=w.reshape(-1),
                               topk=wl.topk, num_pairs=wl.T * wl.topk)
    got = out.cpu().double().numpy()
    want = ref["out"]
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-5


@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_weighted_rows_then_unpermute_sum_matches_oracle(ci):
    """GEMM2 writing router-weighted rows in sorted order, then the j-ordered sum of each token's
    rows, on the oracle's own intermediate codes."""
    wl, layer, perm, A, As, ref, m, w = stage_inputs(GEMM_CASES[ci], 40 + ci)
    rows = A.shape[0]
    A2 = torch.zeros(rows, wl.I, dtype=torch.uint8)
    A2s = torch.ones(rows, wl.I // 128, dtype=torch.float32)
    A2[torch.from_numpy(m)] = torch.from_numpy(ref["a2q"])
    A2s[torch.from_numpy(m)] = torch.from_numpy(ref["a2s"])
    y = torch.full((rows, wl.H), float("nan"), dtype=torch.float32, device=DEV)
    moe.fp8_block_grouped_gemm(A2.to(DEV), A2s.to(DEV), (wl.I // 128, 1), layer.w2q, layer.w2s, perm["tile_expert"],
                               perm["tile_row0"], perm["num_tiles"], "weighted_rows", out_f32=y,
                               sorted_pair_ids=perm["sorted_pair_ids"], topk_weights=w.reshape(-1),
                               topk=wl.topk, num_pairs=wl.T * wl.topk)
    # each real row holds weight * C2 of its pair
    wflat = ref["weights"].reshape(-1).astype(np.float64)
    got_rows = y.cpu().double().numpy()[m]
    want_rows = ref["c2"] * wflat[ref["sorted"]][:, None]
    assert np.linalg.norm(got_rows - want_rows) / np.linalg.norm(want_rows) < 1e-5
    out = moe.moe_unpermute_sum(y, perm["pos"][: wl.T * wl.topk].contiguous(), wl.T, wl.topk)
    got = out.float().cpu().double().numpy()
    want = ref["out"]
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 4e-3      # bf16 output rounding
    assert np.all(np.abs(got - want) <= 2.0 ** -7 * np.abs(want) + 1e-6 * np.abs(want).max())


@pytest.mark.parametrize("epilogue", ["weighted_rows", "weighted_pairs_bf16"])
def test_gemm_weighted_rows_many_tiles_per_cta(epilogue):
    """The w2 GEMM alone on the DeepSeek-V3 decode shapes with T=8 (~20 tiles per CTA, both epilogue
    warpgroups cycling through their accumulators and scale rings many times), fed the oracle's own
    intermediate codes, three launches in a row."""
    wl = mi.WORKLOADS["dsv3_decode"].with_tokens(8)
    layer = Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    oids, ow = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    w13q, w13s, w2q, w2s = layer.oracle_weights(set(oids.reshape(-1).tolist()))
    ref = oracle.moe_forward(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, wl.renormalize, **okw)
    perm = moe.moe_align_permute(torch.from_numpy(oids).to(DEV), wl.E)
    m = unpadded_rows(perm["padded_offsets"].cpu().numpy(), ref["offsets"])
    rows = perm["max_rows"]
    A2 = torch.zeros(rows, wl.I, dtype=torch.uint8)
    A2s = torch.ones(rows, wl.I // 128, dtype=torch.float32)
    A2[torch.from_numpy(m)] = torch.from_numpy(ref["a2q"])
    A2s[torch.from_numpy(m)] = torch.from_numpy(ref["a2s"])
    want = ref["c2"] * ow.reshape(-1).astype(np.float64)[ref["sorted"]][:, None]
    P = wl.T * wl.topk
    for _ in range(3):
        if epilogue == "weighted_rows":
            y = torch.full((rows, wl.H), float("nan"), dtype=torch.float32, device=DEV)
            kw = dict(out_f32=y)
        else:
            y = torch.full((P, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
            kw = dict(out_bf16=y)
        moe.fp8_block_grouped_gemm(A2.to(DEV), A2s.to(DEV), (wl.I // 128, 1), layer.w2q, layer.w2s,
                                   perm["tile_expert"], perm["tile_row0"], perm["num_tiles"], epilogue,
                                   sorted_pair_ids=perm["sorted_pair_ids"],
                                   topk_weights=torch.from_numpy(ow).to(DEV).reshape(-1), topk=wl.topk,
                                   num_pairs=P, **kw)
        if epilogue == "weighted_rows":
            got = y.cpu().double().numpy()[m]
            assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-5
            assert np.abs(got - want).max() <= 1e-4 * np.abs(want).max()
        else:
            got = y.float().cpu().double().numpy()[ref["sorted"]]
            assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-4 * np.abs(want).max())


@pytest.mark.parametrize("T,k,H,rows", [(1, 1, 4, 3), (37, 3, 384, 200), (300, 8, 2048, 2500)])
def test_unpermute_sum_bit_exact_against_fp32_j_order(T, k, H, rows):
    g = torch.Generator().manual_seed(T * k)
    y = torch.randn(rows, H, generator=g)
    pos = torch.randint(0, rows, (T * k,), generator=g, dtype=torch.int32)
    pos[::5] = -1                                    # dropped pairs are skipped
    out = moe.moe_unpermute_sum(y.to(DEV), pos.to(DEV), T, k)
    acc = torch.zeros(T, H, dtype=torch.float32)
    p2 = pos.view(T, k).long()
    for j in range(k):
        valid = p2[:, j] >= 0
        acc[valid] = acc[valid] + y[p2[valid, j]]
    assert torch.equal(out.cpu(), acc.to(torch.bfloat16))


def pair_rows_reference(ref, wl):
    """The oracle's router-weighted w2 rows in pair order ([P, H], fp64) and, per token and
    column, the sum of the magnitudes of its k terms (scale of the bf16 rounding error)."""
    P = wl.T * wl.topk
    wflat = ref["weights"].reshape(-1).astype(np.float64)
    rows = np.zeros((P, wl.H))
    rows[ref["sorted"]] = ref["c2"] * wflat[ref["sorted"]][:, None]
    sum_abs = np.abs(rows).reshape(wl.T, wl.topk, wl.H).sum(axis=1)
    return rows, sum_abs


@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_weighted_pairs_bf16_then_combine_matches_oracle(ci):
    """GEMM2 writing bf16 router-weighted rows in pair order, then the j-ordered sum of each
    token's k contiguous rows, on the oracle's own intermediate codes."""
    wl, layer, perm, A, As, ref, m, w = stage_inputs(GEMM_CASES[ci], 40 + ci)
    rows = A.shape[0]
    P = wl.T * wl.topk
    A2 = torch.zeros(rows, wl.I, dtype=torch.uint8)
    A2s = torch.ones(rows, wl.I // 128, dtype=torch.float32)
    A2[torch.from_numpy(m)] = torch.from_numpy(ref["a2q"])
    A2s[torch.from_numpy(m)] = torch.from_numpy(ref["a2s"])
    y = torch.full((P, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.fp8_block_grouped_gemm(A2.to(DEV), A2s.to(DEV), (wl.I // 128, 1), layer.w2q, layer.w2s, perm["tile_expert"],
                               perm["tile_row0"], perm["num_tiles"], "weighted_pairs_bf16", out_bf16=y,
                               sorted_pair_ids=perm["sorted_pair_ids"], topk_weights=w.reshape(-1),
                               topk=wl.topk, num_pairs=P)
    want_rows, sum_abs = pair_rows_reference(ref, wl)
    got_rows = y.float().cpu().double().numpy()
    # every pair row written once: bf16 rounding (half an ulp, 2^-8 relative) of an fp32 value
    # within the GEMM's fp32 accumulation error of the fp64 reference
    scale = np.abs(want_rows).max()
    assert np.all(np.abs(got_rows - want_rows) <= 2.0 ** -8 * np.abs(want_rows) + 1e-4 * scale)
    out = moe.moe_combine_pairs(y, perm["pos"][:P].contiguous(), wl.T, wl.topk)
    got = out.float().cpu().double().numpy()
    want = ref["out"]
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 6e-3
    # each term rounded to bf16, the sum rounded once more, against the oracle's single rounding
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * (2 * np.abs(want) + sum_abs) * 1.01 + 1e-4 * np.abs(want).max())


@pytest.mark.parametrize("T,k,H", [(1, 1, 8), (37, 3, 384), (300, 8, 2048), (5, 2, 7168), (64, 8, 7168)])
def test_combine_pairs_bit_exact_against_fp32_j_order(T, k, H):
    g = torch.Generator().manual_seed(T * k + H)
    y = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    pos = torch.arange(T * k, dtype=torch.int32)
    pos[::5] = -1                                    # dropped pairs are skipped ...
    y[pos < 0] = float("nan")                        # ... and their rows never read
    out = moe.moe_combine_pairs(y.to(DEV), pos.to(DEV), T, k)
    acc = torch.zeros(T, H, dtype=torch.float32)
    yv, pv = y.view(T, k, H), pos.view(T, k)
    for j in range(k):
        valid = pv[:, j] >= 0
        acc[valid] = acc[valid] + yv[valid, j].float()
    assert torch.equal(out.cpu(), acc.to(torch.bfloat16))


# ----------------------------------------------------------------------------- tile-packed weights

@pytest.mark.parametrize("E,N,K", [(1, 128, 128), (3, 384, 256), (2, 4096, 7168)])
def test_pack_weights_is_the_block_permutation(E, N, K):
    g = torch.Generator().manual_seed(E * N + K)
    w = torch.randint(0, 256, (E, N, K), generator=g, dtype=torch.uint8)
    packed = moe.moe_fp8_block_pack_weights(w.to(DEV))
    want = w.view(E, N // 128, 128, K // 128, 128).permute(0, 1, 3, 2, 4).contiguous()
    assert torch.equal(packed.cpu(), want)


@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_gemm_packed_weights_bit_identical(ci):
    """Every epilogue reads the tile-packed weights to exactly the same bits as the [E, N, K] ones."""
    wl, layer, perm, A, As, ref, m, w = stage_inputs(GEMM_CASES[ci], 40 + ci)
    w13p, w2p = moe.moe_fp8_block_pack_weights(layer.w13q), moe.moe_fp8_block_pack_weights(layer.w2q)
    rows, P = A.shape[0], wl.T * wl.topk
    outs = []
    for b13, b2 in ((layer.w13q, layer.w2q), (w13p, w2p)):
        c1 = torch.zeros(rows, 2 * wl.I, dtype=torch.float32, device=DEV)
        moe.fp8_block_grouped_gemm(A, As, (wl.H // 128, 1), b13, layer.w13s, perm["tile_expert"],
                                   perm["tile_row0"], perm["num_tiles"], "store", out_f32=c1)
        oq = torch.zeros(rows, wl.I, dtype=torch.uint8, device=DEV)
        osc = torch.zeros(rows, wl.I // 128, dtype=torch.float32, device=DEV)
        moe.fp8_block_grouped_gemm(A, As, (wl.H // 128, 1), b13, layer.w13s, perm["tile_expert"],
                                   perm["tile_row0"], perm["num_tiles"], "silu_mul_quant", out_q=oq, out_scale=osc,
                                   out_scale_strides=(wl.I // 128, 1))
        y = torch.zeros(P, wl.H, dtype=torch.bfloat16, device=DEV)
        moe.fp8_block_grouped_gemm(oq, osc, (wl.I // 128, 1), b2, layer.w2s, perm["tile_expert"],
                                   perm["tile_row0"], perm["num_tiles"], "weighted_pairs_bf16", out_bf16=y,
                                   sorted_pair_ids=perm["sorted_pair_ids"], topk_weights=w.reshape(-1),
                                   topk=wl.topk, num_pairs=P)
        outs.append((c1, oq, osc, y))
    mt = torch.from_numpy(m).to(DEV)
    (c1a, oqa, osa, ya), (c1b, oqb, osb, yb) = outs
    assert torch.equal(c1a[mt], c1b[mt]) and torch.equal(oqa[mt], oqb[mt]) and torch.equal(osa[mt], osb[mt])
    assert torch.equal(ya, yb)


# ----------------------------------------------------------------------------- whole layer

def run_layer(wl, tokens=None, layer=None):
    layer = layer or Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = layer.forward(hidden.to(DEV), logits.to(DEV), rp)
    # the same layer on the tile-packed weights gives the same bits
    out_packed = layer.forward(hidden.to(DEV), logits.to(DEV), rp, packed=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out_packed)
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    toks = range(wl.T) if tokens is None else tokens
    experts = set(oids[list(toks)].reshape(-1).tolist())
    w13q, w13s, w2q, w2s = layer.oracle_weights(experts)
    ref = oracle.moe_forward(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, wl.renormalize,
                             tokens=tokens, **okw)
    return out, ref


def test_forward_tiny_all_tokens():
    wl = mi.WORKLOADS["tiny"]
    out, ref = run_layer(wl)
    assert_output_close(out, ref["out"])


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "qwen3_skew"])
def test_forward_full_size_every_tile_sampled(name):
    """The full-size layer against the oracle on a sample that reaches every expert tile of both
    GEMMs: for each 128-row tile the token owning its last real row, and for each expert the token
    owning its first row (DeepSeek-V3 shape: every touched expert; Qwen3 Zipf shape: every tile
    of the hot experts)."""
    wl = mi.WORKLOADS[name]
    _, okw = routing_of(wl)
    oids, _ = oracle.route(mi.router_logits(wl).numpy(), wl.topk, wl.renormalize, **okw)
    tokens = tile_sample_tokens(oids, wl.E, extra=[0, 1, wl.T // 2, wl.T - 1])
    out, ref = run_layer(wl, tokens)
    assert_output_close(out, ref["out"], rows=tokens)


@pytest.mark.parametrize("fmt", ["f32", "ue8m0_packed"])
def test_forward_more_items_than_a_cta_caches(fmt):
    """Both grouped GEMMs with more than 256 work items per CTA on every SM (a CTA caches its first
    256 items' tile, column block, expert and first row in shared memory and looks up later ones
    in global memory).  H=4096, I=2048: 16 column blocks per tile in each GEMM; 50000 tokens, top-8
    over 32 experts: about 3150 tiles, so the items of tiles from 16 x (SM count) on come after a
    CTA's 256th.  Experts 28-31 hold exactly 300 rows each (three tiles, a w13 of 16 MB: the w13
    GEMM visits their tiles column by column) and sit in the last tiles.  Tokens whose rows lie
    past the cached items are compared with the oracle.  With packed UE8M0 scales (12500 rows per
    expert) the GEMMs run on the CTA-pair kernel, whose clusters (at most half the SM count) cache
    their first 256 candidates, i.e. tiles below 16 x (SM count) / 2 x 2: the same bound; the small
    experts' third tiles are pairs whose second CTA has no rows."""
    T, H, I, E, topk = 50000, 4096, 2048, 32, 8
    wl = mi.Workload("items", 95, T, H, I, E, topk)
    logits = mi.router_logits(wl)
    small = torch.arange(E - 4, E)
    logits[:, small] -= 1000.0                 # experts 28-31 never chosen ...
    chosen = torch.arange(0, T, T // 300)[:300]
    logits[chosen.unsqueeze(1), small.unsqueeze(0)] += 2000.0   # ... except by these 300 tokens
    packed = fmt == "ue8m0_packed"
    if packed:
        from test_gpu_block_scaled import PackedLayer
        layer = PackedLayer(wl)
    else:
        layer = Layer(wl)
    rp, _ = routing_of(wl)
    out = layer.forward(mi.hidden(wl).to(DEV), logits.to(DEV), rp)
    oids, _ = oracle.route(logits.numpy(), topk, True)
    counts = np.bincount(oids.reshape(-1), minlength=E)
    assert np.all(counts[E - 4:] == 300)
    tiles_per_expert = (counts + 127) // 128
    first_tile = np.concatenate([[0], np.cumsum(tiles_per_expert)])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cached_tiles = 256 * sms // 16             # tiles whose items are among the CTAs' first 256
    assert first_tile[-1] > cached_tiles + 400
    # tokens with rows in the uncached tiles: every tile's last real row past the cache, thinned,
    # plus the small experts' first and last rows
    off, sorted_, _ = oracle.permute(oids, E)
    toks = set()
    for e in range(E):
        n = int(counts[e])
        for i in range(0, n, 128):
            tile = first_tile[e] + i // 128
            last = min(i + 127, n - 1)
            if tile >= cached_tiles and (e >= E - 4 or tile % 16 == 0):
                toks.add(int(sorted_[off[e] + last]) // topk)
        if e >= E - 4:
            toks.add(int(sorted_[off[e]]) // topk)
    tokens = sorted(toks)
    w13q, w13s, w2q, w2s = layer.oracle_weights(set(oids[tokens].reshape(-1).tolist()))
    ref = oracle.moe_forward(bits(mi.hidden(wl)), logits.numpy(), w13q, w13s, w2q, w2s, topk, True, tokens=tokens,
                             scale_fmt=oracle.SCALE_UE8M0 if packed else oracle.SCALE_F32)
    assert_output_close(out, ref["out"], rows=tokens)


@pytest.mark.parametrize("T", mi.DECODE_TOKENS)
def test_forward_decode_sampled_tokens(T):
    wl = mi.WORKLOADS["dsv3_decode"].with_tokens(T)
    tokens = sorted(set([0, T // 2, T - 1]))
    out, ref = run_layer(wl, tokens)
    assert_output_close(out, ref["out"], rows=tokens)


@pytest.mark.parametrize("T,H,I,E,topk", [(1, 128, 128, 1, 1), (5, 256, 128, 8, 8), (70, 128, 256, 3, 2)])
def test_forward_small_shapes(T, H, I, E, topk):
    wl = mi.Workload("edge", 60 + T, T, H, I, E, topk)
    out, ref = run_layer(wl)
    assert_output_close(out, ref["out"])


@pytest.mark.parametrize("fmt", ["f32", "ue8m0_packed"])
def test_forward_w2_last_wave_in_half_items(fmt):
    """The w2 GEMM runs a last wave that would keep at most half of the CTAs busy as 128-column half
    items.  200 tokens, top-2 over 4 experts, H=768: four tiles of three 256-column items each, all
    in the one partial wave, so every item is split (bands 0..5); every token against the oracle,
    for the fp32-scale and the block-scaled kernel."""
    wl = mi.Workload("halves", 196, 200, 768, 256, 4, 2)
    if fmt == "f32":
        out, ref = run_layer(wl)
    else:
        from test_gpu_block_scaled import run_packed_layer
        out, ref = run_packed_layer(wl)
    assert_output_close(out, ref["out"])


@pytest.mark.parametrize("T,H,I,E,topk", [
    (64, 128, 128, 16, 8),       # 512 routed pairs: the one-launch sort + quantisation
    (65, 128, 128, 16, 8),       # 520 pairs: the three sort kernels and the grid-wide quantiser
    (5, 128, 128, 1024, 4),      # the largest expert count, small batch
    (40, 128, 256, 1024, 16),    # the largest expert count, 640 pairs
])
def test_forward_sort_path_boundaries(T, H, I, E, topk):
    wl = mi.Workload("bounds", 70 + T + E, T, H, I, E, topk)
    out, ref = run_layer(wl)
    assert_output_close(out, ref["out"])


@pytest.mark.parametrize("name,T", [("dsv3_decode", 1), ("dsv3_decode", 2), ("mixtral", 1)])
def test_forward_one_and_two_token_batches(name, T):
    """One or two tokens (each expert's tile holds one or two real rows, 32-row activation
    boxes, fewer GEMM items than SMs): every token matches the oracle."""
    wl = workload(name, T)
    out, ref = run_layer(wl)
    assert_output_close(out, ref["out"])


@pytest.mark.parametrize("T,E,topk", [(640, 4, 1), (300, 2, 2), (900, 4, 2)])
def test_forward_column_order_experts_all_tokens(T, E, topk):
    """Experts whose w13 is 16 MB or more (H=2048, I=4096) with 129-512 rows, the case where the
    w13 GEMM visits an expert's two to four tiles column by column: every token matches."""
    wl = mi.Workload("colorder", 90 + T + E, T, 2048, 4096, E, topk)
    assert 2 * wl.I * wl.H >= 16 << 20
    out, ref = run_layer(wl)
    assert_output_close(out, ref["out"])


def test_forward_two_tokens_small_shape():
    wl = mi.Workload("twotok", 81, 2, 256, 512, 6, 3)
    out, ref = run_layer(wl)
    assert_output_close(out, ref["out"])


def test_forward_all_tokens_to_one_expert():
    """300 tokens, top-1, every token on expert 2: three tiles of one expert, the other experts empty."""
    wl = mi.Workload("skew", 77, 300, 256, 256, 4, 1)
    layer = Layer(wl)
    hidden = mi.hidden(wl)
    logits = mi.router_logits(wl)
    logits[:, 2] += 100.0
    out = layer.forward(hidden.to(DEV), logits.to(DEV), None)
    w13q, w13s, w2q, w2s = layer.oracle_weights([2])
    ref = oracle.moe_forward(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, 1)
    assert_output_close(out, ref["out"])


@pytest.mark.parametrize("name,T", [("tiny", None), ("dsv3_decode", 8), ("mixtral", None), ("dsv3_decode", 1),
                                    ("dsv3_decode", 2)])
def test_forward_replays_from_a_cuda_graph(name, T):
    """The whole layer captured once in a CUDA graph (its kernels linked by programmatic
    dependent launch) and replayed on new inputs copied into the captured buffers: every
    replay equals the eager forward on those inputs, bit for bit."""
    wl = workload(name, T)
    layer = Layer(wl)
    rp, _ = routing_of(wl)
    hid = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    log = torch.empty(wl.T, wl.E, dtype=torch.float32, device=DEV)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.topk), dtype=torch.uint8,
                     device=DEV)
    hid.copy_(mi.hidden(wl).to(DEV))
    log.copy_(mi.router_logits(wl).to(DEV))

    def step():
        moe.moe_fp8_block_forward(hid, log, layer.w13q, layer.w13s, layer.w2q, layer.w2s, wl.topk,
                                  wl.renormalize, rp, out=out, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in range(3):
        wl_s = wl.with_(number=wl.number + 500 + seed)
        h, l = mi.hidden(wl_s).to(DEV), mi.router_logits(wl_s).to(DEV)
        hid.copy_(h)
        log.copy_(l)
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        want = moe.moe_fp8_block_forward(h, l, layer.w13q, layer.w13s, layer.w2q, layer.w2s, wl.topk,
                                         wl.renormalize, rp)
        torch.cuda.synchronize()
        assert torch.equal(got, want)


def test_forward_zero_tokens_is_noop():
    wl = mi.WORKLOADS["tiny"]
    layer = Layer(wl)
    hidden = torch.empty(0, wl.H, dtype=torch.bfloat16, device=DEV)
    logits = torch.empty(0, wl.E, dtype=torch.float32, device=DEV)
    out = layer.forward(hidden, logits, None)
    assert out.shape == (0, wl.H)
