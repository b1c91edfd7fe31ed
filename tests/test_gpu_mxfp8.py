"""MXFP8 (MOE_SCALE_MXFP8) on the GPU: 1x32 groups and blocks with UE8M0 scales ("MXFP8 (block
[1, 32])", page "vllm.model_executor.layers.fused_moe.oracle.fp8", make_fp8_moe_quant_config).

Bit-exact against the oracle: the activation quantiser (codes and scale bytes) and the weight
quantiser; the packed scale tiles against their definition (numpy); one GEMM tile whose scales
change every 32 K (so each MMA of a K block must take its own scale byte) exactly; the GEMM
epilogues and the layer against the oracle's MXFP8 mode within the tests' tolerances.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import block_fp8_mixture_topk_gb300 as moe
from moe_testutil import assert_output_close, routing_of, tile_sample_tokens, unpadded_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def device_status_stays_clean():
    moe.moe_get_device_status(clear=True)
    yield
    assert moe.moe_get_device_status(clear=True) == 0


def bits(t):
    return mi.bf16_bits(t)


def scale_of(byte):
    return np.ldexp(1.0, np.asarray(byte, dtype=np.int64) - 127).astype(np.float32)


def mx_offsets(rows, K):
    """Byte offset of (row r, 32-group g) in the MXFP8 packed tiles of a [rows, K] operand (header)."""
    G = K // 32
    r = np.arange(rows)[:, None]
    g = np.arange(G)[None, :]
    return ((r // 128) * (K // 128) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4


def pack_mx_np(scale_bytes, K):
    rows = scale_bytes.shape[0]
    out = np.full(moe.moe_mxfp8_packed_scale_bytes(rows, K), 127, dtype=np.uint8)
    out[mx_offsets(rows, K)] = scale_bytes
    return out


def to_bytes(scales):
    e = np.frexp(np.asarray(scales, dtype=np.float64))[1] - 1
    assert np.all(np.ldexp(1.0, e) == scales)
    return (e + 127).astype(np.uint8)


# ----------------------------------------------------------------------------- quantisers and packing

@pytest.mark.parametrize("rows,cols", [(1, 128), (200, 640), (4096, 7168)])
def test_mxfp8_activation_quant_bit_exact(rows, cols):
    g = torch.Generator().manual_seed(rows * 7 + cols)
    x = (torch.randn(rows, cols, generator=g) *
         torch.exp2(torch.randint(-20, 20, (rows, cols // 32), generator=g).float()).repeat_interleave(32, 1))
    x[0, :64] = 0.0
    x = x.to(torch.bfloat16)
    q, sb = moe.fp8_group_quant(x.to(DEV), "mxfp8")
    oq, os_ = oracle.quant_1x32_bf16(bits(x))
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(scale_of(sb.cpu().numpy()), os_)


@pytest.mark.parametrize("name", ["tiny", "dsv3"])
def test_mxfp8_weight_quant_bit_exact(name):
    wl = mi.WORKLOADS[name]
    experts = None if name == "tiny" else [0, 255]
    for w in (mi.w13_bf16(wl, DEV, experts), mi.w2_bf16(wl, DEV, experts)):
        q, sb = moe.moe_mxfp8_quant_weight(w)
        oq, os_ = oracle.quant_mxfp8_weight_bf16(bits(w))
        assert np.array_equal(q.cpu().numpy(), oq)
        assert np.array_equal(scale_of(sb.cpu().numpy()), os_)


@pytest.mark.parametrize("rows,K", [(128, 128), (384, 640), (256, 7168)])
def test_mxfp8_pack_scales_layout(rows, K):
    g = torch.Generator().manual_seed(rows + K)
    sb = torch.randint(90, 140, (rows, K // 32), generator=g, dtype=torch.uint8)
    packed = moe.moe_mxfp8_pack_scales(sb.to(DEV)).cpu().numpy()
    assert np.array_equal(packed[:moe.moe_mxfp8_packed_scale_bytes(rows, K)], pack_mx_np(sb.numpy(), K))


# ----------------------------------------------------------------------------- one exact tile

@pytest.mark.parametrize("K,N", [(128, 256), (512, 256), (384, 128)])
def test_mxfp8_gemm_one_tile_is_exact(K, N):
    """Values in {-2..2}, scales 2^-2 .. 2^2 changing with the row / column and with every 32-wide
    K group: the fp32 sums are exact, so the block-scaled MMA must give the fp64 result exactly."""
    rng = np.random.default_rng(K * 3 + N)
    G = K // 32
    A = rng.integers(-2, 3, size=(128, K)).astype(np.float64)
    B = rng.integers(-2, 3, size=(N, K)).astype(np.float64)
    sa = np.ldexp(1.0, (np.arange(128)[:, None] * 3 + np.arange(G)[None, :] * 2) % 5 - 2).astype(np.float32)
    sb = np.ldexp(1.0, (np.arange(N)[:, None] + np.arange(G)[None, :] * 3) % 5 - 2).astype(np.float32)
    want = (A * np.repeat(sa, 32, axis=1)) @ (B * np.repeat(sb, 32, axis=1)).T
    Aq = torch.tensor(A, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).to(DEV)
    Bq = torch.tensor(B, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).reshape(1, N, K).to(DEV)
    a_sf = torch.from_numpy(pack_mx_np(to_bytes(sa), K)).to(DEV)
    b_sf = torch.from_numpy(pack_mx_np(to_bytes(sb), K)).to(DEV)
    one = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((128, N), float("nan"), dtype=torch.float32, device=DEV)
    moe.fp8_block_grouped_gemm(Aq, a_sf, (0, 0), Bq, b_sf, one, one, one + 1, "store", out_f32=out, scale_fmt="mxfp8")
    got = out.cpu().double().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:6].tolist()}"


# ----------------------------------------------------------------------------- layer

class MxLayer:
    """MXFP8 weights of a workload (GPU quantiser, scales packed), and the oracle's own
    quantisation of any subset of experts from the same bf16 weights."""

    def __init__(self, wl, chunk=8):
        self.wl = wl
        E, H, I = wl.E, wl.H, wl.I
        self.w13q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=DEV)
        self.w2q = torch.empty(E, H, I, dtype=torch.uint8, device=DEV)
        s13 = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=DEV)
        s2 = torch.empty(E, H, I // 32, dtype=torch.uint8, device=DEV)
        for e0 in range(0, E, chunk):
            ex = range(e0, min(E, e0 + chunk))
            self.w13q[e0:e0 + len(ex)], s13[e0:e0 + len(ex)] = moe.moe_mxfp8_quant_weight(mi.w13_bf16(wl, DEV, ex))
            self.w2q[e0:e0 + len(ex)], s2[e0:e0 + len(ex)] = moe.moe_mxfp8_quant_weight(mi.w2_bf16(wl, DEV, ex))
        self.s13, self.s2 = s13, s2
        self.w13sf, self.w2sf = moe.moe_mxfp8_pack_scales(s13), moe.moe_mxfp8_pack_scales(s2)
        torch.cuda.synchronize()

    def forward(self, hidden, logits, rp, tiled=False):
        w13, w2 = self.w13q, self.w2q
        if tiled:
            w13, w2 = moe.moe_fp8_block_pack_weights(w13), moe.moe_fp8_block_pack_weights(w2)
        return moe.moe_fp8_block_forward(hidden, logits, w13, self.w13sf, w2, self.w2sf, self.wl.topk,
                                         self.wl.renormalize, rp, scale_fmt="mxfp8")

    def oracle_weights(self, experts):
        wl = self.wl
        E, H, I = wl.E, wl.H, wl.I
        w13q = np.zeros((E, 2 * I, H), np.uint8)
        w13s = np.ones((E, 2 * I, H // 32), np.float32)
        w2q = np.zeros((E, H, I), np.uint8)
        w2s = np.ones((E, H, I // 32), np.float32)
        for e in sorted(set(int(x) for x in experts)):
            q, s_ = oracle.quant_mxfp8_weight_bf16(bits(mi.w13_bf16(wl, DEV, [e])))
            w13q[e], w13s[e] = q[0], s_[0]
            q, s_ = oracle.quant_mxfp8_weight_bf16(bits(mi.w2_bf16(wl, DEV, [e])))
            w2q[e], w2s[e] = q[0], s_[0]
        return w13q, w13s, w2q, w2s


def run_mx_layer(wl, tokens=None):
    layer = MxLayer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = layer.forward(hidden.to(DEV), logits.to(DEV), rp)
    out_tiled = layer.forward(hidden.to(DEV), logits.to(DEV), rp, tiled=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out_tiled)
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    toks = range(wl.T) if tokens is None else tokens
    w13q, w13s, w2q, w2s = layer.oracle_weights(set(oids[list(toks)].reshape(-1).tolist()))
    ref = oracle.moe_forward_mxfp8(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, wl.renormalize,
                                   tokens=tokens, **okw)
    return out, ref


def test_mxfp8_gemm_epilogues_match_the_oracle():
    """The w13 GEMM's requantised intermediate (1x32 groups) against the oracle's: scales within one
    power of two (>= 99% equal), codes of equal-scale groups within one e4m3 step (>= 99% equal)."""
    wl = mi.Workload("mx_stage", 171, 200, 640, 384, 16, 4)
    layer = MxLayer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    oids, _ = oracle.route(logits.numpy(), wl.topk, True)
    perm = moe.moe_align_permute(torch.from_numpy(oids).to(DEV), wl.E)
    q, sb = moe.fp8_group_quant(hidden.to(DEV), "mxfp8")
    used = int(perm["padded_offsets"][-1].item())
    sp = perm["sorted_pair_ids"].cpu().numpy()[:used].astype(np.int64)
    assert np.all(sp < wl.T * wl.topk) and np.all(sp >= -1)
    valid = np.nonzero(sp >= 0)[0]
    tok = sp[valid] // wl.topk
    rows = perm["max_rows"]
    A = torch.zeros(rows, wl.H, dtype=torch.uint8)
    Ab = torch.full((rows, wl.H // 32), 127, dtype=torch.uint8)
    A[torch.from_numpy(valid)] = q.cpu()[torch.from_numpy(tok)]
    Ab[torch.from_numpy(valid)] = sb.cpu()[torch.from_numpy(tok)]
    a_sf = torch.from_numpy(pack_mx_np(Ab.numpy(), wl.H)).to(DEV)
    ts = (perm["tile_expert"], perm["tile_row0"], perm["num_tiles"])
    oq = torch.zeros(rows, wl.I, dtype=torch.uint8, device=DEV)
    osf = torch.zeros(moe.moe_mxfp8_packed_scale_bytes(rows, wl.I), dtype=torch.uint8, device=DEV)
    moe.fp8_block_grouped_gemm(A.to(DEV), a_sf, (0, 0), layer.w13q, layer.w13sf, *ts, "silu_mul_quant", out_q=oq,
                               out_scale=osf, scale_fmt="mxfp8")
    w13q, w13s, w2q, w2s = layer.oracle_weights(range(wl.E))
    ref = oracle.moe_forward_mxfp8(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk)
    m = unpadded_rows(perm["padded_offsets"].cpu().numpy(), ref["offsets"])
    gs = scale_of(osf.cpu().numpy()[mx_offsets(rows, wl.I)])[m]
    ratio = gs / ref["a2s"]
    assert np.all(np.isin(ratio, [0.5, 1.0, 2.0])) and np.mean(ratio == 1.0) >= 0.99
    same_group = np.repeat(ratio == 1.0, 32, axis=1)
    gq = oq.cpu().numpy()[m].astype(np.int32)[same_group]
    rq = ref["a2q"].astype(np.int32)[same_group]
    assert np.mean(gq == rq) >= 0.99
    diff = gq != rq
    mag_g, mag_r = gq[diff] & 0x7F, rq[diff] & 0x7F
    assert np.all(((gq[diff] ^ rq[diff]) & 0x80 == 0) | ((mag_g <= 1) & (mag_r <= 1)))
    assert np.all(np.abs(mag_g - mag_r) <= 1)


@pytest.mark.parametrize("T,H,I,E,topk", [(16, 256, 256, 4, 2), (1, 128, 128, 1, 1), (70, 128, 256, 3, 2),
                                          (300, 640, 384, 4, 1), (65, 128, 128, 16, 8)])
def test_mxfp8_layer_all_tokens(T, H, I, E, topk):
    wl = mi.WORKLOADS["tiny"] if (T, H) == (16, 256) else mi.Workload("mx_edge", 180 + T + E, T, H, I, E, topk)
    out, ref = run_mx_layer(wl)
    assert_output_close(out, ref["out"])


@pytest.mark.parametrize("name,T", [("mixtral", None), ("dsv3", None), ("qwen3_skew", None), ("dsv3_decode", 1)])
def test_mxfp8_layer_full_size_every_tile_sampled(name, T):
    wl = mi.WORKLOADS[name] if T is None else mi.WORKLOADS[name].with_tokens(T)
    _, okw = routing_of(wl)
    oids, _ = oracle.route(mi.router_logits(wl).numpy(), wl.topk, wl.renormalize, **okw)
    tokens = tile_sample_tokens(oids, wl.E, extra=[0, wl.T - 1])
    out, ref = run_mx_layer(wl, tokens)
    assert_output_close(out, ref["out"], rows=tokens)


def test_mxfp8_masked_layout():
    """Rows already grouped by expert in MXFP8: every valid row equals the oracle's MXFP8 expert MLP
    (the routed oracle with one expert and top-1, row by row)."""
    E, M, H, I = 4, 150, 256, 384
    wl = mi.Workload("mx_masked", 185, M, H, I, E, 1)
    layer = MxLayer(wl)
    g = torch.Generator().manual_seed(186)
    hidden = torch.randn(E, M, H, generator=g).to(torch.bfloat16)
    counts = torch.tensor([0, 150, 17, 129], dtype=torch.int32)
    out = moe.moe_fp8_block_forward_masked(hidden.to(DEV), counts.to(DEV), layer.w13q, layer.w13sf, layer.w2q,
                                           layer.w2sf, scale_fmt="mxfp8")
    w13q, w13s, w2q, w2s = layer.oracle_weights(range(E))
    got = out.float().cpu().double().numpy()
    for e in range(E):
        c = int(counts[e])
        if not c:
            continue
        r = oracle.moe_forward_mxfp8(bits(hidden[e, :c]), np.zeros((c, 1), np.float32), w13q[e:e + 1],
                                     w13s[e:e + 1], w2q[e:e + 1], w2s[e:e + 1], 1)
        assert_output_close(torch.from_numpy(got[e, :c]), r["out"])
