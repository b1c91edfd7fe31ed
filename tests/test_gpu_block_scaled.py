"""Packed UE8M0 scales on the block-scaled tensor-core MMA (MOE_SCALE_UE8M0_PACKED).

The packed layout ("UE8M0: packed UE8M0 (4 values per int32) (Blackwell)", page "Quantization and
MoE Optimizations", section DeepGEMM Scale Formats) is rebuilt here with numpy from its definition
in include/moefp8.h, independently of the kernels.  Then:
  - the activation quantiser's packed scales and the weight-scale packing, byte for byte;
  - one GEMM tile with exactly representable products and per-row / per-block power-of-two
    scales (so that fp32 sums are exact): the block-scaled MMA must give the exact result, and a
    wrong scale placement shows up as a power-of-two ratio naming the row or block it came from;
  - the GEMM epilogues and the whole layer against the oracle's UE8M0 mode (the same numbers:
    only the fp32 summation order differs).
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import block_fp8_mixture_topk_gb300 as moe
from moe_testutil import Layer, assert_output_close, routing_of, tile_sample_tokens, unpadded_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
UE8M0 = oracle.SCALE_UE8M0


@pytest.fixture(autouse=True)
def device_status_stays_clean():
    moe.moe_get_device_status(clear=True)
    yield
    assert moe.moe_get_device_status(clear=True) == 0


def bits(t):
    return mi.bf16_bits(t)


def packed_offsets(rows, K):
    """Byte offset of (row r, K block kb) in the packed tiles of a [rows, K] operand (header layout)."""
    KB = K // 128
    kb4 = (KB + 3) // 4
    r = np.arange(rows)[:, None]
    kb = np.arange(KB)[None, :]
    return ((r // 128) * kb4 + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4


def pack_scales_np(scales):
    """fp32 power-of-two scales [rows, K/128] -> packed bytes (numpy, from the definition)."""
    rows, KB = scales.shape
    K = KB * 128
    nbytes = moe.moe_packed_scale_bytes(rows, K)
    e = np.frexp(scales.astype(np.float64))[1] - 1          # scale = 2^e exactly
    assert np.all(np.ldexp(1.0, e) == scales)
    out = np.full(nbytes, 127, dtype=np.uint8)
    out[packed_offsets(rows, K)] = (e + 127).astype(np.uint8)
    return out


def unpack_scales_np(packed, rows, K):
    b = np.asarray(packed, dtype=np.uint8).reshape(-1)[packed_offsets(rows, K)]
    return np.ldexp(1.0, b.astype(np.int64) - 127).astype(np.float32)


# ----------------------------------------------------------------------------- packed layouts

@pytest.mark.parametrize("rows,cols", [(1, 128), (200, 640), (4096, 7168)])
def test_packed_activation_scales_equal_the_oracle(rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    x = (torch.randn(rows, cols, generator=g) *
         torch.exp2(torch.randint(-20, 20, (rows, 1), generator=g).float())).to(torch.bfloat16)
    q, sp = moe.fp8_group_quant(x.to(DEV), "ue8m0_packed")
    oq, os_ = oracle.quant_1x128_bf16(bits(x), UE8M0)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(unpack_scales_np(sp.cpu().numpy(), rows, cols), os_)


@pytest.mark.parametrize("E,N,K", [(1, 128, 128), (3, 384, 640), (2, 256, 7168)])
def test_pack_scales_layout(E, N, K):
    g = torch.Generator().manual_seed(E * N + K)
    s = torch.exp2(torch.randint(-30, 10, (E, N // 128, K // 128), generator=g).float())
    packed = moe.moe_fp8_block_pack_scales(s.to(DEV)).cpu().numpy().reshape(E, -1)
    for e in range(E):
        want = pack_scales_np(np.repeat(s[e].numpy(), 128, axis=0))   # a block's scale on each of its rows
        assert np.array_equal(packed[e], want)


def test_pack_scales_reports_a_scale_that_is_not_a_power_of_two():
    s = torch.full((1, 1, 1), 0.75, device=DEV)
    moe.moe_fp8_block_pack_scales(s)
    assert moe.moe_get_device_status(clear=True) & 0x8


# ----------------------------------------------------------------------------- one exact tile

def e4m3_codes(vals):
    """e4m3 codes of small exact values (torch's cast, exact for these)."""
    return torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


@pytest.mark.parametrize("K,N", [(128, 256), (512, 256), (640, 128)])
def test_block_scaled_gemm_one_tile_is_exact(K, N):
    """128 rows x N columns, values in {-2, -1, 0, 1, 2}, scales 2^-2 .. 2^2 varying with the row, the
    column block and the K block: every fp32 partial sum is exact, so the tensor cores' result must
    equal the fp64 reference bit for bit."""
    rng = np.random.default_rng(K + N)
    KB, NB = K // 128, N // 128
    A = rng.integers(-2, 3, size=(128, K)).astype(np.float64)
    B = rng.integers(-2, 3, size=(N, K)).astype(np.float64)
    r = np.arange(128)[:, None]
    kb = np.arange(KB)[None, :]
    sa = np.ldexp(1.0, (r * 3 + kb * 2) % 5 - 2).astype(np.float32)           # [128, KB]
    nb = np.arange(NB)[:, None]
    sb = np.ldexp(1.0, (nb * 2 + kb * 3 + 1) % 5 - 2).astype(np.float32)      # [NB, KB]
    want = np.zeros((128, N))
    for k in range(KB):
        part = A[:, k * 128:(k + 1) * 128] @ B[:, k * 128:(k + 1) * 128].T
        want += part * sa[:, k:k + 1] * np.repeat(sb[:, k], 128)[None, :]
    Aq = e4m3_codes(A).to(DEV)
    Bq = e4m3_codes(B).reshape(1, N, K).to(DEV)
    a_sf = torch.from_numpy(pack_scales_np(sa)).to(DEV)
    b_sf = torch.from_numpy(pack_scales_np(np.repeat(sb, 128, axis=0))).to(DEV)
    one = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((128, N), float("nan"), dtype=torch.float32, device=DEV)
    moe.fp8_block_grouped_gemm(Aq, a_sf, (0, 0), Bq, b_sf, one, one, one + 1, "store", out_f32=out,
                               scale_fmt="ue8m0_packed")
    got = out.cpu().double().numpy()
    if not np.array_equal(got, want):
        # which power of two went wrong where (rows x column blocks, first mismatching K layout)
        ratio = np.where(want != 0, got / np.where(want == 0, 1, want), 1.0)
        bad = np.argwhere(~np.isclose(ratio, 1.0))
        raise AssertionError(f"{len(bad)} mismatches; first rows/cols {bad[:8].tolist()}; "
                             f"log2 ratio sample {np.log2(np.abs(ratio[bad[:8, 0], bad[:8, 1]])).tolist()}")


# ----------------------------------------------------------------------------- GEMM epilogues

GEMM_CASES = [
    dict(T=24, H=384, I=256, E=4, topk=2),
    dict(T=300, H=256, I=384, E=2, topk=1),           # several tiles per expert
    dict(T=200, H=640, I=128, E=16, topk=4),          # many small experts, some empty; K of 5 blocks
]


def stage_inputs(c, seed):
    wl = mi.Workload("bs_stage", seed, c["T"], c["H"], c["I"], c["E"], c["topk"])
    layer = Layer(wl, scale_fmt="ue8m0")
    hidden = mi.hidden(wl)
    logits = mi.router_logits(wl)
    oids, ow = oracle.route(logits.numpy(), wl.topk, True)
    perm = moe.moe_align_permute(torch.from_numpy(oids).to(DEV), wl.E)
    q, s = moe.fp8_group_quant(hidden.to(DEV), "ue8m0")
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
    a_sf = torch.from_numpy(pack_scales_np(As.numpy())).to(DEV)
    w13q, w13s, w2q, w2s = layer.oracle_weights(range(wl.E))
    ref = oracle.moe_forward(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, want_c1=True,
                             scale_fmt=UE8M0)
    m = unpadded_rows(perm["padded_offsets"].cpu().numpy(), ref["offsets"])
    return wl, layer, perm, A.to(DEV), a_sf, ref, m, torch.from_numpy(ow).to(DEV)


@pytest.mark.parametrize("ci", range(len(GEMM_CASES)))
def test_block_scaled_gemm_epilogues_match_the_oracle(ci):
    """store: C1 within fp32 accumulation error of the oracle's fp64 C1; silu: requantised codes
    within one e4m3 step (>= 99% identical) and UE8M0 scales within one power of two; weighted
    pairs: every pair row of C2 (from the oracle's own intermediate) within bf16 rounding."""
    wl, layer, perm, A, a_sf, ref, m, w = stage_inputs(GEMM_CASES[ci], 140 + ci)
    rows, P = A.shape[0], wl.T * wl.topk
    w13sf, w2sf = moe.moe_fp8_block_pack_scales(layer.w13s), moe.moe_fp8_block_pack_scales(layer.w2s)
    ts = (perm["tile_expert"], perm["tile_row0"], perm["num_tiles"])
    c1 = torch.zeros(rows, 2 * wl.I, dtype=torch.float32, device=DEV)
    moe.fp8_block_grouped_gemm(A, a_sf, (0, 0), layer.w13q, w13sf, *ts, "store", out_f32=c1, scale_fmt="ue8m0_packed")
    got = c1.cpu().double().numpy()[m]
    want = ref["c1"]
    scale = np.abs(want).max(axis=1, keepdims=True)
    assert np.abs(got - want).max() <= 1e-5 * scale.max() and np.all(np.abs(got - want) <= 2e-5 * scale + 1e-30)

    oq = torch.zeros(rows, wl.I, dtype=torch.uint8, device=DEV)
    osf = torch.zeros(moe.moe_packed_scale_bytes(rows, wl.I), dtype=torch.uint8, device=DEV)
    moe.fp8_block_grouped_gemm(A, a_sf, (0, 0), layer.w13q, w13sf, *ts, "silu_mul_quant", out_q=oq, out_scale=osf,
                               scale_fmt="ue8m0_packed")
    gs = unpack_scales_np(osf.cpu().numpy(), rows, wl.I)[m]
    ratio = gs / ref["a2s"]
    assert np.all(np.isin(ratio, [0.5, 1.0, 2.0])) and np.mean(ratio == 1.0) >= 0.99
    # in groups whose scale agrees: >= 99% identical codes, the rest adjacent codes of the same sign
    # (or +-0 around zero)
    same_group = np.repeat(ratio == 1.0, 128, axis=1)
    gq = oq.cpu().numpy()[m].astype(np.int32)[same_group]
    rq = ref["a2q"].astype(np.int32)[same_group]
    assert np.mean(gq == rq) >= 0.99
    diff = gq != rq
    mag_g, mag_r = gq[diff] & 0x7F, rq[diff] & 0x7F
    sign_ok = ((gq[diff] ^ rq[diff]) & 0x80 == 0) | ((mag_g <= 1) & (mag_r <= 1))
    assert np.all(sign_ok) and np.all(np.abs(mag_g - mag_r) <= 1)

    # the w2 GEMM on the oracle's own intermediate, weighted pair rows
    A2 = torch.zeros(rows, wl.I, dtype=torch.uint8)
    A2s = torch.ones(rows, wl.I // 128, dtype=torch.float32)
    A2[torch.from_numpy(m)] = torch.from_numpy(ref["a2q"])
    A2s[torch.from_numpy(m)] = torch.from_numpy(ref["a2s"])
    a2_sf = torch.from_numpy(pack_scales_np(A2s.numpy())).to(DEV)
    y = torch.zeros(P, wl.H, dtype=torch.bfloat16, device=DEV)
    moe.fp8_block_grouped_gemm(A2.to(DEV), a2_sf, (0, 0), layer.w2q, w2sf, *ts, "weighted_pairs_bf16", out_bf16=y,
                               sorted_pair_ids=perm["sorted_pair_ids"], topk_weights=w.reshape(-1), topk=wl.topk,
                               num_pairs=P, scale_fmt="ue8m0_packed")
    wflat = ref["weights"].reshape(-1).astype(np.float64)
    want_rows = np.zeros((P, wl.H))
    want_rows[ref["sorted"]] = ref["c2"] * wflat[ref["sorted"]][:, None]
    got_rows = y.float().cpu().double().numpy()
    tol = np.abs(want_rows) * 2.0 ** -8 + 1e-5 * np.abs(want_rows).max()
    assert np.all(np.abs(got_rows - want_rows) <= tol)


# ----------------------------------------------------------------------------- whole layer

class PackedLayer(Layer):
    """UE8M0 weights (GPU quantiser) with their scales packed for the block-scaled MMA."""

    def __init__(self, wl):
        super().__init__(wl, scale_fmt="ue8m0")
        self.w13sf = moe.moe_fp8_block_pack_scales(self.w13s)
        self.w2sf = moe.moe_fp8_block_pack_scales(self.w2s)

    def forward(self, hidden, logits, rp, packed=False):
        w13, w2 = self.w13q, self.w2q
        if packed:
            w13, w2 = moe.moe_fp8_block_pack_weights(w13), moe.moe_fp8_block_pack_weights(w2)
        return moe.moe_fp8_block_forward(hidden, logits, w13, self.w13sf, w2, self.w2sf, self.wl.topk,
                                         self.wl.renormalize, rp, scale_fmt="ue8m0_packed")


def run_packed_layer(wl, tokens=None):
    layer = PackedLayer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = layer.forward(hidden.to(DEV), logits.to(DEV), rp)
    out_tiled = layer.forward(hidden.to(DEV), logits.to(DEV), rp, packed=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out_tiled)
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    toks = range(wl.T) if tokens is None else tokens
    w13q, w13s, w2q, w2s = layer.oracle_weights(set(oids[list(toks)].reshape(-1).tolist()))
    ref = oracle.moe_forward(bits(hidden), logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, wl.renormalize,
                             tokens=tokens, scale_fmt=UE8M0, **okw)
    return out, ref


@pytest.mark.parametrize("T,H,I,E,topk", [(16, 256, 256, 4, 2), (1, 128, 128, 1, 1), (70, 128, 256, 3, 2),
                                          (300, 640, 384, 4, 1), (65, 128, 128, 16, 8)])
def test_packed_layer_all_tokens(T, H, I, E, topk):
    wl = mi.WORKLOADS["tiny"] if (T, H) == (16, 256) else mi.Workload("bs_edge", 150 + T + E, T, H, I, E, topk)
    out, ref = run_packed_layer(wl)
    assert_output_close(out, ref["out"])


@pytest.mark.parametrize("name,T", [("mixtral", None), ("dsv3", None), ("qwen3_skew", None), ("dsv3_decode", 1),
                                    ("dsv3_decode", 32)])
def test_packed_layer_full_size_every_tile_sampled(name, T):
    wl = mi.WORKLOADS[name] if T is None else mi.WORKLOADS[name].with_tokens(T)
    _, okw = routing_of(wl)
    oids, _ = oracle.route(mi.router_logits(wl).numpy(), wl.topk, wl.renormalize, **okw)
    tokens = tile_sample_tokens(oids, wl.E, extra=[0, wl.T - 1])
    out, ref = run_packed_layer(wl, tokens)
    assert_output_close(out, ref["out"], rows=tokens)


def test_packed_masked_layout():
    E, M, H, I = 5, 200, 256, 384
    wl = mi.Workload("bs_masked", 160, M, H, I, E, 1)
    layer = PackedLayer(wl)
    g = torch.Generator().manual_seed(161)
    hidden = torch.randn(E, M, H, generator=g).to(torch.bfloat16)
    counts = torch.tensor([0, 200, 17, 129, 1], dtype=torch.int32)
    out = moe.moe_fp8_block_forward_masked(hidden.to(DEV), counts.to(DEV), layer.w13q, layer.w13sf, layer.w2q,
                                           layer.w2sf, scale_fmt="ue8m0_packed")
    w13q, w13s, w2q, w2s = layer.oracle_weights(range(E))
    ref, _ = oracle.moe_forward_masked(bits(hidden), counts.numpy(), w13q, w13s, w2q, w2s, UE8M0)
    got = out.float().cpu().double().numpy()
    for e in range(E):
        c = int(counts[e])
        if c:
            assert_output_close(torch.from_numpy(got[e, :c]), ref[e, :c])


def test_packed_layer_rejects_the_decode_kernel_and_nvfp4():
    wl = mi.WORKLOADS["tiny"].with_tokens(2)
    layer = PackedLayer(wl)
    h, l = mi.hidden(wl).to(DEV), mi.router_logits(wl).to(DEV)
    with pytest.raises(moe.MoeError):
        moe.moe_fp8_block_forward(h, l, layer.w13q, layer.w13sf, layer.w2q, layer.w2sf, wl.topk, True, None,
                                  scale_fmt="ue8m0_packed", decode="on")
    # "auto" takes the tile kernels for a 2-token step in this format
    out = moe.moe_fp8_block_forward(h, l, layer.w13q, layer.w13sf, layer.w2q, layer.w2sf, wl.topk, True, None,
                                    scale_fmt="ue8m0_packed")
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("pair", [False, True], ids=["one_cta", "cta_pair"])
@pytest.mark.parametrize("fmt", ["ue8m0_packed", "mxfp8"])
def test_block_scaled_layer_repeats_and_replays_from_a_cuda_graph(fmt, pair):
    """Ten calls on one dirty workspace and a CUDA-graph replay on new inputs give the same bytes
    as a fresh eager call, in both block-scaled formats, on the one-CTA GEMMs (50 rows per expert)
    and on the CTA-pair GEMMs (600 rows per expert)."""
    wl = mi.Workload("bs_graph", 163, 1200, 256, 384, 2, 1) if pair else mi.Workload("bs_graph", 163, 300, 256, 384, 6, 2)
    if fmt == "mxfp8":
        from test_gpu_mxfp8 import MxLayer
        layer = MxLayer(wl)
    else:
        layer = PackedLayer(wl)
    rp, _ = routing_of(wl)
    hid = mi.hidden(wl).to(DEV)
    log = mi.router_logits(wl).to(DEV)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.topk), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)

    def step():
        moe.moe_fp8_block_forward(hid, log, layer.w13q, layer.w13sf, layer.w2q, layer.w2sf, wl.topk, True, rp,
                                  out=out, workspace=ws, scale_fmt=fmt)

    step()
    first = out.clone()
    for _ in range(9):
        step()
        assert torch.equal(out, first)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in range(2):
        wl_s = wl.with_(number=wl.number + 300 + seed)
        h, l = mi.hidden(wl_s).to(DEV), mi.router_logits(wl_s).to(DEV)
        hid.copy_(h)
        log.copy_(l)
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        want = moe.moe_fp8_block_forward(h, l, layer.w13q, layer.w13sf, layer.w2q, layer.w2sf, wl.topk, True, rp,
                                         scale_fmt=fmt)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
