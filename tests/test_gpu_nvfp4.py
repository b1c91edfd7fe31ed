"""NVFP4 expert weights (page "vllm.model_executor.layers.quantization.online.nvfp4",
_quantize_moe_weight_to_nvfp4) on the GPU: the quantiser's codes, block scales and global
scales bit-exact against the oracle, the packed layout element by element, and the layer on
NVFP4 weights (decode-path kernel) against the oracle's layer on the oracle's own
quantisation of the same bf16 weights, for one to eight tokens and for longer steps that run
eight tokens at a time."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import block_fp8_mixture_topk_gb300 as moe
from moe_testutil import assert_output_close, routing_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
UNIT = 16 * 64 + 16 * 8


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def pack_reference(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """[E, N, K/2] codes and [E, N, K/16] scales -> [E, N/16, K/128, 1152] by index arithmetic."""
    E, N, K2 = q.shape
    K = 2 * K2
    codes = q.reshape(E, N // 16, 16, K // 128, 64).transpose(0, 1, 3, 2, 4).reshape(E, N // 16, K // 128, 1024)
    scales = sf.reshape(E, N // 16, 16, K // 128, 8).transpose(0, 1, 3, 2, 4).reshape(E, N // 16, K // 128, 128)
    return np.concatenate([codes, scales], axis=3)


class Fp4Layer:
    """NVFP4 weights of a workload quantised on the GPU (and packed), and the oracle's own
    quantisation of any subset of experts from the same bf16 weights."""

    def __init__(self, wl, chunk=8):
        self.wl = wl
        E, H, I = wl.E, wl.H, wl.I
        self.q13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=DEV)
        self.s13 = torch.empty(E, 2 * I, H // 16, dtype=torch.uint8, device=DEV)
        self.g13 = torch.empty(E, dtype=torch.float32, device=DEV)
        self.q2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=DEV)
        self.s2 = torch.empty(E, H, I // 16, dtype=torch.uint8, device=DEV)
        self.g2 = torch.empty(E, dtype=torch.float32, device=DEV)
        for e0 in range(0, E, chunk):
            ex = range(e0, min(E, e0 + chunk))
            n = len(ex)
            self.q13[e0:e0 + n], self.s13[e0:e0 + n], self.g13[e0:e0 + n] = \
                moe.moe_nvfp4_quant_weight(mi.w13_bf16(wl, DEV, ex))
            self.q2[e0:e0 + n], self.s2[e0:e0 + n], self.g2[e0:e0 + n] = \
                moe.moe_nvfp4_quant_weight(mi.w2_bf16(wl, DEV, ex))
        self.p13 = moe.moe_nvfp4_pack_weights(self.q13, self.s13)
        self.p2 = moe.moe_nvfp4_pack_weights(self.q2, self.s2)
        torch.cuda.synchronize()

    def forward(self, hidden, logits, rp, scale_fmt="f32", workspace=None):
        wl = self.wl
        return moe.moe_nvfp4_forward(hidden, logits, self.p13, self.g13, self.p2, self.g2, wl.topk, wl.renormalize,
                                     rp, scale_fmt=scale_fmt, workspace=workspace)

    def oracle_weights(self, experts):
        wl = self.wl
        E, H, I = wl.E, wl.H, wl.I
        w = dict(q13=np.zeros((E, 2 * I, H // 2), np.uint8), s13=np.zeros((E, 2 * I, H // 16), np.uint8),
                 g13=np.ones(E, np.float32), q2=np.zeros((E, H, I // 2), np.uint8),
                 s2=np.zeros((E, H, I // 16), np.uint8), g2=np.ones(E, np.float32))
        for e in sorted(set(int(x) for x in experts)):
            q, s, g = oracle.quant_nvfp4_bf16(mi.bf16_bits(mi.w13_bf16(wl, DEV, [e])))
            w["q13"][e], w["s13"][e], w["g13"][e] = q[0], s[0], g[0]
            q, s, g = oracle.quant_nvfp4_bf16(mi.bf16_bits(mi.w2_bf16(wl, DEV, [e])))
            w["q2"][e], w["s2"][e], w["g2"][e] = q[0], s[0], g[0]
        return w


def test_nvfp4_quant_bit_exact_against_oracle():
    g = torch.Generator().manual_seed(71)
    E, N, K = 3, 256, 512
    w = torch.randn(E, N, K, generator=g) * 0.02
    w[1] *= 50.0                 # another global scale
    w[2, :, 64:80] = 0.0         # zero blocks: scale 0, codes 0
    w[2, 3, 100] = 3.0e-4        # a tiny block among them
    wb = w.to(torch.bfloat16)
    q, sf, gs = moe.moe_nvfp4_quant_weight(wb.to(DEV))
    torch.cuda.synchronize()
    oq, osf, ogs = oracle.quant_nvfp4_bf16(bits(wb))
    assert np.array_equal(gs.cpu().numpy(), ogs)
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(q.cpu().numpy(), oq)


def test_nvfp4_pack_layout():
    g = torch.Generator().manual_seed(72)
    E, N, K = 2, 48, 384
    q = torch.randint(0, 256, (E, N, K // 2), generator=g, dtype=torch.uint8)
    sf = torch.randint(0, 127, (E, N, K // 16), generator=g, dtype=torch.uint8)
    packed = moe.moe_nvfp4_pack_weights(q.to(DEV), sf.to(DEV))
    torch.cuda.synchronize()
    assert packed.numel() == moe.moe_nvfp4_packed_bytes(E, N, K)
    assert np.array_equal(packed.cpu().numpy(), pack_reference(q.numpy(), sf.numpy()))


CASES = [("dsv3_decode", 1), ("dsv3_decode", 2), ("dsv3_decode", 8), ("mixtral", 1), ("mixtral", 8),
         ("tiny", 5), ("tiny", 13), ("tiny", 16)]


@pytest.mark.parametrize("name,T", CASES)
def test_nvfp4_layer_matches_oracle(name, T):
    wl = mi.WORKLOADS[name].with_tokens(T)
    layer = Fp4Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = layer.forward(hidden.to(DEV), logits.to(DEV), rp)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(clear=True) == 0
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    touched = set(oids.reshape(-1).tolist())
    w = layer.oracle_weights(touched)
    # the GPU's quantisation of the touched experts is the oracle's, byte for byte
    for e in sorted(touched):
        assert np.array_equal(layer.q13[e].cpu().numpy(), w["q13"][e])
        assert np.array_equal(layer.s13[e].cpu().numpy(), w["s13"][e])
        assert np.array_equal(layer.q2[e].cpu().numpy(), w["q2"][e])
        assert layer.g13[e].item() == w["g13"][e] and layer.g2[e].item() == w["g2"][e]
    ref = oracle.moe_forward_nvfp4(bits(hidden), logits.numpy(), w["q13"], w["s13"], w["g13"], w["q2"], w["s2"],
                                   w["g2"], wl.topk, wl.renormalize, **okw)["out"]
    assert_output_close(out, ref)


@pytest.mark.parametrize("T", [32, 128])
def test_nvfp4_dsv3_decode_steps_in_passes_of_eight(T):
    """DeepSeek-V3-shaped decode steps of 32 and 128 tokens on NVFP4 weights (grouped sigmoid
    routing with bias and routed scaling): the forward runs them eight tokens at a time.  Sampled
    tokens from the first, a middle and the last pass of eight against the oracle."""
    wl = mi.WORKLOADS["dsv3_decode"].with_tokens(T)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    tokens = sorted(set([0, 7, 8, T // 2 + 3, T - 9, T - 1]))
    layer = Fp4Layer(wl)
    out = layer.forward(hidden.to(DEV), logits.to(DEV), rp)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(clear=True) == 0
    w = layer.oracle_weights(set(oids[tokens].reshape(-1).tolist()))
    ref = oracle.moe_forward_nvfp4(bits(hidden), logits.numpy(), w["q13"], w["s13"], w["g13"], w["q2"], w["s2"],
                                   w["g2"], wl.topk, wl.renormalize, tokens=tokens, **okw)["out"]
    assert_output_close(out, ref, rows=tokens)


@pytest.mark.parametrize("T,H,I,E,topk", [(1, 128, 128, 1, 1), (8, 128, 256, 1, 1), (6, 256, 128, 3, 3)])
def test_nvfp4_edge_shapes(T, H, I, E, topk):
    """One expert and top-1 (a dense NVFP4 MLP), every token on the single expert, top-k equal to
    the number of experts, K smaller than the MMA warps' K blocks."""
    wl = mi.Workload("fp4_edge", 190 + T + E, T, H, I, E, topk)
    layer = Fp4Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = layer.forward(hidden.to(DEV), logits.to(DEV), rp)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(clear=True) == 0
    w = layer.oracle_weights(range(E))
    ref = oracle.moe_forward_nvfp4(bits(hidden), logits.numpy(), w["q13"], w["s13"], w["g13"], w["q2"], w["s2"],
                                   w["g2"], wl.topk, wl.renormalize, **okw)["out"]
    assert_output_close(out, ref)


def test_nvfp4_ue8m0_activations_and_repeated_calls():
    """Power-of-two activation scales; ten calls on one workspace and a CUDA-graph replay give the
    same bytes (the decode kernel's counters restart from zero every call)."""
    wl = mi.WORKLOADS["dsv3_decode"].with_tokens(2)
    layer = Fp4Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    h, l = hidden.to(DEV), logits.to(DEV)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.topk), dtype=torch.uint8,
                     device=DEV)
    first = layer.forward(h, l, rp, scale_fmt="ue8m0", workspace=ws).clone()
    for _ in range(9):
        again = layer.forward(h, l, rp, scale_fmt="ue8m0", workspace=ws)
        assert torch.equal(again, first)
    out = torch.empty_like(first)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            moe.moe_nvfp4_forward(h, l, layer.p13, layer.g13, layer.p2, layer.g2, wl.topk, wl.renormalize, rp,
                                  out=out, workspace=ws, scale_fmt="ue8m0")
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, first)
    assert moe.moe_get_device_status(clear=True) == 0
    oids, _ = oracle.route(logits.numpy(), wl.topk, wl.renormalize, **okw)
    w = layer.oracle_weights(set(oids.reshape(-1).tolist()))
    ref = oracle.moe_forward_nvfp4(bits(hidden), logits.numpy(), w["q13"], w["s13"], w["g13"], w["q2"], w["s2"],
                                   w["g2"], wl.topk, wl.renormalize, scale_fmt=oracle.SCALE_UE8M0, **okw)["out"]
    assert_output_close(first, ref)
