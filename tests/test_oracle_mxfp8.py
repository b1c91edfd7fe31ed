"""Pins for the oracle's MXFP8 mode ("MXFP8 (block [1, 32])", page
"vllm.model_executor.layers.fused_moe.oracle.fp8", make_fp8_moe_quant_config; weights with "e8m0
group-32 scales", _humming_fp8_weight_schema).

* Rows built from e4m3 grid values times a power of two per 32-wide group quantise back to exactly
  those codes and scales (a group of 128, or a scale that is not rounded up, fails it).
* Random rows: the scales equal 2^ceil(log2(max(amax, 1e-8) / 448)) from numpy, the codes torch's
  float8_e4m3fn cast of x / scale.
* With one expert and top-1 the layer reduces to the dense chain in torch float64 (1x32 groups
  for the activations and the intermediate, weights dequantised with their 32-wide blocks), and
  a per-token brute force of a routed layer agrees.
"""
import numpy as np
import torch

import moe_inputs as mi
import oracle


def bf16_bits(x):
    return oracle.bf16_from_f64(np.asarray(x, dtype=np.float64))


def deq_torch(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double()


def test_mxfp8_groups_quantise_back_to_their_codes():
    rng = np.random.default_rng(31)
    vals = oracle.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(vals[c])])
    R, C = 5, 256
    codes = rng.choice(finite, size=(R, C)).astype(np.uint8)
    exps = rng.integers(-12, 6, size=(R, C // 32))
    for r in range(R):
        for g in range(C // 32):
            codes[r, g * 32 + rng.integers(0, 32)] = 0x7E | (0x80 if rng.random() < 0.5 else 0)   # +-448
    x = vals[codes] * np.exp2(np.repeat(exps, 32, axis=1))
    q, s = oracle.quant_1x32_bf16(bf16_bits(x))
    assert np.array_equal(s, np.exp2(exps).astype(np.float32))
    assert np.array_equal(q, codes)


def test_mxfp8_quant_matches_torch_formulation():
    rng = np.random.default_rng(32)
    R, C = 64, 512
    x = rng.standard_normal((R, C)) * np.exp2(rng.integers(-30, 30, size=(R, 1)))
    x[0] = 0.0                                                    # zero groups: floor scale, zero codes
    xb = bf16_bits(x)
    q, s = oracle.quant_1x32_bf16(xb)
    xf = torch.from_numpy(oracle.bf16_to_f64(xb)).float().view(R, C // 32, 32)
    t = (xf.abs().amax(2).clamp_min(1e-8) / 448.0)                # fp32 quotient
    want_s = torch.exp2(torch.ceil(torch.log2(t.double()))).float()
    assert np.array_equal(s, want_s.numpy())
    want_q = (xf / want_s[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).view(R, C)
    assert np.array_equal(q, want_q.numpy())


def test_mxfp8_weight_quant_is_rowwise_1x32():
    rng = np.random.default_rng(33)
    E, N, K = 2, 128, 256
    w = bf16_bits(rng.standard_normal((E, N, K)) * 0.02)
    q, s = oracle.quant_mxfp8_weight_bf16(w)
    assert q.shape == (E, N, K) and s.shape == (E, N, K // 32)
    q2, s2 = oracle.quant_1x32_bf16(w.reshape(E * N, K))
    assert np.array_equal(q.reshape(E * N, K), q2) and np.array_equal(s.reshape(E * N, K // 32), s2)
    assert np.all(np.frexp(s)[0] == 0.5)                          # powers of two


def _dense_chain_mx(hid_bits, w13q, w13s, w2q, w2s):
    """E=1, top-1 in torch float64: 1x32 UE8M0 quantisation of the hidden state, GEMM with
    per-32 weight scales, SiLU(gate)*up, 1x32 requantisation, GEMM."""
    x = torch.from_numpy(oracle.bf16_to_f64(hid_bits)).float()

    def quant(v):
        g = v.view(v.shape[0], -1, 32)
        s = torch.exp2(torch.ceil(torch.log2((g.abs().amax(2).clamp_min(1e-8) / 448.0).double()))).float()
        q = (g / s[..., None]).to(torch.float8_e4m3fn)
        return q.double().view(v.shape[0], -1) * s.double().repeat_interleave(32, 1)

    I = w2q.shape[2]
    W13 = deq_torch(w13q[0]) * torch.from_numpy(w13s[0]).double().repeat_interleave(32, 1)
    W2 = deq_torch(w2q[0]) * torch.from_numpy(w2s[0]).double().repeat_interleave(32, 1)
    c1 = quant(x) @ W13.T
    h = (torch.nn.functional.silu(c1[:, :I]) * c1[:, I:]).float()
    return (quant(h) @ W2.T).numpy()


def test_mxfp8_single_expert_reduces_to_dense_chain():
    rng = np.random.default_rng(34)
    T, H, I = 7, 256, 384
    hid = bf16_bits(rng.standard_normal((T, H)) * 3.0)
    w13q, w13s = oracle.quant_mxfp8_weight_bf16(bf16_bits(rng.standard_normal((1, 2 * I, H)) * 0.02))
    w2q, w2s = oracle.quant_mxfp8_weight_bf16(bf16_bits(rng.standard_normal((1, H, I)) * 0.02))
    r = oracle.moe_forward_mxfp8(hid, np.zeros((T, 1), np.float32), w13q, w13s, w2q, w2s, 1)
    assert r["a1s"].shape == (T, H // 32) and r["a2s"].shape[1] == I // 32
    ref = _dense_chain_mx(hid, w13q, w13s, w2q, w2s)
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-14)


def test_mxfp8_layer_brute_force_per_token():
    """The tiny workload's shapes (T=16, H=256, I=256, E=4, top-2 softmax) in MXFP8: loop over
    tokens, then over each token's experts, in torch float64."""
    wl = mi.WORKLOADS["tiny"]
    hid = mi.bf16_bits(mi.hidden(wl))
    logits = mi.router_logits(wl).numpy()
    w13q, w13s = oracle.quant_mxfp8_weight_bf16(mi.bf16_bits(mi.w13_bf16(wl)))
    w2q, w2s = oracle.quant_mxfp8_weight_bf16(mi.bf16_bits(mi.w2_bf16(wl)))
    r = oracle.moe_forward_mxfp8(hid, logits, w13q, w13s, w2q, w2s, wl.topk)
    x = torch.from_numpy(oracle.bf16_to_f64(hid)).float()
    ref = np.zeros((wl.T, wl.H))
    for t in range(wl.T):
        top = torch.topk(torch.from_numpy(logits[t]).double(), wl.topk)
        wts = torch.softmax(top.values, 0)
        for j in range(wl.topk):
            e = int(top.indices[j])
            y = _dense_chain_mx(mi.bf16_bits(x[t:t + 1].to(torch.bfloat16)), w13q[e:e + 1], w13s[e:e + 1],
                                w2q[e:e + 1], w2s[e:e + 1])
            ref[t] += float(np.float32(wts[j])) * y[0]
    rel = np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref)
    assert rel < 1e-9, rel


def test_mxfp8_sampled_tokens_match_full_run():
    rng = np.random.default_rng(36)
    T, H, I, E, k = 9, 128, 256, 3, 2
    hid = bf16_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    w13q, w13s = oracle.quant_mxfp8_weight_bf16(bf16_bits(rng.standard_normal((E, 2 * I, H)) * 0.02))
    w2q, w2s = oracle.quant_mxfp8_weight_bf16(bf16_bits(rng.standard_normal((E, H, I)) * 0.02))
    full = oracle.moe_forward_mxfp8(hid, logits, w13q, w13s, w2q, w2s, k)
    part = oracle.moe_forward_mxfp8(hid, logits, w13q, w13s, w2q, w2s, k, tokens=[1, 8])
    assert np.array_equal(part["out"][[1, 8]], full["out"][[1, 8]])
    assert np.all(np.isnan(part["out"][[0, 2, 7]]))
