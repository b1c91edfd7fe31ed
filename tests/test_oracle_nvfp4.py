"""Pins for the oracle's NVFP4 weight format (page "vllm.model_executor.layers.quantization.
online.nvfp4", _quantize_moe_weight_to_nvfp4) and the layer computed with it.

* The 16 e2m1 code values are compared with the hand-derived format facts in tests/golden/.
* Encoding is compared with a brute-force nearest-value search (ties to the even code,
  saturation at 6) over a grid that holds every midpoint.
* Weights built on the format's own grid (code value x power-of-two block scale, one value at
  6 x 448 so that the global scale is 1, or a power of two) must quantise back to exactly the
  codes, block scales and global scale they were built from: a wrong nibble order, block
  index, divisor (448 for 6) or amax scope fails it.
* Random weights stay within the format's rounding bounds.
* With one expert and top-1 the layer equals the dense chain in torch float64 on weights
  dequantised here from the golden table; a routed tiny layer equals a per-token brute force.
"""
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_codes.txt")


def golden_table():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            vals[int(c, 16)] = float(v)
    assert sorted(vals) == list(range(16))
    return np.array([vals[c] for c in range(16)])


def bf16_bits(x):
    return oracle.bf16_from_f64(np.asarray(x, dtype=np.float64))


def e4m3_value(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def dequant(q, sf, gs):
    """[E, N, K/2] codes, [E, N, K/16] scales, [E] global -> fp64 [E, N, K], from the golden table
    (low nibble first) and torch's float8_e4m3fn decoding."""
    tab = golden_table()
    E, N, K2 = q.shape
    codes = np.empty((E, N, 2 * K2), dtype=np.int64)
    codes[..., 0::2] = q & 15
    codes[..., 1::2] = q >> 4
    return tab[codes] * np.repeat(e4m3_value(sf), 16, axis=2) * gs.astype(np.float64)[:, None, None]


def test_e2m1_values_match_golden_facts():
    got = oracle.e2m1_values()
    want = golden_table()
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))
    assert got.max() == 6.0


def test_e2m1_encode_is_nearest_with_ties_to_even_and_saturation():
    tab = golden_table()
    mags = tab[:8]
    # every multiple of 1/64 in [-8, 8]: holds all the format's values and all midpoints
    x = np.arange(-8 * 64, 8 * 64 + 1) / 64.0
    got = oracle.e2m1_encode(x.astype(np.float32))
    for v, c in zip(x, got):
        a = min(abs(v), 6.0)
        d = np.abs(mags - a)
        best = np.nonzero(d == d.min())[0]
        want = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        if np.signbit(v):
            want |= 8
        assert int(c) == want, (v, int(c), want)
    # values round-trip
    assert oracle.e2m1_encode(tab.astype(np.float32)).tolist() == list(range(16))


def _grid_weights(rng, E, N, K, shift):
    """Weights on the NVFP4 grid: w = value(code) * p_block * 2^shift[e], one element of each
    expert at 6 * 448 * 2^shift[e] (its amax).  Returns bf16 bits and the expected codes / scales."""
    tab = golden_table()
    codes = rng.integers(0, 16, size=(E, N, K))
    pw = rng.integers(-6, 6, size=(E, N, K // 16))
    p = np.exp2(pw.astype(np.float64))
    # each block's largest magnitude is 6 (code 7 or 15) so that its scale is exactly p
    codes[..., ::16] = 7 + 8 * rng.integers(0, 2, size=(E, N, K // 16))
    for e in range(E):
        p[e, 0, 0] = 448.0
    w = tab[codes] * np.repeat(p, 16, axis=2)
    w *= np.exp2(np.asarray(shift, dtype=np.float64))[:, None, None]
    q = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    sf_other = (np.log2(p) + 7).astype(np.int64) << 3       # e4m3 bits of 2^k, -6 <= k <= 8
    sf = np.where(p == 448.0, 0x7E, sf_other).astype(np.uint8)
    return bf16_bits(w), q, sf


def test_nvfp4_quant_recovers_grid_weights_exactly():
    rng = np.random.default_rng(31)
    E, N, K = 3, 6, 64
    shift = [0, -5, 3]          # global scales 1, 2^-5 and 2^3 (amax 2688 * 2^shift)
    w, q_want, sf_want = _grid_weights(rng, E, N, K, shift)
    q, sf, gs = oracle.quant_nvfp4_bf16(w)
    assert np.array_equal(gs, np.exp2(np.asarray(shift, dtype=np.float32)))
    assert np.array_equal(sf, sf_want)
    # codes equal, signed zeros included (bf16 and the fp32 quotient keep the sign of a zero)
    assert np.array_equal(q, q_want)
    assert np.array_equal(dequant(q, sf, gs), oracle.bf16_to_f64(w))


def test_nvfp4_quant_random_weights_within_format_bounds():
    rng = np.random.default_rng(32)
    E, N, K = 2, 8, 256
    wf = rng.standard_normal((E, N, K)) * 0.02
    wf[1] *= 37.0
    w = bf16_bits(wf)
    q, sf, gs = oracle.quant_nvfp4_bf16(w)
    x = oracle.bf16_to_f64(w)
    amax = np.abs(x).reshape(E, -1).max(1)
    # global scale: amax / (6 * 448) up to the two fp32 roundings of 1 / (2688 / amax)
    assert np.all(np.abs(gs / (amax / 2688.0) - 1.0) < 2.0 ** -22)
    tab = golden_table()
    codes = np.empty((E, N, K), dtype=np.int64)
    codes[..., 0::2] = q & 15
    codes[..., 1::2] = q >> 4
    gsc = (np.float32(2688.0) / amax.astype(np.float32)).astype(np.float64)
    scaled = oracle.bf16_to_f64(bf16_bits(x * gsc[:, None, None]))
    sfv = np.repeat(e4m3_value(sf), 16, axis=2)
    vmax = np.abs(scaled).reshape(E, N, K // 16, 16).max(3)
    # block scale: e4m3 rounding of vmax / 6 (3 mantissa bits: relative error <= 2^-4)
    assert np.all(np.abs(e4m3_value(sf) - vmax / 6.0) <= 2.0 ** -4 * vmax / 6.0 + 2.0 ** -10)
    # codes: nearest grid value of scaled / scale, i.e. error <= half the local spacing
    r = scaled / np.where(sfv == 0, 1.0, sfv)
    spacing = np.where(np.abs(r) < 2.0, 0.5, np.where(np.abs(r) < 4.0, 1.0, 2.0))
    err = np.abs(np.clip(np.abs(r), 0, 6.0) - np.abs(tab[codes]))
    assert np.all(err <= spacing / 2 + 1e-12)
    assert np.all((np.sign(tab[codes]) == np.sign(r)) | (tab[codes] == 0))


def _dense_chain_nvfp4(hid_bits, W13, W2):
    """E=1, top-1 in torch float64: 1x128 quantisation, x @ W13^T, SiLU(gate)*up in fp32,
    requantisation, @ W2^T."""
    x = torch.from_numpy(oracle.bf16_to_f64(hid_bits)).float()
    I = W2.shape[1]

    def quant(v):
        g = v.view(v.shape[0], -1, 128)
        s = g.abs().amax(2).clamp_min(1e-8) / 448.0
        q = (g / s[..., None]).to(torch.float8_e4m3fn)
        return q.double().view(v.shape[0], -1) * s.double().repeat_interleave(128, 1)

    c1 = quant(x) @ torch.from_numpy(W13).T
    h = (torch.nn.functional.silu(c1[:, :I]) * c1[:, I:]).float()
    return (quant(h) @ torch.from_numpy(W2).T).numpy()


def test_nvfp4_single_expert_top1_reduces_to_dense_chain():
    rng = np.random.default_rng(33)
    T, H, I = 5, 256, 384
    hid = bf16_bits(rng.standard_normal((T, H)))
    q13, s13, g13 = oracle.quant_nvfp4_bf16(bf16_bits(rng.standard_normal((1, 2 * I, H)) * 0.02))
    q2, s2, g2 = oracle.quant_nvfp4_bf16(bf16_bits(rng.standard_normal((1, H, I)) * 0.02))
    r = oracle.moe_forward_nvfp4(hid, np.zeros((T, 1), np.float32), q13, s13, g13, q2, s2, g2, 1)
    ref = _dense_chain_nvfp4(hid, dequant(q13, s13, g13)[0], dequant(q2, s2, g2)[0])
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-14)


def test_nvfp4_routed_layer_brute_force_per_token():
    rng = np.random.default_rng(34)
    T, H, I, E, k = 6, 256, 256, 4, 2
    hid = bf16_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    q13, s13, g13 = oracle.quant_nvfp4_bf16(bf16_bits(rng.standard_normal((E, 2 * I, H)) * 0.02))
    q2, s2, g2 = oracle.quant_nvfp4_bf16(bf16_bits(rng.standard_normal((E, H, I)) * 0.02))
    r = oracle.moe_forward_nvfp4(hid, logits, q13, s13, g13, q2, s2, g2, k)
    W13, W2 = dequant(q13, s13, g13), dequant(q2, s2, g2)
    ref = np.zeros((T, H))
    for t in range(T):
        top = torch.topk(torch.from_numpy(logits[t]).double(), k)
        wts = torch.softmax(top.values, 0)
        for j in range(k):
            e = int(top.indices[j])
            y = _dense_chain_nvfp4(hid[t:t + 1], W13[e], W2[e])
            ref[t] += float(np.float32(wts[j])) * y[0]
    rel = np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref)
    assert rel < 1e-9, rel
    assert np.array_equal(r["out_bf16"], oracle.bf16_from_f64(r["out"]))


def test_nvfp4_sampled_tokens_match_full_run():
    rng = np.random.default_rng(35)
    T, H, I, E, k = 9, 128, 256, 3, 2
    hid = bf16_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    q13, s13, g13 = oracle.quant_nvfp4_bf16(bf16_bits(rng.standard_normal((E, 2 * I, H)) * 0.02))
    q2, s2, g2 = oracle.quant_nvfp4_bf16(bf16_bits(rng.standard_normal((E, H, I)) * 0.02))
    full = oracle.moe_forward_nvfp4(hid, logits, q13, s13, g13, q2, s2, g2, k)
    part = oracle.moe_forward_nvfp4(hid, logits, q13, s13, g13, q2, s2, g2, k, tokens=[1, 8])
    assert np.array_equal(part["out"][[1, 8]], full["out"][[1, 8]])
    assert np.all(np.isnan(part["out"][[0, 2, 7]]))
