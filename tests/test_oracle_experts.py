"""Pins for the oracle's expert computation (GEMM1, SiLU*up + requant, GEMM2, combine).

* GEMM1 on power-of-two scales is compared EXACTLY with an integer computation
  (e4m3 values are multiples of 2^-9, so every product is an integer times a
  power of two): a transposed operand or a wrong scale index fails it.
* SiLU(gate)*up and the requantisation are pinned by closed forms: gate values
  0, +56 and -56 give h = 0, 56*u and ~0, and a single non-zero group quantises
  its maximum to 448 with scale amax/448.
* Random inputs are compared with torch float64 matmuls on tensors dequantised
  through torch's own float8_e4m3fn dtype.
* With one expert and top-1 the layer reduces to the dense block-FP8 chain, and
  a per-token brute force (different loop order, torch arithmetic) agrees.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def deq_torch(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double()


def bf16_bits(x):
    return oracle.bf16_from_f64(np.asarray(x, dtype=np.float64))


def rows_with_known_quant(rng, T, H, exps):
    """bf16 rows whose 1x128 quantisation is exactly (codes, 2^exps)."""
    vals = oracle.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(vals[c])])
    codes = rng.choice(finite, size=(T, H)).astype(np.uint8)
    for t in range(T):
        for g in range(H // 128):
            codes[t, g * 128 + rng.integers(0, 128)] = 0x7E
    x = vals[codes] * np.exp2(np.repeat(exps, 128, axis=1))
    return bf16_bits(x), codes


def test_gemm1_exact_integer_arithmetic():
    rng = np.random.default_rng(21)
    T, H, I, E, k = 3, 256, 128, 2, 2
    a_exp = rng.integers(-3, 1, size=(T, H // 128))
    hid, a_codes = rows_with_known_quant(rng, T, H, a_exp)
    vals = oracle.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(vals[c]) and abs(vals[c]) <= 64])
    w13 = rng.choice(finite, size=(E, 2 * I, H)).astype(np.uint8)
    w_exp = rng.integers(-4, 0, size=(E, 2 * I // 128, H // 128))
    w13s = np.exp2(w_exp).astype(np.float32)
    w2 = rng.choice(finite, size=(E, H, I)).astype(np.uint8)
    w2s = np.full((E, H // 128, I // 128), 2.0 ** -6, dtype=np.float32)
    logits = np.array([[1.0, 0.0], [0.0, 1.0], [0.5, 0.2]], dtype=np.float32)
    r = oracle.moe_forward(hid, logits, w13, w13s, w2, w2s, k, want_c1=True)
    assert np.array_equal(r["a1q"], a_codes)
    assert np.array_equal(r["a1s"], np.exp2(a_exp).astype(np.float32))
    ai = (vals[a_codes] * 512).astype(np.int64)               # integer multiples of 2^-9
    wi = (vals[w13] * 512).astype(np.int64)
    for row in range(T * k):
        p = int(r["sorted"][row])
        t, e = p // k, int(r["ids"].reshape(-1)[p])
        for n in range(2 * I):
            exact = Fraction(0)
            for kb in range(H // 128):
                dot = int(np.dot(ai[t, kb * 128:(kb + 1) * 128], wi[e, n, kb * 128:(kb + 1) * 128]))
                exact += Fraction(dot) * Fraction(2) ** int(a_exp[t, kb] + w_exp[e, n // 128, kb] - 18)
            assert Fraction(r["c1"][row, n]) == exact, (row, n)


def _single_column_case(gate_vals, up_val, w2_code=0x38, T=1):
    """E=1, k=1, H=I=128: hidden = 448*2^-6 at column 0, so a = 7 there and 0 elsewhere.
    Gate row i holds value gate_vals[i]/7 at column 0, every up row holds up_val/7."""
    vals = oracle.e4m3_values()
    code_of = {float(vals[c]): c for c in range(127)}
    H = I = 128
    x = np.zeros((T, H))
    x[:, 0] = 448 * 2.0 ** -6
    w13 = np.zeros((1, 2 * I, H), dtype=np.uint8)
    for i, g in enumerate(gate_vals):
        v = abs(g) / 7
        w13[0, i, 0] = code_of[v] | (0x80 if g < 0 else 0)
    w13[0, I:, 0] = code_of[up_val / 7]
    w13s = np.ones((1, 2, 1), dtype=np.float32)
    w2 = np.full((1, H, I), w2_code, dtype=np.uint8)
    w2s = np.ones((1, 1, 1), dtype=np.float32)
    logits = np.zeros((T, 1), dtype=np.float32)
    return oracle.moe_forward(bf16_bits(x), logits, w13, w13s, w2, w2s, 1, want_c1=True)


def test_silu_up_closed_forms_and_requant():
    gate = np.zeros(128)
    gate[0:10] = 56.0          # silu(56) == 56 in fp64
    gate[10:20] = -56.0        # silu(-56) ~ -2.7e-23
    r = _single_column_case(gate, up_val=7.0)
    assert np.array_equal(r["c1"][0, :128], gate)
    assert np.all(r["c1"][0, 128:] == 7.0)
    # h = 392 on the first ten columns, ~0 on the next ten, 0 elsewhere: amax 392 -> scale 392/448
    assert r["a2s"][0, 0] == np.float32(392.0) / np.float32(448.0)
    assert np.all(r["a2q"][0, 0:10] == 0x7E)
    assert np.all(r["a2q"][0, 10:] & 0x7F == 0)
    # GEMM2 with all-ones w2 sums the ten dequantised values 448*0.875 = 392
    assert np.all(r["c2"][0] == 10 * 448 * float(np.float32(0.875)))
    assert np.all(r["out"][0] == r["c2"][0])     # single expert, weight exactly 1


def test_silu_up_general_value_and_gate_up_order():
    gate = np.zeros(128)
    gate[0] = 3.5
    r = _single_column_case(gate, up_val=14.0)
    h0 = 3.5 / (1 + math.exp(-3.5)) * 14.0        # gate is the first half, up the second
    s = np.float32(np.float32(h0) / np.float32(448.0))
    assert r["a2s"][0, 0] == s
    assert r["a2q"][0, 0] == 0x7E
    swapped = 14.0 / (1 + math.exp(-14.0)) * 3.5
    assert abs(float(s) * 448 - swapped) > 1.0


def test_random_gemms_against_torch_float64():
    rng = np.random.default_rng(5)
    T, H, I, E, k = 12, 384, 256, 3, 2
    hid = bf16_bits(rng.standard_normal((T, H)))
    w13q = rng.integers(0, 256, size=(E, 2 * I, H)).astype(np.uint8)
    w13q[(w13q & 0x7F) == 0x7F] = 0x3F                       # no NaN codes
    w2q = rng.integers(0, 256, size=(E, H, I)).astype(np.uint8)
    w2q[(w2q & 0x7F) == 0x7F] = 0x3F
    w13s = rng.uniform(1e-4, 3e-4, size=(E, 2 * I // 128, H // 128)).astype(np.float32)
    w2s = rng.uniform(1e-4, 3e-4, size=(E, H // 128, I // 128)).astype(np.float32)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle.moe_forward(hid, logits, w13q, w13s, w2q, w2s, k, want_c1=True)
    A = deq_torch(r["a1q"]) * torch.from_numpy(r["a1s"]).double().repeat_interleave(128, 1)
    W13 = deq_torch(w13q) * torch.from_numpy(w13s).double().repeat_interleave(128, 1).repeat_interleave(128, 2)
    W2 = deq_torch(w2q) * torch.from_numpy(w2s).double().repeat_interleave(128, 1).repeat_interleave(128, 2)
    ids = r["ids"].reshape(-1)
    out = torch.zeros(T, H, dtype=torch.float64)
    for row in range(T * k):
        p = int(r["sorted"][row])
        t, e = p // k, int(ids[p])
        c1 = W13[e] @ A[t]
        assert torch.allclose(torch.from_numpy(r["c1"][row]), c1, rtol=1e-12, atol=1e-12)
        h = (torch.nn.functional.silu(c1[:I]) * c1[I:]).float()
        amax = h.view(-1, 128).abs().amax(1).clamp_min(1e-8)
        s = amax / 448.0
        q = (h.view(-1, 128) / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(-1)
        assert np.array_equal(r["a2s"][row], s.numpy())
        assert np.array_equal(r["a2q"][row], q.numpy())
        a2 = deq_torch(r["a2q"][row]) * torch.from_numpy(r["a2s"][row]).double().repeat_interleave(128)
        c2 = W2[e] @ a2
        assert torch.allclose(torch.from_numpy(r["c2"][row]), c2, rtol=1e-12, atol=1e-12)
        out[t] += float(r["weights"].reshape(-1)[p]) * c2
    assert torch.allclose(torch.from_numpy(r["out"]), out, rtol=1e-12, atol=1e-12)
    # unpermute: pos maps each pair back to its sorted row
    assert np.array_equal(r["sorted"][r["pos"]], np.arange(T * k))


def _dense_chain_torch(hid_bits, w13q, w13s, w2q, w2s, ue8m0=False):
    """E=1, top-1: quantise -> GEMM -> SiLU*up -> requantise -> GEMM, all in torch (with ue8m0:
    every activation scale rounded up to a power of two)."""
    x = torch.from_numpy(oracle.bf16_to_f64(hid_bits)).float()
    T, H = x.shape
    I = w2q.shape[2]

    def quant(v):
        g = v.view(v.shape[0], -1, 128)
        s = g.abs().amax(2).clamp_min(1e-8) / 448.0
        if ue8m0:
            s = torch.exp2(torch.ceil(torch.log2(s.double()))).float()
        q = (g / s[..., None]).to(torch.float8_e4m3fn)
        return q.double().view(v.shape[0], -1) * s.double().repeat_interleave(128, 1)

    W13 = deq_torch(w13q[0]) * torch.from_numpy(w13s[0]).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
    W2 = deq_torch(w2q[0]) * torch.from_numpy(w2s[0]).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
    c1 = quant(x) @ W13.T
    h = (torch.nn.functional.silu(c1[:, :I]) * c1[:, I:]).float()
    return (quant(h) @ W2.T).numpy()


def test_single_expert_top1_reduces_to_dense_chain():
    rng = np.random.default_rng(8)
    T, H, I = 9, 256, 384
    hid = bf16_bits(rng.standard_normal((T, H)))
    w13q, w13s = oracle.quant_128x128_bf16(bf16_bits(rng.standard_normal((1, 2 * I, H)) * 0.02))
    w2q, w2s = oracle.quant_128x128_bf16(bf16_bits(rng.standard_normal((1, H, I)) * 0.02))
    r = oracle.moe_forward(hid, np.zeros((T, 1), np.float32), w13q, w13s, w2q, w2s, 1)
    assert np.all(r["weights"] == 1.0)
    ref = _dense_chain_torch(hid, w13q, w13s, w2q, w2s)
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-14)


def test_tiny_layer_brute_force_per_token():
    """The tiny workload (T=16, H=256, I=256, E=4, top-2 softmax): loop over tokens, then over each
    token's experts, in torch float64 with torch's float8 casts."""
    import moe_inputs as mi
    wl = mi.WORKLOADS["tiny"]
    hid = mi.bf16_bits(mi.hidden(wl))
    logits = mi.router_logits(wl).numpy()
    w13q, w13s = oracle.quant_128x128_bf16(mi.bf16_bits(mi.w13_bf16(wl)))
    w2q, w2s = oracle.quant_128x128_bf16(mi.bf16_bits(mi.w2_bf16(wl)))
    r = oracle.moe_forward(hid, logits, w13q, w13s, w2q, w2s, wl.topk)
    x = torch.from_numpy(oracle.bf16_to_f64(hid)).float()
    ref = np.zeros((wl.T, wl.H))
    for t in range(wl.T):
        top = torch.topk(torch.from_numpy(logits[t]).double(), wl.topk)
        wts = torch.softmax(top.values, 0)
        for j in range(wl.topk):
            e = int(top.indices[j])
            y = _dense_chain_torch(mi.bf16_bits(x[t:t + 1].to(torch.bfloat16)), w13q[e:e + 1], w13s[e:e + 1],
                                   w2q[e:e + 1], w2s[e:e + 1])
            ref[t] += float(np.float32(wts[j])) * y[0]      # router weights are stored as fp32
    rel = np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref)
    assert rel < 1e-9, rel
    # final bf16 rounding of the fp64 sum
    assert np.array_equal(r["out_bf16"], oracle.bf16_from_f64(r["out"]))


def test_sampled_tokens_match_full_run():
    rng = np.random.default_rng(17)
    T, H, I, E, k = 10, 128, 128, 4, 2
    hid = bf16_bits(rng.standard_normal((T, H)))
    w13q, w13s = oracle.quant_128x128_bf16(bf16_bits(rng.standard_normal((E, 2 * I, H)) * 0.02))
    w2q, w2s = oracle.quant_128x128_bf16(bf16_bits(rng.standard_normal((E, H, I)) * 0.02))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    full = oracle.moe_forward(hid, logits, w13q, w13s, w2q, w2s, k)
    part = oracle.moe_forward(hid, logits, w13q, w13s, w2q, w2s, k, tokens=[2, 7])
    assert np.array_equal(part["out"][[2, 7]], full["out"][[2, 7]])
    assert np.all(np.isnan(part["out"][[0, 1, 3]]))


def test_masked_layout_equals_dense_chain_per_expert():
    """The masked batched layout ([E, M, H] rows already grouped by expert, counts[e] valid rows):
    every valid row of expert e equals the dense block-FP8 chain through expert e's weights
    (torch float64), rows past the count stay empty, and an empty expert computes nothing."""
    rng = np.random.default_rng(23)
    E, M, H, I = 3, 40, 256, 256
    counts = [0, 40, 17]
    hid = bf16_bits(rng.standard_normal((E, M, H)))
    w13q, w13s = oracle.quant_128x128_bf16(bf16_bits(rng.standard_normal((E, 2 * I, H)) * 0.02))
    w2q, w2s = oracle.quant_128x128_bf16(bf16_bits(rng.standard_normal((E, H, I)) * 0.02))
    out, out_bf16 = oracle.moe_forward_masked(hid, counts, w13q, w13s, w2q, w2s)
    for e, c in enumerate(counts):
        assert np.all(np.isnan(out[e, c:]))
        if c:
            ref = _dense_chain_torch(hid[e, :c], w13q[e:e + 1], w13s[e:e + 1], w2q[e:e + 1], w2s[e:e + 1])
            assert np.allclose(out[e, :c], ref, rtol=1e-12, atol=1e-14)
            assert np.array_equal(out_bf16[e, :c], oracle.bf16_from_f64(out[e, :c]))
    empty, _ = oracle.moe_forward_masked(hid, [0, 0, 0], w13q, w13s, w2q, w2s)
    assert np.all(np.isnan(empty))



def test_ue8m0_single_expert_reduces_to_dense_chain():
    """The FLOAT32_CEIL_UE8M0 mode end to end: weights, activations and the requantised
    intermediate all on power-of-two scales; E=1, top-1 equals the torch chain."""
    rng = np.random.default_rng(9)
    T, H, I = 7, 256, 256
    hid = bf16_bits(rng.standard_normal((T, H)) * 3.0)
    w13q, w13s = oracle.quant_128x128_bf16(bf16_bits(rng.standard_normal((1, 2 * I, H)) * 0.02), oracle.SCALE_UE8M0)
    w2q, w2s = oracle.quant_128x128_bf16(bf16_bits(rng.standard_normal((1, H, I)) * 0.02), oracle.SCALE_UE8M0)
    assert np.all(np.frexp(w13s)[0] == 0.5) and np.all(np.frexp(w2s)[0] == 0.5)
    r = oracle.moe_forward(hid, np.zeros((T, 1), np.float32), w13q, w13s, w2q, w2s, 1, scale_fmt=oracle.SCALE_UE8M0)
    assert np.all(np.frexp(r["a1s"])[0] == 0.5) and np.all(np.frexp(r["a2s"][:T])[0] == 0.5)
    ref = _dense_chain_torch(hid, w13q, w13s, w2q, w2s, ue8m0=True)
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-14)
    # and it differs from the fp32-scale layer on the same weights
    r32 = oracle.moe_forward(hid, np.zeros((T, 1), np.float32), w13q, w13s, w2q, w2s, 1)
    assert not np.array_equal(r["out"], r32["out"])
