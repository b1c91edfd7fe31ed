"""Pins for the oracle's e4m3 codec and its 1x128 / 128x128 quantisers.

The oracle is checked against things other than itself: the e4m3fn format
facts in tests/golden/, torch's float8_e4m3fn dtype (an independent
implementation of the same format), closed forms (groups whose scale is an exact
power of two quantise to known codes) and the rounding error bound of the format.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3fn_codes.txt")


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_table_matches_golden_facts():
    vals = oracle.e4m3_values()
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code_s, val_s = line.split()
        code, want = int(code_s, 16), float(val_s)
        got = vals[code]
        if np.isnan(want):
            assert np.isnan(got), hex(code)
        else:
            assert got == want and np.signbit(got) == np.signbit(want), (hex(code), got, want)
        n += 1
    assert n >= 20


def test_e4m3_table_matches_torch_for_all_256_codes():
    ours, ref = oracle.e4m3_values(), torch_decode_all()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_encode_round_trips_every_finite_code():
    vals = oracle.e4m3_values()
    finite = [c for c in range(256) if not np.isnan(vals[c])]
    enc = oracle.e4m3_encode(vals[finite].astype(np.float32))
    assert enc.tolist() == finite


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(7)
    # magnitudes spanning subnormals to the top binade, both signs
    mags = np.exp2(rng.uniform(-12.0, np.log2(448.0), size=6000))
    x = (mags * rng.choice([-1.0, 1.0], size=mags.size)).astype(np.float32)
    vals = oracle.e4m3_values()
    pos = np.sort(vals[:127])
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)      # exact ties -> even code
    x = np.concatenate([x, mids, -mids, np.float32([0.0, -0.0, 448.0, -448.0])])
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encode_ties_go_to_even_code_and_saturate():
    vals = oracle.e4m3_values()
    for c in range(0, 126):
        mid = np.float32((vals[c] + vals[c + 1]) / 2)
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode([mid])[0] == want
    big = np.float32([448.0, 449.0, 464.0, 500.0, 1e30, -464.0, -1e30])
    assert oracle.e4m3_encode(big).tolist() == [0x7E] * 5 + [0xFE] * 2


def _bf16_bits(x64):
    return oracle.bf16_from_f64(np.asarray(x64, dtype=np.float64))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(4000) * np.exp2(rng.integers(-30, 30, size=4000))
    x32 = x.astype(np.float32)       # torch casts from fp32; use values exact in fp32
    ours = _bf16_bits(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(oracle.bf16_to_f64(ours), torch.from_numpy(x32).to(torch.bfloat16).double().numpy())


def test_group_quant_closed_form_power_of_two_scale():
    """A group holding e4m3 values times 2^a, with one element at +-448*2^a, has scale exactly 2^a
    and quantises to exactly those codes."""
    rng = np.random.default_rng(11)
    vals = oracle.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(vals[c])])
    R, C = 6, 512
    codes = rng.choice(finite, size=(R, C)).astype(np.uint8)
    exps = rng.integers(-20, 10, size=(R, C // 128))
    for r in range(R):
        for g in range(C // 128):
            codes[r, g * 128 + rng.integers(0, 128)] = rng.choice([0x7E, 0xFE])
    x = vals[codes] * np.exp2(np.repeat(exps, 128, axis=1))
    q, s = oracle.quant_1x128_bf16(_bf16_bits(x))
    # -0.0 and +0.0 both encode by sign; compare values and sign
    assert np.array_equal(s, np.exp2(exps).astype(np.float32))
    assert np.array_equal(q, codes)


def test_group_quant_zero_group_and_floor():
    x = np.zeros((2, 256))
    x[1, 128:] = 1e-12                        # amax below the 1e-8 floor
    q, s = oracle.quant_1x128_bf16(_bf16_bits(x))
    floor = np.float32(1e-8) / np.float32(448.0)
    assert np.all(s[0] == floor) and s[1, 0] == floor and s[1, 1] == floor
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0)
    # 1e-12 / (1e-8/448) ~ 4.49e-2 lies in the binade [2^-5, 2^-4), where e4m3 steps by 2^-8
    v = oracle.e4m3_values()[q[1, 128]]
    assert abs(v - np.float32(oracle.bf16_to_f64(_bf16_bits([1e-12]))[0]) / floor) <= 2 ** -9


def test_group_quant_error_bound_and_max_maps_to_448():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((32, 1024)) * np.exp2(rng.integers(-8, 8, size=(32, 1)))
    bits = _bf16_bits(x)
    xb = oracle.bf16_to_f64(bits)
    q, s = oracle.quant_1x128_bf16(bits)
    vals = oracle.e4m3_values()
    deq = vals[q]
    scaled = xb / np.repeat(s.astype(np.float64), 128, axis=1)
    # half a unit in the last place of e4m3 at that magnitude (subnormal spacing 2^-9)
    ex = np.floor(np.log2(np.maximum(np.abs(scaled), 2.0 ** -6)))
    half_ulp = np.exp2(ex - 3) / 2
    assert np.all(np.abs(deq - scaled) <= half_ulp * (1 + 1e-6))
    # the group maximum lands on the top code
    g = xb.reshape(32, 8, 128)
    arg = np.abs(g).argmax(axis=2)
    top = np.take_along_axis(q.reshape(32, 8, 128), arg[..., None], axis=2)[..., 0]
    assert np.all((top == 0x7E) | (top == 0xFE))


def test_group_quant_matches_torch_formulation():
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal((64, 768)).astype(np.float32)).to(torch.bfloat16)
    q, s = oracle.quant_1x128_bf16(x.view(torch.int16).numpy().view(np.uint16))
    xf = x.float().view(64, 6, 128)
    amax = xf.abs().amax(dim=2).clamp_min(1e-8)
    st = amax / 448.0
    qt = (xf / st[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(64, 768)
    assert np.array_equal(s, st.numpy())
    assert np.array_equal(q, qt.numpy())


def test_block_quant_structure():
    """Each 128x128 block gets its own scale; scaling one block by 2 doubles its scale only."""
    rng = np.random.default_rng(13)
    E, N, K = 2, 256, 384
    w = rng.standard_normal((E, N, K)) * 0.02
    q0, s0 = oracle.quant_128x128_bf16(_bf16_bits(w))
    assert s0.shape == (E, 2, 3)
    w2 = w.copy()
    w2[1, 128:256, 256:384] *= 2.0
    q1, s1 = oracle.quant_128x128_bf16(_bf16_bits(w2))
    mask = np.ones_like(s0, dtype=bool)
    mask[1, 1, 2] = False
    assert np.array_equal(s1[mask], s0[mask])
    assert s1[1, 1, 2] == 2 * s0[1, 1, 2]
    assert np.array_equal(q1, q0)
    # block scale = amax over exactly that block / 448 (rows index N, columns index K)
    xb = oracle.bf16_to_f64(_bf16_bits(w)).reshape(E, N, K)
    for e in range(E):
        for nb in range(2):
            for kb in range(3):
                blk = xb[e, nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
                assert s0[e, nb, kb] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))
    # codes agree with torch's cast of x / s
    st = torch.from_numpy(np.repeat(np.repeat(s0, 128, axis=1), 128, axis=2))
    qt = (torch.from_numpy(xb.astype(np.float32)) / st).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q0, qt)


@pytest.mark.parametrize("rows,cols", [(1, 128), (3, 384)])
def test_f32_and_bf16_quantisers_agree(rows, cols):
    rng = np.random.default_rng(rows)
    bits = _bf16_bits(rng.standard_normal((rows, cols)))
    q1, s1 = oracle.quant_1x128_bf16(bits)
    q2, s2 = oracle.quant_1x128_f32(oracle.bf16_to_f64(bits).astype(np.float32))
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_ue8m0_scales_round_the_fp32_scale_up_to_a_power_of_two():
    """FLOAT32_CEIL_UE8M0: each scale is the smallest power of two not below fp32(amax/448)
    (numpy's float32 division and float64 log2, not the oracle's frexp), exact powers stay, and
    the codes are torch's float8 cast of x / scale (exact, the scale being a power of two)."""
    rng = np.random.default_rng(31)
    rows, cols = 64, 512
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-30, 30, (rows, 1)))
    x[0, :128] = 0.0                                       # floor group
    x[1, :128] = 0.0
    x[1, 7] = 448.0 * 2.0 ** 5                             # t = 2^5 exactly: kept
    x[2, 128:256] = 0.0
    x[2, 130] = -(448.0 * 2.0 ** -3) * 1.5                 # t = 1.5 * 2^-3: rounded up to 2^-2
    bits = oracle.bf16_from_f64(x)
    q, s = oracle.quant_1x128_bf16(bits, oracle.SCALE_UE8M0)
    xb = oracle.bf16_to_f64(bits).astype(np.float32)
    amax = np.abs(xb.reshape(rows, -1, 128)).max(axis=2)
    t = np.maximum(amax, np.float32(1e-8)).astype(np.float32) / np.float32(448.0)
    want = np.exp2(np.ceil(np.log2(t.astype(np.float64)))).astype(np.float32)
    assert np.array_equal(s, want)
    assert s[1, 0] == 2.0 ** 5 and s[2, 1] == 2.0 ** -2
    assert np.all(np.frexp(s)[0] == 0.5)
    # codes: float8 cast of the exact quotient
    y = torch.from_numpy(xb.reshape(rows, -1, 128) / s[..., None])
    tq = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(rows, cols)
    assert np.array_equal(q, tq)
    # the fp32 mode on the same rows is unchanged
    q32, s32 = oracle.quant_1x128_bf16(bits)
    assert np.array_equal(s32, t)


def test_ue8m0_weight_blocks():
    rng = np.random.default_rng(32)
    w = oracle.bf16_from_f64(rng.standard_normal((2, 256, 384)) * 0.02)
    q, s = oracle.quant_128x128_bf16(w, oracle.SCALE_UE8M0)
    wf = oracle.bf16_to_f64(w).astype(np.float32)
    amax = np.abs(wf.reshape(2, 2, 128, 3, 128)).max(axis=(2, 4))
    t = np.maximum(amax, np.float32(1e-8)).astype(np.float32) / np.float32(448.0)
    assert np.array_equal(s, np.exp2(np.ceil(np.log2(t.astype(np.float64)))).astype(np.float32))
    y = wf / np.repeat(np.repeat(s, 128, axis=1), 128, axis=2)
    assert np.array_equal(q, torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
