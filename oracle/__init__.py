"""CPU oracle for the block-FP8 fused MoE expert layer (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path (``block_fp8_mixture_topk_gb300``)
never imports it, and it imports nothing from there: the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 sums, OpenMP over
independent rows); this module only compiles it with gcc on first use and
marshals numpy arrays.  Every function cites the passage it follows in the C
source.  bf16 tensors are passed as ``uint16`` arrays holding the bf16 bits.

Parity status: every function is pinned by ``tests/test_oracle_*.py`` except the
bytes of the requantised intermediate (SiLU(gate)*up): those depend on fp32
rounding order and are compared only within +-1 e4m3 code.  The NVFP4 block
step (block scale = e4m3(max|x| / 6), code = e2m1(x / scale)) is a reading of
the pages, which name scaled_fp4_quant without its arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_moe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=gnu11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            L = ctypes.c_long
            I = ctypes.c_int
            lib.orc_e4m3_value.argtypes = [I]
            lib.orc_e4m3_value.restype = ctypes.c_double
            lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_bf16_from_f64.argtypes = [ctypes.c_double]
            lib.orc_bf16_from_f64.restype = ctypes.c_uint16
            lib.orc_quant_1x128_f32.argtypes = [P, L, L, P, P, I]
            lib.orc_quant_1x128_bf16.argtypes = [P, L, L, P, P, I]
            lib.orc_quant_1xg_f32.argtypes = [P, L, L, I, P, P, I]
            lib.orc_quant_1xg_bf16.argtypes = [P, L, L, I, P, P, I]
            lib.orc_experts_mxfp8.argtypes = [P, P, P, P, P, P, P, P, P, L, L, L, I, I, P, P, P, P]
            lib.orc_quant_128x128_bf16.argtypes = [P, L, L, L, P, P, I]
            lib.orc_route.argtypes = [P, P, L, I, I, I, I, I, I, ctypes.c_double, P, P]
            lib.orc_route.restype = I
            lib.orc_permute.argtypes = [P, L, I, P, P, P]
            lib.orc_experts.argtypes = [P, P, P, P, P, P, P, P, P, L, L, L, I, I, P, P, P, P, I]
            lib.orc_experts_nvfp4.argtypes = [P, P, P, P, P, P, P, P, P, P, P, L, L, L, I, I, P, P, P, P, I]
            lib.orc_e2m1_value.argtypes = [I]
            lib.orc_e2m1_value.restype = ctypes.c_double
            lib.orc_e2m1_encode.argtypes = [ctypes.c_float]
            lib.orc_e2m1_encode.restype = ctypes.c_uint8
            lib.orc_quant_nvfp4_bf16.argtypes = [P, L, L, L, P, P, P]
            lib.orc_combine.argtypes = [P, P, P, P, L, L, I, P]
            lib.orc_num_threads.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return _load().orc_num_threads()


# --------------------------------------------------------------------------- e4m3 / bf16

def e4m3_values() -> np.ndarray:
    """Value of each of the 256 e4m3fn codes (NaN for 0x7F / 0xFF)."""
    lib = _load()
    return np.array([lib.orc_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3fn code of each fp32 value (ties to even, saturating)."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.orc_e4m3_encode(float(flat_in[i]))
    return out


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """fp64 value of e4m3 codes."""
    return e4m3_values()[np.asarray(codes, dtype=np.uint8)]


def bf16_from_f64(x) -> np.ndarray:
    """Nearest-even bf16 bits (uint16) of fp64 values."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    fi, fo = x.reshape(-1), out.reshape(-1)
    for i in range(fi.size):
        fo[i] = lib.orc_bf16_from_f64(float(fi[i]))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bits."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- quantisers

# scale formats: fp32 amax/448, or that scale rounded up to a power of two (FLOAT32_CEIL_UE8M0)
SCALE_F32, SCALE_UE8M0 = 0, 1


def quant_1x128_bf16(x_bits: np.ndarray, scale_fmt: int = SCALE_F32):
    """1x128 group quantisation of bf16 rows: returns (codes [R,C] u8, scales [R,C/128] f32)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    assert C % 128 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((R, C // 128), dtype=np.float32)
    _load().orc_quant_1x128_bf16(_ptr(x), R, C, _ptr(q), _ptr(s), scale_fmt)
    return q, s


def quant_1x128_f32(x: np.ndarray, scale_fmt: int = SCALE_F32):
    """1x128 group quantisation of fp32 rows: returns (codes, scales)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    assert C % 128 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((R, C // 128), dtype=np.float32)
    _load().orc_quant_1x128_f32(_ptr(x), R, C, _ptr(q), _ptr(s), scale_fmt)
    return q, s


def quant_1x32_bf16(x_bits: np.ndarray):
    """MXFP8 activation quantisation ("MXFP8 (block [1, 32])", page "vllm.model_executor.layers.
    fused_moe.oracle.fp8", make_fp8_moe_quant_config): groups of 32 along each bf16 row, scale
    max(amax, 1e-8)/448 rounded up to a power of two (UE8M0).  Returns (codes [R, C] u8,
    scales [R, C/32] f32, each a power of two)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((R, C // 32), dtype=np.float32)
    _load().orc_quant_1xg_bf16(_ptr(x), R, C, 32, _ptr(q), _ptr(s), SCALE_UE8M0)
    return q, s


def quant_1x32_f32(x: np.ndarray):
    """The same 1x32 UE8M0 quantisation of fp32 rows."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((R, C // 32), dtype=np.float32)
    _load().orc_quant_1xg_f32(_ptr(x), R, C, 32, _ptr(q), _ptr(s), SCALE_UE8M0)
    return q, s


def quant_mxfp8_weight_bf16(w_bits: np.ndarray):
    """MXFP8 expert weights [E, N, K] (bf16 bits): 1x32 blocks along K with UE8M0 scales ("e8m0
    group-32 scales", _humming_fp8_weight_schema).  Returns (codes [E, N, K], scales [E, N, K/32]
    f32 powers of two)."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    E, N, K = w.shape
    q, s = quant_1x32_bf16(w.reshape(E * N, K))
    return q.reshape(E, N, K), s.reshape(E, N, K // 32)


def e2m1_values() -> np.ndarray:
    """fp64 value of each of the 16 e2m1 (fp4) codes."""
    lib = _load()
    return np.array([lib.orc_e2m1_value(c) for c in range(16)], dtype=np.float64)


def e2m1_encode(x) -> np.ndarray:
    """fp32 values -> e2m1 codes (nearest, ties to even, saturating at +-6), one per uint8."""
    x = np.asarray(x, dtype=np.float32)
    lib = _load()
    return np.array([lib.orc_e2m1_encode(float(v)) for v in x.reshape(-1)], dtype=np.uint8).reshape(x.shape)


def quant_nvfp4_bf16(w_bits: np.ndarray):
    """NVFP4 quantisation of stacked expert weights (page "vllm.model_executor.layers.quantization.
    online.nvfp4", _quantize_moe_weight_to_nvfp4): bf16 bits [E, N, K] (K % 16 == 0) ->
    (codes [E, N, K/2] u8, element 2i in the low nibble; block scales [E, N, K/16] u8 (e4m3 bits);
    global scales [E] f32 = 1 / ((6 * 448) / amax))."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    E, N, K = w_bits.shape
    assert K % 16 == 0
    q = np.zeros((E, N, K // 2), dtype=np.uint8)
    sf = np.zeros((E, N, K // 16), dtype=np.uint8)
    gs = np.zeros(E, dtype=np.float32)
    _load().orc_quant_nvfp4_bf16(_ptr(w_bits), E, N, K, _ptr(q), _ptr(sf), _ptr(gs))
    return q, sf, gs


def quant_128x128_bf16(w_bits: np.ndarray, scale_fmt: int = SCALE_F32):
    """128x128 block quantisation of stacked bf16 weights [E,N,K]: (codes [E,N,K], scales [E,N/128,K/128])."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    E, N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    q = np.empty((E, N, K), dtype=np.uint8)
    s = np.empty((E, N // 128, K // 128), dtype=np.float32)
    _load().orc_quant_128x128_bf16(_ptr(w), E, N, K, _ptr(q), _ptr(s), scale_fmt)
    return q, s


# --------------------------------------------------------------------------- routing / permute

SOFTMAX, SIGMOID = 0, 1


def route(logits: np.ndarray, topk: int, renormalize: bool = True, scoring: int = SOFTMAX,
          bias: np.ndarray | None = None, n_group: int = 1, topk_group: int = 1,
          routed_scaling: float = 1.0):
    """Top-k routing: returns (ids [T,k] int32, weights [T,k] f32)."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = l.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ids = np.empty((T, topk), dtype=np.int32)
    w = np.empty((T, topk), dtype=np.float32)
    rc = _load().orc_route(_ptr(l), _ptr(b), T, E, topk, int(bool(renormalize)), scoring,
                           n_group, topk_group, float(routed_scaling), _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError(f"oracle route rejected the arguments (rc={rc})")
    return ids, w


def permute(ids: np.ndarray, E: int):
    """Stable sort of pairs by expert: returns (offsets [E+1], sorted [P], pos [P])."""
    flat = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    P = flat.size
    offsets = np.empty(E + 1, dtype=np.int32)
    sorted_ = np.empty(P, dtype=np.int32)
    pos = np.empty(P, dtype=np.int32)
    _load().orc_permute(_ptr(flat), P, E, _ptr(offsets), _ptr(sorted_), _ptr(pos))
    return offsets, sorted_, pos


# --------------------------------------------------------------------------- full layer

def moe_forward(hidden_bits, logits, w13, w13_scale, w2, w2_scale, topk, renormalize=True,
                scoring=SOFTMAX, bias=None, n_group=1, topk_group=1, routed_scaling=1.0,
                tokens=None, want_c1=False, scale_fmt=SCALE_F32):
    """The whole layer on the CPU.

    hidden_bits [T,H] uint16 (bf16 bits), logits [T,E] f32, w13 [E,2I,H] u8,
    w13_scale [E,2I/128,H/128] f32, w2 [E,H,I] u8, w2_scale [E,H/128,I/128] f32.
    ``tokens``: optional iterable of token indices to compute (others stay NaN).
    Returns a dict with ids, weights, offsets, sorted, pos, a1q, a1s, a2q, a2s
    (by sorted row), c2 (by sorted row), out (fp64 [T,H]) and out_bf16 bits.  With
    ``tokens`` given, a2q, a2s, c1 and c2 hold only the rows of those tokens' pairs, and
    ``rows`` gives the sorted-row index of each (without, ``rows`` = all P rows).
    """
    E, N1, H2 = w13.shape
    assert N1 % 256 == 0
    I = N1 // 2
    assert w2.shape == (E, H2, I)
    w13c = np.ascontiguousarray(w13, dtype=np.uint8)
    w2c = np.ascontiguousarray(w2, dtype=np.uint8)
    w13s = np.ascontiguousarray(w13_scale, dtype=np.float32)
    w2s = np.ascontiguousarray(w2_scale, dtype=np.float32)

    def experts(a1q, a1s, offsets, sorted_, need, T, H, topk_, a2q, a2s, c1, c2):
        _load().orc_experts(_ptr(a1q), _ptr(a1s), _ptr(w13c), _ptr(w13s), _ptr(w2c), _ptr(w2s),
                            _ptr(offsets), _ptr(sorted_), _ptr(need), T, H, I, E, topk_,
                            _ptr(a2q), _ptr(a2s), _ptr(c1), _ptr(c2), scale_fmt)

    return _routed_layer(experts, hidden_bits, logits, E, I, topk, renormalize, scoring, bias, n_group,
                         topk_group, routed_scaling, tokens, want_c1, scale_fmt)


def moe_forward_nvfp4(hidden_bits, logits, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, topk, renormalize=True,
                      scoring=SOFTMAX, bias=None, n_group=1, topk_group=1, routed_scaling=1.0,
                      tokens=None, want_c1=False, scale_fmt=SCALE_F32):
    """The whole layer with NVFP4 expert weights (page "vllm.model_executor.layers.quantization.
    online.nvfp4", _quantize_moe_weight_to_nvfp4): the same routing, activation quantisation,
    SiLU(gate)*up requantisation and combine as ``moe_forward``; the weight values are
    code * block scale * global scale.

    w13 [E,2I,H/2] u8 (two fp4 codes per byte), w13_sf [E,2I,H/16] u8 (e4m3 bits), w13_gs [E] f32;
    w2 [E,H,I/2], w2_sf [E,H,I/16], w2_gs [E].  Returns the same dict as ``moe_forward``.
    """
    E, N1, H2h = w13.shape
    assert N1 % 256 == 0
    I = N1 // 2
    H = 2 * H2h
    assert w13_sf.shape == (E, N1, H // 16) and w2.shape == (E, H, I // 2) and w2_sf.shape == (E, H, I // 16)
    c = [np.ascontiguousarray(a, dtype=np.uint8) for a in (w13, w13_sf, w2, w2_sf)]
    g = [np.ascontiguousarray(a, dtype=np.float32).reshape(E) for a in (w13_gs, w2_gs)]

    def experts(a1q, a1s, offsets, sorted_, need, T, H_, topk_, a2q, a2s, c1, c2):
        _load().orc_experts_nvfp4(_ptr(a1q), _ptr(a1s), _ptr(c[0]), _ptr(c[1]), _ptr(g[0]), _ptr(c[2]),
                                  _ptr(c[3]), _ptr(g[1]), _ptr(offsets), _ptr(sorted_), _ptr(need), T, H_, I,
                                  E, topk_, _ptr(a2q), _ptr(a2s), _ptr(c1), _ptr(c2), scale_fmt)

    return _routed_layer(experts, hidden_bits, logits, E, I, topk, renormalize, scoring, bias, n_group,
                         topk_group, routed_scaling, tokens, want_c1, scale_fmt)


def moe_forward_mxfp8(hidden_bits, logits, w13, w13_scale, w2, w2_scale, topk, renormalize=True,
                      scoring=SOFTMAX, bias=None, n_group=1, topk_group=1, routed_scaling=1.0,
                      tokens=None, want_c1=False):
    """The whole layer in MXFP8 ("MXFP8 (block [1, 32])", page "vllm.model_executor.layers.
    fused_moe.oracle.fp8", make_fp8_moe_quant_config): activations and the requantised
    intermediate in 1x32 groups with UE8M0 scales, weights w13 [E,2I,H] / w2 [E,H,I] e4m3 with
    w13_scale [E,2I,H/32] / w2_scale [E,H,I/32] (fp32 powers of two).  Same routing, sort, SiLU
    and combine as ``moe_forward``; a1s / a2s in the result are [.., H/32] / [.., I/32]."""
    E, N1, H2 = w13.shape
    assert N1 % 256 == 0
    I = N1 // 2
    assert w2.shape == (E, H2, I) and w13_scale.shape == (E, N1, H2 // 32) and w2_scale.shape == (E, H2, I // 32)
    w13c = np.ascontiguousarray(w13, dtype=np.uint8)
    w2c = np.ascontiguousarray(w2, dtype=np.uint8)
    w13s = np.ascontiguousarray(w13_scale, dtype=np.float32)
    w2s = np.ascontiguousarray(w2_scale, dtype=np.float32)

    def experts(a1q, a1s, offsets, sorted_, need, T, H, topk_, a2q, a2s, c1, c2):
        _load().orc_experts_mxfp8(_ptr(a1q), _ptr(a1s), _ptr(w13c), _ptr(w13s), _ptr(w2c), _ptr(w2s),
                                  _ptr(offsets), _ptr(sorted_), _ptr(need), T, H, I, E, topk_,
                                  _ptr(a2q), _ptr(a2s), _ptr(c1), _ptr(c2))

    return _routed_layer(experts, hidden_bits, logits, E, I, topk, renormalize, scoring, bias, n_group,
                         topk_group, routed_scaling, tokens, want_c1, SCALE_UE8M0, group=32)


def _routed_layer(experts, hidden_bits, logits, E, I, topk, renormalize, scoring, bias, n_group, topk_group,
                  routed_scaling, tokens, want_c1, scale_fmt, group=128):
    hidden_bits = np.ascontiguousarray(hidden_bits, dtype=np.uint16)
    T, H = hidden_bits.shape
    N1 = 2 * I
    ids, wts = route(logits, topk, renormalize, scoring, bias, n_group, topk_group, routed_scaling)
    offsets, sorted_, pos = permute(ids, E)
    a1q, a1s = quant_1x32_bf16(hidden_bits) if group == 32 else quant_1x128_bf16(hidden_bits, scale_fmt)
    P = T * topk
    need = np.zeros(T, dtype=np.uint8)
    if tokens is None:
        need[:] = 1
        rows = np.arange(P, dtype=np.int64)
        r_offsets, r_sorted, r_pos = offsets, sorted_, pos
    else:
        need[np.asarray(list(tokens), dtype=np.int64)] = 1
        # only the sorted rows of the chosen tokens' pairs are held (in sorted order): every row is
        # computed on its own, so leaving the others out changes no value, and a sample of a large
        # step needs no [P, H] buffer
        rows = np.nonzero(need[sorted_ // topk])[0]
        expert_of_row = np.repeat(np.arange(E), np.diff(offsets))
        r_offsets = np.zeros(E + 1, dtype=np.int32)
        r_offsets[1:] = np.cumsum(np.bincount(expert_of_row[rows], minlength=E))
        r_sorted = np.ascontiguousarray(sorted_[rows], dtype=np.int32)
        r_pos = np.zeros(P, dtype=np.int32)
        r_pos[r_sorted] = np.arange(rows.size, dtype=np.int32)
    R = max(int(rows.size), 1)
    a2q = np.zeros((R, I), dtype=np.uint8)
    a2s = np.zeros((R, I // group), dtype=np.float32)
    c1 = np.full((R, N1), np.nan) if want_c1 else None
    c2 = np.full((R, H), np.nan)
    experts(a1q, a1s, r_offsets, r_sorted, need, T, H, topk, a2q, a2s, c1, c2)
    out = np.full((T, H), np.nan)
    _load().orc_combine(_ptr(c2), _ptr(wts), _ptr(r_pos), _ptr(need), T, H, topk, _ptr(out))
    out_bf16 = np.zeros((T, H), dtype=np.uint16)
    toks = np.nonzero(need)[0]
    if toks.size:
        out_bf16[toks] = bf16_from_f64(out[toks])
    # a2q, a2s, c1, c2 are indexed like `rows` (sorted-row indices; all P rows when tokens is None)
    return dict(ids=ids, weights=wts, offsets=offsets, sorted=sorted_, pos=pos, a1q=a1q, a1s=a1s,
                a2q=a2q, a2s=a2s, c1=c1, c2=c2, rows=rows, out=out, out_bf16=out_bf16, need=need)


# --------------------------------------------------------------------------- masked batched layout

def moe_forward_masked(hidden_bits, counts, w13, w13_scale, w2, w2_scale, scale_fmt=SCALE_F32):
    """The expert MLP on rows already grouped by expert ("[num_experts, max_tokens, hidden]"
    with per-expert counts, the batched layout the low-latency expert-parallel path hands to
    the experts, page "Quantization and MoE Optimizations", BatchedDeepGemmExperts): for
    every expert e and row i < counts[e], the same 1x128 quantisation, GEMM over w13,
    SiLU(gate)*up with requantisation and GEMM over w2 as the routed layer computes for a
    pair of that expert, with no router weight (the combine belongs to the dispatcher).

    hidden_bits [E, M, H] uint16 (bf16 bits), counts [E] ints in [0, M].
    Returns (out fp64 [E, M, H] with NaN in rows i >= counts[e], out_bf16 bits [E, M, H]).
    """
    hidden_bits = np.ascontiguousarray(hidden_bits, dtype=np.uint16)
    E, M, H = hidden_bits.shape
    counts = np.asarray(counts, dtype=np.int64)
    assert counts.shape == (E,) and np.all((counts >= 0) & (counts <= M))
    N1 = w13.shape[1]
    I = N1 // 2
    a1q, a1s = quant_1x128_bf16(hidden_bits.reshape(E * M, H), scale_fmt)
    # one pair per valid row (topk = 1): expert e's rows in order
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    sorted_ = np.concatenate([e * M + np.arange(counts[e]) for e in range(E)]).astype(np.int32) \
        if offsets[-1] else np.zeros(0, dtype=np.int32)
    P = int(offsets[-1])
    need = np.ones(E * M, dtype=np.uint8)
    a2q = np.zeros((max(P, 1), I), dtype=np.uint8)
    a2s = np.zeros((max(P, 1), I // 128), dtype=np.float32)
    c2 = np.full((max(P, 1), H), np.nan)
    w13c, w2c = np.ascontiguousarray(w13, dtype=np.uint8), np.ascontiguousarray(w2, dtype=np.uint8)
    w13s = np.ascontiguousarray(w13_scale, dtype=np.float32)
    w2s = np.ascontiguousarray(w2_scale, dtype=np.float32)
    _load().orc_experts(_ptr(a1q), _ptr(a1s), _ptr(w13c), _ptr(w13s), _ptr(w2c), _ptr(w2s),
                        _ptr(offsets), _ptr(sorted_), _ptr(need), E * M, H, I, E, 1,
                        _ptr(a2q), _ptr(a2s), None, _ptr(c2), scale_fmt)
    out = np.full((E * M, H), np.nan)
    out_bf16 = np.zeros((E * M, H), dtype=np.uint16)
    if P:
        out[sorted_] = c2[:P]
        out_bf16[sorted_] = bf16_from_f64(c2[:P])
    return out.reshape(E, M, H), out_bf16.reshape(E, M, H)
