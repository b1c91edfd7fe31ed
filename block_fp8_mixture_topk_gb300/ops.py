"""ctypes binding of libmoefp8 (argument marshalling only).

Function names and argument order follow the C ABI; tensors are torch CUDA
tensors (bf16 as torch.bfloat16, e4m3 codes as torch.uint8 or
torch.float8_e4m3fn), launched on torch's current stream.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading

import torch

from . import build as _build

MOE_BLOCK_M = 128
MOE_WEIGHTS_NK, MOE_WEIGHTS_TILED, MOE_WEIGHTS_NVFP4 = 0, 1, 2
NVFP4_UNIT_BYTES = 16 * 64 + 16 * 8   # one 16-row slab x one 128-wide K block: codes, then block scales
# fp32 amax/448; that scale rounded up to a power of two (FLOAT32_CEIL_UE8M0); the same UE8M0 scales in
# the packed scale-factor tiles of the block-scaled MMA (MOE_SCALE_UE8M0_PACKED)
# the same UE8M0 scales in the packed scale-factor tiles of the block-scaled MMA (MOE_SCALE_UE8M0_PACKED);
# MXFP8: 1x32 groups and blocks along K with UE8M0 scales, on the block-scaled MMA (MOE_SCALE_MXFP8)
SCALE_FMT = {"f32": 0, "ue8m0": 1, "ue8m0_packed": 2, "mxfp8": 3}
_PACKED_SCALES = ("ue8m0_packed", "mxfp8")
SCORING = {"softmax": 0, "sigmoid": 1}
EPILOGUE = {"store": 0, "silu_mul_quant": 1, "weighted_scatter": 2, "weighted_rows": 3, "weighted_pairs_bf16": 4}

_ERRORS = {-1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED_SHAPE", -3: "MOE_ERR_WORKSPACE_TOO_SMALL",
           -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE"}


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {_ERRORS.get(code, code)}")
        self.code = code


class _RoutingParams(ctypes.Structure):
    _fields_ = [("scoring", ctypes.c_int32), ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("routed_scaling", ctypes.c_float), ("bias", ctypes.c_void_p)]


class _Epilogue(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("topk", ctypes.c_int32), ("out_f32", ctypes.c_void_p),
                ("out_q", ctypes.c_void_p), ("out_scale", ctypes.c_void_p),
                ("out_scale_row_stride", ctypes.c_int64), ("out_scale_kb_stride", ctypes.c_int64),
                ("sorted_pair_ids", ctypes.c_void_p), ("topk_weights", ctypes.c_void_p),
                ("num_pairs", ctypes.c_int64), ("out_bf16", ctypes.c_void_p), ("b_layout", ctypes.c_int32),
                ("scale_fmt", ctypes.c_int32)]


class _ForwardOptions(ctypes.Structure):
    _fields_ = [("weight_layout", ctypes.c_int32), ("scale_fmt", ctypes.c_int32), ("decode_path", ctypes.c_int32)]


# MOE_DECODE_*: which kernels run the expert GEMMs of a small step
DECODE_PATH = {"auto": 0, "off": 1, "on": 2}


@dataclasses.dataclass
class RoutingParams:
    """Router options of the C ABI's moe_routing_params (bias: CUDA fp32 [E] or None)."""
    scoring: str = "softmax"
    n_group: int = 1
    topk_group: int = 1
    routed_scaling: float = 1.0
    bias: torch.Tensor | None = None

    def to_c(self) -> _RoutingParams:
        return _RoutingParams(SCORING[self.scoring], self.n_group, self.topk_group, float(self.routed_scaling),
                              _ptr(self.bias))


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded libmoefp8 (built on first use if absent; raises if that fails)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB_PATH):
                _build.build()
            L = ctypes.CDLL(_build.LIB_PATH)
            P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            sig = {
                "moe_route_topk": ([P, I, I, I, I, P, P, P, P], I),
                "moe_max_padded_rows": ([I, I, I, I], I64),
                "moe_max_tiles": ([I, I, I, I], I64),
                "moe_align_permute_workspace_size": ([I, I, I], SZ),
                "moe_align_permute": ([P, I, I, I, I, P, P, P, P, P, P, P, P, SZ, P], I),
                "moe_align_permute_noalloc": ([P, I, I, I, I, P, P, P, P, P, P, P, P], I),
                "fp8_group_quant": ([P, I, I, I, P, P, P], I),
                "fp8_group_quant_ex": ([P, I, I, I, P, P, I, P], I),
                "fp8_block_quant_weight_ex": ([P, I, I, I, P, P, I, P], I),
                "fp8_block_quant_weight": ([P, I, I, I, P, P, P], I),
                "fp8_block_grouped_gemm": ([P, P, I64, I64, I64, P, P, I, I, I, P, P, P, I64, P, P], I),
                "moe_fp8_block_workspace_size": ([I, I, I, I, I], SZ),
                "moe_fp8_block_forward_kernel_count": ([I, I, I, I, I], I),
                "moe_fp8_block_forward_kernel_count_ex": ([I, I, I, I, I, P, P], I),
                "moe_fp8_block_decode_path": ([I, I, I, I, I], I),
                "moe_fp8_block_pair_path": ([I, I, I, I, I], I),
                "moe_fp8_block_forward": ([P, P, P, P, P, P, I, I, I, I, I, I, P, P, SZ, P, P], I),
                "moe_fp8_block_forward_packed": ([P, P, P, P, P, P, I, I, I, I, I, I, P, P, SZ, P, P], I),
                "moe_fp8_block_forward_ex": ([P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, SZ, P, P, P], I),
                "moe_fp8_block_pack_weights": ([P, I, I, I, P, P], I),
                "moe_packed_scale_bytes": ([I64, I], SZ),
                "moe_fp8_block_pack_scales": ([P, I, I, I, P, P], I),
                "moe_mxfp8_packed_scale_bytes": ([I64, I], SZ),
                "moe_mxfp8_quant_weight": ([P, I, I, I, P, P, P], I),
                "moe_mxfp8_pack_scales": ([P, I64, I, P, P], I),
                "moe_nvfp4_quant_weight": ([P, I, I, I, P, P, P, P], I),
                "moe_nvfp4_packed_bytes": ([I, I, I], SZ),
                "moe_nvfp4_pack_weights": ([P, P, I, I, I, P, P], I),
                "moe_fp8_block_masked_workspace_size": ([I, I, I, I], SZ),
                "moe_fp8_block_forward_masked": ([P, P, P, P, P, P, I, I, I, I, P, P, SZ, P, P], I),
                "moe_unpermute_sum": ([P, I64, P, I, I, I, P, P], I),
                "moe_combine_pairs": ([P, P, I, I, I, P, P], I),
                "moe_get_device_status": ([P, I], I),
                "moe_selftest_bounded_wait": ([I, P], I),
                "moe_error_string": ([I], ctypes.c_char_p),
                "moe_device_supported": ([], I),
            }
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(name, rc):
    if rc != 0:
        raise MoeError(name, rc)


def _codes(t: torch.Tensor) -> torch.Tensor:
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"e4m3 codes must be uint8 or float8_e4m3fn, got {t.dtype}")
    return t


def _cuda(t, dtype=None, name="tensor"):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def moe_device_supported() -> bool:
    return bool(lib().moe_device_supported())


def moe_max_padded_rows(T, topk, E, block_m=MOE_BLOCK_M) -> int:
    return int(lib().moe_max_padded_rows(T, topk, E, block_m))


def moe_max_tiles(T, topk, E, block_m=MOE_BLOCK_M) -> int:
    return int(lib().moe_max_tiles(T, topk, E, block_m))


def moe_route_topk(logits, topk, renormalize=True, routing: RoutingParams | None = None):
    """Top-k routing: returns (ids int32 [T,k], weights fp32 [T,k])."""
    _cuda(logits, torch.float32, "logits")
    T, E = logits.shape
    ids = torch.empty(T, topk, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, topk, dtype=torch.float32, device=logits.device)
    rp = routing.to_c() if routing else None
    rc = lib().moe_route_topk(_ptr(logits), T, E, topk, int(bool(renormalize)),
                              ctypes.byref(rp) if rp else None, _ptr(ids), _ptr(w), _stream())
    _check("moe_route_topk", rc)
    return ids, w


def moe_align_permute(topk_ids, num_experts, block_m=MOE_BLOCK_M):
    """Sort pairs by expert; returns a dict of the C ABI's outputs."""
    _cuda(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    dev = topk_ids.device
    rows = moe_max_padded_rows(T, k, num_experts, block_m)
    tiles = moe_max_tiles(T, k, num_experts, block_m)
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(expert_offsets=torch.empty(num_experts + 1, **i32),
               padded_offsets=torch.empty(num_experts + 1, **i32),
               sorted_pair_ids=torch.full((max(rows, 1),), -1, **i32), pos=torch.empty(max(T * k, 1), **i32),
               tile_expert=torch.empty(max(tiles, 1), **i32), tile_row0=torch.empty(max(tiles, 1), **i32),
               num_tiles=torch.empty(1, **i32))
    wsb = int(lib().moe_align_permute_workspace_size(T, k, num_experts))
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    rc = lib().moe_align_permute(_ptr(topk_ids), T, k, num_experts, block_m, _ptr(out["expert_offsets"]),
                                 _ptr(out["padded_offsets"]), _ptr(out["sorted_pair_ids"]), _ptr(out["pos"]),
                                 _ptr(out["tile_expert"]), _ptr(out["tile_row0"]), _ptr(out["num_tiles"]),
                                 _ptr(ws), wsb, _stream())
    _check("moe_align_permute", rc)
    out["max_rows"], out["max_tiles"] = rows, tiles
    return out


def moe_packed_scale_bytes(rows, K) -> int:
    """Bytes of the packed UE8M0 scale tiles of a [rows, K] operand."""
    return int(lib().moe_packed_scale_bytes(rows, K))


def fp8_group_quant(x, scale_fmt="f32"):
    """1x128 group quantisation of bf16 [rows, cols]: returns (codes uint8, scales fp32 [rows, cols/128]).
    scale_fmt: "f32" (amax/448), "ue8m0" (rounded up to a power of two), "ue8m0_packed" (the same
    scales as packed UE8M0 tiles: a uint8 tensor of moe_packed_scale_bytes(rows, cols) bytes) or
    "mxfp8" (groups of 32: the UE8M0 scale bytes, uint8 [rows, cols/32])."""
    _cuda(x, torch.bfloat16, "x")
    rows, cols = x.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
    if scale_fmt == "ue8m0_packed":
        s = torch.zeros(max(moe_packed_scale_bytes(rows, cols), 16), dtype=torch.uint8, device=x.device)
    elif scale_fmt == "mxfp8":
        s = torch.empty(rows, max(cols // 32, 1), dtype=torch.uint8, device=x.device)
    else:
        s = torch.empty(rows, max(cols // 128, 1), dtype=torch.float32, device=x.device)
    rc = lib().fp8_group_quant_ex(_ptr(x), rows, cols, cols, _ptr(q), _ptr(s), SCALE_FMT[scale_fmt], _stream())
    _check("fp8_group_quant", rc)
    return q, s


def fp8_block_quant_weight(w, scale_fmt="f32"):
    """128x128 block quantisation of bf16 [E, N, K]: returns (codes uint8 [E,N,K], scales [E,N/128,K/128])."""
    _cuda(w, torch.bfloat16, "w")
    E, N, K = w.shape
    q = torch.empty(E, N, K, dtype=torch.uint8, device=w.device)
    s = torch.empty(E, max(N // 128, 1), max(K // 128, 1), dtype=torch.float32, device=w.device)
    rc = lib().fp8_block_quant_weight_ex(_ptr(w), E, N, K, _ptr(q), _ptr(s), SCALE_FMT[scale_fmt], _stream())
    _check("fp8_block_quant_weight", rc)
    return q, s


def moe_fp8_block_pack_scales(s):
    """UE8M0 (power-of-two) block scales fp32 [E, N/128, K/128] -> the packed scale tiles of the
    block-scaled GEMMs, uint8 [E, N/128, ceil(K/512), 512] (load-time, once)."""
    _cuda(s, torch.float32, "s")
    E, NB, KB = s.shape
    out = torch.empty(E, NB, (KB + 3) // 4, 512, dtype=torch.uint8, device=s.device)
    _check("moe_fp8_block_pack_scales", lib().moe_fp8_block_pack_scales(_ptr(s), E, NB * 128, KB * 128, _ptr(out),
                                                                          _stream()))
    return out


def moe_mxfp8_quant_weight(w):
    """MXFP8 quantisation of bf16 expert weights [E, N, K]: returns (codes uint8 [E, N, K], UE8M0
    scale bytes uint8 [E, N, K/32]) (load-time)."""
    _cuda(w, torch.bfloat16, "w")
    E, N, K = w.shape
    q = torch.empty(E, N, K, dtype=torch.uint8, device=w.device)
    s = torch.empty(E, N, max(K // 32, 1), dtype=torch.uint8, device=w.device)
    _check("moe_mxfp8_quant_weight", lib().moe_mxfp8_quant_weight(_ptr(w), E, N, K, _ptr(q), _ptr(s), _stream()))
    return q, s


def moe_mxfp8_packed_scale_bytes(rows, K) -> int:
    return int(lib().moe_mxfp8_packed_scale_bytes(rows, K))


def moe_mxfp8_pack_scales(s):
    """UE8M0 scale bytes [..., rows, K/32] (uint8; leading dimensions folded into rows, a multiple of
    128) -> the MXFP8 packed scale tiles, a uint8 tensor of moe_mxfp8_packed_scale_bytes bytes."""
    s = _cuda(s, torch.uint8, "s")
    K = s.shape[-1] * 32
    rows = s.numel() // s.shape[-1]
    out = torch.empty(max(moe_mxfp8_packed_scale_bytes(rows, K), 16), dtype=torch.uint8, device=s.device)
    _check("moe_mxfp8_pack_scales", lib().moe_mxfp8_pack_scales(_ptr(s), rows, K, _ptr(out), _stream()))
    return out


def moe_fp8_block_pack_weights(w):
    """e4m3 expert weights [E, N, K] -> the tile-packed layout, a uint8 tensor of shape
    [E, N/128, K/128, 128, 128] (each 128x128 block contiguous; load-time, once)."""
    w = _codes(_cuda(w, None, "w"))
    E, N, K = w.shape
    packed = torch.empty(E, N // 128, K // 128, 128, 128, dtype=torch.uint8, device=w.device)
    _check("moe_fp8_block_pack_weights", lib().moe_fp8_block_pack_weights(_ptr(w), E, N, K, _ptr(packed), _stream()))
    return packed


def moe_nvfp4_quant_weight(w):
    """NVFP4 quantisation of bf16 expert weights [E, N, K] (page "vllm.model_executor.layers.
    quantization.online.nvfp4", _quantize_moe_weight_to_nvfp4): returns (codes uint8 [E, N, K/2],
    two e2m1 per byte, element 2i in the low nibble; block scales uint8 [E, N, K/16], e4m3 bits;
    global scales fp32 [E], the factor that dequantises)."""
    _cuda(w, torch.bfloat16, "w")
    E, N, K = w.shape
    q = torch.empty(E, N, K // 2, dtype=torch.uint8, device=w.device)
    sf = torch.empty(E, N, K // 16, dtype=torch.uint8, device=w.device)
    gs = torch.empty(E, dtype=torch.float32, device=w.device)
    _check("moe_nvfp4_quant_weight",
           lib().moe_nvfp4_quant_weight(_ptr(w), E, N, K, _ptr(q), _ptr(sf), _ptr(gs), _stream()))
    return q, sf, gs


def moe_nvfp4_pack_weights(q, block_scale):
    """NVFP4 codes [E, N, K/2] and block scales [E, N, K/16] -> the packed layout the forward
    reads (MOE_WEIGHTS_NVFP4): uint8 [E, N/16, K/128, 1152] (load-time, once)."""
    q = _cuda(q, torch.uint8, "q")
    block_scale = _codes(_cuda(block_scale, None, "block_scale"))
    E, N, K2 = q.shape
    K = 2 * K2
    if block_scale.shape != (E, N, K // 16):
        raise ValueError("block_scale must be [E, N, K/16]")
    packed = torch.empty(E, N // 16, K // 128, NVFP4_UNIT_BYTES, dtype=torch.uint8, device=q.device)
    _check("moe_nvfp4_pack_weights",
           lib().moe_nvfp4_pack_weights(_ptr(q), _ptr(block_scale), E, N, K, _ptr(packed), _stream()))
    return packed


def moe_nvfp4_packed_bytes(E, N, K) -> int:
    return int(lib().moe_nvfp4_packed_bytes(E, N, K))


def _weight_shape(w):
    """(E, N, K, layout) of expert weights in any of the layouts."""
    if w.dim() == 5:
        return w.shape[0], w.shape[1] * 128, w.shape[2] * 128, MOE_WEIGHTS_TILED
    if w.dim() == 4 and w.shape[3] == NVFP4_UNIT_BYTES:
        return w.shape[0], w.shape[1] * 16, w.shape[2] * 128, MOE_WEIGHTS_NVFP4
    E, N, K = w.shape
    return E, N, K, MOE_WEIGHTS_NK


def fp8_block_grouped_gemm(A, a_scale, a_scale_strides, B, b_scale, tile_expert, tile_row0, num_tiles,
                           epilogue="store", out_f32=None, out_q=None, out_scale=None, out_scale_strides=(0, 0),
                           sorted_pair_ids=None, topk_weights=None, topk=1, num_pairs=0, out_bf16=None,
                           scale_fmt="f32"):
    """Grouped GEMM of the C ABI.  Outputs are caller-provided tensors (see include/moefp8.h)."""
    A, B = _codes(_cuda(A, None, "A")), _codes(_cuda(B, None, "B"))
    E, N, K, layout = _weight_shape(B)
    ep = _Epilogue(EPILOGUE[epilogue], topk, _ptr(out_f32), _ptr(out_q), _ptr(out_scale),
                   int(out_scale_strides[0]), int(out_scale_strides[1]), _ptr(sorted_pair_ids),
                   _ptr(topk_weights), int(num_pairs), _ptr(out_bf16), layout, SCALE_FMT[scale_fmt])
    rc = lib().fp8_block_grouped_gemm(_ptr(A), _ptr(a_scale), int(a_scale_strides[0]), int(a_scale_strides[1]),
                                      A.shape[0], _ptr(B), _ptr(b_scale), N, K, E, _ptr(tile_expert),
                                      _ptr(tile_row0), _ptr(num_tiles), tile_expert.numel(), ctypes.byref(ep),
                                      _stream())
    _check("fp8_block_grouped_gemm", rc)


def moe_unpermute_sum(y, pos, T, topk, out=None):
    """out[t] = bf16(sum_j y[pos[t*topk + j]]) for y fp32 [rows, H] and pos int32 [T*topk]."""
    _cuda(y, torch.float32, "y")
    _cuda(pos, torch.int32, "pos")
    H = y.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    rc = lib().moe_unpermute_sum(_ptr(y), y.shape[0], _ptr(pos), T, topk, H, _ptr(out), _stream())
    _check("moe_unpermute_sum", rc)
    return out


def moe_combine_pairs(y, pos, T, topk, out=None):
    """out[t] = bf16(sum_j y[t*topk + j]) over pairs with pos >= 0, for y bf16 [T*topk, H] in pair order."""
    _cuda(y, torch.bfloat16, "y")
    _cuda(pos, torch.int32, "pos")
    H = y.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    rc = lib().moe_combine_pairs(_ptr(y), _ptr(pos), T, topk, H, _ptr(out), _stream())
    _check("moe_combine_pairs", rc)
    return out


def moe_fp8_block_pair_path(T, H, E, topk, scale_fmt="f32") -> int:
    """Two-CTA clusters that the step's tile GEMMs launch on the CTA-pair kernel (0: the one-CTA
    kernels)."""
    r = int(lib().moe_fp8_block_pair_path(T, H, E, topk, SCALE_FMT[scale_fmt]))
    if r < 0:
        raise MoeError("moe_fp8_block_pair_path", r)
    return r


def moe_fp8_block_decode_path(T, H, I, topk, decode="auto") -> bool:
    """Whether a step of T tokens takes the decode-path GEMMs under `decode` (auto / off / on)."""
    r = int(lib().moe_fp8_block_decode_path(T, H, I, topk, DECODE_PATH[decode]))
    if r < 0:
        raise ValueError(f"moe_fp8_block_decode_path({T}, {H}, {I}, {topk}, {decode!r})")
    return bool(r)


def moe_fp8_block_forward_kernel_count(T, H, I, E, topk, routing: RoutingParams | None = None, layout=None,
                                       scale_fmt="f32", decode="auto") -> int:
    """Kernels one moe_fp8_block_forward with these routing parameters and options launches
    (layout: MOE_WEIGHTS_NK / _TILED / _NVFP4, default NK)."""
    if routing is None and layout is None and scale_fmt == "f32" and decode == "auto":
        return int(lib().moe_fp8_block_forward_kernel_count(T, H, I, E, topk))
    rp = routing.to_c() if routing else None
    opts = _ForwardOptions(MOE_WEIGHTS_NK if layout is None else layout, SCALE_FMT[scale_fmt], DECODE_PATH[decode])
    return int(lib().moe_fp8_block_forward_kernel_count_ex(T, H, I, E, topk, ctypes.byref(rp) if rp else None,
                                                           ctypes.byref(opts)))


def moe_fp8_block_workspace_size(T, H, I, E, topk) -> int:
    return int(lib().moe_fp8_block_workspace_size(T, H, I, E, topk))


_ws_cache: dict = {}


def _workspace(device, nbytes):
    key = (device.type, device.index)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


FORWARD_STAGES = ("route", "sort", "quant", "gemm_w13", "gemm_w2", "unpermute_sum")


def moe_fp8_block_forward(hidden, router_logits, w13, w13_scale, w2, w2_scale, topk, renormalize=True,
                          routing: RoutingParams | None = None, out=None, workspace=None, events=None,
                          scale_fmt="f32", decode="auto"):
    """The whole layer: returns bf16 [T, H] (written into `out` when given).

    w13 / w2 in the pages' layout [E, N, K] or tile-packed (moe_fp8_block_pack_weights, 5-D), or
    NVFP4-packed (moe_nvfp4_pack_weights, 4-D) with w13_scale / w2_scale the global scales [E].
    scale_fmt "ue8m0_packed": w13_scale / w2_scale are moe_fp8_block_pack_scales outputs and both
    GEMMs run on the block-scaled MMA.
    decode: "auto", "off" or "on" -- the decode-path GEMMs for small steps (MOE_DECODE_*).
    events: optional list of 7 torch.cuda.Event recorded between the stages
    (FORWARD_STAGES) on the current stream, for per-stage timing."""
    _cuda(hidden, torch.bfloat16, "hidden")
    _cuda(router_logits, torch.float32, "router_logits")
    w13, w2 = _codes(_cuda(w13, None, "w13")), _codes(_cuda(w2, None, "w2"))
    sdt = torch.uint8 if scale_fmt in _PACKED_SCALES else torch.float32
    _cuda(w13_scale, sdt, "w13_scale")
    _cuda(w2_scale, sdt, "w2_scale")
    T, H = hidden.shape
    E, N1, _, layout = _weight_shape(w13)
    if _weight_shape(w2)[3] != layout:
        raise ValueError("w13 and w2 must share one layout")
    I = N1 // 2
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=hidden.device)
    nbytes = moe_fp8_block_workspace_size(T, H, I, E, topk)
    if workspace is None:
        workspace = _workspace(hidden.device, nbytes)
    rp = routing.to_c() if routing else None
    opts = _ForwardOptions(layout, SCALE_FMT[scale_fmt], DECODE_PATH[decode])
    arr = None
    if events is not None:
        if len(events) != len(FORWARD_STAGES) + 1:
            raise ValueError("events: one more than the number of stages")
        for ev in events:
            if not ev.cuda_event:       # torch creates the CUDA event on its first record()
                ev.record()
        arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(ev.cuda_event) for ev in events])
    rc = lib().moe_fp8_block_forward_ex(_ptr(hidden), _ptr(router_logits), _ptr(w13), _ptr(w13_scale), _ptr(w2),
                                        _ptr(w2_scale), T, H, I, E, topk, int(bool(renormalize)),
                                        ctypes.byref(rp) if rp else None, ctypes.byref(opts), _ptr(workspace),
                                        workspace.numel(), _ptr(out), _stream(), arr)
    _check("moe_fp8_block_forward", rc)
    return out


def moe_nvfp4_forward(hidden, router_logits, w13, w13_global_scale, w2, w2_global_scale, topk, renormalize=True,
                      routing: RoutingParams | None = None, out=None, workspace=None, events=None, scale_fmt="f32"):
    """The layer on NVFP4 expert weights (moe_nvfp4_pack_weights outputs and their global scales
    [E]); activations and the intermediate in FP8 1x128 groups (scale_fmt)."""
    if _weight_shape(w13)[3] != MOE_WEIGHTS_NVFP4 or _weight_shape(w2)[3] != MOE_WEIGHTS_NVFP4:
        raise ValueError("w13 and w2 must be NVFP4-packed (moe_nvfp4_pack_weights)")
    return moe_fp8_block_forward(hidden, router_logits, w13, w13_global_scale, w2, w2_global_scale, topk,
                                 renormalize, routing, out, workspace, events, scale_fmt, "on")


def moe_fp8_block_masked_workspace_size(E, max_tokens, H, I) -> int:
    return int(lib().moe_fp8_block_masked_workspace_size(E, max_tokens, H, I))


def moe_fp8_block_forward_masked(hidden, counts, w13, w13_scale, w2, w2_scale, out=None, workspace=None,
                                 scale_fmt="f32"):
    """Expert MLP on the masked batched layout: hidden bf16 [E, M, H] with counts int32 [E]
    (CUDA) valid rows per expert; returns bf16 [E, M, H] (rows past the counts not written)."""
    _cuda(hidden, torch.bfloat16, "hidden")
    _cuda(counts, torch.int32, "counts")
    w13, w2 = _codes(_cuda(w13, None, "w13")), _codes(_cuda(w2, None, "w2"))
    sdt = torch.uint8 if scale_fmt in _PACKED_SCALES else torch.float32
    _cuda(w13_scale, sdt, "w13_scale")
    _cuda(w2_scale, sdt, "w2_scale")
    E, M, H = hidden.shape
    _, N1, _, layout = _weight_shape(w13)
    if _weight_shape(w2)[3] != layout:
        raise ValueError("w13 and w2 must share one layout")
    I = N1 // 2
    if out is None:
        out = torch.empty(E, M, H, dtype=torch.bfloat16, device=hidden.device)
    nbytes = moe_fp8_block_masked_workspace_size(E, M, H, I)
    if workspace is None:
        workspace = _workspace(hidden.device, nbytes)
    rc = lib().moe_fp8_block_forward_masked(_ptr(hidden), _ptr(counts), _ptr(w13), _ptr(w13_scale), _ptr(w2),
                                            _ptr(w2_scale), E, M, H, I, ctypes.byref(_ForwardOptions(layout,
                                            SCALE_FMT[scale_fmt], 0)), _ptr(workspace), workspace.numel(),
                                            _ptr(out), _stream())
    _check("moe_fp8_block_forward_masked", rc)
    return out


def moe_selftest_bounded_wait(expire=True):
    """Make one pipeline wait expire (about 2 s, MOE_STATUS_WAIT_TIMEOUT) or complete at once;
    read the outcome with moe_get_device_status."""
    _check("moe_selftest_bounded_wait", lib().moe_selftest_bounded_wait(int(bool(expire)), _stream()))


def moe_get_device_status(clear=False) -> int:
    """Device status bits (synchronises the device)."""
    st = ctypes.c_uint32(0)
    _check("moe_get_device_status", lib().moe_get_device_status(ctypes.byref(st), int(bool(clear))))
    return st.value
