"""The C-ABI library loads without a GPU, exports every function include/moefp8.h
declares, and rejects bad arguments on the host (no compute calls here)."""
import ctypes
import os
import re

import pytest

import block_fp8_mixture_topk_gb300 as moe
from block_fp8_mixture_topk_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moefp8.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["moe_route_topk", "moe_align_permute", "fp8_group_quant", "fp8_block_grouped_gemm",
                 "moe_fp8_block_forward", "moe_fp8_block_workspace_size", "moe_get_device_status"]:
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(moe.library_path() if os.path.exists(moe.library_path()) else ops.lib()._name)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_package_reexports_every_binding():
    """Each C entry point the binding wraps in ops.py is importable from the package."""
    wrapped = [n for n in declared_functions() if callable(getattr(ops, n, None))]
    assert "moe_combine_pairs" in wrapped
    missing = [n for n in wrapped if not hasattr(moe, n)]
    assert not missing, missing


def test_host_only_queries():
    L = ops.lib()
    assert L.moe_error_string(0) == b"MOE_OK"
    assert L.moe_error_string(-3) == b"MOE_ERR_WORKSPACE_TOO_SMALL"
    # P + min(E, P) * (block_m - 1) padded rows, whole tiles
    assert moe.moe_max_padded_rows(4096, 8, 256, 128) == 32768 + 256 * 127
    assert moe.moe_max_padded_rows(1, 8, 256, 128) == 8 + 8 * 127
    assert moe.moe_max_tiles(1, 8, 256, 128) == (8 + 8 * 127) // 128
    assert moe.moe_max_padded_rows(-1, 8, 256, 128) == -1
    ws = moe.moe_fp8_block_workspace_size(4096, 7168, 2048, 256, 8)
    rows = 32768 + 256 * 127
    # sorted activation codes, the sorted intermediate, bf16 weighted rows in pair order
    assert ws >= rows * 7168 + rows * 2048 + 32768 * 7168 * 2
    assert moe.moe_fp8_block_workspace_size(16, 256, 256, 4, 2) > 0
    # decode path (up to 4 tokens by default): its prologue + the decode kernel + the weighted sum
    assert moe.moe_fp8_block_forward_kernel_count(2, 7168, 2048, 256, 8) == 3
    assert moe.moe_fp8_block_forward_kernel_count(4, 7168, 2048, 256, 8) == 3
    # route + sort/quantise (one kernel up to 512 pairs, four above) + two GEMMs + weighted sum
    assert moe.moe_fp8_block_forward_kernel_count(5, 7168, 2048, 256, 8) == 5
    assert moe.moe_fp8_block_forward_kernel_count(64, 7168, 2048, 256, 8) == 5
    assert moe.moe_fp8_block_forward_kernel_count(65, 7168, 2048, 256, 8) == 8
    assert moe.moe_fp8_block_forward_kernel_count(0, 7168, 2048, 256, 8) == 0
    assert moe.moe_fp8_block_forward_kernel_count(-1, 7168, 2048, 256, 8) == -1


def test_forward_kernel_count_with_options():
    """The decode kernel routes in every CTA for E <= 256 (with groups the register-resident
    selection takes); otherwise the routing kernel runs first.  NVFP4 steps count per 8 tokens;
    block-scaled formats always take the tile GEMMs."""
    kc = moe.moe_fp8_block_forward_kernel_count
    dsv3 = moe.RoutingParams("sigmoid", 8, 4, 2.5, None)
    assert kc(1, 7168, 2048, 256, 8, dsv3) == 3
    assert kc(1, 4096, 14336, 8, 2, None, moe.ops.MOE_WEIGHTS_TILED) == 3
    assert kc(1, 2048, 768, 512, 8) == 4                        # 16 experts per lane: routing kernel
    assert kc(1, 256, 256, 96, 4, moe.RoutingParams("softmax", 4, 2)) == 4   # groups of 24 on 4-expert lanes
    assert kc(4, 7168, 2048, 256, 8, dsv3, decode="on") == 3
    assert kc(4, 7168, 2048, 256, 8, dsv3, decode="off") == 5
    assert kc(1, 7168, 2048, 256, 8, dsv3, scale_fmt="ue8m0_packed") == 5
    assert kc(17, 7168, 2048, 256, 8, dsv3, moe.ops.MOE_WEIGHTS_NVFP4) == 3 * 3
    assert kc(0, 7168, 2048, 256, 8, dsv3) == 0
    # the CTA-pair w2 GEMM replaces the one-CTA launch: the same 8 launches per step
    for fmt in ("f32", "ue8m0_packed", "mxfp8"):
        assert kc(16384, 2048, 768, 128, 8, scale_fmt=fmt) == 8


def test_pair_path_selection_without_a_device():
    """The shape rule of the CTA-pair GEMMs is host logic: steps that do not qualify give 0 with or
    without a device; invalid arguments give MOE_ERR_INVALID_ARG."""
    L = ops.lib()
    f32, packed, mx = (ops.SCALE_FMT[k] for k in ("f32", "ue8m0_packed", "mxfp8"))
    assert L.moe_fp8_block_pair_path(16384, 2048, 128, 8, f32) == 0            # fp32 scales
    assert L.moe_fp8_block_pair_path(4096, 7168, 256, 8, packed) == 0          # 128 rows per expert
    assert L.moe_fp8_block_pair_path(16384, 2176, 128, 8, packed) == 0         # H not whole 256-column items
    assert L.moe_fp8_block_pair_path(8191, 2048, 128, 8, mx) == 0              # 511.9 rows per expert
    assert L.moe_fp8_block_pair_path(-1, 2048, 128, 8, packed) == -1
    assert L.moe_fp8_block_pair_path(16, 2048, 0, 8, packed) == -1
    assert L.moe_fp8_block_pair_path(16, 2048, 4, 0, packed) == -1
    assert L.moe_fp8_block_pair_path(16, 2048, 4, 2, 9) == -1


def test_decode_path_selection():
    """"on" takes the decode-path GEMMs for any step they can serve (at most 8 tokens, at most
    512 routed pairs, an expert's w13 under 2^31 bytes), "off" never, "auto" never more than
    "on"."""
    dp = moe.moe_fp8_block_decode_path
    assert dp(1, 7168, 2048, 8, "on") and dp(8, 7168, 2048, 8, "on")
    assert dp(1, 7168, 2048, 8) and dp(4, 7168, 2048, 8) and not dp(5, 7168, 2048, 8)
    assert not dp(9, 7168, 2048, 8) and not dp(4096, 7168, 2048, 8)
    # the decode prologue + the decode kernel (routing, sort, both GEMMs) + the weighted sum
    assert moe.moe_fp8_block_forward_kernel_count(1, 7168, 2048, 256, 8) == 3
    assert not dp(1, 7168, 2048, 8, "off")
    assert dp(8, 256, 256, 32, "on") and not dp(9, 256, 256, 2, "on") and not dp(0, 256, 256, 8, "on")
    assert not dp(1, 65536, 16384, 8, "on")
    L = ops.lib()
    assert L.moe_fp8_block_decode_path(1, 256, 256, 8, 3) == -1
    assert L.moe_fp8_block_decode_path(-1, 256, 256, 8, 0) == -1
    assert L.moe_fp8_block_decode_path(1, 256, 256, 0, 0) == -1


@pytest.mark.parametrize("T,E,topk,rp,code", [
    (-1, 8, 2, None, -1),
    (4, 0, 1, None, -1),
    (4, 2048, 2, None, -2),
    (4, 8, 9, None, -2),
    (4, 64, 33, None, -2),
    (4, 8, 2, (1, 3, 1, 1.0), -2),     # E % n_group != 0
    (4, 8, 2, (0, 2, 1, 1.0), -2),     # grouping with softmax
    (4, 8, 2, (1, 2, 3, 1.0), -1),     # topk_group > n_group
    (4, 8, 2, (7, 1, 1, 1.0), -1),     # unknown scoring
])
def test_route_rejects_bad_arguments_on_host(T, E, topk, rp, code):
    L = ops.lib()
    p = ctypes.c_void_p(0x1000)
    rps = None
    if rp is not None:
        rps = ops._RoutingParams(rp[0], rp[1], rp[2], rp[3], None)
    rc = L.moe_route_topk(p, T, E, topk, 1, ctypes.byref(rps) if rps else None, p, p, None)
    assert rc == code


def test_quant_and_gemm_reject_bad_shapes_on_host():
    L = ops.lib()
    p = ctypes.c_void_p(0x1000)
    assert L.fp8_group_quant(p, 4, 100, 100, p, p, None) == -2          # cols % 128
    assert L.fp8_group_quant(p, 4, 128, 100, p, p, None) == -1          # ld < cols
    assert L.fp8_group_quant(p, 0, 128, 128, p, p, None) == 0           # empty: nothing to do
    assert L.fp8_block_quant_weight(p, 1, 100, 128, p, p, None) == -2
    ep = ops._Epilogue(1, 1, None, None, None, 0, 0, None, None, 0)
    # silu epilogue needs N % 256 == 0
    assert L.fp8_block_grouped_gemm(p, p, 1, 1, 128, p, p, 384, 128, 1, p, p, p, 1, ctypes.byref(ep), None) == -2
    ep.kind = 9
    assert L.fp8_block_grouped_gemm(p, p, 1, 1, 128, p, p, 256, 128, 1, p, p, p, 1, ctypes.byref(ep), None) == -1


def test_forward_rejects_bad_arguments_on_host():
    L = ops.lib()
    p = ctypes.c_void_p(0x1000)
    # H not a multiple of 128
    assert L.moe_fp8_block_forward(p, p, p, p, p, p, 4, 100, 256, 4, 2, 1, None, p, 1 << 30, p, None) == -2
    # T == 0 is a no-op
    assert L.moe_fp8_block_forward(None, None, None, None, None, None, 0, 256, 256, 4, 2, 1, None, None, 0, None,
                                   None) == 0
    # workspace too small
    assert L.moe_fp8_block_forward(p, p, p, p, p, p, 4, 256, 256, 4, 2, 1, None, ctypes.c_void_p(0x10000), 16, p,
                                   None) == -3


def test_newer_entry_points_reject_bad_arguments_on_host():
    """Options, scale formats, packing, the pair sum and the masked layout: argument errors are
    returned before anything touches a device."""
    L = ops.lib()
    p = ctypes.c_void_p(0x1000)
    big = ctypes.c_void_p(0x100000)
    # forward options: unknown weight layout / scale format / decode-path mode
    for layout, fmt, dec in [(7, 0, 0), (0, 5, 0), (0, 0, 3), (0, 0, -1)]:
        opts = ops._ForwardOptions(layout, fmt, dec)
        assert L.moe_fp8_block_forward_ex(p, p, p, p, p, p, 4, 256, 256, 4, 2, 1, None, ctypes.byref(opts), big,
                                          1 << 30, p, None, None) == -1
    # quantisers: unknown scale format
    assert L.fp8_group_quant_ex(p, 4, 128, 128, p, p, 7, None) == -1
    assert L.fp8_block_quant_weight_ex(p, 1, 128, 128, p, p, 3, None) == -1     # weights: f32 / ue8m0 only
    assert L.fp8_block_quant_weight_ex(p, 1, 128, 128, p, p, 2, None) == -1
    # packing: N not a multiple of 128; in place; empty is a no-op
    assert L.moe_fp8_block_pack_weights(p, 1, 100, 128, big, None) == -2
    assert L.moe_fp8_block_pack_weights(big, 2, 128, 128, ctypes.c_void_p(0x100000 + 4096), None) == -1
    assert L.moe_fp8_block_pack_weights(None, 0, 128, 128, None, None) == 0
    # pair sum: H not a multiple of 8
    assert L.moe_combine_pairs(p, p, 4, 2, 100, p, None) == -2
    # grouped GEMM: unknown weight layout / scale format in the epilogue options
    ep = ops._Epilogue(0, 1, p, None, None, 0, 0, None, None, 0, None, 4, 0)
    assert L.fp8_block_grouped_gemm(p, p, 1, 1, 128, p, p, 256, 128, 1, p, p, p, 1, ctypes.byref(ep), None) == -1
    ep = ops._Epilogue(0, 1, p, None, None, 0, 0, None, None, 0, None, 0, 9)
    assert L.fp8_block_grouped_gemm(p, p, 1, 1, 128, p, p, 256, 128, 1, p, p, p, 1, ctypes.byref(ep), None) == -1
    # masked layout
    ws = moe.moe_fp8_block_masked_workspace_size(4, 16, 256, 256)
    assert ws > 0
    assert L.moe_fp8_block_forward_masked(p, p, p, p, p, p, 4, 16, 100, 256, None, big, ws, p, None) == -2
    assert L.moe_fp8_block_forward_masked(p, p, p, p, p, p, 2048, 16, 256, 256, None, big, 1 << 40, p, None) == -2
    assert L.moe_fp8_block_forward_masked(p, p, p, p, p, p, 4, 16, 256, 256, None, big, ws - 256, p, None) == -3
    bad = ops._ForwardOptions(3, 0)
    assert L.moe_fp8_block_forward_masked(p, p, p, p, p, p, 4, 16, 256, 256, ctypes.byref(bad), big, ws, p,
                                          None) == -1
    assert L.moe_fp8_block_forward_masked(None, None, None, None, None, None, 0, 16, 256, 256, None, None, 0, None,
                                          None) == 0


def test_nvfp4_entry_points_reject_bad_arguments_on_host():
    L = ops.lib()
    p = ctypes.c_void_p(0x1000)
    big = ctypes.c_void_p(0x100000)
    # packed layout: [E][N/16][K/128] units of 16 x 64 code bytes + 16 x 8 scale bytes
    assert moe.moe_nvfp4_packed_bytes(2, 256, 512) == 2 * 16 * 4 * 1152
    assert moe.moe_nvfp4_packed_bytes(2, 250, 512) == 0
    assert moe.moe_nvfp4_packed_bytes(2, 256, 200) == 0
    # K not a multiple of 16 (quantiser) or 128 (packing); N not a multiple of 16; empty is a no-op
    assert L.moe_nvfp4_quant_weight(p, 1, 128, 120, p, p, p, None) == -2
    assert L.moe_nvfp4_quant_weight(None, 0, 128, 128, None, None, None, None) == 0
    assert L.moe_nvfp4_pack_weights(p, p, 1, 100, 128, big, None) == -2
    assert L.moe_nvfp4_pack_weights(p, p, 1, 128, 64, big, None) == -2
    assert L.moe_nvfp4_pack_weights(None, None, 0, 128, 128, None, None) == 0
    # NVFP4 weights run on the decode-path kernel: turning it off is an argument error
    opts = ops._ForwardOptions(ops.MOE_WEIGHTS_NVFP4, 0, 1)
    assert L.moe_fp8_block_forward_ex(p, p, p, p, p, p, 4, 256, 256, 4, 2, 1, None, ctypes.byref(opts), big,
                                      1 << 30, p, None, None) == -1
    # more than 8 tokens run 8 at a time: argument errors still come back before any launch
    assert L.moe_fp8_block_forward_ex(None, p, p, p, p, p, 20, 256, 256, 4, 2, 1, None, ctypes.byref(opts), big,
                                      1 << 30, p, None, None) == -1
    assert L.moe_fp8_block_forward_ex(p, p, p, p, p, p, 20, 200, 256, 4, 2, 1, None, ctypes.byref(opts), big,
                                      1 << 30, p, None, None) == -2
    # ... including the weights, the workspace and its size, checked before the first stage event is
    # recorded (the fake event handles below would fail if they were recorded)
    opts = ops._ForwardOptions(ops.MOE_WEIGHTS_NVFP4, 0, 0)
    events = (ctypes.c_void_p * 7)(*([0x40] * 7))
    assert L.moe_fp8_block_forward_ex(p, p, None, p, p, p, 20, 256, 256, 4, 2, 1, None, ctypes.byref(opts), big,
                                      1 << 30, p, None, events) == -1
    assert L.moe_fp8_block_forward_ex(p, p, p, p, p, p, 20, 256, 256, 4, 2, 1, None, ctypes.byref(opts), big,
                                      256, p, None, events) == -3
    assert L.moe_fp8_block_forward_ex(p, p, p, p, p, p, 20, 256, 256, 4, 2, 1, None, ctypes.byref(opts),
                                      ctypes.c_void_p(0x100010), 1 << 30, p, None, events) == -1
    # an expert MLP the decode kernel cannot take (top-k above 64 gives more than 512 pairs)
    opts = ops._ForwardOptions(ops.MOE_WEIGHTS_NVFP4, 0, 0)
    assert L.moe_fp8_block_forward_ex(p, p, p, p, p, p, 8, 256, 256, 128, 65, 1, None, ctypes.byref(opts), big,
                                      1 << 40, p, None, None) == -2


def test_block_scaled_formats_reject_bad_arguments_on_host():
    """Packed UE8M0 and MXFP8 scales: sizes, packing and the layer's options, checked on the host."""
    L = ops.lib()
    p = ctypes.c_void_p(0x1000)
    big = ctypes.c_void_p(0x100000)
    # packed UE8M0 tiles: ceil(rows/128) * ceil(K/512) * 512 bytes; MXFP8: ceil(rows/128) * (K/128) * 512
    assert moe.moe_packed_scale_bytes(128, 7168) == 14 * 512
    assert moe.moe_packed_scale_bytes(129, 640) == 2 * 2 * 512
    assert moe.moe_packed_scale_bytes(128, 100) == 0
    assert moe.moe_mxfp8_packed_scale_bytes(128, 7168) == 56 * 512
    assert moe.moe_mxfp8_packed_scale_bytes(300, 256) == 3 * 2 * 512
    # packing: shapes and alignment
    assert L.moe_fp8_block_pack_scales(p, 1, 100, 128, big, None) == -2
    assert L.moe_fp8_block_pack_scales(p, 1, 128, 128, ctypes.c_void_p(0x100008), None) == -1
    assert L.moe_fp8_block_pack_scales(None, 0, 128, 128, None, None) == 0
    assert L.moe_mxfp8_quant_weight(p, 1, 128, 96, p, p, None) == -2
    assert L.moe_mxfp8_pack_scales(p, 100, 128, big, None) == -2         # whole 128-row tiles
    assert L.moe_mxfp8_pack_scales(p, 128, 96, big, None) == -2
    assert L.moe_mxfp8_pack_scales(None, 0, 128, None, None) == 0
    # the layer: block-scaled formats take neither the decode kernel nor NVFP4 weights
    for fmt in (2, 3):
        opts = ops._ForwardOptions(0, fmt, 2)
        assert L.moe_fp8_block_forward_ex(p, p, p, p, p, p, 4, 256, 256, 4, 2, 1, None, ctypes.byref(opts), big,
                                          1 << 30, p, None, None) == -1
        opts = ops._ForwardOptions(ops.MOE_WEIGHTS_NVFP4, fmt, 0)
        assert L.moe_fp8_block_forward_ex(p, p, p, p, p, p, 4, 256, 256, 4, 2, 1, None, ctypes.byref(opts), big,
                                          1 << 30, p, None, None) == -1
    # grouped GEMM: the block-scaled kernel has the store, SiLU and pair-row epilogues only
    ep = ops._Epilogue(3, 1, p, None, None, 0, 0, p, p, 1, None, 0, 3)
    assert L.fp8_block_grouped_gemm(p, p, 1, 1, 128, p, p, 256, 128, 1, p, p, p, 1, ctypes.byref(ep), None) == -1
