/*
 * moefp8 — block-FP8 fused Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument documented "device" is caller-owned device
 * memory of the current CUDA device; "host" pointers are caller-owned host
 * memory.  The library allocates no memory per call: scratch space is the
 * caller's workspace, whose size the matching *_workspace_size function gives.
 * All calls are asynchronous on the given stream (a cudaStream_t passed as
 * void*, NULL = the legacy default stream) and never synchronise the host.
 *
 * Return value of every int function: MOE_OK (0) or a negative MOE_ERR_* code.
 * Argument errors are detected on the host before anything is enqueued.
 * Problems only the device can see (a routed expert id out of range, a pipeline
 * wait that ran past its time limit) never trap: they set bits in a device
 * status word, read with moe_get_device_status after synchronising.
 *
 * Tensor layouts (row-major, innermost dimension last):
 *   hidden        bf16  [T, H]            (bf16 passed as uint16_t bit patterns)
 *   router_logits fp32  [T, E]
 *   w13           e4m3  [E, 2I, H]        rows [0, I) gate, rows [I, 2I) up
 *   w13_scale     fp32  [E, 2I/128, H/128]
 *   w2            e4m3  [E, H, I]
 *   w2_scale      fp32  [E, H/128, I/128]
 *   out           bf16  [T, H]
 * "e4m3" is float8 e4m3fn (1-4-3, bias 7, max 448, no infinities) stored as
 * uint8_t.  H and I must be multiples of 128.
 *
 * Sources: the pages "Quantization and MoE Optimizations" (vLLM wiki),
 * "vllm.model_executor.layers.fused_moe.oracle.fp8" and
 * "vllm.model_executor.layers.quantization.online.nvfp4" (vLLM API docs).
 */
#ifndef MOEFP8_H
#define MOEFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)          /* null pointer, negative size, bad enum */
#define MOE_ERR_UNSUPPORTED_SHAPE (-2)    /* H or I not a multiple of 128, topk > E, ... */
#define MOE_ERR_WORKSPACE_TOO_SMALL (-3)
#define MOE_ERR_CUDA (-4)                 /* a CUDA runtime call failed */
#define MOE_ERR_DEVICE (-5)               /* current device is not sm_103 (GB300) */

/* device status bits (moe_get_device_status) */
#define MOE_STATUS_WAIT_TIMEOUT 0x1u      /* a pipeline wait gave up; outputs invalid */
#define MOE_STATUS_BAD_EXPERT_ID 0x2u     /* a routed id was outside [0, E); pair dropped */
#define MOE_STATUS_BAD_COUNT 0x4u         /* a masked-layout count was outside [0, max_tokens]; clamped */
#define MOE_STATUS_BAD_SCALE 0x8u         /* a scale packed as UE8M0 was not a positive power of two */

/* Limits of this implementation. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32
#define MOE_MAX_GROUPS 32
#define MOE_BLOCK_M 128                   /* rows per expert tile of the grouped GEMMs */

/* ---- routing -------------------------------------------------------------- */
#define MOE_SCORING_SOFTMAX 0
#define MOE_SCORING_SIGMOID 1

/* Router options ("router — top-K router" of the FusedMoE layer and the
 * "fused grouped top-K routing" switch, page "Quantization and MoE
 * Optimizations", sections FusedMoE Class and Key Environment Variables).
 * A NULL moe_routing_params* means softmax scoring, no grouping, scaling 1.   */
typedef struct moe_routing_params {
    int32_t scoring;        /* MOE_SCORING_SOFTMAX or MOE_SCORING_SIGMOID */
    int32_t n_group;        /* 1 = ungrouped; > 1 (sigmoid only): E/n_group consecutive experts per group */
    int32_t topk_group;     /* groups kept when n_group > 1 */
    float routed_scaling;   /* multiplies the final weights (1.0 = none) */
    const float* bias;      /* device fp32 [E] selection bias, or NULL (sigmoid only) */
} moe_routing_params;

/* Top-k routing of T tokens over E experts.
 *   softmax: the k largest logits (ties: lower index); weight = softmax
 *            probability, renormalised over the chosen k if renormalize != 0.
 *   sigmoid: s = fp32(1/(1+exp(-logit))) evaluated in fp64; b = s + bias
 *            selects; grouped: group score = sum of its two largest b, the
 *            topk_group best groups are kept (ties: lower group), the k largest
 *            b among their experts are chosen; weight = s, renormalised over the
 *            chosen k if renormalize != 0.
 *   Both: weights *= routed_scaling.
 * logits: device fp32 [T, E]; topk_ids: device int32 [T, topk] (descending
 * score order); topk_weights: device fp32 [T, topk].
 * Errors: INVALID_ARG (null pointer, T < 0), UNSUPPORTED_SHAPE (E > 1024,
 * topk > min(E, 32), E % n_group, n_group > 32, grouping with softmax). */
int moe_route_topk(const float* logits, int T, int E, int topk, int renormalize,
                   const moe_routing_params* rp, int32_t* topk_ids, float* topk_weights,
                   void* stream);

/* ---- expert sort ("sorted token" pattern) ------------------------------------
 * Page "Quantization and MoE Optimizations", section Triton Fused MoE Kernel:
 * each program handles a block of tokens sorted by expert.  Pair p = t*topk + j
 * goes to expert topk_ids[p].  Rows are grouped by expert, each expert's rows
 * padded to a multiple of block_m, pairs of one expert in ascending p.
 *
 * Outputs (device):
 *   expert_offsets  int32 [E+1]  exclusive prefix sum of the per-expert counts
 *   padded_offsets  int32 [E+1]  the same with every count rounded up to block_m
 *   sorted_pair_ids int32 [moe_max_padded_rows(...)]  pair of each padded row, -1 in padding
 *   pos             int32 [T*topk]  padded row of each pair (-1 if its id was invalid)
 *   tile_expert     int32 [moe_max_tiles(...)]  expert of each block_m-row tile
 *   tile_row0       int32 [moe_max_tiles(...)]  first padded row of each tile
 *   num_tiles       int32 [1]
 * workspace: device scratch of moe_align_permute_workspace_size(T, topk, E) bytes.
 * block_m: 1..1024.  Invalid ids set MOE_STATUS_BAD_EXPERT_ID and are dropped. */
int64_t moe_max_padded_rows(int T, int topk, int E, int block_m);
int64_t moe_max_tiles(int T, int topk, int E, int block_m);
size_t moe_align_permute_workspace_size(int T, int topk, int E);
int moe_align_permute(const int32_t* topk_ids, int T, int topk, int E, int block_m,
                      int32_t* expert_offsets, int32_t* padded_offsets, int32_t* sorted_pair_ids,
                      int32_t* pos, int32_t* tile_expert, int32_t* tile_row0, int32_t* num_tiles,
                      void* workspace, size_t workspace_bytes, void* stream);

/* The same expert sort without a workspace argument.  The pages have no
 * counterpart to this entry point: it is for callers that cannot allocate device
 * memory when they call (a plugin inside a host program whose pool owns all
 * device memory, or a serving loop that must not call cudaMalloc, which may
 * synchronise the device).  Its scratch is one fixed array of
 * MOE_NOALLOC_SORT_SCRATCH_INTS int32 inside the library, present on every GPU
 * that loads the library until the process exits.
 *   - Arguments, outputs and results are those of moe_align_permute.
 *   - A problem needing more than the fixed scratch, i.e.
 *     ceil(T*topk / 1024) * E > MOE_NOALLOC_SORT_SCRATCH_INTS, is rejected with
 *     MOE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - The first call on a device looks up the array's device address (with that
 *     device current); make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents.  Nothing
 *     in it has to start at zero (each call writes every count it reads), but calls
 *     that overlap on the GPU (e.g. on two streams) race on it: order them.
 *   - Allocates no memory (no cudaMalloc / cudaFree). */
#define MOE_NOALLOC_SORT_SCRATCH_INTS 262144
int moe_align_permute_noalloc(const int32_t* topk_ids, int T, int topk, int E, int block_m,
                              int32_t* expert_offsets, int32_t* padded_offsets, int32_t* sorted_pair_ids,
                              int32_t* pos, int32_t* tile_expert, int32_t* tile_row0, int32_t* num_tiles,
                              void* stream);

/* ---- FP8 quantisation ---------------------------------------------------------
 * Dynamic per-token-group activation quantisation, groups of 1x128 ("computed
 * per-token at runtime", page "Quantization and MoE Optimizations", section
 * Fp8Config; activation key kFp8Dynamic128Sym, page
 * "vllm.model_executor.layers.fused_moe.oracle.fp8", _get_priority_backends):
 *   scale = max(amax, 1e-8) / 448 (fp32), q = e4m3(x / scale), round to
 *   nearest even, saturate to +-448.
 * x: device bf16 [rows, cols] with row stride ld (elements, >= cols, multiple
 * of 8); q: device e4m3 [rows, cols] (dense); s: device fp32 [rows, cols/128].
 * cols must be a multiple of 128. */
int fp8_group_quant(const uint16_t* x, int rows, int cols, int ld, uint8_t* q, float* s,
                    void* stream);

/* 128x128 block weight quantisation of stacked expert weights w [E, N, K]
 * (bf16) with the same rule, amax over each block ("weight_block_size ...
 * [128, 128]", Fp8Config; online quantisation at load time, page
 * "Quantization", section Online quantization).  q: device e4m3 [E, N, K];
 * s: device fp32 [E, N/128, K/128].  N and K multiples of 128. */
int fp8_block_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, float* s,
                           void* stream);

/* Load-time conversion of e4m3 expert weights from the pages' layout [E, N, K]
 * into the tile-packed layout the GEMMs stream fastest: packed[e][nb][kb][r][c] =
 * w[e, nb*128 + r, kb*128 + c], i.e. [E][N/128][K/128][128][128], each 128x128
 * block one contiguous 16 KB run and the K blocks of a 128-row band adjacent.
 * The pages convert checkpoint weights into each kernel's own format once, at
 * load time (process_weights_after_loading -> convert_to_nvfp4_moe_kernel_format,
 * page "vllm.model_executor.layers.quantization.online.nvfp4"); this is that step
 * for the block-FP8 kernels.  The block scales keep their layout.
 * w, packed: device, 16-byte aligned, E*N*K bytes, not overlapping.  N and K
 * multiples of 128, E*N*K/128 < 2^31. */
#define MOE_WEIGHTS_NK 0      /* [E, N, K] row-major, the pages' layout */
#define MOE_WEIGHTS_TILED 1   /* moe_fp8_block_pack_weights output */
#define MOE_WEIGHTS_NVFP4 2   /* NVFP4 weights, moe_nvfp4_pack_weights output */
int moe_fp8_block_pack_weights(const uint8_t* w, int E, int N, int K, uint8_t* packed, void* stream);

/* NVFP4 expert weights (page "vllm.model_executor.layers.quantization.online.nvfp4",
 * _quantize_moe_weight_to_nvfp4; load time).  Per expert: amax over the whole [N, K] weight,
 * floored at 1e-8; global_scale = (FLOAT4_E2M1_MAX * FLOAT8_E4M3_MAX) / amax = 2688 / amax; the
 * weights times global_scale rounded back to bf16 are quantised in blocks of 16 along K with
 * one e4m3 scale per block: block scale = e4m3(max|x| / 6), code = e2m1(x / block scale)
 * (nearest, ties to even, saturating at +-6; the pages name scaled_fp4_quant's inputs, not its
 * arithmetic, and this is the FP8 groups' rule with e2m1's maximum).
 *   w            bf16 [E, N, K], device, 16-byte aligned; K a multiple of 16
 *   q            uint8 [E, N, K/2]: two e2m1 codes per byte, element 2i in the low nibble
 *   block_scale  uint8 [E, N, K/16]: e4m3fn bits
 *   global_scale fp32 [E]: 1 / global_scale, the factor that dequantises
 * Dequantised weight = e2m1(code) * block_scale * global_scale[e].  Three launches on `stream`
 * (amax, quantise, global scales); global_scale serves as the amax scratch until the last. */
int moe_nvfp4_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, uint8_t* block_scale,
                           float* global_scale, void* stream);
/* Bytes of the packed NVFP4 layout of an [E, N, K] weight (N % 16 == 0, K % 128 == 0; else 0):
 * [E][N/16][K/128] units of 1152 bytes, each the 16 rows x 64 code bytes of one 16-row slab over
 * one 128-wide K block followed by their 16 rows x 8 block-scale bytes. */
size_t moe_nvfp4_packed_bytes(int E, int N, int K);
/* Load-time conversion of moe_nvfp4_quant_weight's codes and block scales into that layout (the
 * one the forward reads with MOE_WEIGHTS_NVFP4).  q: 16-byte aligned, block_scale: 8-byte
 * aligned, packed: 16-byte aligned, moe_nvfp4_packed_bytes(E, N, K) bytes, not overlapping. */
int moe_nvfp4_pack_weights(const uint8_t* q, const uint8_t* block_scale, int E, int N, int K, uint8_t* packed,
                           void* stream);

/* ---- scale formats ------------------------------------------------------------------
 * Every 1x128 group and 128x128 block scale is max(amax, 1e-8)/448 in fp32 (MOE_SCALE_F32),
 * or that value rounded up to a power of two (MOE_SCALE_UE8M0: the "FLOAT32_CEIL_UE8M0"
 * format, fp32 scales rounded up to UE8M0, page "Quantization and MoE Optimizations",
 * section DeepGEMM Scale Formats), so that each scale is exactly an 8-bit exponent.  The
 * GEMMs take either (scales are fp32 values); the format decides how the activations and
 * the requantised intermediate are scaled, and should match the weights'. */
#define MOE_SCALE_F32 0
#define MOE_SCALE_UE8M0 1
/* MOE_SCALE_UE8M0_PACKED: the UE8M0 scales stored as 8-bit exponents (value 2^(byte - 127)) in the
 * packed layout the tensor cores read ("UE8M0: packed UE8M0 (4 values per int32) (Blackwell)",
 * page "Quantization and MoE Optimizations", section DeepGEMM Scale Formats).  With it the GEMMs
 * run on the block-scaled MMA (tcgen05.mma kind::mxf8f6f4.block_scale): the tensor cores apply
 * the scales and accumulate the whole K loop, with no per-K-block promotion.  The numbers are those
 * of MOE_SCALE_UE8M0 (the same scales; only the fp32 summation order differs).
 *
 * Packed layout of the scales of a [rows, K] operand (1x128 groups of activations, or a weight's
 * 128x128 blocks repeated over their 128 rows): 512-byte tiles ordered [ceil(rows/128)][ceil(K/512)];
 * the byte of (row r, K block kb = k/128) is at
 *     ((r / 128) * ceil(K/512) + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4
 * i.e. a tile is 32 lines of 16 bytes, line l holding rows l, l+32, l+64, l+96 as four 32-bit
 * words, each word the scales of 4 consecutive K blocks (byte b = K block 4q + b).  Weights: one
 * set of tiles per expert, [E][N/128][ceil(K/512)] tiles (moe_fp8_block_pack_scales). */
#define MOE_SCALE_UE8M0_PACKED 2
/* MOE_SCALE_MXFP8: MXFP8 ("MXFP8 (block [1, 32])", page "vllm.model_executor.layers.fused_moe.oracle.fp8",
 * make_fp8_moe_quant_config; weights with "e8m0 group-32 scales", _humming_fp8_weight_schema): the
 * activations and the requantised intermediate in groups of 32 along K, the weights in 1x32 blocks
 * along K, every scale max(amax, 1e-8)/448 rounded up to a power of two and stored as its UE8M0
 * byte.  The GEMMs run on the block-scaled MMA, one scale per 32 K per row, as the format defines.
 * Packed scale tiles of a [rows, K] operand: the same layout as above with the 32-wide groups as
 * the scale columns, i.e. ceil(rows/128) * (K/128) tiles of 512 bytes, the byte of (row r, group
 * g = k/32) at ((r / 128) * (K/128) + g / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + g % 4. */
#define MOE_SCALE_MXFP8 3
/* Bytes of the MXFP8 packed scale tiles of a [rows, K] operand: ceil(rows/128) * (K/128) * 512. */
size_t moe_mxfp8_packed_scale_bytes(int64_t rows, int K);
/* MXFP8 weight quantisation of stacked bf16 expert weights w [E, N, K] (load time): 1x32 blocks
 * along K, q e4m3 [E, N, K], s the UE8M0 scale bytes [E, N, K/32] (the pages' uint8 layout).  w,
 * q 16-byte aligned; K a multiple of 128. */
int moe_mxfp8_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, uint8_t* s, void* stream);
/* Packing of UE8M0 scale bytes s [rows, K/32] (e.g. moe_mxfp8_quant_weight's, rows = E * N) into the
 * MXFP8 packed tiles: out, moe_mxfp8_packed_scale_bytes(rows, K) bytes, 16-byte aligned.  rows a
 * multiple of 128 (whole tiles), K a multiple of 128. */
int moe_mxfp8_pack_scales(const uint8_t* s, int64_t rows, int K, uint8_t* out, void* stream);
/* Bytes of the packed scale tiles of a [rows, K] operand: ceil(rows/128) * ceil(K/512) * 512
 * (0 for negative sizes or K not a multiple of 128). */
size_t moe_packed_scale_bytes(int64_t rows, int K);
/* Load-time packing of UE8M0 weight block scales s [E, N/128, K/128] (fp32 powers of two, e.g.
 * fp8_block_quant_weight_ex with MOE_SCALE_UE8M0) into the packed layout: out, device,
 * moe_packed_scale_bytes(E * N, K) bytes, 16-byte aligned; K blocks past K in a tile get byte 127.
 * A scale that is not a positive power of two sets MOE_STATUS_BAD_SCALE (device status word; its
 * byte is then its exponent, not a rounding of it).  N and K multiples of 128. */
int moe_fp8_block_pack_scales(const float* s, int E, int N, int K, uint8_t* out, void* stream);
/* fp8_group_quant / fp8_block_quant_weight with a scale format.  fp8_group_quant_ex with
 * MOE_SCALE_UE8M0_PACKED writes the UE8M0 scales as packed tiles: s is then a byte array of
 * moe_packed_scale_bytes(rows, cols) (passed as float*), rows past `rows` in the last tile left as
 * they are.  With MOE_SCALE_MXFP8, groups of 32: s is a byte array of the UE8M0 scales
 * [rows, cols/32] (passed as float*).  fp8_block_quant_weight_ex takes MOE_SCALE_F32 or
 * MOE_SCALE_UE8M0 (pack its scales with moe_fp8_block_pack_scales). */
int fp8_group_quant_ex(const uint16_t* x, int rows, int cols, int ld, uint8_t* q, float* s, int scale_fmt,
                       void* stream);
int fp8_block_quant_weight_ex(const uint16_t* w, int E, int N, int K, uint8_t* q, float* s, int scale_fmt,
                              void* stream);

/* ---- grouped block-FP8 GEMM ------------------------------------------------------
 * For every tile m < *num_tiles (rows tile_row0[m] .. +127 of A, all routed to
 * expert e = tile_expert[m]) and every output column n:
 *   C[r, n] = sum_kb a_scale[r, kb] * b_scale[e, n/128, kb]
 *                   * sum_{k in block kb} A[r, k] * B[e, n, k]
 * with the block scales applied per 128-wide K block in fp32 (tensor cores
 * accumulate each K block, the scales are applied before the next one).
 *   A        device e4m3 [a_rows, K]   (a_rows >= every tile_row0 + 128)
 *   a_scale  device fp32, element (r, kb) at a_scale[r*a_scale_row_stride + kb*a_scale_kb_stride]
 *   B        device e4m3 [E, N, K];  b_scale device fp32 [E, N/128, K/128]
 *   tile_expert / tile_row0 device int32 [max_tiles]; num_tiles device int32 [1]
 * Epilogues:
 *   MOE_EPI_STORE_F32: out_f32[r, n] = C[r, n]  (out_f32: device fp32 [a_rows, N])
 *   MOE_EPI_SILU_MUL_QUANT: h[r, i] = silu(C[r, i]) * C[r, N/2 + i] for i < N/2,
 *       then 1x128 e4m3 quantisation of h ("SiLU(gate)*up with requantisation"):
 *       out_q device e4m3 [a_rows, N/2]; out_scale element (r, g) at
 *       out_scale[r*out_scale_row_stride + g*out_scale_kb_stride].
 *   MOE_EPI_WEIGHTED_SCATTER: for rows with pair = sorted_pair_ids[r] >= 0,
 *       out_f32[pair / topk, n] += topk_weights[pair] * C[r, n]  (out_f32: device
 *       fp32 [T, N], accumulated with atomics; the caller zeroes it first).
 *   MOE_EPI_WEIGHTED_ROWS: for rows with pair = sorted_pair_ids[r] >= 0,
 *       out_f32[r, n] = topk_weights[pair] * C[r, n]  (out_f32: device fp32
 *       [a_rows, N] in sorted-row order; padding rows are not written).
 *   MOE_EPI_WEIGHTED_PAIRS_BF16: for rows with pair = sorted_pair_ids[r] in
 *       [0, num_pairs), out_bf16[pair, n] = bf16_rn(topk_weights[pair] * C[r, n])
 *       (out_bf16: device bf16 [num_pairs, N] in pair order p = t*topk + j, rows
 *       16-byte aligned; rows of pairs that no tile holds are not written).  The
 *       router weight is applied after dequantisation, in fp32, as the pages'
 *       Triton kernel orders it (section Triton Fused MoE Kernel); the weighted
 *       row is then held in the output's own type until the k-way sum
 *       (moe_combine_pairs).
 * K, N multiples of 128 (N multiple of 256 for MOE_EPI_SILU_MUL_QUANT).
 * Optional epilogue field sorted_pair_ids (store / silu epilogues; NULL =
 * unused): rows with id -1 are padding; a group of 32 padding rows is not
 * computed and its output rows are left unspecified (the scatter and rows
 * epilogues always require it and skip padding rows).
 * Otherwise rows of a tile past its expert's count are computed from whatever
 * A holds there and belong to no pair.
 * Scale format (epilogue scale_fmt): MOE_SCALE_F32 / MOE_SCALE_UE8M0: fp32 scales as above, the
 * format only deciding the SiLU epilogue's requantisation scales.  MOE_SCALE_UE8M0_PACKED: the
 * block-scaled MMA; a_scale is A's packed scale tiles (a byte array of
 * moe_packed_scale_bytes(a_rows, K), strides ignored), b_scale the weights' packed tiles
 * (moe_fp8_block_pack_scales), every tile_row0 a multiple of 128 (other tiles are skipped and set
 * MOE_STATUS_BAD_EXPERT_ID), the SiLU epilogue writes out_scale as packed tiles of
 * moe_packed_scale_bytes(a_rows, N/2) bytes, and only MOE_EPI_STORE_F32, MOE_EPI_SILU_MUL_QUANT and
 * MOE_EPI_WEIGHTED_PAIRS_BF16 are available. */
#define MOE_EPI_STORE_F32 0
#define MOE_EPI_SILU_MUL_QUANT 1
#define MOE_EPI_WEIGHTED_SCATTER 2
#define MOE_EPI_WEIGHTED_ROWS 3
#define MOE_EPI_WEIGHTED_PAIRS_BF16 4

typedef struct moe_gemm_epilogue {
    int32_t kind;                     /* MOE_EPI_* */
    int32_t topk;                     /* MOE_EPI_WEIGHTED_SCATTER / _ROWS / _PAIRS_BF16 */
    float* out_f32;
    uint8_t* out_q;
    float* out_scale;
    int64_t out_scale_row_stride;
    int64_t out_scale_kb_stride;
    const int32_t* sorted_pair_ids;   /* MOE_EPI_WEIGHTED_SCATTER / _ROWS / _PAIRS_BF16 */
    const float* topk_weights;        /* MOE_EPI_WEIGHTED_SCATTER / _ROWS / _PAIRS_BF16, [T*topk] */
    int64_t num_pairs;                /* MOE_EPI_WEIGHTED_SCATTER / _ROWS / _PAIRS_BF16: T*topk; other pair ids are skipped */
    uint16_t* out_bf16;               /* MOE_EPI_WEIGHTED_PAIRS_BF16 */
    int32_t b_layout;                 /* layout of B: MOE_WEIGHTS_NK (0) or MOE_WEIGHTS_TILED */
    int32_t scale_fmt;                /* MOE_EPI_SILU_MUL_QUANT: scale format of the requantisation */
} moe_gemm_epilogue;

int fp8_block_grouped_gemm(const uint8_t* A, const float* a_scale, int64_t a_scale_row_stride,
                           int64_t a_scale_kb_stride, int64_t a_rows,
                           const uint8_t* B, const float* b_scale, int N, int K, int E,
                           const int32_t* tile_expert, const int32_t* tile_row0,
                           const int32_t* num_tiles, int64_t max_tiles,
                           const moe_gemm_epilogue* epilogue, void* stream);

/* ---- weighted unpermute-sum -------------------------------------------------------
 * out[t, :] = bf16( sum_{j < topk, pos[t*topk+j] >= 0} y[pos[t*topk+j], :] ), summed in
 * j order in fp32, rounded to nearest even ("gathers results", page
 * "Quantization and MoE Optimizations", section Modular Kernel Architecture).
 * y: device fp32 [y_rows, H] (the router-weighted rows of MOE_EPI_WEIGHTED_ROWS);
 * pos: device int32 [T*topk] (moe_align_permute); out: device bf16 [T, H].
 * H multiple of 4; positions >= y_rows are skipped and set MOE_STATUS_BAD_EXPERT_ID. */
int moe_unpermute_sum(const float* y, int64_t y_rows, const int32_t* pos, int T, int topk, int H,
                      uint16_t* out, void* stream);

/* The same sum over rows held in pair order (MOE_EPI_WEIGHTED_PAIRS_BF16):
 * out[t, :] = bf16( sum_{j < topk, pos[t*topk+j] >= 0} y[t*topk+j, :] ), each term
 * widened to fp32, summed in j order, rounded to nearest even once.
 * y: device bf16 [T*topk, H]; pos: device int32 [T*topk] (used only to skip the
 * pairs that were dropped, pos < 0); out: device bf16 [T, H].  H multiple of 8,
 * y and out 16-byte aligned. */
int moe_combine_pairs(const uint16_t* y, const int32_t* pos, int T, int topk, int H, uint16_t* out,
                      void* stream);

/* ---- the whole layer -------------------------------------------------------------
 * Router -> sort by expert -> 1x128 quantisation of hidden -> GEMM over w13 with
 * SiLU(gate)*up + requantisation -> GEMM over w2 writing each pair's
 * router-weighted row (bf16, pair order) -> per-token sum of its k rows in j
 * order -> bf16 output (the modular pipeline Router -> Prepare/Finalize
 * -> Permute/Experts/Unpermute, page "Quantization and MoE Optimizations",
 * section Modular Kernel Architecture; weights "[num_experts, N, K]", section
 * FusedMoE Class; 128x128 weight blocks with dynamic activations, section
 * Fp8Config).
 * workspace: device scratch of moe_fp8_block_workspace_size(T, H, I, E, topk)
 * bytes (256-byte aligned).  hidden, w13, w2 and out 16-byte aligned.  out may
 * not alias any input.  T == 0 is a no-op. */
size_t moe_fp8_block_workspace_size(int T, int H, int I, int E, int topk);
/* Number of kernels one moe_fp8_block_forward launches for these sizes (host only), with
 * rp == NULL and default options: see moe_fp8_block_forward_kernel_count_ex. */
int moe_fp8_block_forward_kernel_count(int T, int H, int I, int E, int topk);
int moe_fp8_block_forward(const uint16_t* hidden, const float* router_logits,
                          const uint8_t* w13, const float* w13_scale,
                          const uint8_t* w2, const float* w2_scale,
                          int T, int H, int I, int E, int topk, int renormalize,
                          const moe_routing_params* rp, void* workspace, size_t workspace_bytes,
                          uint16_t* out, void* stream);

/* The same layer with w13 and w2 in the tile-packed layout (moe_fp8_block_pack_weights);
 * identical results, the weights streamed as contiguous 16 KB blocks. */
int moe_fp8_block_forward_packed(const uint16_t* hidden, const float* router_logits,
                                 const uint8_t* w13, const float* w13_scale,
                                 const uint8_t* w2, const float* w2_scale,
                                 int T, int H, int I, int E, int topk, int renormalize,
                                 const moe_routing_params* rp, void* workspace, size_t workspace_bytes,
                                 uint16_t* out, void* stream);

/* ---- decode path ---------------------------------------------------------------------
 * Which kernels run the two expert GEMMs of moe_fp8_block_forward_ex.  A step of at most 8
 * tokens (T*topk <= 512, 2*I*H < 2^31) can take the decode path: both GEMMs in one persistent
 * kernel whose work items are 32 weight rows of one expert over the whole K, streamed by TMA
 * and multiplied on the warp-level tensor core MMA, so that every SM streams weights even
 * when only a few experts are touched (a one-token DeepSeek-V3-shaped step touches 8 experts:
 * 1024 w13 items instead of 128 tiles of 128 x 256) and the w2 weights stream while the last
 * w13 items finish.  The same kernel routes the step's tokens in every CTA (the routing
 * kernel's selection, so the same experts and weights; for E <= 256 with groups the register-
 * resident selection takes, otherwise the routing kernel runs first) and sorts the pairs; a small
 * prologue kernel zeroes its counters and quantises the tokens, and the weighted sum follows.
 * Same operands, block scales and epilogues as the tile GEMMs; the sums run in another order, so
 * results agree with the tile path to fp32 rounding, not bit for bit.  With events, the prologue
 * is recorded as the quantisation stage and the decode kernel as the w13 GEMM stage (the routing
 * stage holds the routing kernel or nothing; the sort and w2 stages are empty).
 *   MOE_DECODE_AUTO: the faster path for the step's size as measured on GB300: the decode
 *                    path for steps of up to four tokens, the tile GEMMs otherwise
 *   MOE_DECODE_OFF:  always the tile GEMMs
 *   MOE_DECODE_ON:   the decode path whenever the step qualifies */
#define MOE_DECODE_AUTO 0
#define MOE_DECODE_OFF 1
#define MOE_DECODE_ON 2
/* 1 if a step of T tokens (hidden H, intermediate I, this top-k) takes the decode-path GEMMs
 * under `mode`, 0 if it takes the tile GEMMs, -1 for a negative size, topk < 1 or an unknown
 * mode.  Host only. */
int moe_fp8_block_decode_path(int T, int H, int I, int topk, int mode);
/* Whether the w2 GEMM of a step of T tokens (hidden H, E experts, this top-k) in `scale_fmt`
 * runs on the CTA-pair kernel: two CTAs of a cluster compute two consecutive 128-row tiles of one
 * expert with the two-SM tensor-core MMA (tcgen05.mma.cta_group::2, M = 256), each CTA holding its
 * own rows of the activations and half of the 256 weight rows of the item, so that an SM takes in
 * a third fewer operand bytes per multiply-add.  Taken with the packed block-scaled formats
 * (MOE_SCALE_UE8M0_PACKED, MOE_SCALE_MXFP8) when H is a multiple of 256 and the step routes at
 * least 512 rows per expert on average (the tensor-bound regime, where an expert's tiles pair up
 * with little padding); the w13 GEMM stays on the one-CTA kernel (faster there as measured).
 * Returns the number of two-CTA clusters the w2 GEMM launches (> 0), 0 if the step takes the
 * one-CTA kernels, MOE_ERR_INVALID_ARG for a negative size, E or topk < 1 or an unknown format, or
 * an error code if no usable device is present (the cluster count is the device's: pairs of SMs
 * within a GPC). */
int moe_fp8_block_pair_path(int T, int H, int E, int topk, int scale_fmt);

/* Options of the layer: the expert weights' layout, the scale format of the activations
 * and of the requantised intermediate, and the GEMM kernels of small steps
 * (NULL options = MOE_WEIGHTS_NK, MOE_SCALE_F32, MOE_DECODE_AUTO).
 * MOE_WEIGHTS_NVFP4: w13 / w2 are moe_nvfp4_pack_weights outputs and w13_scale / w2_scale the
 * per-expert global scales [E] (moe_nvfp4_quant_weight); activations and the intermediate keep
 * their FP8 1x128 groups.  Both GEMMs then run on the decode-path kernel (decode_path
 * MOE_DECODE_OFF is rejected with MOE_ERR_INVALID_ARG), a step of more than 8 tokens 8 tokens
 * at a time (3 or 4 launches each); moe_fp8_block_workspace_size(T, ...) still suffices.  Shapes the
 * decode kernel cannot take give MOE_ERR_UNSUPPORTED_SHAPE.
 * MOE_SCALE_UE8M0_PACKED: w13_scale / w2_scale are the packed UE8M0 weight scales
 * (moe_fp8_block_pack_scales outputs, passed as const float*) and both GEMMs run on the block-scaled
 * MMA; the decode-path kernel does not take them (MOE_DECODE_AUTO then takes the tile GEMMs,
 * MOE_DECODE_ON and MOE_WEIGHTS_NVFP4 are rejected with MOE_ERR_INVALID_ARG). */
typedef struct moe_forward_options {
    int32_t weight_layout;            /* MOE_WEIGHTS_NK, MOE_WEIGHTS_TILED or MOE_WEIGHTS_NVFP4 */
    int32_t scale_fmt;                /* MOE_SCALE_F32, MOE_SCALE_UE8M0 or MOE_SCALE_UE8M0_PACKED */
    int32_t decode_path;              /* MOE_DECODE_AUTO, MOE_DECODE_OFF or MOE_DECODE_ON */
} moe_forward_options;

/* Number of kernels one moe_fp8_block_forward_ex with these routing parameters and options
 * (either may be NULL) launches (host only): on the tile path routing, the expert sort and
 * quantisation (one kernel for up to 512 routed pairs, four otherwise), the two grouped GEMMs
 * and the weighted sum; on the decode path the prologue, the decode kernel and the weighted sum,
 * plus the routing kernel when the decode kernel cannot route in every CTA (E > 256, or groups
 * the register-resident selection does not take), per 8 tokens with MOE_WEIGHTS_NVFP4.  0 when T == 0, -1 for
 * invalid sizes. */
int moe_fp8_block_forward_kernel_count_ex(int T, int H, int I, int E, int topk, const moe_routing_params* rp,
                                          const moe_forward_options* opts);

/* The same layer with options, optionally recording CUDA events between its stages for
 * per-stage timing (events: host array of MOE_FORWARD_NUM_EVENTS cudaEvent_t created by the
 * caller, recorded on `stream` in this order: before routing, before the expert
 * sort, before the activation quantisation, before the w13 GEMM, before the w2
 * GEMM, before the weighted unpermute-sum, after it), with options (may be NULL).
 * Other arguments and errors as moe_fp8_block_forward; events == NULL records none. */
#define MOE_FORWARD_NUM_EVENTS 7
int moe_fp8_block_forward_ex(const uint16_t* hidden, const float* router_logits,
                             const uint8_t* w13, const float* w13_scale,
                             const uint8_t* w2, const float* w2_scale,
                             int T, int H, int I, int E, int topk, int renormalize,
                             const moe_routing_params* rp, const moe_forward_options* opts,
                             void* workspace, size_t workspace_bytes, uint16_t* out, void* stream,
                             void* const* events);

/* ---- the masked batched layout -----------------------------------------------------
 * The expert MLP on rows already grouped by expert: hidden [E, max_tokens, H] bf16 with
 * counts[e] valid rows for expert e (the "[num_experts, max_tokens, hidden]" batched format
 * that low-latency expert-parallel dispatch produces, BatchedDeepGemmExperts, page
 * "Quantization and MoE Optimizations").  For every e and i < counts[e]:
 *   out[e, i, :] = bf16( w2-GEMM( requant( SiLU(gate) * up ( w13-GEMM( quant(hidden[e, i]) ) ) ) ) )
 * with the same 1x128 activation groups, 128x128 weight blocks and fp32 block-scale
 * promotion as moe_fp8_block_forward, and no router weight (the combine belongs to the
 * dispatcher).  Rows i >= counts[e] of out are not written.
 * counts: device int32 [E], read on the device (no host synchronisation); a count
 * outside [0, max_tokens] is clamped and sets MOE_STATUS_BAD_COUNT.
 * opts (may be NULL): the weights' layout and the scale format; hidden, w13, w2, out
 * 16-byte aligned; workspace of moe_fp8_block_masked_workspace_size bytes, 256-byte
 * aligned.  H, I multiples of 128, E <= 1024.  max_tokens == 0 or E == 0 is a no-op. */
size_t moe_fp8_block_masked_workspace_size(int E, int max_tokens, int H, int I);
int moe_fp8_block_forward_masked(const uint16_t* hidden, const int32_t* counts,
                                 const uint8_t* w13, const float* w13_scale,
                                 const uint8_t* w2, const float* w2_scale,
                                 int E, int max_tokens, int H, int I, const moe_forward_options* opts,
                                 void* workspace, size_t workspace_bytes, uint16_t* out, void* stream);

/* ---- status -------------------------------------------------------------------- */
/* Reads (and with clear != 0, resets) the device status word of the current
 * device into *status (host).  Synchronises the device. */
int moe_get_device_status(uint32_t* status, int clear);
/* Failure-detection check of the pipelines' bounded wait (every mbarrier wait of the GEMM and
 * decode kernels gives up after 2 s of device time, sets MOE_STATUS_WAIT_TIMEOUT in the status
 * word and lets its kernel return).  expire != 0: one such wait on a phase that nothing completes
 * runs out (about 2 s) and sets MOE_STATUS_WAIT_TIMEOUT; expire == 0: the phase is completed
 * first and the wait returns at once.  Nothing faults; the context stays usable.  Asynchronous
 * on `stream`; read the result with moe_get_device_status. */
int moe_selftest_bounded_wait(int expire, void* stream);
/* Human-readable name of a MOE_* return code. */
const char* moe_error_string(int code);
/* 1 if the current device can run these kernels (compute capability 10.3). */
int moe_device_supported(void);

#ifdef __cplusplus
}
#endif
#endif /* MOEFP8_H */
