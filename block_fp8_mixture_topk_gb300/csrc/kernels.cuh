// Host-side launchers of the sm_103a kernels (one translation unit each) and
// their once-per-device set-up.  All launchers are asynchronous on `stream`
// and return the launch's cudaError_t.
#pragma once

#include <utility>

#include "common.cuh"

namespace mfp8 {

// Launch on `stream` with programmatic stream serialisation allowed (the kernel must call
// grid_dependency_wait before touching data of earlier kernels).
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// route.cu
cudaError_t route_init_device();
cudaError_t launch_route_topk(const float* logits, int T, int E, int topk, int renormalize, int scoring,
                              int n_group, int topk_group, float routed_scaling, const float* bias, int32_t* ids,
                              float* weights, cudaStream_t stream);

// permute.cu
constexpr int kPermuteChunk = 1024;   // pairs per block of the counting / scatter kernels
cudaError_t permute_init_device();
int64_t permute_chunks(int64_t P);
cudaError_t launch_align_permute(const int32_t* ids, int64_t P, int E, int block_m, int32_t* expert_offsets,
                                 int32_t* padded_offsets, int32_t* sorted_pair_ids, int32_t* pos,
                                 int32_t* tile_expert, int32_t* tile_row0, int32_t* num_tiles,
                                 int32_t* chunk_counts, uint32_t* status, cudaStream_t stream);

// The most routed rows per expert the decode-path kernel takes (a step of at most 8 tokens).
constexpr int kDecodeCols = 8;

// prologue.cu: expert sort + scattering quantisation of a small batch in one launch
constexpr int kSmallPairs = 512;   // routed pairs the one-block path takes
cudaError_t launch_sort_quant_small(const int32_t* ids, int P, int E, int block_m, int32_t* expert_offsets,
                                    int32_t* padded_offsets, int32_t* sorted_pair_ids, int32_t* pos,
                                    int32_t* tile_expert, int32_t* tile_row0, int32_t* num_tiles, uint32_t* status,
                                    const uint16_t* x, int T, int H, int topk, uint8_t* q, int64_t q_ld, float* s,
                                    int64_t s_rs, int64_t s_gs, int scale_fmt, cudaStream_t stream,
                                    uint8_t* sf = nullptr);
// prologue.cu: the decode path's prologue (1 <= T <= kDecodeCols): counters[0, ncounters) zeroed,
// the T tokens' 1x128 groups quantised into `copies` copies of token-major rows q [copy][T][H] and
// scales s [copy][H/128][kDecodeCols]; lets the decode kernel launch before it ends
cudaError_t launch_decode_prologue(const uint16_t* x, int T, int H, int copies, uint8_t* q, float* s,
                                   int32_t* counters, int ncounters, int scale_fmt, cudaStream_t stream);

// masked.cu: row maps and tile table of the masked batched layout [E, M, H] (Mp = M rounded
// up to 128): row_map [E*Mp] (input row or -1), pos [E*M] (padded row or -1), ones [E*M]
cudaError_t launch_masked_map(const int32_t* counts, int E, int M, int Mp, int32_t* row_map, int32_t* pos,
                              float* ones, int32_t* tile_expert, int32_t* tile_row0, int32_t* num_tiles,
                              uint32_t* status, cudaStream_t stream);

// quant.cu
// 1x128 group quantisation of bf16 rows.  Row r of x goes to output row r, or
// (when pos != null) to output rows pos[r*topk + j], j < topk, skipping -1.
// Scale of (output row o, group g) is stored at s[o*s_row_stride + g*s_group_stride].
// s may be null (no fp32 scales); sf != null: the scales (then rounded up to powers of two,
// MOE_SCALE_UE8M0) also go out as UE8M0 bytes in packed scale-factor tiles (packed_sf_offset,
// ceil(cols/512) tiles per 128 output rows).
// scale_fmt MOE_SCALE_MXFP8: groups of 32 with UE8M0 scales (s then unused; s8: the scale bytes
// [out rows, cols/32]; sf: packed tiles of the 32-group columns, cols/128 tiles per 128 rows).
cudaError_t launch_group_quant(const uint16_t* x, int64_t rows, int cols, int64_t ld, uint8_t* q, int64_t q_ld,
                               float* s, int64_t s_row_stride, int64_t s_group_stride, const int32_t* pos,
                               int topk, int scale_fmt, cudaStream_t stream, uint8_t* sf = nullptr,
                               uint8_t* s8 = nullptr);
// UE8M0 bytes s [rows, C] -> packed scale-factor tiles (packed_sf_offset(r, c, ceil(C/4)))
cudaError_t launch_pack_scale_bytes(const uint8_t* s, int64_t rows, int C, uint8_t* out, cudaStream_t stream);
// [E, N/128, K/128] power-of-two block scales -> [E][N/128][ceil(K/512)] scale-factor tiles (out
// 16-byte aligned); a scale that is not a positive power of two sets MOE_STATUS_BAD_SCALE
cudaError_t launch_pack_scales(const float* s, int E, int N, int K, uint8_t* out, uint32_t* status,
                               cudaStream_t stream);
cudaError_t launch_block_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, float* s, int scale_fmt,
                                      cudaStream_t stream);
// [E, N, K] e4m3 -> [E][N/128][K/128][128][128] (each 128x128 block contiguous)
cudaError_t launch_pack_weights(const uint8_t* w, int E, int N, int K, uint8_t* packed, cudaStream_t stream);
// out[t] = bf16(sum_j y[pos[t*topk + j]]) in j order (H multiple of 4, y / out 16- / 8-byte aligned)
cudaError_t launch_unpermute_sum(const float* y, int64_t y_rows, const int32_t* pos, int64_t T, int topk, int H,
                                 uint16_t* out, uint32_t* status, cudaStream_t stream);
// out[t] = bf16(sum_j float(y[t*topk + j])) in j order over the pairs with pos >= 0
// (y bf16 [T*topk, H] in pair order; H multiple of 8, y / out 16-byte aligned)
cudaError_t launch_combine_pairs(const uint16_t* y, const int32_t* pos, int64_t T, int topk, int H, uint16_t* out,
                                 cudaStream_t stream);

// nvfp4.cu: NVFP4 expert weights (codes [E, N, K/2], e4m3 block scales [E, N, K/16], per-expert
// 1 / global_scale [E]) and their packed form for the decode kernel: [E][N/16][K/128] units of
// kFp4UnitBytes = 16 rows x 64 code bytes, then 16 rows x 8 scale bytes
constexpr int kFp4UnitBytes = 16 * 64 + 16 * 8;
cudaError_t launch_nvfp4_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, uint8_t* sf, float* gs,
                                      cudaStream_t stream);
size_t nvfp4_packed_bytes(int E, int N, int K);
cudaError_t launch_nvfp4_pack(const uint8_t* q, const uint8_t* sf, int E, int N, int K, uint8_t* packed,
                              cudaStream_t stream);

// selftest.cu: one bounded pipeline wait that expires (expire != 0) or completes at once
cudaError_t launch_bounded_wait_check(int expire, uint32_t* status, cudaStream_t stream);

// gemm.cu
struct GemmArgs {
    const uint8_t* A;
    const float* a_scale;
    int64_t as_row_stride, as_kb_stride;
    int64_t a_rows;
    int a_box_rows;            // rows of A loaded per tile: 128, or 32 when no tile has real rows past 32
    const uint8_t* B;
    int b_tiled;               // B in the tile-packed layout (moe_fp8_block_pack_weights)
    const float* b_scale;
    int N, K, E;
    const int32_t* tile_expert;
    const int32_t* tile_row0;
    const int32_t* num_tiles;
    int64_t max_tiles;
    // optional [E + 1] padded row offsets of a tile table whose tiles are the experts' padded rows
    // in order (tile m = rows [128m, 128m + 128)): lets the SiLU-epilogue GEMM visit an expert's
    // few tiles column by column (see item_of in gemm.cu); nullptr, and the other epilogues, keep
    // the tile-by-tile order
    const int32_t* padded_offsets;
    // optional [E + 1] offsets of each expert's real rows and of its padded rows in the sorted layout
    // (the sort places an expert's real rows first in its padded region): the epilogues then take a
    // tile's real rows from them, cached per work item, instead of loading sorted_pair_ids for
    // every row at the start of an item
    const int32_t* row_offsets;
    const int32_t* row_padded;
    int epi;
    float* out_f32;
    uint8_t* out_q;
    float* out_scale;
    int64_t os_row_stride, os_kb_stride;
    const int32_t* sorted_pair_ids;
    const float* topk_weights;
    int topk;
    int64_t num_pairs;
    uint16_t* out_bf16;
    int scale_fmt;             // MOE_SCALE_*: the SiLU epilogue's requantisation scales
    // packed UE8M0 scale factors (sf_packed != 0): the block-scaled kernel, with scale-factor tiles
    // (common.cuh, packed_sf_offset) instead of fp32 scales.  a_sf: A's, ceil(K/512) tiles per 128
    // rows (tiles start at row 0: tile_row0 must be a multiple of 128); b_sf: B's, [E][N/128]
    // [ceil(K/512)] tiles; out_sf: the SiLU epilogue's requantisation scales, ceil(N/1024) tiles
    // per 128 rows.  a_scale, b_scale and out_scale are then unused.
    int sf_packed;             // 1: packed UE8M0 (4 K blocks per word); 2: MXFP8 (4 32-groups per word, one tile per K block)
    const uint8_t* a_sf;
    const uint8_t* b_sf;
    uint8_t* out_sf;
    // non-null (with sf_packed and the weighted-pairs epilogue): the CTA-pair kernel (gemm.cu),
    // whose items are two consecutive tiles of one expert; [E + 1] padded row offsets of the tile
    // table (tile m = rows [128m, 128m + 128)).  Needs N % 256 == 0 and a_box_rows == 128.
    const int32_t* pair_offsets;
    uint32_t* status;
};
cudaError_t gemm_init_device();
// Clusters of two CTAs of the pair GEMM kernel that are resident at once (0 if it cannot run).
int gemm_pair_clusters();
// Tensor map of a 2-D byte matrix [rows, cols] (row stride = cols bytes), boxes of
// box_cols x box_rows, with the 128-byte swizzle or none.
cudaError_t encode_u8_map(CUtensorMap* map, const uint8_t* ptr, int64_t cols, int64_t rows, uint32_t box_cols,
                          uint32_t box_rows, bool swizzle128);
// Tensor map of a byte tensor of `rank` dimensions (dims[0] innermost; strides[i] = bytes between
// consecutive indices of dimension i+1), boxes `box`, with the 128-byte swizzle (box[0] = 128,
// destinations 1024-byte aligned: 16-byte chunk c of the 128-byte row at shared address A lands
// at chunk c ^ ((A / 128) % 8)) or none.
cudaError_t encode_u8_map_nd(CUtensorMap* map, const uint8_t* ptr, int rank, const uint64_t* dims,
                             const uint64_t* strides, const uint32_t* box, bool swizzle128);

// decode.cu: both expert GEMMs of a step with at most 8 rows per expert in one persistent
// launch, as weight-streaming work items of 32 weight rows (see decode.cu)
struct DecodeMlpArgs {
    const uint8_t* w13;        // [E, 2I, H] or tile-packed (w_fp4: NVFP4-packed)
    const float* w13_scale;    // [E, 2I/128, H/128] (w_fp4: the per-expert 1 / global_scale [E])
    const uint8_t* w2;         // [E, H, I] or tile-packed (w_fp4: NVFP4-packed)
    const float* w2_scale;     // [E, H/128, I/128] (w_fp4: [E])
    int w_tiled;
    int w_fp4;                 // NVFP4 weights in the packed layout of nvfp4.cu
    int H, I, E;
    // the step's routing: T tokens, topk pairs each (pair p = t * topk + j)
    int T, topk;
    int route_v;               // experts per lane of the in-kernel routing (1, 2, 4, 8), 0: ids / wts are inputs
    const float* logits;       // [T, E] router logits (route_v > 0)
    const float* bias;         // [E] selection bias or null
    int renormalize, scoring, n_group, topk_group, vec_loads;
    float routed_scaling;
    int32_t* ids;              // [P] chosen experts: written by CTA 0 (route_v > 0) or read
    float* wts;                // [P] router weights: likewise
    int32_t* pos;              // [P] written by CTA 0: the pair's padded row, -1 for a dropped pair
    const uint8_t* a1;         // activation codes: x_copies copies of the T token rows [copy][T][H]
    const float* a1s;          // their scales [copy][H/128][kDecodeCols] (the decode prologue's)
    int x_copies;
    uint8_t* a2;               // requantised intermediate [rows, I]: tile m's j-th row at padded row m*128 + j
    float* a2s;                // its scales [I/128][rows]
    int64_t rows;
    int max_tiles;             // >= the step's tiles (one per touched expert)
    int cols;                  // the most routed rows an expert can hold, 1..8 (decode_cols: T)
    float* h;                  // h = silu(gate) * up [P, I] fp32 by pair
    int32_t* counters;         // decode_counters(max_tiles, I) ints, zero on entry
    int scale_fmt;
    uint16_t* y;               // [P, H] bf16 = router weight * C2 in pair order
    uint32_t* status;
    int stages, stage_bytes;   // ring geometry (set by launch_decode_mlp)
};
// the most rows an expert holds in a step of T tokens, as the decode kernel takes it (0: T too
// large for it)
int decode_cols(int T);
// tile records a decode CTA can hold in shared memory
size_t decode_max_tiles();
// ints of the decode kernel's counters: per-(tile, group) counts, per-tile ready counts, the ticket
int64_t decode_counters(int max_tiles, int I);
cudaError_t decode_init_device();
cudaError_t launch_decode_mlp(const DecodeMlpArgs& args, int num_sms, cudaStream_t stream);

// api.cu: once-per-device set-up; on MOE_OK, *status = the device status word's address
int device_status_word(uint32_t** status);
cudaError_t launch_grouped_gemm(const GemmArgs& args, int num_sms, cudaStream_t stream);

}  // namespace mfp8
