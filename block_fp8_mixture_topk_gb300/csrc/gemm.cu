// Grouped block-FP8 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// C[r, n] = sum_kb a_scale[r, kb] * b_scale[e, n/128, kb] * sum_{k in kb} A[r, k] * B[e, n, k]
//
// The weights of an expert are "[num_experts, N, K]" with 128x128 blocks
// (page "Quantization and MoE Optimizations", sections FusedMoE Class and
// Fp8Config); the activations carry one scale per 1x128 group.  Each CTA tile is
// 128 sorted rows of one expert (the "sorted token" pattern, section Triton
// Fused MoE Kernel) by 256 output columns.  Because the scales change with
// every 128-wide K block and are fp32 (not the power-of-two scales of the
// hardware block-scaled MMA), every K block is accumulated by the tensor cores
// into its own TMEM buffer and then "promoted": the epilogue warps read it,
// multiply by a_scale * b_scale and add it to fp32 register accumulators.  Two
// TMEM buffers (2 x 256 columns) let the MMA of block kb+1 run while block kb
// is promoted.  (The pages' Triton kernel dequantises after the K loop, which is
// exact only for per-tensor / per-channel scales; blockwise scales vary along K.)
//
// Roles (384 threads, one CTA per SM, persistent over the tile list):
//   warp 0, one thread : TMA producer, 4-stage ring of {A 128x128, B 256x128} e4m3 tiles
//   warp 1, one thread : MMA issuer (4 x tcgen05.mma 128x256x32 per K block), TMEM owner
//   warp 2             : scale producer, an 8-slot ring of each K block's row and weight scales
//   warp 3             : idle (it completes warpgroup 0, which gives registers away)
//   warps 4..11        : promotion + epilogue; warp w reads TMEM lanes 32*(w%4)..+31
//                        (its rows) and 128 of the 256 columns (column half (w-4)/4)
// Epilogues:
//   store     : fp32 rows to out_f32
//   silu      : B tile = 128 gate rows + the 128 matching up rows; h = silu(g)*u in
//               fp32, amax of the 128-wide group exchanged between the two column
//               halves through shared memory, 1x128 e4m3 requantisation
//   scatter   : out_f32[token] += router_weight * C (float4 atomics)
//   rows      : out_f32[row] = router_weight * C in sorted-row order (plain stores); the
//               layer sums each token's k rows afterwards (moe_unpermute_sum), in a fixed order
//   pairs     : out_bf16[pair] = bf16(router_weight * C) in pair order (pair = t*topk + j), so
//               that a token's k rows are contiguous for the sum that follows (moe_combine_pairs)
// Every wait is bounded (mbar_wait); on expiry the CTA records
// MOE_STATUS_WAIT_TIMEOUT, waits (bounded) for its TMA loads and MMAs in flight,
// frees its TMEM and exits.
#include <mutex>

#include "kernels.cuh"

namespace mfp8 {

namespace {

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int STAGES = 4;
constexpr int A_TILE = BM * BK;        // 16 KB
constexpr int B_HALF = 128 * BK;       // 16 KB: 128 weight rows
constexpr int B_TILE = 2 * B_HALF;     // 32 KB: 256 weight rows
constexpr int NUM_EPI_WARPS = 8;
constexpr int FIRST_EPI_WARP = 4;       // warpgroup 0: TMA warp, MMA warp, two idle warps
constexpr int NUM_THREADS = (FIRST_EPI_WARP + NUM_EPI_WARPS) * 32;
// registers per thread: 168 at launch (384 threads).  Warpgroup 0 (the TMA, MMA and
// scale warps) gives some back and the two epilogue warpgroups take them: 128*c + 256*e
// <= 384*168.  The SiLU epilogue holds more live values (gate and up halves); the
// splits are the ones with the fewest spills.  A spill in a control warp is a local-memory
// round trip in the loop that feeds the tensor pipe; with most of the SM's L1 given to shared
// memory it can reach L2.
template <int EPI>
struct RegSplit {
    static constexpr uint32_t control = (EPI == MOE_EPI_SILU_MUL_QUANT) ? 72 : 120;
    static constexpr uint32_t epilogue = (EPI == MOE_EPI_SILU_MUL_QUANT) ? 216 : 184;
    static_assert(128 * control + 256 * epilogue <= 384 * 168, "register split over the launch budget");
};
// the block-scaled kernels (no promotion in the epilogue): the epilogues need fewer registers
// and the control warps more (the SiLU kernel spills nothing at 88 / 208, its control warps did at
// 72 / 216; the pair kernel spills nothing at 136 / 176, 8 / 48 bytes at 104 / 192)
template <int EPI>
struct RegSplitBs {
    static constexpr uint32_t control = (EPI == MOE_EPI_SILU_MUL_QUANT) ? 88 : 136;
    static constexpr uint32_t epilogue = (EPI == MOE_EPI_SILU_MUL_QUANT) ? 208 : 176;
    static_assert(128 * control + 256 * epilogue <= 384 * 168, "register split over the launch budget");
};
constexpr uint32_t TMEM_COLS = 512;    // two 256-column fp32 accumulators
constexpr int SR = 8;                  // slots of the scale ring (K blocks in flight)
constexpr int ITEMS = 256;             // work items of a CTA whose tile and column are cached in shared memory
constexpr int PAIR_TILES = 4;          // experts with at most this many tiles take their tiles column by column
constexpr int SCL = 132;               // floats per slot: 128 row scales, 2 weight-block scales, pad

struct SmemCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t amax_bar[2];
    uint64_t sfull[SR];                // scales of a K block landed (32 producer-lane arrivals)
    uint64_t sempty[SR];               // the epilogue warps have read them (8 arrivals)
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    float amax_x[2][2][BM];            // [tile parity][column half][row]
    alignas(16) float stage[NUM_EPI_WARPS][32 * 20];   // per-warp store staging: 32 rows x 16 floats (+4 pad)
    alignas(16) float scl[SR][SCL];    // scale ring: a_scale of the tile's 128 rows, then the two weight scales
    int item_n[ITEMS];                 // the CTA's work items (see item_of), in its visiting order: column block,
    int item_e[ITEMS];                 // the tile's expert,
    int item_r0[ITEMS];                // first row
    int item_live[ITEMS];              // and real rows (Tile::live)
};
constexpr int STAGE_ROW = 20;          // floats per staged row (80 B: conflict-free 16-byte slots)
constexpr size_t SMEM_BYTES = 1024 + STAGES * (A_TILE + B_TILE) + sizeof(SmemCtl);
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds the sm_103 limit");

struct Tile {
    int64_t row0;
    int e;
    int n;
    int bcol0, bcol1;
    int live;       // real rows of the tile (its first `live` rows), or -1: check sorted_pair_ids
    bool has1;
    bool ok;
};

// Work item w -> (tile m, column block n).  Without expert offsets: m = w / NT, n = w % NT, so
// consecutive CTAs take the column blocks of one tile and share its A rows in L2.  With them,
// the items of an expert whose rows fill c <= PAIR_TILES tiles (its items are w in [f*NT,
// (f+c)*NT) either way, f its first tile) go column by column: n = l / c, m = f + l % c for
// l = w - f*NT, so that its c tiles read each weight block one after the other and the block
// is still in L2 for the second (an expert with 129-256 rows otherwise streamed its weights
// twice when N is large); experts with more tiles keep the tile-by-tile order.
__device__ __forceinline__ void item_of(const GemmArgs& a, int64_t w, int NT, int& m, int& n) {
    const int64_t mt = w / NT;
    m = static_cast<int>(mt);
    n = static_cast<int>(w - mt * NT);
    if (!a.padded_offsets) return;
    const int e = a.tile_expert[mt];
    if (e < 0 || e >= a.E) return;
    const int f = a.padded_offsets[e] / BM;
    const int c = (a.padded_offsets[e + 1] - a.padded_offsets[e]) / BM;
    if (c < 2 || c > PAIR_TILES || mt < f || mt >= f + c) return;
    const int64_t l = w - static_cast<int64_t>(f) * NT;
    n = static_cast<int>(l / c);
    m = f + static_cast<int>(l - static_cast<int64_t>(n) * c);
}

// The w2 GEMM's (router-weighted pair rows) last wave: when its R = total mod gridDim items would
// keep at most half of the CTAs busy, each of them runs as two 128-column half items, so that 2R
// SMs stream half an item's weights each instead of R SMs a whole item's (Mixtral-shaped layer:
// ~190 items of 112 K blocks on 152 SMs).  Only when every unit is among the items the CTAs cache
// (fill_item_cache), so that decode_tile's lookup of a later item never meets a half item.
// Returns R, or 0 for no split.
template <int EPI>
__device__ __forceinline__ int64_t tail_halves(const GemmArgs& a, int64_t total) {
    if constexpr (EPI != MOE_EPI_WEIGHTED_PAIRS_BF16) {
        return 0;
    } else {
        if (a.N % 256 != 0) return 0;
        const int64_t G = gridDim.x, R = total % G;
        return (R > 0 && 2 * R <= G && total + R <= static_cast<int64_t>(ITEMS) * G) ? R : 0;
    }
}

// Unit w of the non-SiLU GEMMs -> tile m and column block n (256 columns), or for a half item of
// the split last wave n = -(128-column band + 1).  Units: total - halves whole items, then two
// units for each of the last `halves` items.
__device__ __forceinline__ void unit_of(int64_t w, int NT, int64_t total, int64_t halves, int& m, int& n) {
    if (halves > 0 && w >= total - halves) {
        const int64_t h = w - (total - halves);
        const int64_t item = total - halves + (h >> 1);
        const int64_t mt = item / NT;
        m = static_cast<int>(mt);
        n = -(2 * static_cast<int>(item - mt * NT) + static_cast<int>(h & 1) + 1);
    } else {
        const int64_t mt = w / NT;
        m = static_cast<int>(mt);
        n = static_cast<int>(w - mt * NT);
    }
}

template <int EPI, class Ctl>
__device__ __forceinline__ Tile decode_tile(const GemmArgs& a, const Ctl* ctl, int64_t k, int64_t w, int NT) {
    Tile t;
    if (k < ITEMS) {
        // cached at the kernel's start: no global load at an item boundary
        t.n = ctl->item_n[k];
        t.e = ctl->item_e[k];
        t.row0 = ctl->item_r0[k];
        t.live = ctl->item_live[k];
    } else {
        // (past the cached items there are no half items: tail_halves)
        int m, n;
        if constexpr (EPI != MOE_EPI_SILU_MUL_QUANT) {
            m = static_cast<int>(w / NT);
            n = static_cast<int>(w - static_cast<int64_t>(m) * NT);
        } else {
            item_of(a, w, NT, m, n);
        }
        t.n = n;
        t.e = a.tile_expert[m];
        t.row0 = a.tile_row0[m];
        t.live = -1;
    }
    t.ok = t.e >= 0 && t.e < a.E && t.row0 >= 0 && t.row0 + BM <= a.a_rows;
    // the packed scale-factor tiles of A cover rows 128q .. 128q + 127
    if (a.sf_packed && (t.row0 & (BM - 1))) t.ok = false;
    if (EPI == MOE_EPI_SILU_MUL_QUANT) {
        t.bcol0 = t.n * 128;
        t.bcol1 = a.N / 2 + t.n * 128;
        t.has1 = true;
    } else if (t.n >= 0) {
        t.bcol0 = t.n * 256;
        t.bcol1 = t.bcol0 + 128;
        t.has1 = t.bcol1 < a.N;
    } else {
        t.bcol0 = (-t.n - 1) * 128;   // a half item of the split last wave
        t.bcol1 = t.bcol0 + 128;
        t.has1 = false;
    }
    return t;
}

// Both 128-row weight bands of a work item for K block kb in one 32 KB TMA box (rows bcol0 .. +127
// land first, rows bcol1 .. +127 16 KB later, as two 128-row boxes would put them): an SM streams
// many more bytes per second with fewer, larger boxes (a probe with every SM streaming L2-resident
// tiles: 79 GB/s per SM with three 16 KB boxes per stage, 125 GB/s with two 32 KB boxes).  The box
// steps from one band to the other with its outermost dimension (map: make_pair_map).
//   silu:   gate band n and up band N/256 + n of expert e
//   others: bands 2n and 2n + 1
template <int EPI>
__device__ __forceinline__ void load_b_pair(uint32_t dst, const CUtensorMap* m, const GemmArgs& a, const Tile& t,
                                            int kb, uint32_t bar) {
    if constexpr (EPI == MOE_EPI_SILU_MUL_QUANT) {
        if (a.b_tiled)
            tma_load_5d(dst, m, 0, 0, kb, t.n, 2 * t.e, bar);
        else
            tma_load_4d(dst, m, kb * BK, 0, t.n, 2 * t.e, bar);
    } else {
        if (a.b_tiled)
            tma_load_4d(dst, m, 0, 0, kb, t.e * (a.N / 128) + 2 * t.n, bar);
        else
            tma_load_2d(dst, m, kb * BK, t.e * a.N + t.n * 256, bar);
    }
}

// This CTA's first ITEMS work items (w = blockIdx.x + k * gridDim.x): tile, column block, expert
// and first row looked up once (all threads, one round of global loads), so that no role waits on
// a global load when it starts an item.  Only the w13 GEMM reorders (item_of); the w2 GEMM keeps the
// tile-by-tile order (its column blocks of one expert run in the same wave for the shapes served,
// and the reorder gained nothing measurable there).
template <int EPI, class Ctl>
__device__ __forceinline__ void fill_item_cache(const GemmArgs& a, Ctl* ctl, int64_t total, int64_t halves, int NT) {
    for (int64_t k = threadIdx.x; k < ITEMS; k += blockDim.x) {
        const int64_t w = blockIdx.x + k * gridDim.x;
        if (w >= total + halves) break;
        int m, n;
        if constexpr (EPI == MOE_EPI_SILU_MUL_QUANT) {
            item_of(a, w, NT, m, n);
        } else {
            unit_of(w, NT, total, halves, m, n);
        }
        const int e = a.tile_expert[m];
        const int32_t r0 = a.tile_row0[m];
        int live = -1;
        if (a.row_offsets && a.row_padded && e >= 0 && e < a.E) {
            const int64_t l = static_cast<int64_t>(a.row_offsets[e + 1]) - a.row_offsets[e] - (r0 - a.row_padded[e]);
            live = static_cast<int>(l < 0 ? 0 : (l > BM ? BM : l));
        }
        ctl->item_n[k] = n;
        ctl->item_e[k] = e;
        ctl->item_r0[k] = r0;
        ctl->item_live[k] = live;
    }
}

// The epilogue of one finished work item, run by each of the 8 epilogue warps on its share:
// acc holds the warp's 32 rows (TMEM lane quarter sp, row = sp * 32 + lane) by 128 columns
// (silu: gate columns g*64 .. +63 in acc[0, 64) and the matching up columns in acc[64, 128);
// otherwise columns g*128 .. +127 of the tile).  SiLU(gate)*up with 1x128 requantisation (the
// group amax exchanged between the two column halves through shared memory; with sf_packed the
// scale goes out as its UE8M0 byte in packed tiles), or the router-weighted / plain row stores.
// Returns false if the amax exchange's wait gave up.
template <int EPI, class Ctl>
__device__ __forceinline__ bool finish_item(const GemmArgs& a, Ctl* ctl, const Tile& t, float* acc, int warp, int lane,
                                            int g, int row, int64_t grow, bool active, uint32_t tile_iter,
                                            volatile int* abort_flag) {
    const int sp = warp & 3;
    if (EPI == MOE_EPI_SILU_MUL_QUANT && a.sf_packed == 2) {
        // MXFP8: this thread's 64 values are two whole 1x32 groups of its row; no exchange
        uint4* dst = reinterpret_cast<uint4*>(a.out_q + grow * (a.N / 2) + t.n * 128 + g * 64);
#pragma unroll
        for (int hg = 0; hg < 2; ++hg) {
            float amax = 0.0f;
#pragma unroll
            for (int j = hg * 32; j < hg * 32 + 32; ++j) {
                const float gate = acc[j];
                const float h = __fdividef(gate * acc[64 + j], 1.0f + __expf(-gate));
                acc[j] = h;
                amax = fmaxf(amax, fabsf(h));
            }
            const float sc = group_scale_fmt(amax, MOE_SCALE_UE8M0);
            const float rsc = __frcp_rn(sc);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t wv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float* h = acc + hg * 32 + c * 16 + j * 4;
                    const uint32_t lo = e4m3x2(div_by_scale(h[0], sc, rsc), div_by_scale(h[1], sc, rsc));
                    const uint32_t hi = e4m3x2(div_by_scale(h[2], sc, rsc), div_by_scale(h[3], sc, rsc));
                    wv[j] = lo | (hi << 16);
                }
                dst[hg * 2 + c] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
            a.out_sf[packed_sf_offset(grow, t.n * 4 + g * 2 + hg, a.N / 256)] = ue8m0_byte(sc);
        }
    } else if (EPI == MOE_EPI_SILU_MUL_QUANT) {
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            // silu(g) * u = g * u / (1 + e^-g); its fp32 rounding is not part of the
            // definition (the requantised bytes are compared within one code)
            const float gate = acc[j];
            const float h = __fdividef(gate * acc[64 + j], 1.0f + __expf(-gate));
            acc[j] = h;
            amax = fmaxf(amax, fabsf(h));
        }
        const uint32_t par = tile_iter & 1u;
        ctl->amax_x[par][g][row] = amax;
        mbar_arrive(smem_addr(&ctl->amax_bar[par]));
        if (!mbar_wait(smem_addr(&ctl->amax_bar[par]), (tile_iter >> 1) & 1u, abort_flag, a.status)) return false;
        amax = fmaxf(ctl->amax_x[par][0][row], ctl->amax_x[par][1][row]);
        const float sc = group_scale_fmt(amax, a.sf_packed ? MOE_SCALE_UE8M0 : a.scale_fmt);
        const float rsc = __frcp_rn(sc);
        uint4* dst = reinterpret_cast<uint4*>(a.out_q + grow * (a.N / 2) + t.n * 128 + g * 64);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float* h = acc + c * 16 + j * 4;
                const uint32_t lo = e4m3x2(div_by_scale(h[0], sc, rsc), div_by_scale(h[1], sc, rsc));
                const uint32_t hi = e4m3x2(div_by_scale(h[2], sc, rsc), div_by_scale(h[3], sc, rsc));
                wv[j] = lo | (hi << 16);
            }
            dst[c] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        if (g == 0) {
            if (a.sf_packed)
                a.out_sf[packed_sf_offset(grow, t.n, (a.N / 256 + 3) / 4)] = ue8m0_byte(sc);
            else
                a.out_scale[grow * a.os_row_stride + static_cast<int64_t>(t.n) * a.os_kb_stride] = sc;
        }
    } else if (EPI == MOE_EPI_WEIGHTED_SCATTER) {
        if (active) {
            const int32_t pair = a.sorted_pair_ids[grow];
            if (pair >= 0 && pair < a.num_pairs) {
                const int64_t tok = pair / a.topk;
                const float wgt = a.topk_weights[pair];
                float* dst = a.out_f32 + tok * a.N + t.bcol0 + g * 128;
#pragma unroll
                for (int j = 0; j < 128; j += 4)
                    atomicAdd(reinterpret_cast<float4*>(dst + j),
                              make_float4(wgt * acc[j], wgt * acc[j + 1], wgt * acc[j + 2], wgt * acc[j + 3]));
            }
        }
    } else if (EPI == MOE_EPI_WEIGHTED_PAIRS_BF16) {
        // bf16 rows (times the router weight) to out_bf16[pair], through a per-warp
        // staging buffer of 32 rows x 32 columns (64 B per row, 16-byte chunks swizzled
        // by row so that both the row-wise writes and the column-wise reads are free
        // of bank conflicts): each store instruction covers 8 rows x 64 contiguous bytes
        if (active) {
            const int32_t pair = a.sorted_pair_ids[grow];
            const bool keep = pair >= 0 && pair < a.num_pairs;
            const float wgt = keep ? a.topk_weights[pair] : 0.0f;
            const uint32_t keep_mask = __ballot_sync(0xffffffffu, keep);
            uint32_t* stg = reinterpret_cast<uint32_t*>(ctl->stage[warp - FIRST_EPI_WARP]);
            const int r_out = lane >> 2, q_out = lane & 3;
            uint16_t* dst[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t p = __shfl_sync(0xffffffffu, pair, i * 8 + r_out);
                dst[i] = a.out_bf16 + p * a.N + t.bcol0 + g * 128 + q_out * 8;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float* v = acc + c * 32 + q * 8;
                    const int slot = q ^ ((lane >> 1) & 3);
                    *reinterpret_cast<uint4*>(stg + lane * 16 + slot * 4) =
                        make_uint4(bf16x2(wgt * v[0], wgt * v[1]), bf16x2(wgt * v[2], wgt * v[3]),
                                   bf16x2(wgt * v[4], wgt * v[5]), bf16x2(wgt * v[6], wgt * v[7]));
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = i * 8 + r_out;
                    const int slot = q_out ^ ((r >> 1) & 3);
                    const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 16 + slot * 4);
                    if ((keep_mask >> r) & 1u) *reinterpret_cast<uint4*>(dst[i] + c * 32) = v;
                }
                __syncwarp();
            }
        }
    } else {
        // fp32 rows (times the router weight for the rows epilogue) written through a
        // per-warp staging buffer, 16 columns at a time, so that each store instruction
        // covers 8 rows x 64 contiguous bytes instead of 32 rows x 16 bytes
        if (active) {
            bool keep = true;
            float wgt = 1.0f;
            if (EPI == MOE_EPI_WEIGHTED_ROWS) {
                const int32_t pair = a.sorted_pair_ids[grow];
                keep = pair >= 0 && pair < a.num_pairs;
                wgt = keep ? a.topk_weights[pair] : 0.0f;
            }
            const uint32_t keep_mask = __ballot_sync(0xffffffffu, keep);
            float* stg = ctl->stage[warp - FIRST_EPI_WARP];
            const int r_out = lane >> 2, q_out = lane & 3;
            float* gbase = a.out_f32 + (t.row0 + sp * 32) * a.N + t.bcol0 + g * 128 + q_out * 4;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float* v = acc + c * 16 + q * 4;
                    *reinterpret_cast<float4*>(stg + lane * STAGE_ROW + q * 4) =
                        make_float4(wgt * v[0], wgt * v[1], wgt * v[2], wgt * v[3]);
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = i * 8 + r_out;
                    const float4 v = *reinterpret_cast<const float4*>(stg + r * STAGE_ROW + q_out * 4);
                    if ((keep_mask >> r) & 1u)
                        *reinterpret_cast<float4*>(gbase + static_cast<int64_t>(r) * a.N + c * 16) = v;
                }
                __syncwarp();
            }
        }
    }
    return true;
}

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmB2, const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* smA = base;
    uint8_t* smB = base + STAGES * A_TILE;
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smB + STAGES * B_TILE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (EPI == MOE_EPI_SILU_MUL_QUANT) ? a.N / 256 : (a.N + 255) / 256;
    const int KB = a.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            mbar_init(smem_addr(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&ctl->tfull[b]), 1);
            mbar_init(smem_addr(&ctl->tempty[b]), NUM_EPI_WARPS);
            mbar_init(smem_addr(&ctl->amax_bar[b]), NUM_EPI_WARPS * 32);
        }
        for (int r = 0; r < SR; ++r) {
            mbar_init(smem_addr(&ctl->sfull[r]), 32);
            mbar_init(smem_addr(&ctl->sempty[r]), NUM_EPI_WARPS);
        }
        mbar_init(smem_addr(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmB2);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the set-up above overlaps the previous kernel's tail; its outputs are read from here on
    grid_dependency_wait();
    int64_t ntiles = *a.num_tiles;
    if (ntiles < 0) ntiles = 0;
    if (ntiles > a.max_tiles) ntiles = a.max_tiles;
    const int64_t total = ntiles * NT;
    const int64_t halves = tail_halves<EPI>(a, total);
    const int64_t units = total + halves;
    fill_item_cache<EPI>(a, ctl, total, halves, NT);
    __syncthreads();
    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort_flag;
    if (warp < FIRST_EPI_WARP) {
      regs_decrease<RegSplit<EPI>::control>();
      if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            // one thread, nothing but the tile loads: the 4-stage ring refills as soon as
            // the MMAs release a stage
            int stage = 0;
            uint32_t phase = 0, issued = 0;
            bool ok = true;
            int64_t k = 0;
            for (int64_t w = blockIdx.x; w < units && ok; w += gridDim.x, ++k) {
                const Tile t = decode_tile<EPI>(a, ctl, k, w, NT);
                if (!t.ok) {
                    status_set(a.status, MOE_STATUS_BAD_EXPERT_ID);
                    continue;
                }
                // weight tile coordinates: [E*N, K] rows in the pages' layout (x advances along
                // K), or one 128-row block per 128 map rows in the tile-packed layout (each
                // 128x128 block a contiguous 16 KB, consecutive K blocks adjacent: y advances)
                int32_t by0, bdx, bdy;
                if (a.b_tiled) {
                    by0 = ((t.e * (a.N / 128) + t.bcol0 / 128) * KB) * 128;
                    bdx = 0;
                    bdy = 128;
                } else {
                    by0 = t.e * a.N + t.bcol0;
                    bdx = BK;
                    bdy = 0;
                }
                // decode tiles (a_box_rows = 32): only the first 32 rows of A hold real rows;
                // the MMA reads whatever rows 32..127 of the stage hold, for padding rows only
                const uint32_t bytes = a.a_box_rows * BK + (t.has1 ? B_TILE : B_HALF);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_addr(&ctl->full[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    tma_load_2d(smem_addr(smA + stage * A_TILE), &tmA, kb * BK, static_cast<int32_t>(t.row0), fb);
                    if (t.has1)
                        load_b_pair<EPI>(smem_addr(smB + stage * B_TILE), &tmB2, a, t, kb, fb);
                    else
                        tma_load_2d(smem_addr(smB + stage * B_TILE), &tmB, kb * bdx, by0 + kb * bdy, fb);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let every tile load already issued land before the CTA exits
                for (int s = 0; s < STAGES; ++s) {
                    const uint32_t n_s = (issued + STAGES - 1 - s) / STAGES;
                    if (n_s > 0) mbar_wait(smem_addr(&ctl->full[s]), (n_s - 1) & 1u, nullptr, a.status);
                }
            }
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------------- scale producer
        // all 32 lanes copy each K block's scales (the tile's 128 row scales and its two
        // weight-block scales) into the scale ring with cp.async, so that the epilogue
        // reads them from shared memory
        const bool vec = a.as_row_stride == 1 && (a.as_kb_stride & 3) == 0 &&
                         (reinterpret_cast<uintptr_t>(a.a_scale) & 15) == 0;
        const int NBn = a.N / 128;
        uint32_t q = 0;
        bool ok = true;
        int64_t k = 0;
        for (int64_t w = blockIdx.x; w < units && ok; w += gridDim.x, ++k) {
            const Tile t = decode_tile<EPI>(a, ctl, k, w, NT);
            if (!t.ok) continue;
            const int nb0 = (EPI == MOE_EPI_SILU_MUL_QUANT) ? t.n : t.bcol0 / 128;
            const int nb1 = (EPI == MOE_EPI_SILU_MUL_QUANT) ? NBn / 2 + t.n : (t.has1 ? nb0 + 1 : nb0);
            const float* bsa = a.b_scale + (static_cast<int64_t>(t.e) * NBn + nb0) * KB;
            const float* bsb = a.b_scale + (static_cast<int64_t>(t.e) * NBn + nb1) * KB;
            const float* asr = a.a_scale + t.row0 * a.as_row_stride;
            for (int kb = 0; kb < KB; ++kb) {
                const uint32_t slot = q % SR, use = q / SR;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->sempty[slot]), (use & 1u) ^ 1u,
                                                       abort_flag, a.status))) {
                    ok = false;
                    break;
                }
                const uint32_t dst = smem_addr(&ctl->scl[slot][0]);
                const float* src = asr + static_cast<int64_t>(kb) * a.as_kb_stride;
                if (vec) {
                    cp_async_16(dst + lane * 16, src + lane * 4);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        cp_async_4(dst + (lane * 4 + i) * 4, src + (lane * 4 + i) * a.as_row_stride);
                }
                if (lane == 0) cp_async_4(dst + 128 * 4, bsa + kb);
                if (lane == 1) cp_async_4(dst + 129 * 4, bsb + kb);
                cp_async_arrive(smem_addr(&ctl->sfull[slot]));
                ++q;
            }
        }
        cp_async_wait_all();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            const uint32_t idesc_full = idesc_e4m3_f32(BM, 256);
            const uint32_t idesc_half = idesc_e4m3_f32(BM, 128);
            int stage = 0;
            uint32_t phase = 0, buf = 0, bphase = 0;
            bool ok = true;
            int64_t k = 0;
            for (int64_t w = blockIdx.x; w < units && ok; w += gridDim.x, ++k) {
                const Tile t = decode_tile<EPI>(a, ctl, k, w, NT);
                if (!t.ok) continue;
                const uint32_t idesc = t.has1 ? idesc_full : idesc_half;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_addr(&ctl->tempty[buf]), bphase ^ 1u, abort_flag, a.status) ||
                        !mbar_wait(smem_addr(&ctl->full[stage]), phase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_addr(smA + stage * A_TILE);
                    const uint32_t b0 = smem_addr(smB + stage * B_TILE);
                    const uint32_t d = tmem + buf * 256;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_e4m3(d, smem_desc_k128_sw128(a0 + k * 32), smem_desc_k128_sw128(b0 + k * 32), idesc,
                                 k > 0 ? 1u : 0u);
                    mma_commit(smem_addr(&ctl->empty[stage]));
                    mma_commit(smem_addr(&ctl->tfull[buf]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    buf ^= 1u;
                    if (buf == 0) bphase ^= 1u;
                }
            }
            if (!ok) {
                mma_commit(smem_addr(&ctl->drain));
                mbar_wait(smem_addr(&ctl->drain), 0, nullptr, a.status);
            }
        }
      }
    } else {
        regs_increase<RegSplit<EPI>::epilogue>();
        // ---------------------------------------------------------------- epilogue
        const int g = (warp - FIRST_EPI_WARP) >> 2;   // column half
        const int sp = warp & 3;                // TMEM lane quarter
        const int row = sp * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(sp * 32) << 16);
        uint32_t buf = 0, bphase = 0, tile_iter = 0, q = 0;
        bool ok = true;
        int64_t k = 0;
        for (int64_t w = blockIdx.x; w < units && ok; w += gridDim.x, ++k) {
            const Tile t = decode_tile<EPI>(a, ctl, k, w, NT);
            if (!t.ok) continue;
            const int64_t grow = t.row0 + row;
            // rows whose sorted pair id is -1 are padding: a warp with no real row skips the
            // promotion (decode tiles hold a few real rows out of 128)
            const bool row_real = t.live >= 0 ? row < t.live
                                              : (a.sorted_pair_ids == nullptr || a.sorted_pair_ids[grow] >= 0);
            const bool warp_live = __any_sync(0xffffffffu, row_real);
            const bool active = ((EPI == MOE_EPI_SILU_MUL_QUANT) || g == 0 || t.has1) && warp_live;
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.0f;

            for (int kb = 0; kb < KB; ++kb) {
                const uint32_t slot = q % SR;
                if (!mbar_wait(smem_addr(&ctl->sfull[slot]), (q / SR) & 1u, abort_flag, a.status) ||
                    !mbar_wait(smem_addr(&ctl->tfull[buf]), bphase, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const float sa = ctl->scl[slot][row];
                // silu: s0 = gate block, s1 = up block; otherwise column half g's weight block
                const float s0 = sa * ctl->scl[slot][128 + ((EPI == MOE_EPI_SILU_MUL_QUANT) ? 0 : g)];
                const float s1 = sa * ctl->scl[slot][129];
                tc_fence_after();
                const uint32_t col = lane_base + buf * 256;
                if (active) {
                    // two rounds of 64 columns: two 32-column TMEM loads, one wait, 32 packed FMAs.
                    // silu: round 0 = gate columns g*64.. (scale s0) -> acc[0, 64),
                    //       round 1 = up columns 128+g*64.. (scale s1) -> acc[64, 128)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const uint32_t c0 = (EPI == MOE_EPI_SILU_MUL_QUANT) ? col + r * 128 + g * 64
                                                                            : col + g * 128 + r * 64;
                        const float sc = (EPI == MOE_EPI_SILU_MUL_QUANT && r == 1) ? s1 : s0;
                        float va[32], vb[32];
                        tmem_ld32x2(c0, c0 + 32, va, vb);
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            ffma2(acc + r * 64 + j, va + j, sc);
                            ffma2(acc + r * 64 + 32 + j, vb + j, sc);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_addr(&ctl->tempty[buf]));
                    mbar_arrive(smem_addr(&ctl->sempty[slot]));
                }
                buf ^= 1u;
                if (buf == 0) bphase ^= 1u;
                ++q;
            }
            if (!ok) break;
            if (!finish_item<EPI>(a, ctl, t, acc, warp, lane, g, row, grow, active, tile_iter, abort_flag)) {
                ok = false;
                break;
            }
            ++tile_iter;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ block-scaled variant
// With packed UE8M0 scales ("UE8M0: packed UE8M0, 4 values per int32, Blackwell", page
// "Quantization and MoE Optimizations", section DeepGEMM Scale Formats) every scale is a power of
// two, so the tensor cores apply them: tcgen05.mma kind::mxf8f6f4.block_scale multiplies each
// product by the UE8M0 scales of its row of A and its column of B for that K range, and the whole K
// loop accumulates in one TMEM accumulator with no promotion step.  A 128-wide K block is four MMAs
// of K = 32 that all use the K block's scale byte (the 128-wide groups and 128x128 blocks span 4
// scale vectors of 32 each: the same value).  Scale-factor tiles (512 bytes, common.cuh) come with
// the stage of every fourth K block (one TMA bulk copy for A's 128 rows, one for each of B's 128-
// column blocks) and are copied into tensor memory by the MMA thread before its MMAs (tcgen05.cp).
//
// Tensor memory: columns 0..255 hold the accumulator of the current item; 4 slots of 16 columns
// from column 256 hold scale factors (A: 4 columns, B: 8 columns).  A slot is reused 4 scale loads
// later: the stage that brings the new tiles was refilled only after the MMAs of the K block 4
// stages back completed, and each load covers at least one K block, so the MMAs reading the slot's
// old contents are complete.  With one accumulator the epilogue first moves its share into
// registers and frees the accumulator at once; the next item's MMAs run while it finishes the
// previous item from registers.
constexpr int SF_STAGE = 3 * kSfTileBytes;   // per stage: A's tile, then B's two
constexpr uint32_t TMEM_SF = 256;
constexpr int SF_SLOTS = 4;

struct SmemCtlBs {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull;                    // the accumulator holds a finished item
    uint64_t tempty;                   // the epilogue warps have moved it to registers (8 arrivals)
    uint64_t amax_bar[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    float amax_x[2][2][BM];
    alignas(16) float stage[NUM_EPI_WARPS][32 * 20];
    int item_n[ITEMS];
    int item_e[ITEMS];
    int item_r0[ITEMS];
    int item_live[ITEMS];
};
constexpr size_t SMEM_BYTES_BS = 1024 + STAGES * (A_TILE + B_TILE + SF_STAGE) + sizeof(SmemCtlBs);
static_assert(SMEM_BYTES_BS <= 232448, "shared memory per CTA exceeds the sm_103 limit");

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmB2, const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* smA = base;
    uint8_t* smB = base + STAGES * A_TILE;
    uint8_t* smSF = smB + STAGES * B_TILE;
    SmemCtlBs* ctl = reinterpret_cast<SmemCtlBs*>(smSF + STAGES * SF_STAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (EPI == MOE_EPI_SILU_MUL_QUANT) ? a.N / 256 : (a.N + 255) / 256;
    const int KB = a.K / BK;
    // scale-factor tiles per 128 rows of A or per 128 columns of B: one per 4 K blocks (packed UE8M0),
    // or one per K block (MXFP8: a word holds the K block's four 32-wide groups)
    const bool mx = a.sf_packed == 2;
    const int KB4 = mx ? KB : (KB + 3) / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            mbar_init(smem_addr(&ctl->empty[s]), 1);
        }
        mbar_init(smem_addr(&ctl->tfull), 1);
        mbar_init(smem_addr(&ctl->tempty), NUM_EPI_WARPS);
        for (int b = 0; b < 2; ++b) mbar_init(smem_addr(&ctl->amax_bar[b]), NUM_EPI_WARPS * 32);
        mbar_init(smem_addr(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmB2);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_dependency_wait();
    int64_t ntiles = *a.num_tiles;
    if (ntiles < 0) ntiles = 0;
    if (ntiles > a.max_tiles) ntiles = a.max_tiles;
    const int64_t total = ntiles * NT;
    const int64_t halves = tail_halves<EPI>(a, total);
    const int64_t units = total + halves;
    fill_item_cache<EPI>(a, ctl, total, halves, NT);
    __syncthreads();
    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort_flag;
    if (warp < FIRST_EPI_WARP) {
      regs_decrease<RegSplitBs<EPI>::control>();
      if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, issued = 0;
            bool ok = true;
            int64_t k = 0;
            const int NBn = a.N / 128;
            for (int64_t w = blockIdx.x; w < units && ok; w += gridDim.x, ++k) {
                const Tile t = decode_tile<EPI>(a, ctl, k, w, NT);
                if (!t.ok) {
                    status_set(a.status, MOE_STATUS_BAD_EXPERT_ID);
                    continue;
                }
                int32_t by0, bdx, bdy;
                if (a.b_tiled) {
                    by0 = ((t.e * (a.N / 128) + t.bcol0 / 128) * KB) * 128;
                    bdx = 0;
                    bdy = 128;
                } else {
                    by0 = t.e * a.N + t.bcol0;
                    bdx = BK;
                    bdy = 0;
                }
                const uint8_t* sfa = a.a_sf + (t.row0 >> 7) * KB4 * kSfTileBytes;
                const uint8_t* sfb0 = a.b_sf + (static_cast<int64_t>(t.e) * NBn + t.bcol0 / 128) * KB4 * kSfTileBytes;
                const uint8_t* sfb1 = a.b_sf + (static_cast<int64_t>(t.e) * NBn + t.bcol1 / 128) * KB4 * kSfTileBytes;
                const uint32_t bytes = a.a_box_rows * BK + (t.has1 ? B_TILE : B_HALF);
                const uint32_t sf_bytes = (t.has1 ? 3 : 2) * kSfTileBytes;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_addr(&ctl->full[stage]);
                    const bool load_sf = mx || (kb & 3) == 0;
                    mbar_arrive_expect_tx(fb, bytes + (load_sf ? sf_bytes : 0u));
                    tma_load_2d(smem_addr(smA + stage * A_TILE), &tmA, kb * BK, static_cast<int32_t>(t.row0), fb);
                    if (t.has1)
                        load_b_pair<EPI>(smem_addr(smB + stage * B_TILE), &tmB2, a, t, kb, fb);
                    else
                        tma_load_2d(smem_addr(smB + stage * B_TILE), &tmB, kb * bdx, by0 + kb * bdy, fb);
                    if (load_sf) {
                        const uint32_t dst = smem_addr(smSF + stage * SF_STAGE);
                        const int64_t q = static_cast<int64_t>(mx ? kb : kb >> 2) * kSfTileBytes;
                        bulk_load(dst, sfa + q, kSfTileBytes, fb);
                        bulk_load(dst + kSfTileBytes, sfb0 + q, kSfTileBytes, fb);
                        if (t.has1) bulk_load(dst + 2 * kSfTileBytes, sfb1 + q, kSfTileBytes, fb);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < STAGES; ++s) {
                    const uint32_t n_s = (issued + STAGES - 1 - s) / STAGES;
                    if (n_s > 0) mbar_wait(smem_addr(&ctl->full[s]), (n_s - 1) & 1u, nullptr, a.status);
                }
            }
        }
      } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0, items = 0, sf_loads = 0;
            bool ok = true;
            int64_t k = 0;
            for (int64_t w = blockIdx.x; w < units && ok; w += gridDim.x, ++k) {
                const Tile t = decode_tile<EPI>(a, ctl, k, w, NT);
                if (!t.ok) continue;
                const int n = t.has1 ? 256 : 128;
                // the accumulator is free once the epilogue warps moved the previous item out
                if (!mbar_wait(smem_addr(&ctl->tempty), (items & 1u) ^ 1u, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sfa_t = 0, sfb_t = 0;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_addr(&ctl->full[stage]), phase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (mx || (kb & 3) == 0) {
                        const uint32_t col = TMEM_SF + (sf_loads % SF_SLOTS) * 16;
                        const uint32_t src = smem_addr(smSF + stage * SF_STAGE);
                        sfa_t = tmem + col;
                        sfb_t = tmem + col + 4;
                        tmem_copy_sf_tile(sfa_t, smem_desc_sf_tile(src));
                        tmem_copy_sf_tile(sfb_t, smem_desc_sf_tile(src + kSfTileBytes));
                        if (t.has1) tmem_copy_sf_tile(sfb_t + 4, smem_desc_sf_tile(src + 2 * kSfTileBytes));
                        ++sf_loads;
                    }
                    const uint32_t a0 = smem_addr(smA + stage * A_TILE);
                    const uint32_t b0 = smem_addr(smB + stage * B_TILE);
#pragma unroll
                    for (int s = 0; s < BK / 32; ++s) {
                        // the scale byte: the K block's (packed UE8M0) or the 32-group's (MXFP8)
                        const uint32_t idesc = idesc_e4m3_ue8m0(BM, n, mx ? s : (kb & 3));
                        mma_e4m3_block_scaled(tmem, smem_desc_k128_sw128(a0 + s * 32), smem_desc_k128_sw128(b0 + s * 32),
                                              idesc, sfa_t, sfb_t, (kb | s) != 0 ? 1u : 0u);
                    }
                    mma_commit(smem_addr(&ctl->empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(smem_addr(&ctl->tfull));
                ++items;
            }
            if (!ok) {
                mma_commit(smem_addr(&ctl->drain));
                mbar_wait(smem_addr(&ctl->drain), 0, nullptr, a.status);
            }
        }
      }
    } else {
        regs_increase<RegSplitBs<EPI>::epilogue>();
        // ---------------------------------------------------------------- epilogue
        const int g = (warp - FIRST_EPI_WARP) >> 2;   // column half
        const int sp = warp & 3;                      // TMEM lane quarter
        const int row = sp * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(sp * 32) << 16);
        uint32_t tile_iter = 0;
        bool ok = true;
        int64_t k = 0;
        for (int64_t w = blockIdx.x; w < units && ok; w += gridDim.x, ++k) {
            const Tile t = decode_tile<EPI>(a, ctl, k, w, NT);
            if (!t.ok) continue;
            const int64_t grow = t.row0 + row;
            const bool row_real = t.live >= 0 ? row < t.live
                                              : (a.sorted_pair_ids == nullptr || a.sorted_pair_ids[grow] >= 0);
            const bool warp_live = __any_sync(0xffffffffu, row_real);
            const bool active = ((EPI == MOE_EPI_SILU_MUL_QUANT) || g == 0 || t.has1) && warp_live;
            float acc[128];
            if (!mbar_wait(smem_addr(&ctl->tfull), tile_iter & 1u, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (active) {
                // silu: gate columns g*64 .. +63 -> acc[0, 64), up columns 128 + g*64 .. -> acc[64, 128)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t c0 = (EPI == MOE_EPI_SILU_MUL_QUANT) ? lane_base + r * 128 + g * 64
                                                                        : lane_base + g * 128 + r * 64;
                    tmem_ld32x2(c0, c0 + 32, acc + r * 64, acc + r * 64 + 32);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl->tempty));
            if (!finish_item<EPI>(a, ctl, t, acc, warp, lane, g, row, grow, active, tile_iter, abort_flag)) {
                ok = false;
                break;
            }
            ++tile_iter;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ CTA-pair block-scaled variant
// The block-scaled w2 GEMM (router-weighted pair rows) on the two-SM MMA, for batches with many
// rows per expert (the layer takes it from 512 routed rows per expert on average).  A cluster of
// two CTAs computes a 256-row x 256-column
// work item (two 128-row tiles of one expert): each CTA keeps its own 128 rows of A and one of the
// item's two 128-row weight bands in its shared memory, and CTA 0 issues tcgen05.mma.cta_group::2
// (M = 256), which reads both CTAs' operands and accumulates each CTA's 128 rows x 256 columns in
// that CTA's tensor memory.  A K block then brings 32 KB into each SM instead of 48 KB for the same
// multiply-adds: the operand feed that bounds the one-CTA kernel on batches with many rows per
// expert drops by a third.
// Facts about the pair forms that this layout relies on (checked on GB300 with one 256 x 256 x 128
// item, exact against a host computation): the allocation is collective (both CTAs allocate and get
// the same base); tcgen05.cp.cta_group::2 copies each CTA's shared memory into its own tensor
// memory; each CTA needs the weight scale factors of all 256 columns (both bands' tiles) beside its
// own rows' activation scale factors; CTA 0's band supplies columns 0..127.
// Synchronisation: the ring holds P_SUPER stages of P_SUB K blocks.  Both CTAs' loads of a stage
// (TMA with .cta_group::2: operand and scale-factor tiles into each CTA's own shared memory)
// complete their bytes on CTA 0's full barrier, which CTA 0's producer armed with the stage's bytes
// of both CTAs.  A second thread of CTA 0 copies the scale-factor tiles of the stage into a ring of
// tensor-memory slots (tcgen05.cp.cta_group::2) and signals each slot on its own barrier; the MMA
// thread waits for the stage and the slots it reads, issues the stage's MMAs and commits them to
// both CTAs' empty barriers (multicast), so each producer refills its own stage; an item's last
// commit arrives on both CTAs' tfull; the epilogue warps of both CTAs arrive on CTA 0's tempty
// before the next item's MMAs overwrite the accumulators.
// The single MMA thread bounds these kernels: issuing a pair MMA takes 60-80 cycles of its time
// against 128 for the tensor pipe to run it, and each barrier wait, commit and scale-factor copy
// another 100-200 (cycle counts of an instrumented copy on GB300).  Hence two K blocks (eight MMAs)
// per barrier wait and commit, and the copies on another thread.  (Forwarding each stage from a
// thread of CTA 1 to CTA 0 instead of the .cta_group::2 loads cost about 0.3 us per stage.)
// Work: candidate w of the tile-major order (tile m, column block n) is an item when tile m sits at
// an even position among its expert's tiles; CTA 0 takes tile m and CTA 1 tile m + 1, or, when
// the expert has no tile m + 1, a copy of tile m's rows whose results it discards.
constexpr int P_SUB = 2;                       // K blocks per stage
constexpr int P_SUPER = 3;                     // stages
constexpr int P_STAGES = P_SUB * P_SUPER;      // K-block buffers
constexpr int P_SF_STAGE = 3 * kSfTileBytes;   // per K block: this CTA's rows' A tile, then both bands' B tiles
constexpr int P_SF_SLOTS = 8;                  // > P_STAGES: a slot's last MMAs completed before its reuse
constexpr int P_ITEMS = 128;                   // candidates of a cluster cached in shared memory

struct SmemCtlPair {
    uint64_t full[P_SUPER];            // (CTA 0) both CTAs' loads of the stage landed
    uint64_t empty[P_SUPER];           // the stage's MMAs completed (commit from CTA 0, both CTAs)
    uint64_t sf_ready[P_SF_SLOTS];     // (CTA 0) the slot's scale-factor copies completed
    uint64_t sf_drain;                 // (CTA 0) all scale-factor copies completed
    uint64_t tfull;                    // the item's accumulators are complete (both CTAs)
    uint64_t tempty;                   // (CTA 0) both CTAs' epilogue warps moved them out (16 arrivals)
    uint64_t amax_bar[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    float amax_x[2][2][BM];
    alignas(16) float stage[NUM_EPI_WARPS][32 * 20];
    int item_n[P_ITEMS];               // the cluster's candidates in visiting order: column block,
    int item_e[P_ITEMS];               // expert (-1: not an item, -2: an item with a bad tile entry),
    int item_r0[P_ITEMS];              // first row of this CTA's tile,
    int item_live[P_ITEMS];            // and whether that tile is one of the expert's
};
constexpr size_t SMEM_BYTES_PAIR = 1024 + P_STAGES * (A_TILE + B_HALF + P_SF_STAGE) + sizeof(SmemCtlPair);
static_assert(SMEM_BYTES_PAIR <= 232448, "shared memory per CTA exceeds the sm_103 limit");
static_assert(TMEM_SF + P_SF_SLOTS * 16 <= TMEM_COLS, "scale-factor slots exceed the tensor-memory allocation");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// TMA tile loads into this CTA's shared memory whose bytes complete on `bar`, a shared::cluster
// address that may be the other CTA's barrier (the .cta_group::2 form).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 int32_t z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
// Arrive on a barrier of either CTA of the pair (shared::cluster address).  CTA-scope release, like
// the waits (mbar_wait): the arrivals hand over tensor memory (ordered by the tcgen05 fences around
// the barrier) and shared-memory stages (written by TMA, completion counted on the barrier), never
// data the arriving thread wrote itself; a cluster-scope release made every arrival of the
// epilogue warps wait for their earlier global stores.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// All threads of both CTAs.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Each CTA's 512-byte scale-factor tile at this shared-memory address into its own tensor memory.
__device__ __forceinline__ void tmem_copy_sf_tile_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// D (256 x N over both CTAs) (+)= (A * sfA) * (B * sfB)^T, K = 32, issued by one thread of CTA 0.
__device__ __forceinline__ void mma_e4m3_block_scaled_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                           uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
            "r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at this offset in each CTA of `mask` when the MMAs issued so far complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

struct PairItem {
    int64_t row0;   // this CTA's tile's first row
    int e, n;
    bool take;      // candidate is an item
    bool ok;        // its tile entries are valid
    bool live;      // this CTA's tile is one of the expert's
};

// Candidate w (tile m, column block n) from the tile table and the experts' padded row offsets.
// Everything but row0 and live is the same in both CTAs, so both skip the same candidates.
__device__ __forceinline__ PairItem pair_item_lookup(const GemmArgs& a, int64_t w, int NT, uint32_t rank,
                                                     int64_t ntiles) {
    PairItem p;
    const int64_t mt = w / NT;
    const int m = static_cast<int>(mt);
    p.n = static_cast<int>(w - mt * NT);
    p.e = a.tile_expert[m];
    p.take = true;
    p.ok = false;
    p.live = false;
    p.row0 = 0;
    if (p.e < 0 || p.e >= a.E) return p;
    const int f = a.pair_offsets[p.e] / BM, end = a.pair_offsets[p.e + 1] / BM;
    if (m < f || m >= end) return p;
    if (((m - f) & 1) != 0) {
        p.take = false;
        return p;
    }
    const bool has2 = m + 1 < end && m + 1 < ntiles;
    const int64_t r_first = a.tile_row0[m];
    const int64_t r_second = has2 ? a.tile_row0[m + 1] : r_first;
    const auto valid = [&](int64_t r) { return r >= 0 && (r & (BM - 1)) == 0 && r + BM <= a.a_rows; };
    p.ok = valid(r_first) && valid(r_second);
    p.live = rank == 0 || has2;
    p.row0 = rank == 0 ? r_first : r_second;
    return p;
}

__device__ __forceinline__ PairItem pair_item(const GemmArgs& a, const SmemCtlPair* ctl, int64_t k, int64_t w, int NT,
                                              uint32_t rank, int64_t ntiles) {
    if (k < P_ITEMS) {
        PairItem p;
        const int ce = ctl->item_e[k];
        p.n = ctl->item_n[k];
        p.e = ce;
        p.take = ce != -1;
        p.ok = ce >= 0;
        p.row0 = ctl->item_r0[k];
        p.live = ctl->item_live[k] != 0;
        return p;
    }
    return pair_item_lookup(a, w, NT, rank, ntiles);
}

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                             const GemmArgs a) {
    // the w2 GEMM's epilogue only (the w13 GEMM ran faster on the one-CTA kernel, whose epilogue
    // does not spill; this kernel's SiLU epilogue did at every register split)
    static_assert(EPI == MOE_EPI_WEIGHTED_PAIRS_BF16, "the pair kernel runs the weighted-pairs epilogue");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* smA = base;
    uint8_t* smB = base + P_STAGES * A_TILE;
    uint8_t* smSF = smB + P_STAGES * B_HALF;
    SmemCtlPair* ctl = reinterpret_cast<SmemCtlPair*>(smSF + P_STAGES * P_SF_STAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int64_t cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    const int NT = a.N / 256;   // item n: weight bands 2n (CTA 0) and 2n + 1 (CTA 1)
    const int KB = a.K / BK;
    const bool mx = a.sf_packed == 2;
    const int KB4 = mx ? KB : (KB + 3) / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_SUPER; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            mbar_init(smem_addr(&ctl->empty[s]), 1);
        }
        for (int s = 0; s < P_SF_SLOTS; ++s) mbar_init(smem_addr(&ctl->sf_ready[s]), 1);
        mbar_init(smem_addr(&ctl->sf_drain), 1);
        mbar_init(smem_addr(&ctl->tfull), 1);
        mbar_init(smem_addr(&ctl->tempty), 2 * NUM_EPI_WARPS);
        for (int b = 0; b < 2; ++b) mbar_init(smem_addr(&ctl->amax_bar[b]), NUM_EPI_WARPS * 32);
        mbar_init(smem_addr(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmSFA);
        tma_prefetch_map(&tmSFB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_barrier();   // both CTAs' barriers initialised before any arrival from the other
    tc_fence_after();
    grid_dependency_wait();
    int64_t ntiles = *a.num_tiles;
    if (ntiles < 0) ntiles = 0;
    if (ntiles > a.max_tiles) ntiles = a.max_tiles;
    const int64_t total = ntiles * NT;
    for (int64_t k = threadIdx.x; k < P_ITEMS; k += blockDim.x) {
        const int64_t w = cid + k * ncl;
        if (w >= total) break;
        const PairItem p = pair_item_lookup(a, w, NT, rank, ntiles);
        ctl->item_n[k] = p.n;
        ctl->item_e[k] = !p.take ? -1 : (p.ok ? p.e : -2);
        ctl->item_r0[k] = static_cast<int>(p.row0);
        ctl->item_live[k] = p.live ? 1 : 0;
    }
    __syncthreads();
    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort_flag;
    if (warp < FIRST_EPI_WARP) {
      regs_decrease<RegSplitBs<EPI>::control>();
      if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0, issued = 0;
            bool ok = true;
            int64_t k = 0;
            const int NBn = a.N / 128;
            for (int64_t w = cid; w < total && ok; w += ncl, ++k) {
                const PairItem p = pair_item(a, ctl, k, w, NT, rank, ntiles);
                if (!p.take) continue;
                if (!p.ok) {
                    status_set(a.status, MOE_STATUS_BAD_EXPERT_ID);
                    continue;
                }
                const int bcol0 = p.n * 256, bcol1 = bcol0 + 128;
                const int band = rank == 0 ? bcol0 : bcol1;   // the weight rows this CTA holds
                int32_t by0, bdx, bdy;
                if (a.b_tiled) {
                    by0 = ((p.e * NBn + band / 128) * KB) * 128;
                    bdx = 0;
                    bdy = 128;
                } else {
                    by0 = p.e * a.N + band;
                    bdx = BK;
                    bdy = 0;
                }
                // scale-factor tiles (index into the packed arrays, tensor maps of 512-byte tiles)
                const int32_t sfa = static_cast<int32_t>((p.row0 >> 7) * KB4);
                const int32_t sfb0 = (p.e * NBn + bcol0 / 128) * KB4;
                const int32_t sfb1 = (p.e * NBn + bcol1 / 128) * KB4;
                for (int kb0 = 0; kb0 < KB; kb0 += P_SUB) {
                    const int nsub = KB - kb0 < P_SUB ? KB - kb0 : P_SUB;
                    if (!mbar_wait(smem_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb0 = smem_addr(&ctl->full[stage]);
                    const uint32_t fb = cluster_map(fb0, 0);   // CTA 0's full barrier
                    uint32_t bytes = 0;
                    for (int j = 0; j < nsub; ++j)
                        bytes += A_TILE + B_HALF + ((mx || ((kb0 + j) & 3) == 0) ? P_SF_STAGE : 0u);
                    if (rank == 0) mbar_arrive_expect_tx(fb0, 2 * bytes);
                    for (int j = 0; j < nsub; ++j) {
                        const int kb = kb0 + j, buf = stage * P_SUB + j;
                        tma_load_2d_pair(smem_addr(smA + buf * A_TILE), &tmA, kb * BK, static_cast<int32_t>(p.row0), fb);
                        tma_load_2d_pair(smem_addr(smB + buf * B_HALF), &tmB, kb * bdx, by0 + kb * bdy, fb);
                        if (mx || (kb & 3) == 0) {
                            const uint32_t dst = smem_addr(smSF + buf * P_SF_STAGE);
                            const int32_t q = mx ? kb : kb >> 2;
                            tma_load_3d_pair(dst, &tmSFA, 0, 0, sfa + q, fb);
                            tma_load_3d_pair(dst + kSfTileBytes, &tmSFB, 0, 0, sfb0 + q, fb);
                            tma_load_3d_pair(dst + 2 * kSfTileBytes, &tmSFB, 0, 0, sfb1 + q, fb);
                        }
                    }
                    ++issued;
                    if (++stage == P_SUPER) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // after an abort, CTA 0 waits (bounded) for the loads of the stages it armed, both
            // CTAs' bytes; CTA 1 cannot see its loads' completion, and waits at the closing
            // cluster barrier for CTA 0 (its own loads land within microseconds, its producer
            // leaves the loop only after a wait of kWaitLimitNs gave up or after its last stage)
            if (!ok && rank == 0) {
                for (int s = 0; s < P_SUPER; ++s) {
                    const uint32_t n_s = (issued + P_SUPER - 1 - s) / P_SUPER;
                    if (n_s > 0) mbar_wait(smem_addr(&ctl->full[s]), (n_s - 1) & 1u, nullptr, a.status);
                }
            }
        }
      } else if (warp == 2 && lane == 0 && rank == 0) {
        // ---------------------------------------------------------------- CTA 0: scale factors
        // Slot u % P_SF_SLOTS takes the u-th scale-factor load.  It is rewritten P_SF_SLOTS loads
        // (at least P_SF_SLOTS K blocks) later, after this thread waited for the stage bringing the
        // new tiles, which was refilled only once the MMAs P_STAGES K blocks back had completed.
        int stage = 0;
        uint32_t phase = 0, sf_loads = 0;
        bool ok = true;
        int64_t k = 0;
        for (int64_t w = cid; w < total && ok; w += ncl, ++k) {
            const PairItem p = pair_item(a, ctl, k, w, NT, rank, ntiles);
            if (!p.take || !p.ok) continue;
            for (int kb0 = 0; kb0 < KB; kb0 += P_SUB) {
                const int nsub = KB - kb0 < P_SUB ? KB - kb0 : P_SUB;
                bool any = false;
                for (int j = 0; j < nsub; ++j) any = any || mx || ((kb0 + j) & 3) == 0;
                if (any) {
                    if (!mbar_wait(smem_addr(&ctl->full[stage]), phase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int j = 0; j < nsub; ++j) {
                        if (!(mx || ((kb0 + j) & 3) == 0)) continue;
                        const uint32_t slot = sf_loads % P_SF_SLOTS;
                        const uint32_t t_sf = tmem + TMEM_SF + slot * 16;
                        const uint32_t src = smem_addr(smSF + (stage * P_SUB + j) * P_SF_STAGE);
                        tmem_copy_sf_tile_pair(t_sf, smem_desc_sf_tile(src));
                        tmem_copy_sf_tile_pair(t_sf + 4, smem_desc_sf_tile(src + kSfTileBytes));
                        tmem_copy_sf_tile_pair(t_sf + 8, smem_desc_sf_tile(src + 2 * kSfTileBytes));
                        mma_commit_pair(smem_addr(&ctl->sf_ready[slot]), 1);
                        ++sf_loads;
                    }
                }
                if (++stage == P_SUPER) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        mma_commit_pair(smem_addr(&ctl->sf_drain), 1);
        mbar_wait(smem_addr(&ctl->sf_drain), 0, nullptr, a.status);
      } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------------------------------------------------------- CTA 0: MMA issuer
        int stage = 0;
        uint32_t phase = 0, items = 0, sf_loads = 0;
        bool ok = true;
        int64_t k = 0;
        for (int64_t w = cid; w < total && ok; w += ncl, ++k) {
            const PairItem p = pair_item(a, ctl, k, w, NT, rank, ntiles);
            if (!p.take || !p.ok) continue;
            if (!mbar_wait(smem_addr(&ctl->tempty), (items & 1u) ^ 1u, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sfa_t = 0, sfb_t = 0;
            for (int kb0 = 0; kb0 < KB && ok; kb0 += P_SUB) {
                const int nsub = KB - kb0 < P_SUB ? KB - kb0 : P_SUB;
                if (!mbar_wait(smem_addr(&ctl->full[stage]), phase, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int j = 0; j < nsub; ++j) {
                    const int kb = kb0 + j;
                    if (mx || (kb & 3) == 0) {
                        const uint32_t slot = sf_loads % P_SF_SLOTS;
                        if (!mbar_wait(smem_addr(&ctl->sf_ready[slot]), (sf_loads / P_SF_SLOTS) & 1u, abort_flag,
                                       a.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        sfa_t = tmem + TMEM_SF + slot * 16;
                        sfb_t = sfa_t + 4;
                        ++sf_loads;
                    }
                    const uint32_t a0 = smem_addr(smA + (stage * P_SUB + j) * A_TILE);
                    const uint32_t b0 = smem_addr(smB + (stage * P_SUB + j) * B_HALF);
#pragma unroll
                    for (int s = 0; s < BK / 32; ++s) {
                        const uint32_t idesc = idesc_e4m3_ue8m0(2 * BM, 256, mx ? s : (kb & 3));
                        mma_e4m3_block_scaled_pair(tmem, smem_desc_k128_sw128(a0 + s * 32),
                                                   smem_desc_k128_sw128(b0 + s * 32), idesc, sfa_t, sfb_t,
                                                   (kb | s) != 0 ? 1u : 0u);
                    }
                }
                if (!ok) break;
                mma_commit_pair(smem_addr(&ctl->empty[stage]), 3);
                if (++stage == P_SUPER) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            mma_commit_pair(smem_addr(&ctl->tfull), 3);
            ++items;
        }
        // every MMA complete before the CTAs can leave (they read both CTAs' shared memory)
        mma_commit_pair(smem_addr(&ctl->drain), 1);
        mbar_wait(smem_addr(&ctl->drain), 0, nullptr, a.status);
      }
    } else {
        regs_increase<RegSplitBs<EPI>::epilogue>();
        // ---------------------------------------------------------------- epilogue (both CTAs)
        const int g = (warp - FIRST_EPI_WARP) >> 2;   // column half
        const int sp = warp & 3;                      // TMEM lane quarter
        const int row = sp * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(sp * 32) << 16);
        const uint32_t tempty0 = cluster_map(smem_addr(&ctl->tempty), 0);
        uint32_t acc_iter = 0, epi_iter = 0;
        bool ok = true;
        int64_t k = 0;
        for (int64_t w = cid; w < total && ok; w += ncl, ++k) {
            const PairItem p = pair_item(a, ctl, k, w, NT, rank, ntiles);
            if (!p.take || !p.ok) continue;
            Tile t;
            t.row0 = p.row0;
            t.e = p.e;
            t.n = p.n;
            t.bcol0 = p.n * 256;
            t.bcol1 = t.bcol0 + 128;
            t.has1 = true;
            t.ok = true;
            const int64_t grow = t.row0 + row;
            const bool row_real = p.live && (a.sorted_pair_ids == nullptr || a.sorted_pair_ids[grow] >= 0);
            const bool active = __any_sync(0xffffffffu, row_real);
            float acc[128];
            if (!mbar_wait(smem_addr(&ctl->tfull), acc_iter & 1u, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (active) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t c0 = lane_base + g * 128 + r * 64;
                    tmem_ld32x2(c0, c0 + 32, acc + r * 64, acc + r * 64 + 32);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0);
            ++acc_iter;
            if (p.live) {
                if (!finish_item<EPI>(a, ctl, t, acc, warp, lane, g, row, grow, active, epi_iter, abort_flag)) {
                    ok = false;
                    break;
                }
                ++epi_iter;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_barrier();   // neither CTA leaves while the other's MMAs or arrivals may still reach it
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
int g_pair_clusters = 0;   // clusters of two CTAs of the pair kernel resident at once (0: unavailable)
std::once_flag g_encode_once;

cudaError_t get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// 2-D e4m3 matrix [rows, cols] (row stride = cols bytes), boxes of 128 bytes x box_rows rows,
// 128-byte swizzle
cudaError_t make_map(CUtensorMap* map, const uint8_t* ptr, int64_t cols, int64_t rows, uint32_t box_rows = 128) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t elem[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(ptr), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t encode_u8_map_nd(CUtensorMap* map, const uint8_t* ptr, int rank, const uint64_t* dims,
                             const uint64_t* strides, const uint32_t* box, bool swizzle128);

namespace {

// Map of the 32 KB boxes of load_b_pair: both 128-row bands of an item for one K block.
cudaError_t make_pair_map(CUtensorMap* map, const GemmArgs& g) {
    const uint64_t KB = g.K / 128, E = g.E, N = g.N, K = g.K;
    if (g.epi == MOE_EPI_SILU_MUL_QUANT) {
        const uint64_t NBh = N / 256;   // bands per half (gate / up)
        if (g.b_tiled) {
            // [E][2][NBh][KB][128 rows][128 B]: the outermost index is 2e + half
            const uint64_t dims[5] = {128, 128, KB, NBh, 2 * E};
            const uint64_t strides[4] = {128, 16384, KB * 16384, NBh * KB * 16384};
            const uint32_t box[5] = {128, 128, 1, 1, 2};
            return encode_u8_map_nd(map, g.B, 5, dims, strides, box, true);
        }
        // rows e*2I + half*I + j*128 + r of [E*N, K]
        const uint64_t dims[4] = {K, 128, NBh, 2 * E};
        const uint64_t strides[3] = {K, 128 * K, (N / 2) * K};
        const uint32_t box[4] = {128, 128, 1, 2};
        return encode_u8_map_nd(map, g.B, 4, dims, strides, box, true);
    }
    if (g.b_tiled) {
        // [E*N/128 bands][KB][128 rows][128 B]
        const uint64_t dims[4] = {128, 128, KB, E * (N / 128)};
        const uint64_t strides[3] = {128, 16384, KB * 16384};
        const uint32_t box[4] = {128, 128, 1, 2};
        return encode_u8_map_nd(map, g.B, 4, dims, strides, box, true);
    }
    const uint64_t dims[2] = {K, E * N};
    const uint64_t strides[1] = {K};
    const uint32_t box[2] = {128, 256};
    return encode_u8_map_nd(map, g.B, 2, dims, strides, box, true);
}

}  // namespace

cudaError_t encode_u8_map_nd(CUtensorMap* map, const uint8_t* ptr, int rank, const uint64_t* dims,
                             const uint64_t* strides, const uint32_t* box, bool swizzle128) {
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], elem[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        elem[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank), const_cast<uint8_t*>(ptr),
                          d, st, b, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_u8_map(CUtensorMap* map, const uint8_t* ptr, int64_t cols, int64_t rows, uint32_t box_cols,
                          uint32_t box_rows, bool swizzle128) {
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t elem[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(ptr), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t gemm_init_device() {
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    const int bytes = static_cast<int>(SMEM_BYTES);
    err = cudaFuncSetAttribute(grouped_gemm_kernel<MOE_EPI_STORE_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               bytes);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(grouped_gemm_kernel<MOE_EPI_SILU_MUL_QUANT>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(grouped_gemm_kernel<MOE_EPI_WEIGHTED_SCATTER>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(grouped_gemm_kernel<MOE_EPI_WEIGHTED_ROWS>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(grouped_gemm_kernel<MOE_EPI_WEIGHTED_PAIRS_BF16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    const int bytes_bs = static_cast<int>(SMEM_BYTES_BS);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(grouped_gemm_bs_kernel<MOE_EPI_STORE_F32>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, bytes_bs);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(grouped_gemm_bs_kernel<MOE_EPI_SILU_MUL_QUANT>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, bytes_bs);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(grouped_gemm_bs_kernel<MOE_EPI_WEIGHTED_PAIRS_BF16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, bytes_bs);
    const int bytes_pair = static_cast<int>(SMEM_BYTES_PAIR);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(grouped_gemm_pair_kernel<MOE_EPI_WEIGHTED_PAIRS_BF16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, bytes_pair);
    if (err == cudaSuccess) {
        // clusters of two that fit on the device at once (one CTA per SM; pairs within a GPC)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES_PAIR;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<MOE_EPI_WEIGHTED_PAIRS_BF16>, &cfg) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        g_pair_clusters = n;
    }
    return err;
}

int gemm_pair_clusters() { return g_pair_clusters; }

// The CTA-pair kernel: clusters of two CTAs, launched like the others with programmatic serialisation.
template <int EPI>
cudaError_t launch_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                        const CUtensorMap& tmSFB, const GemmArgs& args, unsigned clusters, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES_PAIR;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<EPI>, tmA, tmB, tmSFA, tmSFB, args);
}

cudaError_t launch_grouped_gemm(const GemmArgs& args, int num_sms, cudaStream_t stream) {
    const int NT = (args.epi == MOE_EPI_SILU_MUL_QUANT) ? args.N / 256 : (args.N + 255) / 256;
    const int64_t bound = args.max_tiles * NT;
    if (bound == 0) return cudaSuccess;
    CUtensorMap tmA, tmB;
    if (args.pair_offsets) {
        if (!args.sf_packed || args.N % 256 != 0 || args.a_box_rows != 128 || args.epi != MOE_EPI_WEIGHTED_PAIRS_BF16)
            return cudaErrorInvalidValue;
        if (g_pair_clusters < 1) return cudaErrorNotSupported;
        cudaError_t err = make_map(&tmA, args.A, args.K, args.a_rows, 128);
        if (err != cudaSuccess) return err;
        if (args.b_tiled)
            err = make_map(&tmB, args.B, 128, static_cast<int64_t>(args.E) * args.N * (args.K / 128));
        else
            err = make_map(&tmB, args.B, args.K, static_cast<int64_t>(args.E) * args.N);
        if (err != cudaSuccess) return err;
        // the packed scale-factor arrays as rows of 512-byte tiles (box: one tile)
        if (args.a_rows % 128 != 0) return cudaErrorInvalidValue;
        const uint64_t KB = args.K / 128, kb4 = args.sf_packed == 2 ? KB : (KB + 3) / 4;
        const uint64_t sf_strides[2] = {256, 512};
        const uint32_t sf_box[3] = {256, 2, 1};
        const uint64_t a_dims[3] = {256, 2, static_cast<uint64_t>(args.a_rows / 128) * kb4};
        const uint64_t b_dims[3] = {256, 2, static_cast<uint64_t>(args.E) * (args.N / 128) * kb4};
        CUtensorMap tmSFA, tmSFB;
        err = encode_u8_map_nd(&tmSFA, args.a_sf, 3, a_dims, sf_strides, sf_box, false);
        if (err == cudaSuccess) err = encode_u8_map_nd(&tmSFB, args.b_sf, 3, b_dims, sf_strides, sf_box, false);
        if (err != cudaSuccess) return err;
        const unsigned clusters = static_cast<unsigned>(bound < g_pair_clusters ? bound : g_pair_clusters);
        return launch_pair<MOE_EPI_WEIGHTED_PAIRS_BF16>(tmA, tmB, tmSFA, tmSFB, args, clusters, stream);
    }
    if (args.a_box_rows != 32 && args.a_box_rows != 128) return cudaErrorInvalidValue;
    cudaError_t err = make_map(&tmA, args.A, args.K, args.a_rows, static_cast<uint32_t>(args.a_box_rows));
    if (err != cudaSuccess) return err;
    if (args.b_tiled)   // [E][N/128][K/128] blocks of 128 rows x 128 bytes, stacked
        err = make_map(&tmB, args.B, 128, static_cast<int64_t>(args.E) * args.N * (args.K / 128));
    else
        err = make_map(&tmB, args.B, args.K, static_cast<int64_t>(args.E) * args.N);
    if (err != cudaSuccess) return err;
    // (with N = 128 no item has two bands: the pair map is never read)
    CUtensorMap tmB2 = tmB;
    if (args.N >= 256) err = make_pair_map(&tmB2, args);
    if (err != cudaSuccess) return err;
    const unsigned grid = static_cast<unsigned>(bound < num_sms ? bound : num_sms);
    if (args.sf_packed) {
        switch (args.epi) {
            case MOE_EPI_STORE_F32:
                return launch_pdl(grouped_gemm_bs_kernel<MOE_EPI_STORE_F32>, dim3(grid), dim3(NUM_THREADS),
                                  SMEM_BYTES_BS, stream, tmA, tmB, tmB2, args);
            case MOE_EPI_SILU_MUL_QUANT:
                return launch_pdl(grouped_gemm_bs_kernel<MOE_EPI_SILU_MUL_QUANT>, dim3(grid), dim3(NUM_THREADS),
                                  SMEM_BYTES_BS, stream, tmA, tmB, tmB2, args);
            case MOE_EPI_WEIGHTED_PAIRS_BF16:
                return launch_pdl(grouped_gemm_bs_kernel<MOE_EPI_WEIGHTED_PAIRS_BF16>, dim3(grid), dim3(NUM_THREADS),
                                  SMEM_BYTES_BS, stream, tmA, tmB, tmB2, args);
            default:
                return cudaErrorInvalidValue;
        }
    }
    switch (args.epi) {
        case MOE_EPI_STORE_F32:
            err = launch_pdl(grouped_gemm_kernel<MOE_EPI_STORE_F32>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, tmA,
                             tmB, tmB2, args);
            break;
        case MOE_EPI_SILU_MUL_QUANT:
            err = launch_pdl(grouped_gemm_kernel<MOE_EPI_SILU_MUL_QUANT>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, tmA,
                             tmB, tmB2, args);
            break;
        case MOE_EPI_WEIGHTED_SCATTER:
            err = launch_pdl(grouped_gemm_kernel<MOE_EPI_WEIGHTED_SCATTER>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, tmA,
                             tmB, tmB2, args);
            break;
        case MOE_EPI_WEIGHTED_ROWS:
            err = launch_pdl(grouped_gemm_kernel<MOE_EPI_WEIGHTED_ROWS>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, tmA,
                             tmB, tmB2, args);
            break;
        case MOE_EPI_WEIGHTED_PAIRS_BF16:
            err = launch_pdl(grouped_gemm_kernel<MOE_EPI_WEIGHTED_PAIRS_BF16>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, tmA,
                             tmB, tmB2, args);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return err;
}

}  // namespace mfp8
