// Decode-regime expert MLP: the routing, the expert sort and both grouped block-FP8 GEMMs of
// the layer in one persistent launch, for steps of up to 8 tokens (so every expert holds at
// most 8 routed rows).  A small prologue kernel (prologue.cu) zeroes the counters and quantises
// the tokens; it lets this kernel launch at once, and this kernel waits for it only before it
// takes work.  The weighted k-way sum (moe_combine_pairs) follows as its own launch.
//
// The same products as the tile GEMMs (gemm.cu),
//   C[r, n] = sum_kb a_scale[r, kb] * w_scale[e, n/128, kb] * sum_{k in kb} A[r, k] * W[e, n, k],
// with the "[num_experts, N, K]" weights in 128x128 blocks (page "Quantization and MoE
// Optimizations", sections FusedMoE Class and Fp8Config), shaped for weight streaming.  With
// a few rows per expert the layer reads each touched expert's weights once and does two
// flops per weight byte and row: its time is the weight bytes over HBM bandwidth, so every
// SM has to stream weights from the first to the last microsecond.  The 128-row tiles of
// the tile GEMMs give a one-token DeepSeek-V3-shaped step only 128 w13 work items for 152
// SMs (a w13 tile cannot be split further: its 1x128 requantisation groups need all 256 of
// its gate and up rows), and the w2 launch cannot start streaming before the w13 launch has
// drained.  For the same reason the steps before the GEMMs run inside this kernel: with separate
// launches for routing and sort, a one-token step spent 18 us before its first weight load.
//
// Prologue of every CTA (before any weight load): warps 1..T each route one token with the
// routing kernel's selection (route_select.cuh: the same choices, the same arithmetic); the
// CTA sorts the T*topk pairs by (expert, pair) in shared memory into one tile record per
// touched expert (expert, rows, their pairs and tokens), the small-batch sort's order.  The
// fp64 router weights (a few microseconds of dependent fp64 operations on this GPU) are formed
// afterwards by the epilogue warps, idle until the first item is done; on an MMA warp they held
// up the ring for all eight.
// (Shapes whose scores do not fit the register-resident selection take the routing kernel's
// ids and weights instead.)  CTA 0 writes the ids, the weights and each pair's row (-1 for a
// dropped pair) for the k-way sum.
//
// Work items (tickets, taken in order from one counter by the CTAs' producers):
//   first every w13 item: 16 gate rows [16u, 16u+16) and the matching 16 up rows [I+16u, ...)
//   of one expert over the whole K = H;
//   then every w2 item: 32 rows [32u, 32u+32) of one expert over K = I.
// (A one-token DeepSeek-V3 step: 1024 w13 items, then 1792 w2 items.)  A w2 item needs its
// expert's whole requantised intermediate: its producer streams the item's weights at once
// but loads the activation rows only after the expert's I/128 groups are counted as done.
// Tickets are taken in that order by running CTAs, so every w13 item a w2 item waits for is
// held by a running CTA that waits for nothing: the waits end without any assumption about
// how many CTAs are resident.  Dynamic tickets also balance the items over the SMs.
//
// Roles of a CTA (one per SM, 384 threads):
//   warp 0      producer: per group of 16 K blocks of an item, TMA loads of its weight rows
//               over the 16 blocks (w13: two boxes of 16 rows, 32 KB each; w2: one box of 32
//               rows, 64 KB) and of the activation rows over them (w13: the step's token rows,
//               from one of the prologue's copies of them, so that the CTAs' reads of these few
//               lines spread over L2; w2: the tile's rows of the intermediate; a box of 1, 2, 4
//               or 8 rows, the fewest that hold them) into a ring of 2-4 stages, and
//               the blocks' weight-block and activation scales by cp.async, all completing
//               on the stage's mbarrier.  The ring runs on across items and across the two
//               GEMMs.  (On GB300 an SM streams at the HBM share only with large boxes: a
//               probe streaming 16 KB weight boxes lost 16% when each stage added a 1 KB box,
//               none with 32 KB boxes; boxes of one K block, 2 KB each, or activation copies
//               by cp.async were several times slower.)
//   warps 1..8  MMA warps: warp w takes K blocks w-1 and w+7 of every stage; it reads its
//               16-byte pieces from shared memory into registers, releases the stage, and
//               runs the tensor cores' warp-level MMA (mma.sync m16n8k32 e4m3 x e4m3 -> fp32:
//               16 weight rows as the A operand, up to 8 activation rows as B) and promotes
//               the K block's product with its two scales into fp32 accumulators, as the tile
//               GEMM does.  At the end of an item each warp stores its partial sums
//               to one of two reduction buffers and goes on with the next item.
//   warps 9..11 epilogue: add the eight partial sums in warp order (deterministic) and
//               finish the item while the MMA warps stream the next ones.
// The k order inside an MMA is free as long as A and B agree: lane (g, t) gives bytes
// 16t..16t+7 (and 64+16t..) of weight rows g and g+8 and of the tile's activation row g (w13:
// the row of its token) to one MMA and bytes 16t+8..16t+15 to the next, so all lanes with the
// same t hold the same K.
//
// w13 epilogue: h = silu(gate) * up in fp32 for the item's 16 columns, stored to an fp32
// buffer by routed pair.  The eight items of a 1x128 requantisation group count their
// completion on a per-(expert tile, group) counter (a barrier, then one acq_rel atomic add);
// the item that completes the group re-reads the group's 128 values, requantises them
// (amax/448, e4m3 codes) into the expert's padded rows, as the tile GEMM's fused epilogue
// does, and counts the group on the tile's ready counter.  No w13 item waits for another.
// w2 epilogue: bf16(router weight * C) to the pair's row of the [T*topk, H] buffer that the
// k-way sum (moe_combine_pairs) reads, as the tile GEMM's pairs epilogue.  (Forming the sum here
// -- the item that completes 32 output columns adds them up -- took 13 us more on a one-token
// step: the count's release and round trip on every short w2 item held up the epilogue.)
// The counters and the ticket are zeroed by the decode prologue of the same call.  Every wait
// is bounded (mbar_wait, wait_count); on expiry the CTA records MOE_STATUS_WAIT_TIMEOUT,
// lets its loads in flight land and exits.
#include "kernels.cuh"
#include "route_select.cuh"

namespace mfp8 {

namespace {

constexpr int kCols = kDecodeCols;              // routed rows per expert at most: the MMA's 8 B columns
constexpr int kMmaWarps = 8;
constexpr int kEpiWarps = 3;
constexpr int kFirstEpiWarp = 1 + kMmaWarps;
constexpr int kThreads = (1 + kMmaWarps + kEpiWarps) * 32;
constexpr int kMaxStages = 4;
constexpr int kGroupKB = 16;                    // K blocks per stage: two per MMA warp
constexpr int kTileBytes = 16 * 128 * kGroupKB; // 16 weight rows over 16 K blocks
constexpr int kWeightBytes = 2 * kTileBytes;    // a stage's weights: 32 rows over 16 K blocks
// NVFP4 weights: a 16-row slab over 16 K blocks is 16 packed units (codes and block scales)
constexpr int kTileBytes4 = kFp4UnitBytes * kGroupKB;
constexpr int kWeightBytes4 = 2 * kTileBytes4;
constexpr int kStageScales = 2 * kGroupKB + kCols * kGroupKB;   // [tile][kb] weight scales, [kb][row] activation scales
constexpr int kGroupItems = 128 / 16;           // w13 items per 1x128 group of the intermediate
constexpr int kRedBufs = 2;                     // items whose partial sums await the epilogue
constexpr int kTileRows = 128;                  // padded rows per expert tile in a2 (MOE_BLOCK_M)

// Per-expert-tile record of a decode step, built by every CTA in shared memory: the tile's expert,
// its first padded row (m * 128), its routed rows and, for row j < cnt, the pair index, its token
// and its router weight (-1, 0, 0 from cnt on).
struct DecodeTile {
    int32_t e, poff, cnt, pad;   // pad: set once the tile's intermediate was seen complete
    int32_t pair[kCols];
    int32_t tok[kCols];
    float weight[kCols];
};

struct Ctl {
    uint64_t full[kMaxStages];                  // a stage landed (1 + 32 arrivals, tx bytes)
    uint64_t empty[kMaxStages];                 // the MMA warps have read it (8 arrivals)
    uint64_t red_full[kRedBufs];                // all MMA warps stored their partials (8 arrivals)
    uint64_t red_empty[kRedBufs];               // the epilogue has read them (4 arrivals)
    int abort_flag;
    int last;
    int ntiles;                                 // tiles of the step (touched experts)
    double zall[kCols];                         // softmax without renormalisation: each token's sum
    int stage_item[kMaxStages];                 // the stage's item (ticket), -1: no more work
    int stage_grp[kMaxStages];                  // its group of K blocks
    int stage_rows[kMaxStages];                 // activation rows it holds (1, 2, 4 or 8)
    uint32_t stage_tok[kMaxStages];             // w13: B column j reads stage row (tok >> 4j) & 15 (j < cnt)
    int stage_cnt[kMaxStages];                  // the tile's routed rows
    int red_item[kRedBufs];                     // the reduction buffer's item, -1: no more work
    alignas(16) float scl[kMaxStages][kStageScales];
    alignas(16) float red[kRedBufs][kMmaWarps][2][32][4];
};
// shared memory: alignment slack, the control block, the ring (stages x stage bytes: a stage's
// weights, then its activation rows), the step's tile records, the sort's three ints per pair
constexpr size_t kCtlBytes = (sizeof(Ctl) + 1023) / 1024 * 1024;
constexpr size_t kSmemLimit = 232448;
// a stage holds up to `cols` activation rows in a box of the next power of two rows
size_t stage_bytes(int cols, bool fp4 = false) {
    int r = 1;
    while (r < cols) r <<= 1;
    return ((fp4 ? kWeightBytes4 : kWeightBytes) + static_cast<size_t>(r) * 128 * kGroupKB + 1023) / 1024 * 1024;
}
size_t smem_bytes(int max_tiles, int stages, int cols, int pairs, bool fp4 = false) {
    return 1024 + kCtlBytes + static_cast<size_t>(stages) * stage_bytes(cols, fp4) +
           static_cast<size_t>(max_tiles) * sizeof(DecodeTile) + static_cast<size_t>(pairs) * 3 * sizeof(int);
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// d += A(16x32, e4m3) * B(32x8, e4m3), fp32 accumulators
__device__ __forceinline__ void mma_16x8x32(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                            uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d += A(16x16, f16) * B(16x8, f16), fp32 accumulators
__device__ __forceinline__ void mma_16x8x16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                            uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the four bytes of w, each two e2m1 codes (low nibble first), as four f16x2 (byte i -> r[i],
// low nibble in the low half); exact
__device__ __forceinline__ void e2m1x8_f16x2(uint32_t w, uint32_t* r) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(w));
}
// the four e4m3 codes of w as two f16x2 (bytes 0, 1 -> lo; 2, 3 -> hi); exact
__device__ __forceinline__ void e4m3x4_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, h0;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ void epilogue_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

// The counters follow the release / acquire pattern of a CTA-wide barrier: the epilogue
// threads' stores, a barrier among them, then one thread's atomic with release (or acq_rel)
// semantics at GPU scope; the reader acquires, then a barrier among its threads.
__device__ __forceinline__ int atom_add_acq_rel(int32_t* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void red_add_release(int32_t* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded, like mbar_wait) until *p >= target, with acquire ordering.
__device__ __forceinline__ bool wait_count(const int32_t* p, int target, volatile int* abort_flag, uint32_t* status) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        if (ld_acquire(p) >= target) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) break;
        __nanosleep(64);
    }
    *abort_flag = 1;
    status_set(status, MOE_STATUS_WAIT_TIMEOUT);
    return false;
}

// The two GEMMs' shapes: w13 (first) [2I, H], w2 (second) [H, I].
struct Gemm {
    int N, K, KB, GKB, NG, per_tile;
};
__device__ __forceinline__ Gemm gemm_of(const DecodeMlpArgs& a, bool second) {
    Gemm g;
    g.N = second ? a.H : 2 * a.I;
    g.K = second ? a.I : a.H;
    g.KB = g.K / 128;
    g.GKB = g.KB < kGroupKB ? g.KB : kGroupKB;   // K blocks per stage (fewer only when K has fewer)
    g.NG = (g.KB + g.GKB - 1) / g.GKB;           // stages per item
    g.per_tile = g.N / 32;                       // items per expert tile
    return g;
}

// Activation rows of a stage come in boxes of 1, 2, 4 or 8 rows (the fewest that hold the
// item's rows): maps [gemm][log2 rows], gemm 0 = w13 (a1), 1 = w2 (a2).
struct ActMaps {
    CUtensorMap m[2][4];
};

// The step's routing, out of line: called once per token and CTA, these functions hold the
// selection's instantiations and the fp64 exp and division.  Inlined into the kernel they made
// its weight stream slower by 10% at one token (TMA issue-to-landing time per stage 2.2 us
// instead of 1.9 us, measured with the kernel instrumented), and the routing itself slower too.
__device__ __noinline__ int route_token(int route_v, const float* lrow, int E, int topk, int renormalize,
                                        bool sigmoid, int n_group, int topk_group, const float* bias, bool vec_loads,
                                        int lane, double* zall) {
    switch (route_v) {
        case 1:
            return route_token_reg<1, false>(lrow, E, topk, renormalize, sigmoid, n_group, topk_group, bias,
                                             vec_loads, lane, zall);
        case 2:
            return route_token_reg<2, false>(lrow, E, topk, renormalize, sigmoid, n_group, topk_group, bias,
                                             vec_loads, lane, zall);
        case 4:
            return route_token_reg<4, false>(lrow, E, topk, renormalize, sigmoid, n_group, topk_group, bias,
                                             vec_loads, lane, zall);
        default:
            return route_token_reg<8, false>(lrow, E, topk, renormalize, sigmoid, n_group, topk_group, bias,
                                             vec_loads, lane, zall);
    }
}
__device__ __noinline__ float route_weight(const float* lrow, int my_id, bool active, int base, int topk,
                                           int renormalize, bool sigmoid, double zall, float routed_scaling) {
    return route_weight_group(lrow, my_id, active, base, topk, renormalize, sigmoid, zall, routed_scaling);
}

// FP4: NVFP4 weights (nvfp4.cu's packed units); the MMA warps expand each code times its block
// scale to f16 (exact: at most 6 significant bits, |w| <= 6 * 448) and the activation codes to
// f16 (exact), and run f16 MMAs; the expert's 1 / global_scale joins the promotion's scale.
template <bool FP4>
__global__ void __launch_bounds__(kThreads, 1)
    decode_mlp_kernel(const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmW2,
                      const __grid_constant__ ActMaps tmX, const DecodeMlpArgs a) {
    constexpr int kWB = FP4 ? kWeightBytes4 : kWeightBytes;   // a stage's weight bytes: activations follow
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    Ctl* ctl = reinterpret_cast<Ctl*>(base);
    uint8_t* ring = base + kCtlBytes;
    const int S = a.stages;
    const int SB = a.stage_bytes;
    DecodeTile* tab = reinterpret_cast<DecodeTile*>(ring + static_cast<size_t>(S) * SB);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int I = a.I;
    const int GPT = I / 128;                     // 1x128 groups of the intermediate per expert tile
    const int P = a.T * a.topk;                  // routed pairs of the step
    int32_t* group_count = a.counters;           // [max_tiles][I/128]
    int32_t* ready = a.counters + static_cast<int64_t>(a.max_tiles) * GPT;   // [max_tiles]
    int32_t* ticket = ready + a.max_tiles;
    int* s_ids = reinterpret_cast<int*>(tab + a.max_tiles);   // [P] chosen expert of pair p
    int* s_rank = s_ids + P;                     // [P] row of pair p in its tile (-1: dropped)
    int* s_slot = s_rank + P;                    // [P] tile << 8 | row (-1: dropped)

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1 + 32);
            mbar_init(smem_addr(&ctl->empty[s]), kMmaWarps);
        }
        for (int b = 0; b < kRedBufs; ++b) {
            mbar_init(smem_addr(&ctl->red_full[b]), kMmaWarps);
            mbar_init(smem_addr(&ctl->red_empty[b]), kEpiWarps);
        }
        ctl->abort_flag = 0;
        ctl->ntiles = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmW13);
        tma_prefetch_map(&tmW2);
    }
    // The step's routing, in every CTA while the decode prologue still runs: warps 1..T take
    // token warp - 1 with the routing kernel's selection (route_select.cuh).  The scores are the
    // caller's input, complete before the prologue let this grid launch.  Without in-kernel
    // routing (route_v == 0) the routing kernel's ids are read once the earlier grids are done.
    const bool route_here = a.route_v > 0;
    const bool router = route_here && warp >= 1 && warp <= a.T;
    const bool sigmoid = a.scoring == MOE_SCORING_SIGMOID;
    if (router) {
        const float* lrow = a.logits + static_cast<int64_t>(warp - 1) * a.E;
        double zall = 0.0;
        const int my_id = route_token(a.route_v, lrow, a.E, a.topk, a.renormalize, sigmoid, a.n_group, a.topk_group,
                                      a.bias, a.vec_loads != 0, lane, &zall);
        if (lane < a.topk) s_ids[(warp - 1) * a.topk + lane] = my_id;
        if (lane == 0) ctl->zall[warp - 1] = zall;
    }
    if (!route_here) {
        grid_dependency_wait();
        for (int p = threadIdx.x; p < P; p += blockDim.x) s_ids[p] = __ldcg(a.ids + p);
    }
    __syncthreads();
    // the decode prologue's outputs (zeroed counters, quantised tokens) from here on; the first two
    // tickets go out now, their round trip under the sort
    if (route_here) grid_dependency_wait();
    int ticket0 = 0, ticket1 = 0;
    if (warp == 0 && lane == 0) {
        ticket0 = atomicAdd(ticket, 1);
        ticket1 = atomicAdd(ticket, 1);
    }
    // The expert sort, in shared memory: pair p's row is the number of earlier pairs with its
    // expert (a stable order by (expert, pair)); one tile per touched expert, in expert order, at
    // padded row m * 128 of the intermediate -- the small-batch sort's layout.  An id out of range
    // drops its pair and is reported.
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int id = s_ids[p];
        int rank = -1;
        if (id >= 0 && id < a.E) {
            rank = 0;
            for (int o = 0; o < p; ++o) rank += s_ids[o] == id ? 1 : 0;
            if (rank == 0) atomicAdd(&ctl->ntiles, 1);
        } else {
            status_set(a.status, MOE_STATUS_BAD_EXPERT_ID);
        }
        s_rank[p] = rank;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int id = s_ids[p], rank = s_rank[p];
        int slot = -1;
        if (rank >= 0) {
            int m = 0, cnt = 0;
            for (int o = 0; o < P; ++o) {
                m += (s_rank[o] == 0 && s_ids[o] < id) ? 1 : 0;
                cnt += s_ids[o] == id ? 1 : 0;
            }
            if (m < a.max_tiles) {
                // (an expert with more rows than the kernel takes is reported by the epilogue)
                if (rank < kCols) slot = (m << 8) | rank;
                if (rank == 0) {
                    DecodeTile& d = tab[m];
                    d.e = id;
                    d.poff = m * kTileRows;
                    d.cnt = cnt;
                    d.pad = 0;
                    for (int j = cnt; j < kCols; ++j) {
                        d.pair[j] = -1;
                        d.tok[j] = 0;
                        d.weight[j] = 0.0f;
                    }
                }
            }
        }
        s_slot[p] = slot;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int slot = s_slot[p];
        if (blockIdx.x == 0) a.pos[p] = slot < 0 ? -1 : (slot >> 8) * kTileRows + (slot & 255);
        if (slot < 0) continue;
        DecodeTile& d = tab[slot >> 8];
        d.pair[slot & 255] = p;
        d.tok[slot & 255] = p / a.topk;
        d.weight[slot & 255] = route_here ? 0.0f : __ldcg(a.wts + p);
    }
    __syncthreads();
    int64_t ntiles = ctl->ntiles;
    if (ntiles > a.max_tiles) ntiles = a.max_tiles;
    const Gemm G1 = gemm_of(a, false), G2 = gemm_of(a, true);
    const int total1 = static_cast<int>(ntiles * G1.per_tile);
    const int total = total1 + static_cast<int>(ntiles * G2.per_tile);
    volatile int* abort_flag = &ctl->abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        const int xcopy = static_cast<int>(blockIdx.x) % a.x_copies;   // this CTA's copy of the token rows
        uint32_t q = 0;
        bool ok = true;
        // tickets are taken two items ahead: an atomic's round trip is longer than a w2 item's issue
        int item = __shfl_sync(0xffffffffu, ticket0, 0);
        int next = ticket1;
        while (ok) {
            if (item >= total) {
                // no more work: a stage that says so
                const uint32_t stage = q % S, use = q / S;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->empty[stage]), (use & 1u) ^ 1u, abort_flag,
                                                       a.status)))
                    ok = false;
                if (ok) {
                    const uint32_t fb = smem_addr(&ctl->full[stage]);
                    if (lane == 0) {
                        ctl->stage_item[stage] = -1;
                        mbar_arrive(fb);
                    }
                    cp_async_arrive(fb);
                    ++q;
                }
                break;
            }
            const int next2 = lane == 0 ? atomicAdd(ticket, 1) : 0;
            const bool second = item >= total1;
            const Gemm& G = second ? G2 : G1;
            const int w = second ? item - total1 : item;
            const int m = w / G.per_tile, u = w - m * G.per_tile;
            // (a record with an expert out of range -- the sort writes none -- streams expert 0
            // and its item's output is dropped by the epilogue)
            const int e = (tab[m].e >= 0 && tab[m].e < a.E) ? tab[m].e : 0;
            const int poff = tab[m].poff;
            const int row0 = second ? u * 32 : u * 16;
            const int row1 = second ? u * 32 + 16 : I + u * 16;
            const int NB = G.N / 128;
            const CUtensorMap* tmW = second ? &tmW2 : &tmW13;
            const float* wsc = second ? a.w2_scale : a.w13_scale;
            const float* ws[2] = {wsc + (static_cast<int64_t>(e) * NB + row0 / 128) * G.KB,
                                  wsc + (static_cast<int64_t>(e) * NB + row1 / 128) * G.KB};
            // activation scales of K block kb: w13 [copy][kb][token] (ld kCols), w2 [kb][padded row]
            const float* xsc = second ? a.a2s + poff : a.a1s + static_cast<int64_t>(xcopy) * (a.H / 128) * kCols;
            const int64_t xs_ld = second ? a.rows : kCols;
            uint32_t tokmap = 0;
            if (!second)
                for (int j = 0; j < kCols; ++j) tokmap |= static_cast<uint32_t>(tab[m].tok[j] & 15) << (4 * j);
            // activation rows: w13 the step's T token rows, w2 the tile's rows of the intermediate,
            // rounded up to a power of two
            int cnt = second ? tab[m].cnt : a.T;
            cnt = cnt < 1 ? 1 : (cnt > a.cols ? a.cols : cnt);
            const int lg = cnt <= 1 ? 0 : cnt <= 2 ? 1 : cnt <= 4 ? 2 : 3;
            const CUtensorMap* tmA = &tmX.m[second ? 1 : 0][lg];
            // bytes per stage: weights (w13: two 16-row boxes; w2: one 32-row box; NVFP4: two 16-row
            // slabs of packed units) + activations
            const uint32_t stage_tx = FP4 ? static_cast<uint32_t>((2 * kFp4UnitBytes + (1 << lg) * 128) * G.GKB)
                                          : static_cast<uint32_t>((32 + (1 << lg)) * 128 * G.GKB);
            for (int grp = 0; grp < G.NG; ++grp, ++q) {
                const uint32_t stage = q % S, use = q / S;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->empty[stage]), (use & 1u) ^ 1u, abort_flag,
                                                       a.status))) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_addr(&ctl->full[stage]);
                uint8_t* st = ring + static_cast<size_t>(stage) * SB;
                const uint32_t dst = smem_addr(st);
                const int kb0 = grp * G.GKB;
                if (lane == 0) {
                    ctl->stage_item[stage] = item;
                    ctl->stage_grp[stage] = grp;
                    ctl->stage_rows[stage] = 1 << lg;
                    ctl->stage_tok[stage] = tokmap;
                    ctl->stage_cnt[stage] = tab[m].cnt;
                    // K blocks past K are out of the tensor: zero-filled (and counted), and skipped
                    // by the MMA warps
                    mbar_arrive_expect_tx(fb, stage_tx);
                    // the item's weight rows over the stage's K blocks: w2 one box of 32 rows, w13
                    // a box of its 16 gate rows and one of its 16 up rows (I rows apart)
                    if constexpr (FP4) {
                        // slabs of 16 rows: w2 rows [32u, 32u + 32), w13 gate [16u, ...) and up [I + 16u, ...)
                        const int slab0 = e * (G.N / 16) + row0 / 16, slab1 = e * (G.N / 16) + row1 / 16;
                        tma_load_4d(dst, tmW, 0, 0, kb0, slab0, fb);
                        tma_load_4d(dst + kTileBytes4, tmW, 0, 0, kb0, slab1, fb);
                    } else if (second) {
                        if (a.w_tiled)
                            tma_load_4d(dst, tmW, 0, row0 % 128, kb0, e * NB + row0 / 128, fb);
                        else
                            tma_load_3d(dst, tmW, 0, kb0, e * G.N + row0, fb);
                    } else if (a.w_tiled) {
                        tma_load_4d(dst, tmW, 0, row0 % 128, kb0, e * NB + row0 / 128, fb);
                        tma_load_4d(dst + kTileBytes, tmW, 0, row1 % 128, kb0, e * NB + row1 / 128, fb);
                    } else {
                        tma_load_3d(dst, tmW, 0, kb0, e * G.N + row0, fb);
                        tma_load_3d(dst + kTileBytes, tmW, 0, kb0, e * G.N + row1, fb);
                    }
                }
                bool got = true;
                if (second && grp == 0 && tab[m].pad == 0) {
                    // the expert's requantised intermediate is complete once its I/128 groups are
                    // counted; every lane acquires it before its loads of the activations, once
                    // per tile (the record's spare field remembers it)
                    got = lane == 0 ? wait_count(ready + m, GPT, abort_flag, a.status) : true;
                    got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                    if (got) got = ld_acquire(ready + m) >= GPT;
                    got = __all_sync(0xffffffffu, got);
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __syncwarp();
                    if (got && lane == 0) tab[m].pad = 1;
                    __syncwarp();
                }
                // the activation rows of the stage's K blocks (after a failed wait the load still
                // goes out, so that the stage's phase completes and the drain below can wait for
                // it; the status word marks the outputs invalid)
                if (lane == 0) tma_load_3d(dst + kWB, tmA, 0, kb0, second ? poff : xcopy * a.T, fb);
                if constexpr (FP4) {
                    // the expert's 1 / global_scale (the block scales came with the codes)
                    if (lane == 0) cp_async_4(smem_addr(&ctl->scl[stage][0]), wsc + e);
                } else {
                    // weight-block scales (read-only here: 4-byte copies through L1), lane = tile * 16 + kbi
                    const int kbi = lane % kGroupKB, kb = kb0 + kbi;
                    if (kbi < G.GKB && kb < G.KB)
                        cp_async_4(smem_addr(&ctl->scl[stage][lane]), ws[lane / kGroupKB] + kb);
                }
                {
                    // activation scales of a K block's 8 rows, two 16-byte copies that bypass L1 (the
                    // w13 items of other SMs write the intermediate's scales during the kernel)
                    const int kbi = lane >> 1, c = lane & 1, kb = kb0 + kbi;
                    if (kbi < G.GKB && kb < G.KB)
                        cp_async_16(smem_addr(&ctl->scl[stage][2 * kGroupKB + kbi * kCols + 4 * c]),
                                    xsc + static_cast<int64_t>(kb) * xs_ld + 4 * c);
                }
                cp_async_arrive(fb);
                if (!got) {
                    ok = false;
                    ++q;
                    break;
                }
            }
            item = __shfl_sync(0xffffffffu, next, 0);
            next = next2;
        }
        if (!ok) {
            // let every stage load already issued land before the CTA exits
            for (uint32_t s = 0; s < static_cast<uint32_t>(S) && lane == 0; ++s) {
                const uint32_t n_s = (q + S - 1 - s) / S;
                if (n_s > 0) mbar_wait(smem_addr(&ctl->full[s]), (n_s - 1) & 1u, nullptr, a.status);
            }
        }
        cp_async_wait_all();
    } else if (warp < kFirstEpiWarp) {
        // ------------------------------------------------------------------ MMA warps
        const int cw = warp - 1;
        const int g = lane >> 2, t = lane & 3;
        uint32_t q = 0, iter = 0;
        float acc[2][4];
#pragma unroll
        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[tile][i] = 0.0f;
        while (true) {
            const uint32_t stage = q % S;
            if (!mbar_wait(smem_addr(&ctl->full[stage]), (q / S) & 1u, abort_flag, a.status)) break;
            ++q;
            const int item = ctl->stage_item[stage];
            if (item < 0) {
                // no more work: pass that on to the epilogue
                const uint32_t buf = iter % kRedBufs, use = iter / kRedBufs;
                if (use > 0 && !mbar_wait(smem_addr(&ctl->red_empty[buf]), (use - 1) & 1u, abort_flag, a.status))
                    break;
                if (cw == 0 && lane == 0) ctl->red_item[buf] = -1;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->red_full[buf]));
                break;
            }
            const int grp = ctl->stage_grp[stage];
            const bool second = item >= total1;
            const Gemm& G = second ? G2 : G1;
            const uint8_t* st = ring + static_cast<size_t>(stage) * SB;
            const int xr = ctl->stage_rows[stage];
            // B column g is the tile's row g: for w13 the row of its token among the stage's token
            // rows (columns past the tile's rows are zero, their results never read), for w2 row g
            const uint32_t tokmap = ctl->stage_tok[stage];
            const int xrow = second ? g : static_cast<int>((tokmap >> (4 * g)) & 15u);
            const bool xlive = second ? g < xr : g < ctl->stage_cnt[stage];
            const int sc0 = second ? 2 * t : static_cast<int>((tokmap >> (8 * t)) & 15u);
            const int sc1 = second ? 2 * t + 1 : static_cast<int>((tokmap >> (8 * t + 4)) & 15u);
            if constexpr (FP4) {
                // this warp's K blocks of the stage, cw and cw + 8.  Lane (g, t) feeds K positions
                // [32t, 32t + 32) of a block (any K order works when A and B agree): MMA j takes
                // positions 32t + 4j + {0, 1} (A/B registers 0) and + {2, 3} (registers 1), i.e.
                // code bytes 2j and 2j + 1 of the lane's 16 and activation bytes 4j .. 4j + 3 of its
                // 32; positions below 32t + 16 use block scale 2t, the others 2t + 1.
                uint4 cv[2][2][2], xq[2][2];   // [half][tile][row g / g+8] codes, [half][16-byte half] activations
                uint32_t sv[2][2][2];          // [half][tile][row] the two block scales' bytes
                float xa[2], xb[2];
                bool live[2];
                const float gsc = ctl->scl[stage][0];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int kbi = cw + 8 * half, kb = grp * G.GKB + kbi;
                    live[half] = kbi < G.GKB && kb < G.KB;
                    if (!live[half]) continue;
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const uint8_t* up = st + tile * kTileBytes4 + kbi * kFp4UnitBytes;
                            const int r16 = g + 8 * hr;
                            cv[half][tile][hr] = *reinterpret_cast<const uint4*>(up + r16 * 64 + 16 * t);
                            sv[half][tile][hr] = *reinterpret_cast<const uint16_t*>(up + 16 * 64 + r16 * 8 + 2 * t);
                        }
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        xq[half][c] = xlive ? *reinterpret_cast<const uint4*>(st + kWB + (xrow * G.GKB + kbi) * 128 +
                                                                              32 * t + 16 * c)
                                            : make_uint4(0u, 0u, 0u, 0u);
                    xa[half] = ctl->scl[stage][2 * kGroupKB + kbi * kCols + sc0];
                    xb[half] = ctl->scl[stage][2 * kGroupKB + kbi * kCols + sc1];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (!live[half]) continue;
                    uint32_t s2[2][2][2];   // [tile][row][block 2t / 2t+1] the scale in both f16 halves
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            uint32_t sc, unused;
                            e4m3x4_f16x2(sv[half][tile][hr], sc, unused);
                            s2[tile][hr][0] = __byte_perm(sc, 0u, 0x1010);
                            s2[tile][hr][1] = __byte_perm(sc, 0u, 0x3232);
                        }
                    float f[2][2][4];   // [tile][chain: j even / odd]
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int i = 0; i < 4; ++i) f[tile][c][i] = 0.0f;
#pragma unroll
                    for (int jw = 0; jw < 4; ++jw) {
                        // code word jw of each row holds MMAs 2jw and 2jw + 1 (two bytes each)
                        uint32_t r[2][2][4];   // [tile][row] the word's four bytes as f16x2
#pragma unroll
                        for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                            for (int hr = 0; hr < 2; ++hr) e2m1x8_f16x2(word(cv[half][tile][hr], jw), r[tile][hr]);
                        const int blk = jw >> 1;
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int j = 2 * jw + jj;
                            uint32_t b0, b1;
                            e4m3x4_f16x2(word(xq[half][j >> 2], j & 3), b0, b1);
#pragma unroll
                            for (int tile = 0; tile < 2; ++tile)
                                mma_16x8x16(f[tile][jj], hmul2(r[tile][0][2 * jj], s2[tile][0][blk]),
                                            hmul2(r[tile][1][2 * jj], s2[tile][1][blk]),
                                            hmul2(r[tile][0][2 * jj + 1], s2[tile][0][blk]),
                                            hmul2(r[tile][1][2 * jj + 1], s2[tile][1][blk]), b0, b1);
                        }
                    }
                    // accumulator (row g / g+8, column 2t / 2t+1): the expert's 1 / global_scale times
                    // the column's activation scale
                    const float s0 = gsc * xa[half], s1 = gsc * xb[half];
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        acc[tile][0] = fmaf(f[tile][0][0] + f[tile][1][0], s0, acc[tile][0]);
                        acc[tile][1] = fmaf(f[tile][0][1] + f[tile][1][1], s1, acc[tile][1]);
                        acc[tile][2] = fmaf(f[tile][0][2] + f[tile][1][2], s0, acc[tile][2]);
                        acc[tile][3] = fmaf(f[tile][0][3] + f[tile][1][3], s1, acc[tile][3]);
                    }
                }
            } else {
                // this warp's K blocks of the stage, cw and cw + 8: both into registers, the stage
                // released, then their MMAs
                uint4 wv[2][2][2][2], xv[2][2];   // [half][tile][row g / g+8][K half c], [half][K half c]
                float ws[2][2], xa[2], xb[2];
                bool live[2];
    #pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int kbi = cw + 8 * half, kb = grp * G.GKB + kbi;
                    live[half] = kbi < G.GKB && kb < G.KB;
                    if (!live[half]) continue;
                    // 128-byte rows of the stage's weight boxes, tile-packed with the 128-byte swizzle:
                    //   w2: [K block][32 rows]       w13: gate box, up box, each [K block][16 rows]
                    // [E, N, K] without swizzle:
                    //   w2: [32 rows][K block]       w13: gate box, up box, each [16 rows][K block]
    #pragma unroll
                    for (int tile = 0; tile < 2; ++tile)
    #pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int r16 = g + 8 * hr;   // row within the 16-row tile
                            int box, srow;   // the box's offset in the stage, the row within the box
                            if (second) {
                                box = 0;
                                srow = a.w_tiled ? kbi * 32 + 16 * tile + r16 : (16 * tile + r16) * G.GKB + kbi;
                            } else {
                                box = tile * kTileBytes;
                                srow = a.w_tiled ? kbi * 16 + r16 : r16 * G.GKB + kbi;
                            }
                            const int x = a.w_tiled ? (r16 & 7) : 0;   // == srow & 7 when tiled
                            const uint8_t* rp = st + box + srow * 128;
    #pragma unroll
                            for (int c = 0; c < 2; ++c)
                                wv[half][tile][hr][c] = *reinterpret_cast<const uint4*>(rp + 16 * ((4 * c + t) ^ x));
                        }
    #pragma unroll
                    for (int c = 0; c < 2; ++c)
                        xv[half][c] = xlive ? *reinterpret_cast<const uint4*>(st + kWB + (xrow * G.GKB + kbi) * 128 +
                                                                              64 * c + 16 * t)
                                            : make_uint4(0u, 0u, 0u, 0u);
                    ws[half][0] = ctl->scl[stage][kbi];
                    ws[half][1] = ctl->scl[stage][kGroupKB + kbi];
                    xa[half] = ctl->scl[stage][2 * kGroupKB + kbi * kCols + sc0];
                    xb[half] = ctl->scl[stage][2 * kGroupKB + kbi * kCols + sc1];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
    #pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (!live[half]) continue;
                    // four independent chains (tile, K half c) of two MMAs each
                    float f[2][2][4];
    #pragma unroll
                    for (int tile = 0; tile < 2; ++tile)
    #pragma unroll
                        for (int c = 0; c < 2; ++c)
    #pragma unroll
                            for (int i = 0; i < 4; ++i) f[tile][c][i] = 0.0f;
    #pragma unroll
                    for (int h = 0; h < 2; ++h)
    #pragma unroll
                        for (int tile = 0; tile < 2; ++tile)
    #pragma unroll
                            for (int c = 0; c < 2; ++c)
                                mma_16x8x32(f[tile][c], word(wv[half][tile][0][c], 2 * h),
                                            word(wv[half][tile][1][c], 2 * h), word(wv[half][tile][0][c], 2 * h + 1),
                                            word(wv[half][tile][1][c], 2 * h + 1), word(xv[half][c], 2 * h),
                                            word(xv[half][c], 2 * h + 1));
    #pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        // accumulator (row g / g+8, column 2t / 2t+1): the weight block's scale times the
                        // column's activation scale
                        const float s0 = ws[half][tile] * xa[half], s1 = ws[half][tile] * xb[half];
                        acc[tile][0] = fmaf(f[tile][0][0] + f[tile][1][0], s0, acc[tile][0]);
                        acc[tile][1] = fmaf(f[tile][0][1] + f[tile][1][1], s1, acc[tile][1]);
                        acc[tile][2] = fmaf(f[tile][0][2] + f[tile][1][2], s0, acc[tile][2]);
                        acc[tile][3] = fmaf(f[tile][0][3] + f[tile][1][3], s1, acc[tile][3]);
                    }
                }
            }
            if (grp == G.NG - 1) {
                // the item's last stage: partial sums to a reduction buffer
                const uint32_t buf = iter % kRedBufs, use = iter / kRedBufs;
                if (use > 0 && !mbar_wait(smem_addr(&ctl->red_empty[buf]), (use - 1) & 1u, abort_flag, a.status))
                    break;
#pragma unroll
                for (int tile = 0; tile < 2; ++tile) {
                    *reinterpret_cast<float4*>(&ctl->red[buf][cw][tile][lane][0]) =
                        make_float4(acc[tile][0], acc[tile][1], acc[tile][2], acc[tile][3]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[tile][i] = 0.0f;
                }
                if (cw == 0 && lane == 0) ctl->red_item[buf] = item;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->red_full[buf]));
                ++iter;
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue warps
        const int et = threadIdx.x - kFirstEpiWarp * 32;   // 0..95
        const int ew = warp - kFirstEpiWarp;
        if (route_here) {
            // the router weights in fp64, as the routing kernel forms them: lane groups of topk
            // lanes take one token each (all of a step's tokens in one round for topk <= 8); read
            // by the w2 epilogue after the barrier below; CTA 0 writes ids and weights out
            const int per_warp = 32 / a.topk;
            for (int t0 = ew * per_warp; t0 < a.T; t0 += kEpiWarps * per_warp) {
                const int j = lane % a.topk, t = t0 + lane / a.topk;
                const bool active = lane / a.topk < per_warp && t < a.T;
                const int p = active ? t * a.topk + j : 0;
                const int id = active ? s_ids[p] : -1;
                const float wgt = route_weight(a.logits + static_cast<int64_t>(active ? t : 0) * a.E, id, active,
                                               lane - j, a.topk, a.renormalize, sigmoid, ctl->zall[active ? t : 0],
                                               a.routed_scaling);
                if (active) {
                    const int slot = s_slot[p];
                    if (slot >= 0) tab[slot >> 8].weight[slot & 255] = wgt;
                    if (blockIdx.x == 0) {
                        a.ids[p] = id;
                        a.wts[p] = wgt;
                    }
                }
            }
            epilogue_barrier();
        }
        uint32_t iter = 0;
        while (true) {
            const uint32_t buf = iter % kRedBufs;
            if (!mbar_wait(smem_addr(&ctl->red_full[buf]), (iter / kRedBufs) & 1u, abort_flag, a.status)) break;
            const int item = ctl->red_item[buf];
            if (item < 0) break;
            const bool second = item >= total1;
            const Gemm& G = second ? G2 : G1;
            const int w = second ? item - total1 : item;
            const int m = w / G.per_tile, u = w - m * G.per_tile;
            const DecodeTile& tl = tab[m];
            const bool valid = tl.e >= 0 && tl.e < a.E;
            const int poff = tl.poff;
            int cnt = valid ? tl.cnt : 0;
            if (!valid || cnt > a.cols) {
                // the sort lists valid experts with at most one row per token, and a.cols is the
                // step's token count (at most 8)
                status_set(a.status, MOE_STATUS_BAD_EXPERT_ID);
                cnt = cnt > a.cols ? a.cols : cnt;
            }
            // partial sums of (row rr of a 16-row tile, column jj): lane (rr % 8) * 4 + jj / 2,
            // register (rr >= 8 ? 2 : 0) + (jj & 1), added in warp order
            auto total_of = [&](int tile, int rr, int jj) {
                const int l = (rr & 7) * 4 + (jj >> 1), c = ((rr >> 3) << 1) + (jj & 1);
                float s = 0.0f;
#pragma unroll
                for (int cw = 0; cw < kMmaWarps; ++cw) s += ctl->red[buf][cw][tile][l][c];
                return s;
            };
            // the item's outputs, consecutive threads on consecutive rows of one column: w2 32 rows
            // x 8 columns (bf16(router weight * C) to the pair's row of y), w13 16 rows x 8 columns
            // (h = silu(gate) * up by pair; silu(g) * up = g * up / (1 + e^-g), as the tile GEMM)
            const int rows = second ? 32 : 16;
            for (int idx = et; idx < rows * kCols; idx += kEpiWarps * 32) {
                const int r = idx % rows, j = idx / rows;
                if (j >= cnt) continue;
                if (second) {
                    const float v = total_of(r >> 4, r & 15, j);
                    a.y[static_cast<int64_t>(tl.pair[j]) * a.H + u * 32 + r] =
                        static_cast<uint16_t>(bf16x2(tl.weight[j] * v, 0.0f) & 0xFFFFu);
                } else {
                    const float gate = total_of(0, r, j), up = total_of(1, r, j);
                    a.h[static_cast<int64_t>(tl.pair[j]) * I + u * 16 + r] =
                        __fdividef(gate * up, 1.0f + __expf(-gate));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl->red_empty[buf]));
            ++iter;
            if (second) continue;
            // the item that completes a 1x128 group requantises it
            epilogue_barrier();
            const int grp = u / kGroupItems;
            if (et == 0) {
                int32_t* counter = group_count + static_cast<int64_t>(m) * GPT + grp;
                ctl->last = atom_add_acq_rel(counter, 1) == kGroupItems - 1;
            }
            epilogue_barrier();
            const int last = ctl->last;
            epilogue_barrier();   // ctl->last is rewritten by the next item
            if (!last) continue;
            for (int jj = ew; jj < cnt; jj += kEpiWarps) {
                const int64_t p = tl.pair[jj];
                const float4 v = __ldcg(reinterpret_cast<const float4*>(a.h + p * I + grp * 128 + lane * 4));
                float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const float sc = group_scale_fmt(amax, a.scale_fmt);
                const float rsc = __frcp_rn(sc);
                const uint32_t lo = e4m3x2(div_by_scale(v.x, sc, rsc), div_by_scale(v.y, sc, rsc));
                const uint32_t hi = e4m3x2(div_by_scale(v.z, sc, rsc), div_by_scale(v.w, sc, rsc));
                const int64_t row = poff + jj;
                *reinterpret_cast<uint32_t*>(a.a2 + row * I + grp * 128 + lane * 4) = lo | (hi << 16);
                if (lane == 0) a.a2s[static_cast<int64_t>(grp) * a.rows + row] = sc;
            }
            // count the group on the tile: its w2 items may load it once all I/128 are counted
            epilogue_barrier();
            if (et == 0) red_add_release(ready + m, 1);
        }
    }
}

}  // namespace

int decode_cols(int T) { return T >= 1 && T <= kCols ? T : 0; }

size_t decode_max_tiles() {
    // room for two stages of 8 activation rows and the sort of the most pairs a step can have
    return (kSmemLimit - smem_bytes(0, 2, kCols, kSmallPairs)) / sizeof(DecodeTile);
}

int64_t decode_counters(int max_tiles, int I) { return static_cast<int64_t>(max_tiles) * (I / 128 + 1) + 1; }

cudaError_t decode_init_device() {
    cudaError_t e = cudaFuncSetAttribute(decode_mlp_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemLimit));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_mlp_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemLimit));
    return e;
}

namespace {

// Weight boxes of `rows` rows x GKB K blocks.  Tile-packed weights [E*N/128 blocks][K/128][128
// rows][128 bytes] get the 128-byte swizzle: in shared memory the rows of a box are consecutive,
// so lanes reading the same 16 bytes of 8 consecutive rows hit 8 different bank groups.  The
// pages' [E*N rows][K/128][128 bytes] get none.
cudaError_t weight_map(CUtensorMap* map, const uint8_t* w, bool tiled, int E, int N, int K, uint32_t rows) {
    const uint64_t KB = static_cast<uint64_t>(K / 128);
    const uint32_t GKB = static_cast<uint32_t>(KB < kGroupKB ? KB : kGroupKB);
    if (tiled) {
        const uint64_t dims[4] = {128, 128, KB, static_cast<uint64_t>(E) * (N / 128)};
        const uint64_t strides[3] = {128, 128 * 128, KB * 128 * 128};
        const uint32_t box[4] = {128, rows, GKB, 1};
        return encode_u8_map_nd(map, w, 4, dims, strides, box, true);
    }
    const uint64_t dims[3] = {128, KB, static_cast<uint64_t>(E) * N};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(K)};
    const uint32_t box[3] = {128, GKB, rows};
    return encode_u8_map_nd(map, w, 3, dims, strides, box, false);
}

// NVFP4-packed weights [E*N/16 slabs][K/128][9][128 bytes] (nvfp4.cu's units): boxes of one slab
// x GKB K blocks, one contiguous run; in shared memory each unit's 16 rows of 64 code bytes are
// consecutive, so the 8 lanes of a quarter-warp (two rows, four 16-byte pieces) read 128
// consecutive bytes
cudaError_t fp4_weight_map(CUtensorMap* map, const uint8_t* w, int E, int N, int K) {
    const uint64_t KB = static_cast<uint64_t>(K / 128);
    const uint32_t GKB = static_cast<uint32_t>(KB < kGroupKB ? KB : kGroupKB);
    const uint64_t dims[4] = {128, kFp4UnitBytes / 128, KB, static_cast<uint64_t>(E) * (N / 16)};
    const uint64_t strides[3] = {128, kFp4UnitBytes, KB * kFp4UnitBytes};
    const uint32_t box[4] = {128, kFp4UnitBytes / 128, GKB, 1};
    return encode_u8_map_nd(map, w, 4, dims, strides, box, false);
}

// activations [rows][K/128][128 bytes]: boxes of `r` rows x GKB K blocks
cudaError_t act_map(CUtensorMap* map, const uint8_t* x, int64_t rows, int K, uint32_t r) {
    const uint64_t KB = static_cast<uint64_t>(K / 128);
    const uint32_t GKB = static_cast<uint32_t>(KB < kGroupKB ? KB : kGroupKB);
    const uint64_t dims[3] = {128, KB, static_cast<uint64_t>(rows)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(K)};
    const uint32_t box[3] = {128, GKB, r};
    return encode_u8_map_nd(map, x, 3, dims, strides, box, false);
}

}  // namespace

cudaError_t launch_decode_mlp(const DecodeMlpArgs& args, int num_sms, cudaStream_t stream) {
    if (args.max_tiles <= 0) return cudaSuccess;
    if (args.cols < 1 || args.cols > kCols || args.H % 128 != 0 || args.I % 128 != 0) return cudaErrorInvalidValue;
    if (args.T < 1 || args.T > kCols || args.topk < 1 || args.T * args.topk > kSmallPairs) return cudaErrorInvalidValue;
    if (args.route_v != 0 && args.route_v != 1 && args.route_v != 2 && args.route_v != 4 && args.route_v != 8)
        return cudaErrorInvalidValue;
    if (args.x_copies < 1 || static_cast<int64_t>(args.x_copies) * args.T + kCols > args.rows) return cudaErrorInvalidValue;
    DecodeMlpArgs a = args;
    // as many ring stages as fit next to the control block and the tile records
    const bool fp4 = a.w_fp4 != 0;
    a.stage_bytes = static_cast<int>(stage_bytes(a.cols, fp4));
    const int pairs = a.T * a.topk;
    const size_t fixed = smem_bytes(a.max_tiles, 0, a.cols, pairs, fp4);
    if (fixed + 2 * static_cast<size_t>(a.stage_bytes) > kSmemLimit) return cudaErrorInvalidValue;
    a.stages = static_cast<int>((kSmemLimit - fixed) / a.stage_bytes);
    if (a.stages > kMaxStages) a.stages = kMaxStages;
    const size_t smem = smem_bytes(a.max_tiles, a.stages, a.cols, pairs, fp4);
    CUtensorMap tmW13, tmW2;
    cudaError_t err;
    if (fp4) {
        err = fp4_weight_map(&tmW13, a.w13, a.E, 2 * a.I, a.H);
        if (err == cudaSuccess) err = fp4_weight_map(&tmW2, a.w2, a.E, a.H, a.I);
    } else {
        err = weight_map(&tmW13, a.w13, a.w_tiled != 0, a.E, 2 * a.I, a.H, 16);
        if (err == cudaSuccess) err = weight_map(&tmW2, a.w2, a.w_tiled != 0, a.E, a.H, a.I, 32);
    }
    ActMaps tmX;
    for (int lg = 0; lg < 4 && err == cudaSuccess; ++lg) {
        err = act_map(&tmX.m[0][lg], a.a1, a.rows, a.H, 1u << lg);
        if (err == cudaSuccess) err = act_map(&tmX.m[1][lg], a.a2, a.rows, a.I, 1u << lg);
    }
    if (err != cudaSuccess) return err;
    const int64_t items = static_cast<int64_t>(a.max_tiles) * (2 * a.I / 32 + a.H / 32);
    const unsigned grid = static_cast<unsigned>(items < num_sms ? items : num_sms);
    if (fp4) return launch_pdl(decode_mlp_kernel<true>, dim3(grid), dim3(kThreads), smem, stream, tmW13, tmW2, tmX, a);
    return launch_pdl(decode_mlp_kernel<false>, dim3(grid), dim3(kThreads), smem, stream, tmW13, tmW2, tmX, a);
}

}  // namespace mfp8
