// Decode-regime expert GEMMs: the two grouped block-FP8 GEMMs of the layer when every
// expert holds at most 8 routed rows (a decode step of up to 8 tokens).
//
// The same products as the tensor-core grouped GEMM (gemm.cu),
//   C[r, n] = sum_kb a_scale[r, kb] * w_scale[e, n/128, kb] * sum_{k in kb} A[r, k] * W[e, n, k],
// with the "[num_experts, N, K]" weights in 128x128 blocks (page "Quantization and MoE
// Optimizations", sections FusedMoE Class and Fp8Config), shaped for weight streaming.
// With a few rows per expert the layer reads each touched expert's weights once and does
// two flops per weight byte and row: its time is the weight bytes over HBM bandwidth, so
// every SM has to stream weights for the whole kernel.  The 128-row tiles of the tile
// GEMM give a one-token DeepSeek-V3-shaped step only 128 w13 work items (8 experts x 16
// groups of 128 gate + 128 up rows) for 152 SMs, and a w13 tile cannot be split further
// because its 1x128 requantisation group needs all 256 of its rows.
//
// Here a work item is 32 weight rows of one expert over the whole K:
//   w13: 16 gate rows [16u, 16u+16) and the matching 16 up rows [I+16u, ...)
//   w2 : 32 rows [32u, 32u+32)
// (a one-token DeepSeek-V3 step: 1024 w13 items and 1792 w2 items).  One persistent CTA
// per SM takes every gridDim-th item.  Roles (416 threads):
//   warp 0      producer: per group of 8 K blocks of an item, one TMA load of each 16-row
//               weight tile over the 8 blocks (16 KB each) and one of the expert's 8
//               activation rows over them (8 KB) into a 4-stage ring (40 KB a stage, 160 KB
//               in flight), and the blocks' weight-block and activation scales by cp.async,
//               all completing on the stage's mbarrier.  The ring runs on across items.
//               (Boxes of one K block, 2 KB each, kept too few bytes in flight per SM.)
//   warps 1..8  MMA warps: warp w takes K block w-1 of every stage; it reads its 16-byte
//               pieces from shared memory, releases the stage, and runs the tensor cores'
//               warp-level MMA (mma.sync m16n8k32 e4m3 x e4m3 -> fp32: 16 weight rows as the
//               A operand, the 8 activation rows as B) and promotes the K block's product
//               with its two scales into fp32 accumulators, as the tile GEMM does.  At the
//               end of an item each warp stores its partial sums to one of three reduction
//               buffers and goes on with the next item.
//   warps 9..12 epilogue: add the eight partial sums in warp order (deterministic) and
//               finish the item while the MMA warps stream the next ones.
// The k order inside an MMA is free as long as A and B agree: lane (g, t) gives bytes
// 16t..16t+7 (and 64+16t..) of weight rows g and g+8 and of activation row g to one MMA
// and bytes 16t+8..16t+15 to the next, so all lanes with the same t hold the same K.
//
// w13 epilogue: h = silu(gate) * up in fp32 for the item's 16 columns, stored to an fp32
// buffer by routed pair.  The eight items of a 1x128 requantisation group count their
// completion on a per-(expert tile, group) counter (release fence, then one atomic add);
// the item that completes the group re-reads the group's 128 values and requantises them
// (amax/448, e4m3 codes) into the expert's padded rows, the layout the w2 GEMM reads, as
// the tile GEMM's fused epilogue does.  No item waits for another.  The counters are
// zeroed by the expert sort of the same call.
// w2 epilogue: bf16(router weight * C) to the pair's row of the [T*topk, H] buffer that
// the k-way sum (moe_combine_pairs) reads, as the tile GEMM's pairs epilogue.
// Every wait is bounded (mbar_wait); on expiry the CTA records MOE_STATUS_WAIT_TIMEOUT,
// lets its loads in flight land and exits.
#include "kernels.cuh"

namespace mfp8 {

namespace {

constexpr int kCols = kDecodeCols;              // routed rows per expert: the MMA's 8 B columns
constexpr int kMmaWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kFirstEpiWarp = 1 + kMmaWarps;
constexpr int kThreads = (1 + kMmaWarps + kEpiWarps) * 32;
constexpr int kStages = 4;
constexpr int kGroupKB = 8;                     // K blocks per stage: one per MMA warp
constexpr int kTileBytes = 16 * 128 * kGroupKB; // 16 weight rows over 8 K blocks
constexpr int kActBytes = kCols * 128 * kGroupKB;   // 8 activation rows over 8 K blocks
constexpr int kStageBytes = 2 * kTileBytes + kActBytes;
constexpr int kStageScales = 2 * kGroupKB + kCols * kGroupKB;   // [tile][kb] weight scales, [kb][row] activation scales
constexpr int kGroupItems = 128 / 16;           // w13 items per 1x128 group of the intermediate
constexpr int kRedBufs = 3;                     // items whose partial sums await the epilogue

struct Ctl {
    uint64_t full[kStages];                     // a stage landed (1 + 32 arrivals, tx bytes)
    uint64_t empty[kStages];                    // the MMA warps have read it (8 arrivals)
    uint64_t red_full[kRedBufs];                // all MMA warps stored their partials (8 arrivals)
    uint64_t red_empty[kRedBufs];               // the epilogue has read them (4 arrivals)
    int abort_flag;
    int last;
    float scl[kStages][kStageScales];
    alignas(16) float red[kRedBufs][kMmaWarps][2][32][4];
};
// ring, control block, then the step's tile records (max_tiles of them)
constexpr size_t kSmemFixed = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(Ctl);
constexpr size_t kSmemLimit = 232448;
static_assert(kSmemFixed + 64 * sizeof(DecodeTile) <= kSmemLimit, "shared memory per CTA exceeds the sm_103 limit");
size_t smem_bytes(int max_tiles) { return kSmemFixed + static_cast<size_t>(max_tiles) * sizeof(DecodeTile); }

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

__device__ __forceinline__ void epilogue_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

template <bool SILU>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const DecodeGemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* ring = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    Ctl* ctl = reinterpret_cast<Ctl*>(ring + kStages * kStageBytes);
    DecodeTile* tab = reinterpret_cast<DecodeTile*>(ctl + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = a.K / 128;
    const int NB = a.N / 128;
    // K blocks per stage (fewer than 8 only when K has fewer) and stages per item
    const int GKB = KB < kGroupKB ? KB : kGroupKB;
    const int NG = (KB + GKB - 1) / GKB;
    // activation rows loaded per stage: the most rows an expert can hold (a.cols <= 8); the
    // B columns past them hold stale shared memory and their results are never read
    const uint32_t stage_tx = static_cast<uint32_t>((2 * 16 + a.cols) * 128 * GKB);
    const int per_tile = a.N / 32;   // w13: (N/2)/16 items of 16 gate + 16 up rows; w2: N/32 items of 32 rows

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1 + 32);
            mbar_init(smem_addr(&ctl->empty[s]), kMmaWarps);
        }
        for (int b = 0; b < kRedBufs; ++b) {
            mbar_init(smem_addr(&ctl->red_full[b]), kMmaWarps);
            mbar_init(smem_addr(&ctl->red_empty[b]), kEpiWarps);
        }
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmW);
        tma_prefetch_map(&tmX);
    }
    // the set-up above overlaps the previous kernel's tail; its outputs are read from here on
    grid_dependency_wait();
    // the step's tile records, all of them in one load (no item looks anything up in global memory)
    {
        const int4* src = reinterpret_cast<const int4*>(a.tiles);
        int4* dst = reinterpret_cast<int4*>(tab);
        const int n = a.max_tiles * static_cast<int>(sizeof(DecodeTile) / sizeof(int4));
        for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
    }
    int64_t ntiles = *a.num_tiles;
    if (ntiles < 0) ntiles = 0;
    if (ntiles > a.max_tiles) ntiles = a.max_tiles;
    const int64_t total = ntiles * per_tile;
    volatile int* abort_flag = &ctl->abort_flag;
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        uint32_t q = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
            const int m = static_cast<int>(w / per_tile), u = static_cast<int>(w % per_tile);
            // (a record with an expert out of range -- the sort writes none -- streams expert 0
            // and its item's output is dropped by the epilogue)
            const int e = (tab[m].e >= 0 && tab[m].e < a.E) ? tab[m].e : 0;
            const int poff = tab[m].poff;
            const int row0 = SILU ? u * 16 : u * 32;
            const int row1 = SILU ? a.N / 2 + u * 16 : u * 32 + 16;
            const float* ws[2] = {a.w_scale + (static_cast<int64_t>(e) * NB + row0 / 128) * KB,
                                  a.w_scale + (static_cast<int64_t>(e) * NB + row1 / 128) * KB};
            for (int grp = 0; grp < NG; ++grp, ++q) {
                const uint32_t stage = q % kStages, use = q / kStages;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->empty[stage]), (use & 1u) ^ 1u, abort_flag,
                                                       a.status))) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_addr(&ctl->full[stage]);
                const uint32_t dst = smem_addr(ring + stage * kStageBytes);
                const int kb0 = grp * GKB;
                if (lane == 0) {
                    // K blocks past K are out of the tensor: zero-filled (and counted), and skipped
                    // by the MMA warps
                    mbar_arrive_expect_tx(fb, stage_tx);
                    if (a.w_tiled) {   // [E*N/128][K/128][128 rows][128 bytes]: box 16 rows x 8 K blocks
                        tma_load_4d(dst, &tmW, 0, row0 % 128, kb0, e * NB + row0 / 128, fb);
                        tma_load_4d(dst + kTileBytes, &tmW, 0, row1 % 128, kb0, e * NB + row1 / 128, fb);
                    } else {           // [E*N rows][K/128][128 bytes]: box 8 K blocks x 16 rows
                        tma_load_3d(dst, &tmW, 0, kb0, e * a.N + row0, fb);
                        tma_load_3d(dst + kTileBytes, &tmW, 0, kb0, e * a.N + row1, fb);
                    }
                    tma_load_3d(dst + 2 * kTileBytes, &tmX, 0, kb0, poff, fb);
                }
                for (int i = lane; i < kStageScales; i += 32) {
                    const int kbi = i < 2 * kGroupKB ? (i % kGroupKB) : (i - 2 * kGroupKB) / kCols;
                    const int kb = kb0 + kbi;
                    if (kbi >= GKB || kb >= KB) continue;
                    const float* src = i < 2 * kGroupKB
                                           ? ws[i / kGroupKB] + kb
                                           : a.act_scale + static_cast<int64_t>(kb) * a.rows + poff +
                                                 (i - 2 * kGroupKB) % kCols;
                    cp_async_4(smem_addr(&ctl->scl[stage][i]), src);
                }
                cp_async_arrive(fb);
            }
        }
        if (!ok) {
            // let every stage load already issued land before the CTA exits
            for (uint32_t s = 0; s < kStages && lane == 0; ++s) {
                const uint32_t n_s = (q + kStages - 1 - s) / kStages;
                if (n_s > 0) mbar_wait(smem_addr(&ctl->full[s]), (n_s - 1) & 1u, nullptr, a.status);
            }
        }
        cp_async_wait_all();
    } else if (warp < kFirstEpiWarp) {
        // ------------------------------------------------------------------ MMA warps
        const int cw = warp - 1;
        const int g = lane >> 2, t = lane & 3;
        uint32_t q0 = 0, iter = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
            float acc[2][4];
#pragma unroll
            for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[tile][i] = 0.0f;
            for (int grp = 0; grp < NG; ++grp) {
                const uint32_t q = q0 + grp;
                const uint32_t stage = q % kStages;
                if (!mbar_wait(smem_addr(&ctl->full[stage]), (q / kStages) & 1u, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const int kb = grp * GKB + cw;   // this warp's K block of the stage
                const uint8_t* st = ring + stage * kStageBytes;
                uint4 wv[2][2][2], xv[2];
                float ws[2] = {0.0f, 0.0f}, xa = 0.0f, xb = 0.0f;
                const bool live = cw < GKB && kb < KB;
                if (live) {
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            // tile-packed boxes are [K block][row][128 B], [E, N, K] boxes [row][K block][128 B]
                            const int row = g + 8 * hr;
                            const int off = a.w_tiled ? (cw * 16 + row) * 128 : (row * GKB + cw) * 128;
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                wv[tile][hr][c] =
                                    *reinterpret_cast<const uint4*>(st + tile * kTileBytes + off + 64 * c + 16 * t);
                        }
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        xv[c] = *reinterpret_cast<const uint4*>(st + 2 * kTileBytes + (g * GKB + cw) * 128 +
                                                                64 * c + 16 * t);
                    ws[0] = ctl->scl[stage][cw];
                    ws[1] = ctl->scl[stage][kGroupKB + cw];
                    xa = ctl->scl[stage][2 * kGroupKB + cw * kCols + 2 * t];
                    xb = ctl->scl[stage][2 * kGroupKB + cw * kCols + 2 * t + 1];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
                if (!live) continue;
#pragma unroll
                for (int tile = 0; tile < 2; ++tile) {
                    float f[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            mma_16x8x32(f, word(wv[tile][0][c], 2 * h), word(wv[tile][1][c], 2 * h),
                                        word(wv[tile][0][c], 2 * h + 1), word(wv[tile][1][c], 2 * h + 1),
                                        word(xv[c], 2 * h), word(xv[c], 2 * h + 1));
                    // accumulator (row g / g+8, column 2t / 2t+1): the weight block's scale
                    // times the column's activation scale
                    const float s0 = ws[tile] * xa, s1 = ws[tile] * xb;
                    acc[tile][0] = fmaf(f[0], s0, acc[tile][0]);
                    acc[tile][1] = fmaf(f[1], s1, acc[tile][1]);
                    acc[tile][2] = fmaf(f[2], s0, acc[tile][2]);
                    acc[tile][3] = fmaf(f[3], s1, acc[tile][3]);
                }
            }
            if (!ok) break;
            const uint32_t buf = iter % kRedBufs, use = iter / kRedBufs;
            if (use > 0 && !mbar_wait(smem_addr(&ctl->red_empty[buf]), (use - 1) & 1u, abort_flag, a.status))
                break;
#pragma unroll
            for (int tile = 0; tile < 2; ++tile)
                *reinterpret_cast<float4*>(&ctl->red[buf][cw][tile][lane][0]) =
                    make_float4(acc[tile][0], acc[tile][1], acc[tile][2], acc[tile][3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl->red_full[buf]));
            q0 += NG;
            ++iter;
        }
    } else {
        // ------------------------------------------------------------------ epilogue warps
        const int et = threadIdx.x - kFirstEpiWarp * 32;   // 0..127
        const int ew = warp - kFirstEpiWarp;
        uint32_t iter = 0;
        for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
            const int m = static_cast<int>(w / per_tile), u = static_cast<int>(w % per_tile);
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
            // this thread's outputs: w13 (row r of 16, column j); w2 (row r of 32, columns j, j+4)
            const int r = SILU ? (et & 15) : (et & 31);
            const int j = SILU ? (et >> 4) : (et >> 5);
            const int pair0 = j < cnt ? tl.pair[j] : -1;
            const int pair1 = (!SILU && j + 4 < cnt) ? tl.pair[j + 4] : -1;
            const uint32_t buf = iter % kRedBufs;
            if (!mbar_wait(smem_addr(&ctl->red_full[buf]), (iter / kRedBufs) & 1u, abort_flag, a.status)) break;
            // partial sums of (row rr of a 16-row tile, column jj): lane (rr % 8) * 4 + jj / 2,
            // register (rr >= 8 ? 2 : 0) + (jj & 1), added in warp order
            auto total_of = [&](int tile, int rr, int jj) {
                const int l = (rr & 7) * 4 + (jj >> 1), c = ((rr >> 3) << 1) + (jj & 1);
                float s = 0.0f;
#pragma unroll
                for (int cw = 0; cw < kMmaWarps; ++cw) s += ctl->red[buf][cw][tile][l][c];
                return s;
            };
            float v0, v1;
            if (SILU) {
                v0 = total_of(0, r, j);    // gate
                v1 = total_of(1, r, j);    // up
            } else {
                v0 = total_of(r >> 4, r & 15, j);
                v1 = total_of(r >> 4, r & 15, j + 4);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl->red_empty[buf]));
            ++iter;

            if (SILU) {
                const int I = a.N / 2;
                if (pair0 >= 0) {
                    // silu(g) * up = g * up / (1 + e^-g), as the tile GEMM's epilogue
                    a.h[static_cast<int64_t>(pair0) * I + u * 16 + r] = __fdividef(v0 * v1, 1.0f + __expf(-v0));
                }
                // the item that completes a 1x128 group requantises it
                __threadfence();
                epilogue_barrier();
                const int grp = u / kGroupItems;
                if (et == 0) {
                    int32_t* counter = a.group_count + static_cast<int64_t>(m) * (I / 128) + grp;
                    const int done = atomicAdd(counter, 1);
                    const int last = done == kGroupItems - 1;
                    if (last) *counter = 0;
                    ctl->last = last;
                }
                epilogue_barrier();
                const int last = ctl->last;
                epilogue_barrier();   // ctl->last is rewritten by the next item
                if (!last) continue;
                __threadfence();
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
                    *reinterpret_cast<uint32_t*>(a.out_q + row * I + grp * 128 + lane * 4) = lo | (hi << 16);
                    if (lane == 0) a.out_scale[static_cast<int64_t>(grp) * a.rows + row] = sc;
                }
            } else {
                // consecutive threads take consecutive rows of one pair's output row
                if (pair0 >= 0)
                    a.y[static_cast<int64_t>(pair0) * a.N + u * 32 + r] =
                        static_cast<uint16_t>(bf16x2(tl.weight[j] * v0, 0.0f) & 0xFFFFu);
                if (pair1 >= 0)
                    a.y[static_cast<int64_t>(pair1) * a.N + u * 32 + r] =
                        static_cast<uint16_t>(bf16x2(tl.weight[j + 4] * v1, 0.0f) & 0xFFFFu);
            }
        }
    }
}

}  // namespace

int decode_cols(int T) { return T >= 1 && T <= kCols ? T : 0; }

cudaError_t decode_init_device() {
    cudaError_t err = cudaFuncSetAttribute(decode_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSmemLimit));
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(decode_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(kSmemLimit));
    return err;
}

cudaError_t launch_decode_gemm(const DecodeGemmArgs& a, bool silu, int num_sms, cudaStream_t stream) {
    if (a.max_tiles <= 0) return cudaSuccess;
    if (a.cols < 1 || a.cols > kCols || a.N % 128 != 0 || a.K % 128 != 0 || (silu && a.N % 256 != 0))
        return cudaErrorInvalidValue;
    const size_t smem = smem_bytes(a.max_tiles);
    if (smem > kSmemLimit) return cudaErrorInvalidValue;
    CUtensorMap tmW, tmX;
    const uint64_t KB = static_cast<uint64_t>(a.K / 128);
    const uint32_t GKB = static_cast<uint32_t>(KB < kGroupKB ? KB : kGroupKB);   // K blocks per box
    const uint64_t E = static_cast<uint64_t>(a.E), N = static_cast<uint64_t>(a.N), K = static_cast<uint64_t>(a.K);
    cudaError_t err;
    if (a.w_tiled) {
        // [E*N/128 blocks][K/128][128 rows][128 bytes]
        const uint64_t dims[4] = {128, 128, KB, E * (N / 128)};
        const uint64_t strides[3] = {128, 128 * 128, KB * 128 * 128};
        const uint32_t box[4] = {128, 16, GKB, 1};
        err = encode_u8_map_nd(&tmW, a.W, 4, dims, strides, box);
    } else {
        // [E*N rows][K/128][128 bytes]
        const uint64_t dims[3] = {128, KB, E * N};
        const uint64_t strides[2] = {128, K};
        const uint32_t box[3] = {128, GKB, 16};
        err = encode_u8_map_nd(&tmW, a.W, 3, dims, strides, box);
    }
    if (err == cudaSuccess) {
        // activations [rows][K/128][128 bytes]
        const uint64_t dims[3] = {128, KB, static_cast<uint64_t>(a.rows)};
        const uint64_t strides[2] = {128, K};
        const uint32_t box[3] = {128, GKB, static_cast<uint32_t>(a.cols)};
        err = encode_u8_map_nd(&tmX, a.act, 3, dims, strides, box);
    }
    if (err != cudaSuccess) return err;
    const int64_t items = static_cast<int64_t>(a.max_tiles) * (a.N / 32);
    const unsigned grid = static_cast<unsigned>(items < num_sms ? items : num_sms);
    if (silu) return launch_pdl(decode_gemm_kernel<true>, dim3(grid), dim3(kThreads), smem, stream, tmW, tmX, a);
    return launch_pdl(decode_gemm_kernel<false>, dim3(grid), dim3(kThreads), smem, stream, tmW, tmX, a);
}

size_t decode_max_tiles() { return (kSmemLimit - kSmemFixed) / sizeof(DecodeTile); }

}  // namespace mfp8
