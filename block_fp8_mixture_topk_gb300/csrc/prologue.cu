// Expert sort and activation quantisation of a small batch in one launch.
//
// For up to kSmallPairs routed pairs, one launch of 1024-thread blocks does what the
// three sort kernels (permute.cu) and the scattering quantiser (quant.cu) do for large
// batches.  Every block sorts the (few) pairs itself in shared memory, block 0 writes the
// sort's outputs, and the blocks share the quantisation of the tokens' groups:
// the "sorted token" layout of the pages' Triton fused-MoE kernel (page "Quantization
// and MoE Optimizations", section Triton Fused MoE Kernel) with each expert's rows
// padded to whole tiles, then each token's 1x128 group quantisation (section Fp8Config;
// kFp8Dynamic128Sym) written to the sorted rows of its pairs.  The results are the
// same, element for element: per-expert counts, exclusive scans, the stable order by
// (expert, pair) -- a pair's rank is the number of earlier pairs with its expert,
// counted, so no atomics -- the tile table, and the codes and scales.  In a decode step
// this removes three launches and the gaps between them.
//
// decode_prologue_kernel is the decode path's own prologue (below).
#include "kernels.cuh"

namespace mfp8 {

namespace {

// Lets the next kernel of the stream (launched with programmatic serialisation) start before this
// one ends; it still sees this grid's writes only after its own grid_dependency_wait.
__device__ __forceinline__ void grid_dependency_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__global__ void __launch_bounds__(1024, 1) sort_quant_small_kernel(
    const int32_t* __restrict__ ids, int P, int E, int block_m, int32_t* __restrict__ expert_offsets,
    int32_t* __restrict__ padded_offsets, int32_t* __restrict__ sorted_pair_ids, int32_t* __restrict__ pos,
    int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row0, int32_t* __restrict__ num_tiles,
    uint32_t* status, const uint16_t* __restrict__ x, int T, int H, int topk, uint8_t* __restrict__ q,
    int64_t q_ld, float* __restrict__ s, int64_t s_rs, int64_t s_gs, int scale_fmt, uint8_t* __restrict__ sf,
    int sf_kb4) {
    grid_dependency_wait();
    __shared__ int s_id[kSmallPairs];
    __shared__ int s_pos[kSmallPairs];
    __shared__ int s_poff[MOE_MAX_EXPERTS];
    __shared__ int warp_sums[32];
    const int tid = threadIdx.x;

    // routed ids (an id out of range drops its pair and is reported, as in the large sort)
    for (int p = tid; p < P; p += blockDim.x) {
        int id = ids[p];
        if (id < 0 || id >= E) {
            status_set(status, MOE_STATUS_BAD_EXPERT_ID);
            id = -1;
        }
        s_id[p] = id;
    }
    __syncthreads();

    // per-expert counts and padded counts; exclusive scans over the experts (E <= 1024)
    int total = 0;
    if (tid < E)
        for (int p = 0; p < P; ++p) total += s_id[p] == tid ? 1 : 0;
    const int padded = (total + block_m - 1) / block_m * block_m;
    const int off = block_exclusive_scan(total, warp_sums);
    const int poff = block_exclusive_scan(padded, warp_sums);
    const bool writer = blockIdx.x == 0;
    if (tid < E) s_poff[tid] = poff;
    if (writer && tid < E) {
        expert_offsets[tid] = off;
        padded_offsets[tid] = poff;
        if (tid == E - 1) {
            expert_offsets[E] = off + total;
            padded_offsets[E] = poff + padded;
            *num_tiles = (poff + padded) / block_m;
        }
        for (int i = poff / block_m; i < (poff + padded) / block_m; ++i) {
            tile_expert[i] = tid;
            tile_row0[i] = i * block_m;
        }
        for (int r = poff + total; r < poff + padded; ++r) sorted_pair_ids[r] = -1;
    }
    __syncthreads();

    // stable order: pair p goes after the earlier pairs of its expert
    for (int p = tid; p < P; p += blockDim.x) {
        const int id = s_id[p];
        int r = -1;
        if (id >= 0) {
            int before = 0;
            for (int o = 0; o < p; ++o) before += s_id[o] == id ? 1 : 0;
            r = s_poff[id] + before;
            if (writer) sorted_pair_ids[r] = p;
        }
        if (writer) pos[p] = r;
        s_pos[p] = r;
    }
    __syncthreads();

    // 1x128 groups of each token: 16 threads per group (8 values each), codes and scale
    // written to the sorted rows of the token's pairs
    const int G = H / 128;
    const int half = (tid >> 4) & 1, sub = tid & 15;
    const int per_pass = (blockDim.x >> 5) * 2;   // groups per block and pass
    for (int gi0 = blockIdx.x * per_pass + (tid >> 5) * 2; gi0 < T * G; gi0 += gridDim.x * per_pass) {
        const int gi = gi0 + half;
        const bool active = gi < T * G;
        float f[8];
        float amax = 0.0f;
        int t = 0, g = 0;
        if (active) {
            t = gi / G;
            g = gi - t * G;
            unpack8(__ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H + g * 128 + sub * 8)), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        }
        // MXFP8: groups of 32 = 4 threads; otherwise 128 = 16 threads
        const bool mx = scale_fmt == MOE_SCALE_MXFP8;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
            if (!mx || o < 4) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (active) {
            const float sc = group_scale_fmt(amax, mx ? MOE_SCALE_UE8M0 : scale_fmt);
            const uint2 code = encode8(f, sc, __frcp_rn(sc));
            const int sc_col = mx ? g * 4 + (sub >> 2) : g;
            const bool writer = mx ? (sub & 3) == 0 : sub == 0;
            for (int j = 0; j < topk; ++j) {
                const int64_t o = s_pos[t * topk + j];
                if (o < 0) continue;
                *reinterpret_cast<uint2*>(q + o * q_ld + g * 128 + sub * 8) = code;
                if (writer) {
                    if (s) s[o * s_rs + g * s_gs] = sc;
                    if (sf) sf[packed_sf_offset(o, sc_col, sf_kb4)] = ue8m0_byte(sc);
                }
            }
        }
    }
}

// The decode path's prologue: zeroes the decode kernel's counters and quantises the step's T
// tokens in 1x128 groups (section Fp8Config; kFp8Dynamic128Sym) into `copies` copies of
// token-major rows q [copy][T][H] with their scales s [copy][H/128][kDecodeCols]
// (s[(copy * H/128 + g) * kDecodeCols + t]); 16 threads per group, as the small sort's quantiser.
// Every CTA of the decode kernel reads these few rows; the copies spread those reads over L2.
// Right after its own dependency wait it lets the decode kernel launch: that kernel routes and
// sorts the step's tokens itself in every CTA meanwhile, and waits for this grid only before it
// takes work.
__global__ void __launch_bounds__(1024) decode_prologue_kernel(const uint16_t* __restrict__ x, int T, int H,
                                                               int copies, uint8_t* __restrict__ q,
                                                               float* __restrict__ s, int32_t* __restrict__ counters,
                                                               int ncounters, int scale_fmt) {
    grid_dependency_wait();
    grid_dependency_trigger();
    const int tid = threadIdx.x;
    if (blockIdx.x == 0)
        for (int i = tid; i < ncounters; i += blockDim.x) counters[i] = 0;
    const int G = H / 128;
    const int half = (tid >> 4) & 1, sub = tid & 15;
    const int per_pass = (blockDim.x >> 5) * 2;   // groups per block and pass
    for (int gi0 = blockIdx.x * per_pass + (tid >> 5) * 2; gi0 < T * G; gi0 += gridDim.x * per_pass) {
        const int gi = gi0 + half;
        const bool active = gi < T * G;
        float f[8];
        float amax = 0.0f;
        int t = 0, g = 0;
        if (active) {
            t = gi / G;
            g = gi - t * G;
            unpack8(__ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H + g * 128 + sub * 8)), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (active) {
            const float sc = group_scale_fmt(amax, scale_fmt);
            const uint2 code = encode8(f, sc, __frcp_rn(sc));
            for (int c = 0; c < copies; ++c) {
                *reinterpret_cast<uint2*>(q + (static_cast<int64_t>(c) * T + t) * H + g * 128 + sub * 8) = code;
                if (sub == 0) s[(static_cast<int64_t>(c) * G + g) * kDecodeCols + t] = sc;
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode_prologue(const uint16_t* x, int T, int H, int copies, uint8_t* q, float* s,
                                   int32_t* counters, int ncounters, int scale_fmt, cudaStream_t stream) {
    if (T < 1 || T > kDecodeCols || H % 128 != 0 || copies < 1) return cudaErrorInvalidValue;
    int blocks = (T * (H / 128) + 63) / 64;
    if (blocks < 1) blocks = 1;
    if (blocks > 148) blocks = 148;
    return launch_pdl(decode_prologue_kernel, dim3(blocks), dim3(1024), 0, stream, x, T, H, copies, q, s, counters,
                      ncounters, scale_fmt);
}

cudaError_t launch_sort_quant_small(const int32_t* ids, int P, int E, int block_m, int32_t* expert_offsets,
                                    int32_t* padded_offsets, int32_t* sorted_pair_ids, int32_t* pos,
                                    int32_t* tile_expert, int32_t* tile_row0, int32_t* num_tiles, uint32_t* status,
                                    const uint16_t* x, int T, int H, int topk, uint8_t* q, int64_t q_ld, float* s,
                                    int64_t s_rs, int64_t s_gs, int scale_fmt, cudaStream_t stream,
                                    uint8_t* sf) {
    const int groups = T * (H / 128);
    int blocks = (groups + 63) / 64;
    if (blocks < 1) blocks = 1;
    if (blocks > 148) blocks = 148;
    return launch_pdl(sort_quant_small_kernel, dim3(blocks), dim3(1024), 0, stream, ids, P, E, block_m, expert_offsets,
                      padded_offsets, sorted_pair_ids, pos, tile_expert, tile_row0, num_tiles, status, x, T, H, topk,
                      q, q_ld, s, s_rs, s_gs,
                      scale_fmt == MOE_SCALE_MXFP8 ? MOE_SCALE_MXFP8 : (sf ? MOE_SCALE_UE8M0 : scale_fmt), sf,
                      scale_fmt == MOE_SCALE_MXFP8 ? H / 128 : (H / 128 + 3) / 4);
}

}  // namespace mfp8
