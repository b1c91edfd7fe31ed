// Sort of routed pairs by expert ("sorted token" pattern, page "Quantization and
// MoE Optimizations", section Triton Fused MoE Kernel), with each expert's rows
// padded to whole block_m tiles and a tile -> (expert, first row) table, so the
// grouped GEMMs visit only real tiles (the "tile-level skipping" of padding
// rows, page "vllm.model_executor.layers.fused_moe.oracle.fp8",
// _get_priority_backends).
//
// Three kernels, no atomics:
//   1. per chunk of 1024 pairs, a histogram over experts: each warp counts its
//      pairs with a warp match (the lowest lane of each set of equal ids writes
//      the set's size into the warp's own row of counts), then the block sums
//      the warp rows;
//   2. one block scans the chunk histograms (per expert over chunks, then over
//      experts), producing offsets, padded offsets, the tile table and the
//      first row of every (chunk, expert) relative to its expert's padded start;
//   3. per chunk, each pair's rank among the pairs of its expert in that chunk
//      (warp match + per-warp counts), which keeps pairs of one expert in
//      ascending pair order: the sort is stable and deterministic.
#include "kernels.cuh"

namespace mfp8 {

namespace {

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

constexpr int kCountWarps = 8;

__global__ void __launch_bounds__(kCountWarps * 32) chunk_count_kernel(const int32_t* __restrict__ ids, int64_t P,
                                                                       int E, int32_t* __restrict__ counts,
                                                                       uint32_t* status) {
    grid_dependency_wait();
    extern __shared__ int warp_hist[];  // [kCountWarps][E]
    for (int i = threadIdx.x; i < kCountWarps * E; i += blockDim.x) warp_hist[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int* hist = warp_hist + warp * E;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kPermuteChunk;
    // the warp's pairs: 32 at a time, kPermuteChunk / kCountWarps of them
    for (int i = warp * 32; i < kPermuteChunk; i += kCountWarps * 32) {
        const int64_t p = base + i + lane;
        int id = -1;
        if (p < P) {
            id = ids[p];
            if (id < 0 || id >= E) {
                status_set(status, MOE_STATUS_BAD_EXPERT_ID);
                id = -1;
            }
        }
        const uint32_t same = __match_any_sync(0xffffffffu, id);
        if (id >= 0 && (same & lanemask_lt()) == 0) hist[id] += __popc(same);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kCountWarps; ++w) c += warp_hist[w * E + e];
        counts[static_cast<int64_t>(blockIdx.x) * E + e] = c;
    }
}

__global__ void __launch_bounds__(1024) scan_kernel(int64_t n_chunks, int E, int block_m,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ expert_offsets,
                                                    int32_t* __restrict__ padded_offsets,
                                                    int32_t* __restrict__ sorted_pair_ids,
                                                    int32_t* __restrict__ tile_expert,
                                                    int32_t* __restrict__ tile_row0, int32_t* __restrict__ num_tiles) {
    grid_dependency_wait();
    __shared__ int warp_sums[32];
    const int e = threadIdx.x;
    int total = 0;
    if (e < E) {
        // exclusive prefix over chunks, in place; 8 loads in flight at a time
        for (int64_t c0 = 0; c0 < n_chunks; c0 += 8) {
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = (c0 + i < n_chunks) ? counts[(c0 + i) * E + e] : 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (c0 + i < n_chunks) counts[(c0 + i) * E + e] = total;
                total += v[i];
            }
        }
    }
    const int padded = ((total + block_m - 1) / block_m) * block_m;
    const int off = block_exclusive_scan(total, warp_sums);
    const int poff = block_exclusive_scan(padded, warp_sums);
    if (e < E) {
        expert_offsets[e] = off;
        padded_offsets[e] = poff;
        if (e == E - 1) {
            expert_offsets[E] = off + total;
            padded_offsets[E] = poff + padded;
            *num_tiles = (poff + padded) / block_m;
        }
        for (int i = poff / block_m; i < (poff + padded) / block_m; ++i) {
            tile_expert[i] = e;
            tile_row0[i] = i * block_m;
        }
        for (int r = poff + total; r < poff + padded; ++r) sorted_pair_ids[r] = -1;
    }
}

__global__ void __launch_bounds__(kPermuteChunk) scatter_kernel(const int32_t* __restrict__ ids, int64_t P, int E,
                                                                const int32_t* __restrict__ bases,
                                                                const int32_t* __restrict__ padded_offsets,
                                                                int32_t* __restrict__ sorted_pair_ids,
                                                                int32_t* __restrict__ pos) {
    grid_dependency_wait();
    extern __shared__ int16_t warp_count[];  // [32][E]
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) warp_count[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t p = static_cast<int64_t>(blockIdx.x) * kPermuteChunk + threadIdx.x;
    const bool valid = p < P;
    int id = valid ? ids[p] : -1;
    if (id >= E) id = -1;
    if (id < 0) id = -1;
    const uint32_t same = __match_any_sync(0xffffffffu, id);
    const int rank = __popc(same & lanemask_lt());
    if (id >= 0 && rank == 0) warp_count[warp * E + id] = static_cast<int16_t>(__popc(same));
    __syncthreads();
    (void)lane;
    if (id >= 0) {
        int before = 0;
        for (int w = 0; w < warp; ++w) before += warp_count[w * E + id];
        const int r = padded_offsets[id] + bases[static_cast<int64_t>(blockIdx.x) * E + id] + before + rank;
        pos[p] = r;
        sorted_pair_ids[r] = static_cast<int32_t>(p);
    } else if (valid) {
        pos[p] = -1;
    }
}

}  // namespace

int64_t permute_chunks(int64_t P) { return (P + kPermuteChunk - 1) / kPermuteChunk; }

cudaError_t permute_init_device() {
    cudaError_t e = cudaFuncSetAttribute(scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         32 * MOE_MAX_EXPERTS * static_cast<int>(sizeof(int16_t)));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kCountWarps * MOE_MAX_EXPERTS * static_cast<int>(sizeof(int)));
    return e;
}

cudaError_t launch_align_permute(const int32_t* ids, int64_t P, int E, int block_m, int32_t* expert_offsets,
                                 int32_t* padded_offsets, int32_t* sorted_pair_ids, int32_t* pos,
                                 int32_t* tile_expert, int32_t* tile_row0, int32_t* num_tiles,
                                 int32_t* chunk_counts, uint32_t* status, cudaStream_t stream) {
    const int64_t n_chunks = permute_chunks(P);
    cudaError_t e = cudaSuccess;
    if (n_chunks > 0)
        e = launch_pdl(chunk_count_kernel, dim3(static_cast<unsigned>(n_chunks)), dim3(kCountWarps * 32),
                       kCountWarps * E * sizeof(int), stream, ids, P, E, chunk_counts, status);
    if (e == cudaSuccess)
        e = launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, stream, n_chunks, E, block_m, chunk_counts,
                       expert_offsets, padded_offsets, sorted_pair_ids, tile_expert, tile_row0, num_tiles);
    if (e == cudaSuccess && n_chunks > 0)
        e = launch_pdl(scatter_kernel, dim3(static_cast<unsigned>(n_chunks)), dim3(kPermuteChunk),
                       32 * E * sizeof(int16_t), stream, ids, P, E, chunk_counts, padded_offsets, sorted_pair_ids,
                       pos);
    return e;
}

}  // namespace mfp8
