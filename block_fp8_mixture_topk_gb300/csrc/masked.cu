// The expert layer on the masked batched layout: rows already grouped by expert,
// hidden [E, M, H] with counts[e] valid rows per expert (the "[num_experts, max_tokens,
// hidden]" format that low-latency expert-parallel dispatch hands to the experts,
// BatchedDeepGemmExperts on page "Quantization and MoE Optimizations").  No routing and
// no combine: each valid row goes through the expert's block-FP8 MLP and its bf16
// result lands in the same place of out [E, M, H].
//
// masked_map_kernel turns the device-side counts into what the grouped GEMMs read: each
// expert's rows padded to whole 128-row tiles (Mp = M rounded up to 128 rows per
// expert), the tile table (block 0, one scan over the experts), the padded row of every
// valid input row (for the quantiser), the input row of every padded row (-1 for
// padding, for the GEMM epilogues) and unit router weights.
#include "kernels.cuh"

namespace mfp8 {

namespace {

__global__ void __launch_bounds__(1024) masked_map_kernel(const int32_t* __restrict__ counts, int E, int M, int Mp,
                                                          int32_t* __restrict__ row_map, int32_t* __restrict__ pos,
                                                          float* __restrict__ ones, int32_t* __restrict__ tile_expert,
                                                          int32_t* __restrict__ tile_row0,
                                                          int32_t* __restrict__ num_tiles, uint32_t* status) {
    grid_dependency_wait();
    __shared__ int warp_sums[32];
    auto count_of = [&](int e) {
        const int c = counts[e];
        return c < 0 ? 0 : (c > M ? M : c);
    };
    if (blockIdx.x == 0) {
        // tiles of each expert, in expert order (E <= 1024: one expert per thread)
        const int e = threadIdx.x;
        int c = 0;
        if (e < E) {
            const int raw = counts[e];
            if (raw < 0 || raw > M) status_set(status, MOE_STATUS_BAD_COUNT);
            c = count_of(e);
        }
        const int tiles = (c + 127) / 128;
        const int base = block_exclusive_scan(tiles, warp_sums);
        if (e < E) {
            for (int i = 0; i < tiles; ++i) {
                tile_expert[base + i] = e;
                tile_row0[base + i] = e * Mp + i * 128;
            }
            if (e == E - 1) *num_tiles = base + tiles;
        }
    }
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t r = first; r < static_cast<int64_t>(E) * Mp; r += stride) {
        const int e = static_cast<int>(r / Mp), i = static_cast<int>(r - static_cast<int64_t>(e) * Mp);
        row_map[r] = i < count_of(e) ? e * M + i : -1;
    }
    for (int64_t r = first; r < static_cast<int64_t>(E) * M; r += stride) {
        const int e = static_cast<int>(r / M), i = static_cast<int>(r - static_cast<int64_t>(e) * M);
        pos[r] = i < count_of(e) ? e * Mp + i : -1;
        ones[r] = 1.0f;
    }
}

}  // namespace

cudaError_t launch_masked_map(const int32_t* counts, int E, int M, int Mp, int32_t* row_map, int32_t* pos,
                              float* ones, int32_t* tile_expert, int32_t* tile_row0, int32_t* num_tiles,
                              uint32_t* status, cudaStream_t stream) {
    const int64_t work = static_cast<int64_t>(E) * Mp;
    int64_t blocks = (work + 1023) / 1024;
    if (blocks < 1) blocks = 1;
    if (blocks > 4 * 152) blocks = 4 * 152;
    return launch_pdl(masked_map_kernel, dim3(static_cast<unsigned>(blocks)), dim3(1024), 0, stream, counts, E, M,
                      Mp, row_map, pos, ones, tile_expert, tile_row0, num_tiles, status);
}

}  // namespace mfp8
