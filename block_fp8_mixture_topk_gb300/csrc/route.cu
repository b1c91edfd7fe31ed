// Top-k routing: one warp per token.
//
// The router of the FusedMoE layer ("router — top-K router", page "Quantization
// and MoE Optimizations", section FusedMoE Class) with the fused grouped top-k
// variant ("VLLM_USE_FUSED_MOE_GROUPED_TOPK", section Key Environment
// Variables).  Scores live in shared memory (E floats per warp, two arrays for
// sigmoid scoring); the k winners are found by k rounds of a warp-shuffle
// argmax with ties resolved to the lower expert index, so the chosen ids are
// exactly those of the definition.  Sigmoid scores are evaluated in fp64 and
// rounded to fp32; weights are formed in fp64 and rounded to fp32.
#include "kernels.cuh"

namespace mfp8 {

namespace {

constexpr int kWarps = 4;

struct Cand {
    float v;
    int idx;  // INT32_MAX when empty
};

__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
    if (a.idx == INT32_MAX) return false;
    if (b.idx == INT32_MAX) return true;
    return a.v > b.v || (a.v == b.v && a.idx < b.idx);
}

__device__ __forceinline__ Cand warp_argmax(Cand c) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Cand other;
        other.v = __shfl_xor_sync(0xffffffffu, c.v, o);
        other.idx = __shfl_xor_sync(0xffffffffu, c.idx, o);
        if (better(other, c)) c = other;
    }
    return c;
}

__global__ void __launch_bounds__(kWarps * 32) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int topk, int renormalize, int scoring, int n_group,
    int topk_group, float routed_scaling, const float* __restrict__ bias, int32_t* __restrict__ ids,
    float* __restrict__ weights) {
    extern __shared__ float route_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long t = static_cast<long>(blockIdx.x) * kWarps + warp;
    if (t >= T) return;
    float* sel = route_smem + static_cast<size_t>(warp) * 2 * E;  // selection score
    float* sig = sel + E;                                        // sigmoid score (weights)
    const float* lrow = logits + t * E;
    const bool sigmoid = scoring == MOE_SCORING_SIGMOID;

    for (int e = lane; e < E; e += 32) {
        const float l = lrow[e];
        if (sigmoid) {
            const float s = static_cast<float>(1.0 / (1.0 + exp(-static_cast<double>(l))));
            sig[e] = s;
            sel[e] = bias ? s + bias[e] : s;
        } else {
            sel[e] = l;
        }
    }
    __syncwarp();

    // bit j of `taken`: expert lane + 32*j is chosen or excluded (E <= 1024)
    uint32_t taken = 0;
    const int per_lane = (E + 31) / 32;

    if (n_group > 1) {
        const int G = E / n_group;
        Cand gs{0.0f, INT32_MAX};
        if (lane < n_group) {
            int i1 = -1, i2 = -1;
            for (int e = lane * G; e < lane * G + G; ++e)
                if (i1 < 0 || sel[e] > sel[i1]) i1 = e;
            for (int e = lane * G; e < lane * G + G; ++e)
                if (e != i1 && (i2 < 0 || sel[e] > sel[i2])) i2 = e;
            gs.v = sel[i1] + sel[i2];
            gs.idx = lane;
        }
        uint32_t kept = 0;
        for (int r = 0; r < topk_group; ++r) {
            Cand c = gs;
            if (c.idx != INT32_MAX && ((kept >> c.idx) & 1u)) c.idx = INT32_MAX;
            const Cand win = warp_argmax(c);
            kept |= 1u << win.idx;
        }
        // experts outside the kept groups are never candidates
        for (int j = 0; j < per_lane; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((kept >> (e / G)) & 1u)) taken |= 1u << j;
        }
    }

    int my_id = -1;  // lane j < topk ends up holding the j-th chosen expert
    for (int j = 0; j < topk; ++j) {
        Cand c{0.0f, INT32_MAX};
        for (int jj = 0; jj < per_lane; ++jj) {
            const int e = lane + 32 * jj;
            if (e < E && !((taken >> jj) & 1u)) {
                const Cand x{sel[e], e};
                if (better(x, c)) c = x;
            }
        }
        const Cand win = warp_argmax(c);
        if ((win.idx & 31) == lane) taken |= 1u << (win.idx >> 5);
        if (lane == j) my_id = win.idx;
    }

    // weights (fp64, sums in the order of the chosen list / expert index)
    __shared__ int chosen_s[kWarps][MOE_MAX_TOPK];
    if (lane < topk) chosen_s[warp][lane] = my_id;
    __syncwarp();
    double z = 0.0, mine = 0.0;
    if (sigmoid) {
        for (int j = 0; j < topk; ++j) z += static_cast<double>(sig[chosen_s[warp][j]]);
        if (lane < topk) mine = static_cast<double>(sig[my_id]);
        if (!renormalize) z = 1.0;
    } else {
        const double lmax = static_cast<double>(sel[chosen_s[warp][0]]);
        if (renormalize) {
            for (int j = 0; j < topk; ++j) z += exp(static_cast<double>(sel[chosen_s[warp][j]]) - lmax);
        } else {
            double part = 0.0;
            for (int e = lane; e < E; e += 32) part += exp(static_cast<double>(sel[e]) - lmax);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            z = part;
        }
        if (lane < topk) mine = exp(static_cast<double>(sel[my_id]) - lmax);
    }
    if (lane < topk) {
        ids[t * topk + lane] = my_id;
        weights[t * topk + lane] = static_cast<float>(mine / z * static_cast<double>(routed_scaling));
    }
}

}  // namespace

cudaError_t route_init_device() {
    return cudaFuncSetAttribute(route_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kWarps * 2 * MOE_MAX_EXPERTS * static_cast<int>(sizeof(float)));
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int topk, int renormalize, int scoring,
                              int n_group, int topk_group, float routed_scaling, const float* bias, int32_t* ids,
                              float* weights, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(kWarps) * 2 * E * sizeof(float);
    const int blocks = (T + kWarps - 1) / kWarps;
    route_topk_kernel<<<blocks, kWarps * 32, smem, stream>>>(logits, T, E, topk, renormalize, scoring, n_group,
                                                              topk_group, routed_scaling, bias, ids, weights);
    return cudaGetLastError();
}

}  // namespace mfp8
