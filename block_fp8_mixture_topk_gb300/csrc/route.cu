// Top-k routing: one warp per token.
//
// The router of the FusedMoE layer ("router — top-K router", page "Quantization
// and MoE Optimizations", section FusedMoE Class) with the fused grouped top-k
// variant ("VLLM_USE_FUSED_MOE_GROUPED_TOPK", section Key Environment
// Variables).  Scores live in shared memory (E floats per warp); the k winners are
// found by k rounds of a warp-shuffle argmax with ties resolved to the lower
// expert index, so the chosen ids are exactly those of the definition.  Sigmoid
// scores are defined as fp64 sigmoids rounded to fp32; the selection first runs on
// fp32 sigmoids and keeps the result when every decision clears the fp32 error
// (nearly always), else repeats the token on the exact scores.  Weights are formed
// in fp64 from the exact scores of the chosen experts and rounded to fp32.  The register-
// resident selection (route_select.cuh) is shared with the decode-path kernel.
#include "kernels.cuh"
#include "route_select.cuh"

namespace mfp8 {

namespace {

constexpr int kWarps = 4;

// Chooses the experts from the scores sel[0..E) (shared memory): with n_group > 1,
// the topk_group groups with the largest sum of their two best scores are kept
// first (ties: lower group), then the topk best experts among them (ties: lower
// index).  Returns, on lane j < topk, the j-th chosen expert.  With check set,
// *thin tells whether a decision was closer than the error of the scores: two
// consecutive chosen scores (down to the first one not chosen), or the last kept
// and the first dropped group score, within their error bound.
__device__ int select_experts(const float* sel, int E, int topk, int n_group, int topk_group, int lane, bool check,
                              bool* thin) {
    uint32_t taken = 0;  // bit j: expert lane + 32*j is chosen or excluded (E <= 1024)
    const int per_lane = (E + 31) / 32;
    bool close = false;
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
        float last = 0.0f;
        for (int r = 0; r < topk_group; ++r) {
            Cand c = gs;
            if (c.idx != INT32_MAX && ((kept >> c.idx) & 1u)) c.idx = INT32_MAX;
            const Cand win = warp_argmax(c);
            kept |= 1u << win.idx;
            last = win.v;
        }
        if (check && topk_group < n_group) {
            Cand c = gs;
            if (c.idx != INT32_MAX && ((kept >> c.idx) & 1u)) c.idx = INT32_MAX;
            const Cand next = warp_argmax(c);
            const float bound = 0x1p-17f + 0x1p-19f * fmaxf(fabsf(last), fabsf(next.v));
            if (last - next.v <= bound) close = true;
        }
        for (int j = 0; j < per_lane; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((kept >> (e / G)) & 1u)) taken |= 1u << j;
        }
    }
    int my_id = -1;
    float prev = 0.0f;
    const int rounds = check ? topk + 1 : topk;
    for (int j = 0; j < rounds; ++j) {
        Cand c{0.0f, INT32_MAX};
        for (int jj = 0; jj < per_lane; ++jj) {
            const int e = lane + 32 * jj;
            if (e < E && !((taken >> jj) & 1u)) {
                const Cand x{sel[e], e};
                if (better(x, c)) c = x;
            }
        }
        const Cand win = warp_argmax(c);
        if (win.idx == INT32_MAX) break;  // fewer candidates than rounds (only the extra round)
        if (check && j > 0) {
            const float bound = 0x1p-19f + 0x1p-20f * fmaxf(fabsf(prev), fabsf(win.v));
            if (prev - win.v <= bound) close = true;
        }
        prev = win.v;
        if (j < topk) {
            if ((win.idx & 31) == lane) taken |= 1u << (win.idx >> 5);
            if (lane == j) my_id = win.idx;
        }
    }
    if (thin) *thin = close;
    return my_id;
}

__global__ void __launch_bounds__(kWarps * 32) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int topk, int renormalize, int scoring, int n_group,
    int topk_group, float routed_scaling, const float* __restrict__ bias, int32_t* __restrict__ ids,
    float* __restrict__ weights) {
    grid_dependency_wait();
    extern __shared__ float route_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long t = static_cast<long>(blockIdx.x) * kWarps + warp;
    if (t >= T) return;
    float* sel = route_smem + static_cast<size_t>(warp) * E;  // selection scores
    const float* lrow = logits + t * E;
    const bool sigmoid = scoring == MOE_SCORING_SIGMOID;

    int my_id;
    if (sigmoid) {
        // Fast path: fp32 scores 1/(1+expf(-l)) (expf is within 2 ulp, so each biased score is
        // within 2^-21 + 1 ulp of the exact one).  The choice is kept only if every decision had
        // a margin above that error; otherwise the token is redone with the exact scores.
        for (int e = lane; e < E; e += 32) {
            const float s = 1.0f / (1.0f + expf(-lrow[e]));
            sel[e] = bias ? s + bias[e] : s;
        }
        __syncwarp();
        bool thin = false;
        my_id = select_experts(sel, E, topk, n_group, topk_group, lane, true, &thin);
        if (__any_sync(0xffffffffu, thin)) {
            __syncwarp();
            for (int e = lane; e < E; e += 32) {
                const float s = sigmoid_exact(lrow[e]);
                sel[e] = bias ? s + bias[e] : s;
            }
            __syncwarp();
            my_id = select_experts(sel, E, topk, n_group, topk_group, lane, false, nullptr);
        }
    } else {
        for (int e = lane; e < E; e += 32) sel[e] = lrow[e];
        __syncwarp();
        my_id = select_experts(sel, E, topk, n_group, topk_group, lane, false, nullptr);
    }

    // weights (fp64; sums in the order of the chosen list, or of the expert index)
    double mine = 0.0, z = 0.0;
    if (sigmoid) {
        if (lane < topk) mine = static_cast<double>(sigmoid_exact(lrow[my_id]));
        for (int j = 0; j < topk; ++j) z += __shfl_sync(0xffffffffu, mine, j);
        if (!renormalize) z = 1.0;
    } else {
        const double lmax = static_cast<double>(lrow[__shfl_sync(0xffffffffu, my_id, 0)]);
        if (lane < topk) mine = exp(static_cast<double>(lrow[my_id]) - lmax);
        if (renormalize) {
            for (int j = 0; j < topk; ++j) z += __shfl_sync(0xffffffffu, mine, j);
        } else {
            double part = 0.0;
            for (int e = lane; e < E; e += 32) part += exp(static_cast<double>(lrow[e]) - lmax);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            z = part;
        }
    }
    if (lane < topk) {
        ids[t * topk + lane] = my_id;
        weights[t * topk + lane] = static_cast<float>(mine / z * static_cast<double>(routed_scaling));
    }
}

// One warp selects the experts of one token (fp32 registers); the fp64 weights of the
// block's kWarps tokens are then formed together, one thread per (token, choice), so that
// the fp64 instructions (a small fraction of the fp32 rate on this GPU) run on full warps.
template <int V>
__global__ void __launch_bounds__(kWarps * 32) route_topk_reg_kernel(
    const float* __restrict__ logits, int T, int E, int topk, int renormalize, int scoring, int n_group,
    int topk_group, float routed_scaling, const float* __restrict__ bias, int32_t* __restrict__ ids,
    float* __restrict__ weights, bool vec_loads) {
    grid_dependency_wait();
    __shared__ int s_id[kWarps * MOE_MAX_TOPK];
    __shared__ double s_val[kWarps * MOE_MAX_TOPK];
    __shared__ double s_zall[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long tb = static_cast<long>(blockIdx.x) * kWarps;      // first token of the block
    const long t = tb + warp;
    const bool sigmoid = scoring == MOE_SCORING_SIGMOID;
    if (t < T) {
        double zall = 0.0;
        const int my_id = route_token_reg<V, true>(logits + t * E, E, topk, renormalize, sigmoid, n_group,
                                             topk_group, bias, vec_loads, lane, &zall);
        if (!sigmoid && !renormalize && lane == 0) s_zall[warp] = zall;
        if (lane < topk) s_id[warp * topk + lane] = my_id;
    }
    __syncthreads();

    // fp64 weight terms, one thread per (token, choice) of the block
    const long left = T - tb;
    const int ntok = static_cast<int>(left < kWarps ? left : kWarps);
    const int slots = ntok * topk;
    for (int sl = threadIdx.x; sl < slots; sl += blockDim.x) {
        const int w = sl / topk;
        const float* lrow = logits + (tb + w) * E;
        const int id = s_id[sl];
        s_val[sl] = sigmoid ? static_cast<double>(sigmoid_exact(lrow[id]))
                            : exp(static_cast<double>(lrow[id]) - static_cast<double>(lrow[s_id[w * topk]]));
    }
    __syncthreads();
    // sums in the order of the chosen list; weights rounded once to fp32
    for (int sl = threadIdx.x; sl < slots; sl += blockDim.x) {
        const int w = sl / topk;
        double z = 0.0;
        for (int jj = 0; jj < topk; ++jj) z += s_val[w * topk + jj];
        if (!renormalize) z = sigmoid ? 1.0 : s_zall[w];
        ids[tb * topk + sl] = s_id[sl];
        weights[tb * topk + sl] = static_cast<float>(s_val[sl] / z * static_cast<double>(routed_scaling));
    }
}

}  // namespace

cudaError_t route_init_device() {
    return cudaFuncSetAttribute(route_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kWarps * MOE_MAX_EXPERTS * static_cast<int>(sizeof(float)));
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int topk, int renormalize, int scoring,
                              int n_group, int topk_group, float routed_scaling, const float* bias, int32_t* ids,
                              float* weights, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int blocks = (T + kWarps - 1) / kWarps;
    const int V = reg_experts_per_lane(E, n_group);
    if (V > 0) {
        const bool vec = V >= 4 && E == 32 * V && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
#define MOE_ROUTE_REG(VV)                                                                                    \
    return launch_pdl(route_topk_reg_kernel<VV>, dim3(blocks), dim3(kWarps * 32), 0, stream, logits, T, E, topk, \
                      renormalize, scoring, n_group, topk_group, routed_scaling, bias, ids, weights, vec)
        switch (V) {
            case 1: MOE_ROUTE_REG(1);
            case 2: MOE_ROUTE_REG(2);
            case 4: MOE_ROUTE_REG(4);
            case 8: MOE_ROUTE_REG(8);
            case 16: MOE_ROUTE_REG(16);
            default: MOE_ROUTE_REG(32);
        }
#undef MOE_ROUTE_REG
    }
    const size_t smem = static_cast<size_t>(kWarps) * E * sizeof(float);
    return launch_pdl(route_topk_kernel, dim3(blocks), dim3(kWarps * 32), smem, stream, logits, T, E, topk,
                      renormalize, scoring, n_group, topk_group, routed_scaling, bias, ids, weights);
}

}  // namespace mfp8
