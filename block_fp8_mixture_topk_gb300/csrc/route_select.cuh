// Top-k selection of one token by one warp, with the scores in registers: shared by the routing
// kernel (route.cu) and the decode-path kernel (decode.cu), which routes a step's few tokens in
// every CTA, so that both make the same choices with the same arithmetic.
//
// The router of the FusedMoE layer ("router — top-K router", page "Quantization and MoE
// Optimizations", section FusedMoE Class) with the fused grouped top-k variant
// ("VLLM_USE_FUSED_MOE_GROUPED_TOPK", section Key Environment Variables).  Sigmoid scores are
// defined as fp64 sigmoids rounded to fp32; the selection first runs on fp32 sigmoids and keeps
// the result when every decision clears the fp32 error (nearly always), else repeats the token on
// the exact scores.  Weights are formed in fp64 from the exact scores of the chosen experts and
// rounded to fp32.  The routing kernel reads scores and bias through L1 (every token of a block
// reads the same bias); the decode kernel reads them through L2 (ld.global.cg), before it waits
// for the grids ahead of it.
#pragma once
#include "common.cuh"

namespace mfp8 {

namespace {

// a read-only load through L1 (L1 = true) or through L2 only
template <bool L1>
__device__ __forceinline__ float ld_score(const float* p) {
    if constexpr (L1) return __ldg(p);
    else return __ldcg(p);
}
template <bool L1>
__device__ __forceinline__ float4 ld_score4(const float4* p) {
    if constexpr (L1) return __ldg(p);
    else return __ldcg(p);
}


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

// Sigmoid score of a logit as the layer defines it: evaluated in fp64, rounded to fp32.
__device__ __forceinline__ float sigmoid_exact(float l) {
    return static_cast<float>(1.0 / (1.0 + exp(-static_cast<double>(l))));
}

// ---------------------------------------------------------------- register-resident variant
// The same routing with each lane holding V consecutive experts (e = lane*V + v) in
// registers: for E <= 32*V and groups that are whole runs of lanes (n_group == 1, or a
// group's G = E/n_group experts a multiple of V spanning a power-of-two number of lanes).
// A group's two best scores are merged across its lanes with shuffles (the group score
// is the fp32 sum of the two largest values, whichever experts hold them); the topk_group
// best groups are found by ranking the group scores; the k winners by k rounds of a lane
// maximum plus a warp argmax (ties to the lower expert index).  Same fast path, margin
// checks and exact fallback as route_topk_kernel.
template <int V>
__device__ int select_experts_reg(const float (&sel)[V], uint32_t live, int E, int topk, int n_group,
                                  int topk_group, int lane, bool check, bool* thin) {
    bool close = false;
    if (n_group > 1) {
        const int lpg = (E / n_group) / V;   // lanes per group
        float a1 = -INFINITY, a2 = -INFINITY;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            if (!((live >> v) & 1u)) continue;
            if (sel[v] > a1) {
                a2 = a1;
                a1 = sel[v];
            } else if (sel[v] > a2) {
                a2 = sel[v];
            }
        }
        for (int o = 1; o < lpg; o <<= 1) {
            const float b1 = __shfl_xor_sync(0xffffffffu, a1, o);
            const float b2 = __shfl_xor_sync(0xffffffffu, a2, o);
            const float hi = fmaxf(a1, b1);
            a2 = fmaxf(fminf(a1, b1), fmaxf(a2, b2));
            a1 = hi;
        }
        const float gs = a1 + a2;
        const int my_group = lane / lpg;
        int rank = 0;
        for (int g = 0; g < n_group; ++g) {
            const float o = __shfl_sync(0xffffffffu, gs, g * lpg);
            rank += (o > gs || (o == gs && g < my_group)) ? 1 : 0;
        }
        if (check && topk_group < n_group) {
            float last = (my_group < n_group && rank == topk_group - 1) ? gs : -INFINITY;
            float next = (my_group < n_group && rank == topk_group) ? gs : -INFINITY;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                last = fmaxf(last, __shfl_xor_sync(0xffffffffu, last, o));
                next = fmaxf(next, __shfl_xor_sync(0xffffffffu, next, o));
            }
            const float bound = 0x1p-17f + 0x1p-19f * fmaxf(fabsf(last), fabsf(next));
            if (last - next <= bound) close = true;
        }
        if (my_group >= n_group || rank >= topk_group) live = 0;
    }
    int my_id = -1;
    float prev = 0.0f;
    const int rounds = check ? topk + 1 : topk;
    if constexpr (V <= 16) {
        // Each lane sorts its live candidates (value descending, expert index ascending) once;
        // a round is then one warp-wide unsigned max over the lanes' heads (values mapped to
        // order-preserving keys; -0 counted as +0, 0 = no candidate), a ballot for the lowest lane
        // holding it (lanes hold consecutive experts, so the lowest lane has the lowest index
        // among equal values), and the winning lane dropping its head: the same winners, in the
        // same order, as the argmax rounds below.
        uint32_t key[V];
        int ix[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const uint32_t b = __float_as_uint(sel[v] + 0.0f);
            key[v] = ((live >> v) & 1u) ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
            ix[v] = v;
        }
#pragma unroll
        for (int k = 2; k <= V; k <<= 1)
#pragma unroll
            for (int jj = k >> 1; jj > 0; jj >>= 1)
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    const int l = i ^ jj;
                    if (l <= i) continue;
                    // first / second: the pair's required order ((i & k) == 0: i before l)
                    const int f = (i & k) == 0 ? i : l, g2 = (i & k) == 0 ? l : i;
                    const bool ok = key[f] > key[g2] || (key[f] == key[g2] && ix[f] < ix[g2]);
                    if (!ok) {
                        const uint32_t tk = key[i];
                        key[i] = key[l];
                        key[l] = tk;
                        const int ti = ix[i];
                        ix[i] = ix[l];
                        ix[l] = ti;
                    }
                }
        for (int j = 0; j < rounds; ++j) {
            const uint32_t m = __reduce_max_sync(0xffffffffu, key[0]);
            if (m == 0u) break;   // fewer candidates than rounds (only the extra round)
            const int wl = __ffs(__ballot_sync(0xffffffffu, key[0] == m)) - 1;
            const int widx = wl * V + __shfl_sync(0xffffffffu, ix[0], wl);
            const float wv = __uint_as_float((m & 0x80000000u) ? (m & 0x7FFFFFFFu) : ~m);
            if (check && j > 0) {
                const float bound = 0x1p-19f + 0x1p-20f * fmaxf(fabsf(prev), fabsf(wv));
                if (prev - wv <= bound) close = true;
            }
            prev = wv;
            if (j < topk) {
                if (lane == wl) {
#pragma unroll
                    for (int v = 0; v + 1 < V; ++v) {
                        key[v] = key[v + 1];
                        ix[v] = ix[v + 1];
                    }
                    key[V - 1] = 0u;
                }
                if (lane == j) my_id = widx;
            }
        }
        if (thin) *thin = close;
        return my_id;
    }
    for (int j = 0; j < rounds; ++j) {
        Cand c{0.0f, INT32_MAX};
#pragma unroll
        for (int v = 0; v < V; ++v)
            if (((live >> v) & 1u) && (c.idx == INT32_MAX || sel[v] > c.v)) c = Cand{sel[v], lane * V + v};
        const Cand win = warp_argmax(c);
        if (win.idx == INT32_MAX) break;  // fewer candidates than rounds (only the extra round)
        if (check && j > 0) {
            const float bound = 0x1p-19f + 0x1p-20f * fmaxf(fabsf(prev), fabsf(win.v));
            if (prev - win.v <= bound) close = true;
        }
        prev = win.v;
        if (j < topk) {
            if (win.idx / V == lane) live &= ~(1u << (win.idx % V));
            if (lane == j) my_id = win.idx;
        }
    }
    if (thin) *thin = close;
    return my_id;
}

// One warp routes the token whose E scores start at lrow: lane l holds experts l*V .. l*V+V-1
// (vec_loads: E == 32*V, V >= 4, lrow 16-byte aligned).  Returns, on lane j < topk, the j-th
// chosen expert.  zall: for softmax scoring without renormalisation, the fp64 sum over all experts
// of exp(l - l_first) (each lane's experts in order, then a shuffle tree), on every lane.
template <int V, bool L1>
__device__ __forceinline__ int route_token_reg(const float* lrow, int E, int topk, int renormalize, bool sigmoid,
                                               int n_group, int topk_group, const float* bias, bool vec_loads,
                                               int lane, double* zall) {
    const int e0 = lane * V;
    uint32_t live = 0;
    float x[V];
    if (vec_loads) {
        // E == 32*V, V >= 4, rows 16-byte aligned
#pragma unroll
        for (int v = 0; v < V; v += 4) {
            const float4 q = ld_score4<L1>(reinterpret_cast<const float4*>(lrow + e0 + v));
            x[v] = q.x;
            x[v + 1] = q.y;
            x[v + 2] = q.z;
            x[v + 3] = q.w;
        }
        live = V >= 32 ? 0xffffffffu : (1u << V) - 1u;
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const bool ok = e0 + v < E;
            x[v] = ok ? ld_score<L1>(lrow + e0 + v) : 0.0f;
            if (ok) live |= 1u << v;
        }
    }
    float sel[V];
    int my_id;
    if (sigmoid) {
        // fast path on fp32 sigmoids, kept only when every decision clears their error
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float sg = 1.0f / (1.0f + expf(-x[v]));
            sel[v] = (bias && ((live >> v) & 1u)) ? sg + ld_score<L1>(bias + e0 + v) : sg;
        }
        bool thin = false;
        my_id = select_experts_reg<V>(sel, live, E, topk, n_group, topk_group, lane, true, &thin);
        if (__any_sync(0xffffffffu, thin)) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float sg = sigmoid_exact(x[v]);
                sel[v] = (bias && ((live >> v) & 1u)) ? sg + ld_score<L1>(bias + e0 + v) : sg;
            }
            my_id = select_experts_reg<V>(sel, live, E, topk, n_group, topk_group, lane, false, nullptr);
        }
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) sel[v] = x[v];
        my_id = select_experts_reg<V>(sel, live, E, topk, n_group, topk_group, lane, false, nullptr);
        if (!renormalize) {
            const double lmax = static_cast<double>(ld_score<L1>(lrow + __shfl_sync(0xffffffffu, my_id, 0)));
            double part = 0.0;
#pragma unroll
            for (int v = 0; v < V; ++v)
                if ((live >> v) & 1u) part += exp(static_cast<double>(x[v]) - lmax);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            *zall = part;
        }
    }
    return my_id;
}

// The router weight of one token's j-th choice, for the tokens of lane groups: lanes
// [base, base + topk) of the warp hold one token's choices, lane base + j its j-th expert my_id
// (as route_token_reg returns it on lane j) and that token's score row lrow; the first choice is
// lane base's.  The fp64 terms of the chosen experts (sigmoid: the exact score; softmax:
// exp(l - l_first)), summed in the order of the chosen list (renormalize) or 1 / zall, times
// routed_scaling, rounded once to fp32 -- the same operations in the same order as the routing
// kernel's weight stage.  Every lane of the warp takes part (shuffles); a lane outside any group
// passes active = false and gets 0.
__device__ __forceinline__ float route_weight_group(const float* lrow, int my_id, bool active, int base, int topk,
                                                    int renormalize, bool sigmoid, double zall,
                                                    float routed_scaling) {
    const int first = __shfl_sync(0xffffffffu, my_id, base & 31);
    double v = 0.0;
    if (active && my_id >= 0) {
        const float l = __ldcg(lrow + my_id);
        v = sigmoid ? static_cast<double>(sigmoid_exact(l))
                    : exp(static_cast<double>(l) - static_cast<double>(__ldcg(lrow + first)));
    }
    double z = 0.0;
    for (int jj = 0; jj < topk; ++jj) z += __shfl_sync(0xffffffffu, v, (base + jj) & 31);
    if (!renormalize) z = sigmoid ? 1.0 : zall;
    return active ? static_cast<float>(v / z * static_cast<double>(routed_scaling)) : 0.0f;
}

}  // namespace

// experts per lane of the register-resident selection for this shape, or 0 when it does not apply
__host__ __device__ inline int reg_experts_per_lane(int E, int n_group) {
    int V = 1;
    while (32 * V < E) V *= 2;
    if (V > 32) return 0;
    if (n_group > 1) {
        const int G = E / n_group;
        if (G % V != 0) return 0;
        const int lpg = G / V;
        if (lpg > 32 || (lpg & (lpg - 1)) != 0) return 0;
    }
    return V;
}

}  // namespace mfp8
