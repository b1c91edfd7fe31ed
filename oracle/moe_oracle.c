/*
 * CPU oracle for the block-FP8 fused MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA path and the CUDA path never calls it.
 *
 * Plain, slow, obviously correct: every step is written out from its
 * definition, floating point is fp64 except where a quantisation decision is
 * made (those steps are fp32, the precision the quantised format fixes).
 *
 * Sources (web pages on vLLM's quantisation / MoE system):
 *  [QMO]  "Quantization and MoE Optimizations" (vLLM wiki page)
 *  [FP8O] "vllm.model_executor.layers.fused_moe.oracle.fp8" (vLLM API docs)
 *  [NVFP4] "vllm.model_executor.layers.quantization.online.nvfp4" (vLLM API docs)
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes with its justification):
 *  - activation scale of a 1x128 group = max(amax, 1e-8) / 448 in fp32, codes
 *    = e4m3fn round-to-nearest-even of x / scale with saturation to +-448;
 *  - sigmoid routing: score s = fp32(sigma(logit)) evaluated in fp64; the bias
 *    only steers selection; group score = sum of the two largest biased scores;
 *  - ties in every top-k resolve to the lower index;
 *  - w13 rows [0, I) are the gate projection, rows [I, 2I) the up projection;
 *  - the intermediate SiLU(gate)*up is requantised from fp32 values;
 *  - NVFP4 block step: block scale = e4m3(max|x| / 6), code = e2m1(x / block scale);
 *  - MXFP8 (block [1, 32], UE8M0 scales): the same group rule on groups of 32 along the
 *    contiguous dimension, each scale rounded up to a power of two.
 *
 * Parity pins: every function here is checked by tests against closed forms,
 * exhaustive enumeration, brute force on tiny inputs or an independent
 * library; see tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* e4m3fn format ("FLOAT8_E4M3_MAX" = 448, [NVFP4] _quantize_moe_weight_to_nvfp4).
 * 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
 * S.1111.111 is NaN.  Normal: (1 + m/8) * 2^(e-7); subnormal (e = 0): m/8 * 2^-6. */

static double e4m3_val[256];
static int e4m3_ready = 0;

static void e4m3_build(void) {
    if (e4m3_ready) return;
    for (int c = 0; c < 256; ++c) {
        int sign = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
        double v;
        if (e == 15 && m == 7) v = NAN;
        else if (e == 0) v = ldexp((double)m, -9);          /* m/8 * 2^-6 */
        else v = ldexp((double)(8 + m), e - 7 - 3);          /* (8+m)/8 * 2^(e-7) */
        e4m3_val[c] = sign ? -v : v;
    }
    e4m3_ready = 1;
}

double orc_e4m3_value(int code) {
    e4m3_build();
    return e4m3_val[code & 255];
}

/* Round an fp32 value to the nearest e4m3fn value, ties to the even code,
 * saturating at +-448 (no NaN from overflow). */
uint8_t orc_e4m3_encode(float xf) {
    e4m3_build();
    double x = (double)xf;
    if (isnan(x)) return 0x7F;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs(x);
    uint8_t code;
    if (a >= 448.0) {
        code = 0x7E;
    } else {
        /* codes 0..126 hold the non-negative finite values in increasing order:
         * find the largest c with value(c) <= a */
        int lo = 0, hi = 126;
        while (lo < hi) {
            int mid = (lo + hi + 1) / 2;
            if (e4m3_val[mid] <= a) lo = mid; else hi = mid - 1;
        }
        int c = lo;
        if (e4m3_val[c] == a) {
            code = (uint8_t)c;
        } else {
            double below = a - e4m3_val[c], above = e4m3_val[c + 1] - a;
            if (below < above) code = (uint8_t)c;
            else if (above < below) code = (uint8_t)(c + 1);
            else code = (uint8_t)((c & 1) ? c + 1 : c);   /* tie: even mantissa */
        }
    }
    return (uint8_t)(code | (neg ? 0x80 : 0));
}

/* bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits. */
static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Nearest-even rounding of an fp64 value to bf16: 8 significant bits, the
 * fp32 exponent range, subnormal spacing 2^-133, overflow to infinity. */
uint16_t orc_bf16_from_f64(double x) {
    if (isnan(x)) return 0x7FC0;
    double a = fabs(x), y;
    if (a == 0.0 || isinf(a)) {
        y = a;
    } else {
        int ex;
        frexp(a, &ex);                       /* a = m * 2^ex, m in [0.5, 1) */
        int q = ex - 8;                      /* exponent of one unit in the last place */
        if (q < -133) q = -133;
        y = ldexp(nearbyint(ldexp(a, -q)), q);   /* nearbyint: ties to even */
        if (y > 0x1.FEp127) y = INFINITY;    /* above the largest finite bf16 */
    }
    float f = (float)(signbit(x) ? -y : y);  /* exact: y has at most 8 bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------- */
/* Group quantisation: one fp32 scale per group, scale = max(amax, 1e-8)/448,
 * code = e4m3(x / scale).  Dynamic per-token activation scales are "computed
 * per-token at runtime" ([QMO] Fp8Config); the group of 128 is the activation
 * key kFp8Dynamic128Sym ([FP8O] _get_priority_backends); the 1e-8 floor on amax
 * follows [NVFP4] _quantize_moe_weight_to_nvfp4. */

/* Scale formats: 0 = fp32 (amax/448 as computed); 1 = FLOAT32_CEIL_UE8M0, the fp32
 * scale rounded up to a power of two ("Float32 scales rounded up to UE8M0", DeepGEMM
 * scale formats, [QMO] DeepGEMM Scale Formats), so that every scale is exactly
 * representable as an 8-bit exponent. */
static float ceil_pow2(float t) {
    int e;
    float m = frexpf(t, &e);                       /* t = m * 2^e, 0.5 <= m < 1 */
    return m == 0.5f ? t : ldexpf(1.0f, e);
}

static float group_scale(float amax, int fmt) {
    float floored = amax > 1e-8f ? amax : 1e-8f;
    float t = floored / 448.0f;                    /* fp32 IEEE division */
    return fmt == 1 ? ceil_pow2(t) : t;
}

/* x: fp32 [rows, cols] (cols % gs == 0) -> q [rows, cols], s [rows, cols/gs]: groups of gs
 * values along a row (gs = 128: the layer's activation groups; gs = 32: MXFP8's [1, 32] blocks) */
void orc_quant_1xg_f32(const float* x, long rows, long cols, int gs, uint8_t* q, float* s, int fmt) {
    long G = cols / gs;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        for (long g = 0; g < G; ++g) {
            const float* xg = x + r * cols + g * gs;
            float amax = 0.0f;
            for (int i = 0; i < gs; ++i) {
                float a = fabsf(xg[i]);
                if (a > amax) amax = a;
            }
            float sc = group_scale(amax, fmt);
            s[r * G + g] = sc;
            for (int i = 0; i < gs; ++i) q[r * cols + g * gs + i] = orc_e4m3_encode(xg[i] / sc);
        }
    }
}

/* bf16 input version */
void orc_quant_1xg_bf16(const uint16_t* x, long rows, long cols, int gs, uint8_t* q, float* s, int fmt) {
    long G = cols / gs;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        float row[128];
        for (long g = 0; g < G; ++g) {
            float amax = 0.0f;
            for (int i = 0; i < gs; ++i) {
                row[i] = bf16_to_f32(x[r * cols + g * gs + i]);
                float a = fabsf(row[i]);
                if (a > amax) amax = a;
            }
            float sc = group_scale(amax, fmt);
            s[r * G + g] = sc;
            for (int i = 0; i < gs; ++i) q[r * cols + g * gs + i] = orc_e4m3_encode(row[i] / sc);
        }
    }
}

void orc_quant_1x128_f32(const float* x, long rows, long cols, uint8_t* q, float* s, int fmt) {
    orc_quant_1xg_f32(x, rows, cols, 128, q, s, fmt);
}

void orc_quant_1x128_bf16(const uint16_t* x, long rows, long cols, uint8_t* q, float* s, int fmt) {
    orc_quant_1xg_bf16(x, rows, cols, 128, q, s, fmt);
}

/* 128x128 block weight quantisation of stacked expert weights [E, N, K]
 * ("weight_block_size ... [128, 128]", [QMO] Fp8Config; the static block key
 * kFp8Static128BlockSym, [FP8O] _get_priority_backends).  Same rule as the
 * groups, amax over the whole block.  s: [E, N/128, K/128]. */
void orc_quant_128x128_bf16(const uint16_t* w, long E, long N, long K, uint8_t* q, float* s, int fmt) {
    long NB = N / 128, KB = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (long e = 0; e < E; ++e) {
        for (long nb = 0; nb < NB; ++nb) {
            for (long kb = 0; kb < KB; ++kb) {
                float amax = 0.0f;
                for (long n = nb * 128; n < nb * 128 + 128; ++n)
                    for (long k = kb * 128; k < kb * 128 + 128; ++k) {
                        float a = fabsf(bf16_to_f32(w[(e * N + n) * K + k]));
                        if (a > amax) amax = a;
                    }
                float sc = group_scale(amax, fmt);
                s[(e * NB + nb) * KB + kb] = sc;
                for (long n = nb * 128; n < nb * 128 + 128; ++n)
                    for (long k = kb * 128; k < kb * 128 + 128; ++k) {
                        long i = (e * N + n) * K + k;
                        q[i] = orc_e4m3_encode(bf16_to_f32(w[i]) / sc);
                    }
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* e2m1 (fp4) format ("FLOAT4_E2M1_MAX" = 6, [NVFP4] _quantize_moe_weight_to_nvfp4):
 * 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no infinities or NaN.
 * Normal (e > 0): (1 + m/2) * 2^(e-1); subnormal (e = 0): m/2.  Two codes per byte in the
 * packed [.., K/2] tensors: element 2i in the low nibble, 2i + 1 in the high nibble. */
double orc_e2m1_value(int code) {
    int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* Round an fp32 value to the nearest e2m1 value, ties to the even code, saturating at +-6;
 * the sign bit follows the input's (a negative value that rounds to zero gives -0). */
uint8_t orc_e2m1_encode(float xf) {
    double x = (double)xf;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs(x);
    int c;
    if (isnan(x)) {
        c = 0;                                   /* e2m1 has no NaN; not produced by the quantiser */
    } else if (a >= 6.0) {
        c = 7;
    } else {
        /* codes 0..7 hold the non-negative values in increasing order */
        c = 0;
        while (c < 7 && orc_e2m1_value(c + 1) <= a) ++c;
        if (orc_e2m1_value(c) != a) {
            double below = a - orc_e2m1_value(c), above = orc_e2m1_value(c + 1) - a;
            if (above < below || (above == below && (c & 1))) ++c;   /* tie: even mantissa */
        }
    }
    return (uint8_t)(c | (neg ? 8 : 0));
}

/* NVFP4 quantisation of stacked expert weights [E, N, K] as [NVFP4]
 * _quantize_moe_weight_to_nvfp4 states it: per expert, amax over the whole [N, K] (floored at
 * 1e-8), global_scale = (FLOAT4_E2M1_MAX * FLOAT8_E4M3_MAX) / amax, the weights multiplied by it
 * in fp32 and rounded back to bf16; those quantised in blocks of 16 along K with one FP8 (e4m3)
 * scale per block; stored: fp4 codes [E, N, K/2], block scales [E, N, K/16] and the per-expert
 * global scale 1 / global_scale [E].  The block step (scaled_fp4_quant with a unit global scale)
 * is not printed on the pages; its reading here, as for the FP8 groups: block scale =
 * e4m3(max|x| / 6), code = e2m1(x / block scale) (fp32 divisions; a zero scale gives code 0). */
void orc_quant_nvfp4_bf16(const uint16_t* w, long E, long N, long K, uint8_t* q, uint8_t* sf, float* gs2) {
    e4m3_build();
    long KB16 = K / 16;
    for (long e = 0; e < E; ++e) {
        float amax = 0.0f;
#pragma omp parallel for reduction(max : amax) schedule(static)
        for (long i = 0; i < N * K; ++i) {
            float a = fabsf(bf16_to_f32(w[e * N * K + i]));
            if (a > amax) amax = a;
        }
        if (amax < 1e-8f) amax = 1e-8f;
        float gsc = (6.0f * 448.0f) / amax;             /* fp32 IEEE division */
        gs2[e] = 1.0f / gsc;
#pragma omp parallel for schedule(static)
        for (long n = 0; n < N; ++n) {
            for (long b = 0; b < KB16; ++b) {
                float v[16];
                float vmax = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    long idx = (e * N + n) * K + b * 16 + i;
                    uint16_t bits = orc_bf16_from_f64((double)(bf16_to_f32(w[idx]) * gsc));   /* fp32 product -> bf16 */
                    v[i] = bf16_to_f32(bits);
                    if (fabsf(v[i]) > vmax) vmax = fabsf(v[i]);
                }
                uint8_t s = orc_e4m3_encode(vmax / 6.0f);
                float sv = (float)e4m3_val[s];
                sf[(e * N + n) * KB16 + b] = s;
                for (int i = 0; i < 16; i += 2) {
                    uint8_t lo = sv == 0.0f ? 0 : orc_e2m1_encode(v[i] / sv);
                    uint8_t hi = sv == 0.0f ? 0 : orc_e2m1_encode(v[i + 1] / sv);
                    q[((e * N + n) * K + b * 16 + i) / 2] = (uint8_t)((lo & 15) | ((hi & 15) << 4));
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Top-k routing ("router — top-K router", [QMO] FusedMoE Class; "fused grouped
 * top-K routing", [QMO] Key Environment Variables).
 *
 * scoring 0 (softmax): choose the k largest logits (ties: lower index); the
 *   weight of a chosen expert is its softmax probability, renormalised over the
 *   chosen k when renormalize != 0.
 * scoring 1 (sigmoid): s_e = fp32(1/(1+exp(-l_e))) computed in fp64;
 *   b_e = s_e + bias_e in fp32 steers selection only.  With n_group > 1 the
 *   experts are split into n_group consecutive groups, a group's score is the
 *   sum of its two largest b, the topk_group best groups are kept (ties: lower
 *   group) and the k largest b among their experts are chosen (ties: lower
 *   index).  Weight = s_j, renormalised over the chosen k when renormalize != 0.
 * Both modes multiply the final weights by routed_scaling.
 * Returns 0, or -1 on arguments the definition does not cover. */

/* index of the largest value among cand[0..E) with allowed[e] != 0;
 * ties resolve to the lower index */
static int argmax_allowed(const float* v, const unsigned char* allowed, int E) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
        if (!allowed[e]) continue;
        if (best < 0 || v[e] > v[best]) best = e;
    }
    return best;
}

int orc_route(const float* logits, const float* bias, long T, int E, int topk, int renormalize,
              int scoring, int n_group, int topk_group, double routed_scaling,
              int32_t* ids, float* weights) {
    if (topk < 1 || topk > E || E < 1 || topk > 1024) return -1;
    if (scoring != 0 && scoring != 1) return -1;
    if (n_group < 1 || E % n_group != 0) return -1;
    if (n_group > 1) {
        if (scoring != 1) return -1;
        if (topk_group < 1 || topk_group > n_group) return -1;
        if (E / n_group < 2) return -1;
        if (topk > topk_group * (E / n_group)) return -1;
    }
    int fail = 0;
#pragma omp parallel
    {
        float* sel_score = (float*)malloc(sizeof(float) * E);
        float* sig = (float*)malloc(sizeof(float) * E);
        unsigned char* allowed = (unsigned char*)malloc(E);
        float* gscore = (float*)malloc(sizeof(float) * (n_group > 0 ? n_group : 1));
        unsigned char* gallowed = (unsigned char*)malloc(n_group > 0 ? n_group : 1);
        if (!sel_score || !sig || !allowed || !gscore || !gallowed) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(static)
            for (long t = 0; t < T; ++t) {
                const float* l = logits + t * E;
                for (int e = 0; e < E; ++e) {
                    if (scoring == 0) {
                        sel_score[e] = l[e];
                    } else {
                        sig[e] = (float)(1.0 / (1.0 + exp(-(double)l[e])));
                        sel_score[e] = bias ? sig[e] + bias[e] : sig[e];
                    }
                    allowed[e] = 1;
                }
                if (n_group > 1) {
                    int G = E / n_group;
                    for (int g = 0; g < n_group; ++g) {
                        /* two largest b in the group (ties: lower index) */
                        int i1 = -1, i2 = -1;
                        for (int e = g * G; e < g * G + G; ++e)
                            if (i1 < 0 || sel_score[e] > sel_score[i1]) i1 = e;
                        for (int e = g * G; e < g * G + G; ++e)
                            if (e != i1 && (i2 < 0 || sel_score[e] > sel_score[i2])) i2 = e;
                        gscore[g] = sel_score[i1] + sel_score[i2];
                        gallowed[g] = 1;
                    }
                    unsigned char* keep = allowed;   /* reuse: mark kept groups' experts */
                    for (int e = 0; e < E; ++e) keep[e] = 0;
                    for (int r = 0; r < topk_group; ++r) {
                        int g = argmax_allowed(gscore, gallowed, n_group);
                        gallowed[g] = 0;
                        for (int e = g * G; e < g * G + G; ++e) keep[e] = 1;
                    }
                }
                double wsum = 0.0;
                double wj[1024];
                for (int j = 0; j < topk; ++j) {
                    int e = argmax_allowed(sel_score, allowed, E);
                    allowed[e] = 0;
                    ids[t * topk + j] = e;
                }
                if (scoring == 0) {
                    double lmax = -INFINITY;
                    for (int e = 0; e < E; ++e) if ((double)l[e] > lmax) lmax = l[e];
                    double zall = 0.0;
                    for (int e = 0; e < E; ++e) zall += exp((double)l[e] - lmax);
                    for (int j = 0; j < topk; ++j) {
                        wj[j] = exp((double)l[ids[t * topk + j]] - lmax);
                        wsum += wj[j];
                    }
                    double z = renormalize ? wsum : zall;
                    for (int j = 0; j < topk; ++j)
                        weights[t * topk + j] = (float)(wj[j] / z * routed_scaling);
                } else {
                    for (int j = 0; j < topk; ++j) {
                        wj[j] = (double)sig[ids[t * topk + j]];
                        wsum += wj[j];
                    }
                    for (int j = 0; j < topk; ++j) {
                        double w = renormalize ? wj[j] / wsum : wj[j];
                        weights[t * topk + j] = (float)(w * routed_scaling);
                    }
                }
            }
        }
        free(sel_score); free(sig); free(allowed); free(gscore); free(gallowed);
    }
    return fail ? -2 : 0;
}

/* ------------------------------------------------------------------------- */
/* Sort routed pairs by expert ("sorted token" pattern, [QMO] Triton Fused MoE
 * Kernel).  Pair p = t*topk + j is routed to ids[p].  counts[e] = #pairs of
 * expert e; offsets = exclusive prefix sum of counts ([E+1]); within an expert
 * the pairs keep ascending p; sorted[offsets[e] + r] = r-th such pair;
 * pos[p] = the index of pair p in sorted. */
void orc_permute(const int32_t* ids, long P, int E, int32_t* offsets, int32_t* sorted, int32_t* pos) {
    long* count = (long*)calloc((size_t)E, sizeof(long));
    for (long p = 0; p < P; ++p) count[ids[p]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + (int32_t)count[e];
    long* fill = (long*)calloc((size_t)E, sizeof(long));
    for (long p = 0; p < P; ++p) {
        int e = ids[p];
        long idx = offsets[e] + fill[e]++;
        sorted[idx] = (int32_t)p;
        pos[p] = (int32_t)idx;
    }
    free(count);
    free(fill);
}

/* ------------------------------------------------------------------------- */
/* Expert computation on the sorted rows ("permute -> GEMM -> unpermute",
 * [QMO] Modular Kernel Architecture), weights w13 (gate+up) and w2 (down) of
 * shape [num_experts, N, K] ([QMO] FusedMoE Class), 128x128 block scales.
 *
 * For sorted row r (pair p, token t = p / topk, expert e):
 *   a[h]      = code(a1q[t,h]) * a1s[t, h/128]
 *   C1[n]     = sum_h a[h] * code(w13[e,n,h]) * w13s[e, n/128, h/128],  n < 2I
 *   h1[i]     = silu(C1[i]) * C1[I+i],  silu(g) = g / (1 + exp(-g))
 *   (a2q, a2s)= 1x128 quantisation of fp32(h1)
 *   C2[r, n]  = sum_i code(a2q[i]) * a2s[i/128] * code(w2[e,n,i]) * w2s[e, n/128, i/128]
 * all sums in fp64.  Only rows whose token has need[t] != 0 are computed (the
 * others are left untouched), so large configurations can be sampled.
 *
 * a2q: [P, I], a2s: [P, I/128], c1: [P, 2I] (may be NULL), c2: [P, H] fp64,
 * each indexed by sorted row.  With NVFP4 weights (orc_experts_nvfp4) only the
 * weight values change: code(w) * block scale * global scale, see dequant_nvfp4. */

/* dequantised weights of expert e: which 0 = w13 as [2I][H], 1 = w2 as [H][I], in fp64 */
typedef void (*dequant_fn)(const void* ctx, int e, int which, long N1, long H, long I, double* wdq);

static void experts_core(const uint8_t* a1q, const float* a1s, dequant_fn dq, const void* ctx,
                         const int32_t* offsets, const int32_t* sorted, const unsigned char* need,
                         long H, long I, int E, int topk, uint8_t* a2q, float* a2s, double* c1, double* c2,
                         int fmt, int ga) {
    e4m3_build();
    long N1 = 2 * I, HB = H / ga, IB = I / ga;   /* activation groups of ga values (128, or 32 for MXFP8) */
    double* wdq = (double*)malloc(sizeof(double) * (size_t)(N1 * H > H * I ? N1 * H : H * I));
    for (int e = 0; e < E; ++e) {
        long r0 = offsets[e], r1 = offsets[e + 1];
        long nrows = 0;
        for (long r = r0; r < r1; ++r) if (need[sorted[r] / topk]) nrows++;
        if (nrows == 0) continue;
        dq(ctx, e, 0, N1, H, I, wdq);
#pragma omp parallel for schedule(dynamic, 1)
        for (long r = r0; r < r1; ++r) {
            long p = sorted[r], t = p / topk;
            if (!need[t]) continue;
            double* a = (double*)malloc(sizeof(double) * (size_t)H);
            double* g = (double*)malloc(sizeof(double) * (size_t)N1);
            float* h1 = (float*)malloc(sizeof(float) * (size_t)I);
            for (long h = 0; h < H; ++h) a[h] = e4m3_val[a1q[t * H + h]] * (double)a1s[t * HB + h / ga];
            for (long n = 0; n < N1; ++n) {
                double acc = 0.0;
                const double* wr = wdq + n * H;
                for (long h = 0; h < H; ++h) acc += a[h] * wr[h];
                g[n] = acc;
                if (c1) c1[r * N1 + n] = acc;
            }
            for (long i = 0; i < I; ++i) {
                double gate = g[i], up = g[I + i];
                h1[i] = (float)(gate / (1.0 + exp(-gate)) * up);
            }
            orc_quant_1xg_f32(h1, 1, I, ga, a2q + r * I, a2s + r * IB, fmt);
            free(a); free(g); free(h1);
        }
        dq(ctx, e, 1, N1, H, I, wdq);
#pragma omp parallel for schedule(dynamic, 1)
        for (long r = r0; r < r1; ++r) {
            long p = sorted[r], t = p / topk;
            if (!need[t]) continue;
            double* a2 = (double*)malloc(sizeof(double) * (size_t)I);
            for (long i = 0; i < I; ++i) a2[i] = e4m3_val[a2q[r * I + i]] * (double)a2s[r * IB + i / ga];
            for (long n = 0; n < H; ++n) {
                double acc = 0.0;
                const double* wr = wdq + n * I;
                for (long i = 0; i < I; ++i) acc += a2[i] * wr[i];
                c2[r * H + n] = acc;
            }
            free(a2);
        }
    }
    free(wdq);
}

/* 128x128-block FP8 weights: code value times its block's fp32 scale */
struct fp8_weights {
    const uint8_t *w13, *w2;
    const float *w13s, *w2s;
};

static void dequant_fp8(const void* ctx, int e, int which, long N1, long H, long I, double* wdq) {
    const struct fp8_weights* W = (const struct fp8_weights*)ctx;
    long HB = H / 128, IB = I / 128;
    if (which == 0) {
#pragma omp parallel for schedule(static)
        for (long n = 0; n < N1; ++n)
            for (long h = 0; h < H; ++h)
                wdq[n * H + h] = e4m3_val[W->w13[((long)e * N1 + n) * H + h]] *
                                 (double)W->w13s[((long)e * (N1 / 128) + n / 128) * HB + h / 128];
    } else {
#pragma omp parallel for schedule(static)
        for (long n = 0; n < H; ++n)
            for (long i = 0; i < I; ++i)
                wdq[n * I + i] = e4m3_val[W->w2[((long)e * H + n) * I + i]] *
                                 (double)W->w2s[((long)e * HB + n / 128) * IB + i / 128];
    }
}

/* NVFP4 weights ([NVFP4] _quantize_moe_weight_to_nvfp4): code value times its 16-block's e4m3
 * scale times the expert's global scale (the products are exact in fp64) */
struct nvfp4_weights {
    const uint8_t *w13, *w2, *w13sf, *w2sf;
    const float *w13gs, *w2gs;
};

static void dequant_nvfp4(const void* ctx, int e, int which, long N1, long H, long I, double* wdq) {
    const struct nvfp4_weights* W = (const struct nvfp4_weights*)ctx;
    long N = which == 0 ? N1 : H, K = which == 0 ? H : I;
    const uint8_t* q = which == 0 ? W->w13 : W->w2;
    const uint8_t* sf = which == 0 ? W->w13sf : W->w2sf;
    double gs = (double)(which == 0 ? W->w13gs : W->w2gs)[e];
#pragma omp parallel for schedule(static)
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k) {
            long i = ((long)e * N + n) * K + k;
            int code = (q[i / 2] >> (4 * (k & 1))) & 15;
            wdq[n * K + k] = orc_e2m1_value(code) * e4m3_val[sf[i / 16]] * gs;
        }
}

void orc_experts(const uint8_t* a1q, const float* a1s,
                 const uint8_t* w13, const float* w13s, const uint8_t* w2, const float* w2s,
                 const int32_t* offsets, const int32_t* sorted, const unsigned char* need,
                 long T, long H, long I, int E, int topk,
                 uint8_t* a2q, float* a2s, double* c1, double* c2, int fmt) {
    (void)T;
    struct fp8_weights W = {w13, w2, w13s, w2s};
    experts_core(a1q, a1s, dequant_fp8, &W, offsets, sorted, need, H, I, E, topk, a2q, a2s, c1, c2, fmt, 128);
}

/* The same expert MLP with NVFP4 weights: codes [E, N, K/2], block scales [E, N, K/16] (e4m3),
 * global scales [E] (fp32) for w13 and w2. */
void orc_experts_nvfp4(const uint8_t* a1q, const float* a1s,
                       const uint8_t* w13, const uint8_t* w13sf, const float* w13gs,
                       const uint8_t* w2, const uint8_t* w2sf, const float* w2gs,
                       const int32_t* offsets, const int32_t* sorted, const unsigned char* need,
                       long T, long H, long I, int E, int topk,
                       uint8_t* a2q, float* a2s, double* c1, double* c2, int fmt) {
    (void)T;
    struct nvfp4_weights W = {w13, w2, w13sf, w2sf, w13gs, w2gs};
    experts_core(a1q, a1s, dequant_nvfp4, &W, offsets, sorted, need, H, I, E, topk, a2q, a2s, c1, c2, fmt, 128);
}

/* MXFP8 weights ("MXFP8 (block [1, 32])", [FP8O] make_fp8_moe_quant_config; "e8m0 group-32
 * scales", [FP8O] _humming_fp8_weight_schema): code value times the UE8M0 scale of its row's
 * 32-wide K group, w13s [E, 2I, H/32] and w2s [E, H, I/32] (the scales as fp32 powers of two) */
struct mxfp8_weights {
    const uint8_t *w13, *w2;
    const float *w13s, *w2s;
};

static void dequant_mxfp8(const void* ctx, int e, int which, long N1, long H, long I, double* wdq) {
    const struct mxfp8_weights* W = (const struct mxfp8_weights*)ctx;
    long N = which == 0 ? N1 : H, K = which == 0 ? H : I;
    const uint8_t* q = which == 0 ? W->w13 : W->w2;
    const float* sc = which == 0 ? W->w13s : W->w2s;
#pragma omp parallel for schedule(static)
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k) {
            long i = ((long)e * N + n) * K + k;
            wdq[n * K + k] = e4m3_val[q[i]] * (double)sc[((long)e * N + n) * (K / 32) + k / 32];
        }
}

/* The expert MLP in MXFP8: activations and the requantised intermediate in 1x32 groups with UE8M0
 * scales (a1s [T, H/32], a2s [P, I/32]), MXFP8 weights as above. */
void orc_experts_mxfp8(const uint8_t* a1q, const float* a1s,
                       const uint8_t* w13, const float* w13s, const uint8_t* w2, const float* w2s,
                       const int32_t* offsets, const int32_t* sorted, const unsigned char* need,
                       long T, long H, long I, int E, int topk,
                       uint8_t* a2q, float* a2s, double* c1, double* c2) {
    (void)T;
    struct mxfp8_weights W = {w13, w2, w13s, w2s};
    experts_core(a1q, a1s, dequant_mxfp8, &W, offsets, sorted, need, H, I, E, topk, a2q, a2s, c1, c2, 1, 32);
}

/* Weighted unpermute-sum ("gathers results", [QMO] Modular Kernel Architecture;
 * router weight multiply after dequantisation, [QMO] Triton Fused MoE Kernel):
 * out[t, n] = sum_j weights[t, j] * C2[pos[t*topk + j], n], summed in j order in
 * fp64; rows with need[t] == 0 are left untouched. */
void orc_combine(const double* c2, const float* weights, const int32_t* pos, const unsigned char* need,
                 long T, long H, int topk, double* out) {
#pragma omp parallel for schedule(static)
    for (long t = 0; t < T; ++t) {
        if (!need[t]) continue;
        for (long n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int j = 0; j < topk; ++j) acc += (double)weights[t * topk + j] * c2[(long)pos[t * topk + j] * H + n];
            out[t * H + n] = acc;
        }
    }
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
