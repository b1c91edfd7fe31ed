// FP8 quantisation kernels (HBM-bound).
//
// Activation groups of 1x128 ("computed per-token at runtime", page
// "Quantization and MoE Optimizations", section Fp8Config; key
// kFp8Dynamic128Sym, page "vllm.model_executor.layers.fused_moe.oracle.fp8"):
// scale = max(amax, 1e-8)/448 in fp32, codes = e4m3(x / scale) with the
// correctly rounded quotient and the hardware's round-to-nearest-even, saturating
// conversion.
// Sixteen threads own one group (8 bf16 = one 16-byte load each), reduce the
// amax with four shuffles, and write 8 code bytes each.  The scatter form
// writes each token's codes to the sorted rows of its top-k pairs, so the
// expert GEMM reads one dense [rows, H] operand (the token is quantised once).
//
// Weight blocks of 128x128 ("weight_block_size ... [128, 128]", Fp8Config)
// use the same rule with the amax over the whole block: one 256-thread CTA per
// block keeps its 32 KB of bf16 in registers between the amax and the encode.
//
// The weighted unpermute-sum adds each token's k router-weighted expert rows
// in a fixed order (j) and rounds to bf16: from fp32 rows in sorted order
// (unpermute_sum_kernel), or from bf16 rows in pair order, where a token's k
// rows are contiguous (combine_pairs_kernel, the layer's path).
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace mfp8 {

namespace {

__global__ void __launch_bounds__(256) group_quant_kernel(const uint16_t* __restrict__ x, int64_t rows, int cols,
                                                          int64_t ld, uint8_t* __restrict__ q, int64_t q_ld,
                                                          float* __restrict__ s, int64_t s_rs, int64_t s_gs,
                                                          const int32_t* __restrict__ pos, int topk, int scale_fmt,
                                                          uint8_t* __restrict__ sf, int sf_kb4,
                                                          uint8_t* __restrict__ s8) {
    grid_dependency_wait();
    const int G = cols / 128;
    const int64_t total = rows * G;
    const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w * 2 < total;
         w += nwarps) {
        const int64_t gi = w * 2 + half;
        const bool active = gi < total;
        float f[8];
        float amax = 0.0f;
        int64_t r = 0;
        int g = 0;
        if (active) {
            r = gi / G;
            g = static_cast<int>(gi - r * G);
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + r * ld + g * 128 + sub * 8));
            unpack8(v, f);
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
            // the scale's column: the 128-group, or (MXFP8) the 32-group g*4 + sub/4
            const int sc_col = mx ? g * 4 + (sub >> 2) : g;
            const bool writer = mx ? (sub & 3) == 0 : sub == 0;
            const int sc_cols = mx ? cols / 32 : cols / 128;
            const int64_t n_rows = pos ? topk : 1;
            for (int j = 0; j < n_rows; ++j) {
                const int64_t o = pos ? pos[r * topk + j] : r;
                if (o < 0) continue;
                *reinterpret_cast<uint2*>(q + o * q_ld + g * 128 + sub * 8) = code;
                if (writer) {
                    if (s) s[o * s_rs + g * s_gs] = sc;
                    if (s8) s8[o * sc_cols + sc_col] = ue8m0_byte(sc);
                    if (sf) sf[packed_sf_offset(o, sc_col, sf_kb4)] = ue8m0_byte(sc);
                }
            }
        }
    }
}

// The same quantisation for the layer's common case, written to keep the instruction count low
// (the general kernel above issued about 580 warp instructions per two groups and was bound by
// instruction issue, not HBM): 1x128 groups with fp32 or UE8M0 scales (s [groups][rows]), or
// UE8M0 scale bytes in packed tiles (PACKED: sf, sf_kb4 as the general kernel's), or MXFP8 (MX:
// 1x32 groups of four threads, their UE8M0 bytes in packed tiles), every token's
// codes scattered to the K sorted rows pos[r*K + j] (K fixed at compile time, the K row indices
// loaded as vectors once per group; pos 16-byte aligned), 32-bit index arithmetic where the
// sizes allow (checked by the launcher).
template <int K, bool UE8M0, bool PACKED, bool MX = false>
__global__ void __launch_bounds__(256) group_quant_scatter_kernel(const uint16_t* __restrict__ x, int rows, int G,
                                                                  int ld, uint8_t* __restrict__ q, int q_ld,
                                                                  float* __restrict__ s, int s_gs,
                                                                  const int32_t* __restrict__ pos,
                                                                  uint8_t* __restrict__ sf, int sf_kb4) {
    grid_dependency_wait();
    const int total = rows * G;
    const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; w * 2 < total; w += nwarps) {
        const int gi = w * 2 + half;
        const bool active = gi < total;
        const int r = active ? gi / G : 0;
        const int g = active ? gi - r * G : 0;
        int o[K];
        if constexpr (K % 4 == 0) {
#pragma unroll
            for (int j = 0; j < K; j += 4) {
                const int4 v = __ldg(reinterpret_cast<const int4*>(pos + r * K + j));
                o[j] = v.x;
                o[j + 1] = v.y;
                o[j + 2] = v.z;
                o[j + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < K; j += 2) {
                const int2 v = __ldg(reinterpret_cast<const int2*>(pos + r * K + j));
                o[j] = v.x;
                o[j + 1] = v.y;
            }
        }
        float f[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(r) * ld + g * 128 + sub * 8)), f);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o2 = MX ? 2 : 8; o2 > 0; o2 >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
        if (!active) continue;
        const float sc = group_scale_fmt(amax, UE8M0 ? MOE_SCALE_UE8M0 : MOE_SCALE_F32);
        const uint2 code = encode8(f, sc, __frcp_rn(sc));
        uint8_t* qg = q + g * 128 + sub * 8;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (o[j] < 0) continue;
            *reinterpret_cast<uint2*>(qg + static_cast<int64_t>(o[j]) * q_ld) = code;
            if constexpr (MX) {
                if ((sub & 3) == 0) sf[packed_sf_offset(o[j], g * 4 + (sub >> 2), sf_kb4)] = ue8m0_byte(sc);
            } else if (sub == 0) {
                if constexpr (PACKED)
                    sf[packed_sf_offset(o[j], g, sf_kb4)] = ue8m0_byte(sc);
                else
                    s[g * s_gs + o[j]] = sc;
            }
        }
    }
}

__global__ void __launch_bounds__(256) block_quant_weight_kernel(const uint16_t* __restrict__ w, int N, int K,
                                                                 uint8_t* __restrict__ q, float* __restrict__ s,
                                                                 int scale_fmt) {
    grid_dependency_wait();
    __shared__ float warp_max[8];
    const int kb = blockIdx.x, nb = blockIdx.y, e = blockIdx.z;
    const int NB = N / 128, KB = K / 128;
    const int row = threadIdx.x >> 1, part = threadIdx.x & 1;
    const int64_t off = (static_cast<int64_t>(e) * N + nb * 128 + row) * K + kb * 128 + part * 64;
    uint4 v[8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = __ldg(reinterpret_cast<const uint4*>(w + off) + i);
        float f[8];
        unpack8(v[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);
    const float sc = group_scale_fmt(amax, scale_fmt);
    const float rsc = __frcp_rn(sc);
    uint2 out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float f[8];
        unpack8(v[i], f);
        out[i] = encode8(f, sc, rsc);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
        reinterpret_cast<uint4*>(q + off)[i] = make_uint4(out[2 * i].x, out[2 * i].y, out[2 * i + 1].x,
                                                          out[2 * i + 1].y);
    if (threadIdx.x == 0) s[(static_cast<int64_t>(e) * NB + nb) * KB + kb] = sc;
}

// Load-time packing of 128x128 block scales [E, N/128, K/128] (powers of two) into the
// scale-factor tiles of the block-scaled GEMM: [E][N/128][ceil(K/512)] tiles, each line of a tile
// holding the 4 K blocks' bytes once per 32-row quarter (a block's scale is the scale of all its
// 128 rows).  One thread per 16-byte line; K blocks past the end get byte 127 (scale 1).  A scale
// that is not a positive power of two sets MOE_STATUS_BAD_SCALE (its byte is then its exponent).
__global__ void __launch_bounds__(256) pack_scales_kernel(const float* __restrict__ s, int64_t nblocks, int KB,
                                                          uint4* __restrict__ out, uint32_t* status) {
    grid_dependency_wait();
    const int KB4 = (KB + 3) / 4;
    const int64_t lines = nblocks * KB4 * 32;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < lines;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = i >> 5;
        const int64_t blk = tile / KB4;
        const int q = static_cast<int>(tile - blk * KB4);
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int kb = q * 4 + b;
            uint32_t byte = 127u;
            if (kb < KB) {
                const float v = s[blk * KB + kb];
                const uint32_t bits = __float_as_uint(v);
                if ((bits & 0x007FFFFFu) || !(v > 0.0f) || bits >= 0x7F800000u) status_set(status, MOE_STATUS_BAD_SCALE);
                byte = (bits >> 23) & 0xFFu;
            }
            word |= byte << (8 * b);
        }
        out[i] = make_uint4(word, word, word, word);
    }
}

// out[t] = bf16(sum_j y[pos[t*topk + j]]): thread = 4 consecutive columns of one token,
// the k rows summed in j order in fp32.
__global__ void __launch_bounds__(256) unpermute_sum_kernel(const float4* __restrict__ y, int64_t y_rows,
                                                            const int32_t* __restrict__ pos, int64_t T, int topk,
                                                            int H4, uint2* __restrict__ out, uint32_t* status) {
    grid_dependency_wait();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= H4) return;
    for (int64_t t = blockIdx.y; t < T; t += gridDim.y) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int j = 0; j < topk; ++j) {
            const int64_t r = pos[t * topk + j];
            if (r < 0) continue;
            if (r >= y_rows) {
                if (c == 0) status_set(status, MOE_STATUS_BAD_EXPERT_ID);
                continue;
            }
            const float4 v = __ldg(y + r * H4 + c);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(acc.x));
        const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(acc.y));
        const uint32_t cc = __bfloat16_as_ushort(__float2bfloat16_rn(acc.z));
        const uint32_t d = __bfloat16_as_ushort(__float2bfloat16_rn(acc.w));
        out[t * H4 + c] = make_uint2(a | (b << 16), cc | (d << 16));
    }
}

// out[t] = bf16(sum_j float(y[t*topk + j])) over the pairs with pos >= 0: one thread per 8
// consecutive columns of one token, the token's k rows (contiguous in pair order) loaded
// together and summed in j order in fp32.
template <int K>
__global__ void __launch_bounds__(256) combine_pairs_kernel(const uint4* __restrict__ y,
                                                            const int32_t* __restrict__ pos, int64_t T, int topk,
                                                            int H8, uint4* __restrict__ out) {
    grid_dependency_wait();
    const int64_t total = T * H8;
    const int kk = K > 0 ? K : topk;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / H8;
        const int c = static_cast<int>(i - t * H8);
        const uint4* src = y + t * kk * H8 + c;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        if (K > 0) {
            // all k rows in flight at once
            bool live[K > 0 ? K : 1];
            uint4 v[K > 0 ? K : 1];
#pragma unroll
            for (int j = 0; j < K; ++j) live[j] = __ldg(pos + t * K + j) >= 0;
#pragma unroll
            for (int j = 0; j < K; ++j) v[j] = live[j] ? __ldg(src + static_cast<int64_t>(j) * H8) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (!live[j]) continue;
                float f[8];
                unpack8(v[j], f);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += f[q];
            }
        } else {
            for (int j = 0; j < kk; ++j) {
                if (__ldg(pos + t * kk + j) < 0) continue;
                float f[8];
                unpack8(__ldg(src + static_cast<int64_t>(j) * H8), f);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += f[q];
            }
        }
        out[i] = make_uint4(bf16x2(acc[0], acc[1]), bf16x2(acc[2], acc[3]), bf16x2(acc[4], acc[5]),
                            bf16x2(acc[6], acc[7]));
    }
}

// [E, N, K] -> [E][N/128][K/128][128 rows][128 bytes]: one thread per 16 bytes of the output
// (coalesced writes; each source row segment of 128 bytes is read by 8 consecutive threads)
__global__ void __launch_bounds__(256) pack_weights_kernel(const uint4* __restrict__ w, int64_t N, int64_t K,
                                                           int64_t total16, uint4* __restrict__ out) {
    grid_dependency_wait();
    const int64_t NB = N / 128, KB = K / 128;
    for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < total16;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t blk = o >> 10;                 // 1024 x 16 B per block
        const int r = static_cast<int>((o >> 3) & 127), c = static_cast<int>(o & 7);
        const int64_t kb = blk % KB, nb = (blk / KB) % NB, e = blk / (KB * NB);
        out[o] = __ldg(w + (((e * N + nb * 128 + r) * K + kb * 128) >> 4) + c);
    }
}

int grid_for(int64_t work_items, int per_block) {
    int64_t b = (work_items + per_block - 1) / per_block;
    if (b < 1) b = 1;
    if (b > 152 * 32) b = 152 * 32;
    return static_cast<int>(b);
}

}  // namespace

cudaError_t launch_group_quant(const uint16_t* x, int64_t rows, int cols, int64_t ld, uint8_t* q, int64_t q_ld,
                               float* s, int64_t s_row_stride, int64_t s_group_stride, const int32_t* pos,
                               int topk, int scale_fmt, cudaStream_t stream, uint8_t* sf, uint8_t* s8) {
    const int64_t groups = rows * (cols / 128);
    if (groups == 0) return cudaSuccess;
    // packed tiles: 4 scale columns per 32-bit word (MXFP8: 32-groups, 4 per 128-wide K block)
    const int sf_kb4 = scale_fmt == MOE_SCALE_MXFP8 ? cols / 128 : (cols / 128 + 3) / 4;
    // the common case on its lean kernel: fp32 or UE8M0 scales [groups][rows] (row stride 1), or
    // only packed UE8M0 tiles, rows scattered to pos with top-k 2 or 8, every offset within 32 bits
    const bool packed_only = sf && !s;   // packed UE8M0 tiles, or MXFP8 (its 32-group tiles)
    const bool mx = scale_fmt == MOE_SCALE_MXFP8;
    const bool lean = pos && ((s && !sf) || packed_only) && !s8 && s_row_stride == 1 && (topk == 2 || topk == 8) &&
                      (scale_fmt == MOE_SCALE_F32 || scale_fmt == MOE_SCALE_UE8M0 || packed_only) && ld <= INT32_MAX &&
                      q_ld <= INT32_MAX && s_group_stride <= INT32_MAX && groups < (int64_t(1) << 30) &&
                      rows * topk < INT32_MAX && rows * ld < INT32_MAX && (cols / 128) * s_group_stride < INT32_MAX &&
                      (reinterpret_cast<uintptr_t>(pos) & 15) == 0;
    if (lean) {
        const int r32 = static_cast<int>(rows), G = cols / 128;
#define MOE_QUANT_LEAN(KK, U8, PK)                                                                           \
    return launch_pdl(group_quant_scatter_kernel<KK, U8, PK>, dim3(grid_for(groups, 16)), dim3(256), 0, stream, \
                      x, r32, G, static_cast<int>(ld), q, static_cast<int>(q_ld), s,                              \
                      static_cast<int>(s_group_stride), pos, sf, sf_kb4)
        if (topk == 8) {
            if (mx) return launch_pdl(group_quant_scatter_kernel<8, true, true, true>, dim3(grid_for(groups, 16)),
                                      dim3(256), 0, stream, x, r32, G, static_cast<int>(ld), q, static_cast<int>(q_ld),
                                      s, static_cast<int>(s_group_stride), pos, sf, sf_kb4);
            if (packed_only) MOE_QUANT_LEAN(8, true, true);
            if (scale_fmt == MOE_SCALE_UE8M0) MOE_QUANT_LEAN(8, true, false);
            MOE_QUANT_LEAN(8, false, false);
        }
        if (mx) return launch_pdl(group_quant_scatter_kernel<2, true, true, true>, dim3(grid_for(groups, 16)),
                                  dim3(256), 0, stream, x, r32, G, static_cast<int>(ld), q, static_cast<int>(q_ld), s,
                                  static_cast<int>(s_group_stride), pos, sf, sf_kb4);
        if (packed_only) MOE_QUANT_LEAN(2, true, true);
        if (scale_fmt == MOE_SCALE_UE8M0) MOE_QUANT_LEAN(2, true, false);
        MOE_QUANT_LEAN(2, false, false);
#undef MOE_QUANT_LEAN
    }
    const int fmt = scale_fmt == MOE_SCALE_MXFP8 ? MOE_SCALE_MXFP8 : (sf ? MOE_SCALE_UE8M0 : scale_fmt);
    return launch_pdl(group_quant_kernel, dim3(grid_for(groups, 16)), dim3(256), 0, stream, x, rows, cols, ld, q,
                      q_ld, s, s_row_stride, s_group_stride, pos, topk, fmt, sf, sf_kb4, s8);
}

// Packing of UE8M0 scale bytes s [rows, C] (row-major) into scale-factor tiles: out at
// packed_sf_offset(r, c, ceil(C/4)); missing bytes of a last partial word or tile are left alone.
__global__ void __launch_bounds__(256) pack_scale_bytes_kernel(const uint8_t* __restrict__ s, int64_t rows, int C,
                                                               uint8_t* __restrict__ out) {
    grid_dependency_wait();
    const int C4 = (C + 3) / 4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < rows * C;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / C;
        const int c = static_cast<int>(i - r * C);
        out[packed_sf_offset(r, c, C4)] = s[i];
    }
}

cudaError_t launch_pack_scale_bytes(const uint8_t* s, int64_t rows, int C, uint8_t* out, cudaStream_t stream) {
    const int64_t n = rows * C;
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    return launch_pdl(pack_scale_bytes_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, s, rows,
                      C, out);
}

cudaError_t launch_pack_scales(const float* s, int E, int N, int K, uint8_t* out, uint32_t* status,
                               cudaStream_t stream) {
    const int64_t nblocks = static_cast<int64_t>(E) * (N / 128);
    const int KB = K / 128;
    const int64_t lines = nblocks * ((KB + 3) / 4) * 32;
    if (lines == 0) return cudaSuccess;
    int64_t blocks = (lines + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    return launch_pdl(pack_scales_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, s, nblocks, KB,
                      reinterpret_cast<uint4*>(out), status);
}

cudaError_t launch_block_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, float* s, int scale_fmt,
                                      cudaStream_t stream) {
    if (E == 0 || N == 0 || K == 0) return cudaSuccess;
    dim3 grid(K / 128, N / 128, E);
    return launch_pdl(block_quant_weight_kernel, grid, dim3(256), 0, stream, w, N, K, q, s, scale_fmt);
}

cudaError_t launch_unpermute_sum(const float* y, int64_t y_rows, const int32_t* pos, int64_t T, int topk, int H,
                                 uint16_t* out, uint32_t* status, cudaStream_t stream) {
    if (T == 0 || H == 0) return cudaSuccess;
    const int H4 = H / 4;
    dim3 grid((H4 + 255) / 256, static_cast<unsigned>(T < 65535 ? T : 65535));
    return launch_pdl(unpermute_sum_kernel, grid, dim3(256), 0, stream, reinterpret_cast<const float4*>(y), y_rows,
                      pos, T, topk, H4, reinterpret_cast<uint2*>(out), status);
}

}  // namespace mfp8

namespace mfp8 {

cudaError_t launch_combine_pairs(const uint16_t* y, const int32_t* pos, int64_t T, int topk, int H, uint16_t* out,
                                 cudaStream_t stream) {
    if (T == 0 || H == 0) return cudaSuccess;
    const int H8 = H / 8;
    const int grid = grid_for(T * H8, 256);
    const uint4* y4 = reinterpret_cast<const uint4*>(y);
    uint4* o4 = reinterpret_cast<uint4*>(out);
    switch (topk) {
        case 8:
            return launch_pdl(combine_pairs_kernel<8>, dim3(grid), dim3(256), 0, stream, y4, pos, T, topk, H8, o4);
        case 2:
            return launch_pdl(combine_pairs_kernel<2>, dim3(grid), dim3(256), 0, stream, y4, pos, T, topk, H8, o4);
        default:
            return launch_pdl(combine_pairs_kernel<0>, dim3(grid), dim3(256), 0, stream, y4, pos, T, topk, H8, o4);
    }
}

}  // namespace mfp8

namespace mfp8 {

cudaError_t launch_pack_weights(const uint8_t* w, int E, int N, int K, uint8_t* packed, cudaStream_t stream) {
    const int64_t total16 = static_cast<int64_t>(E) * N * K / 16;
    if (total16 == 0) return cudaSuccess;
    return launch_pdl(pack_weights_kernel, dim3(grid_for(total16, 256)), dim3(256), 0, stream,
                      reinterpret_cast<const uint4*>(w), N, K, total16, reinterpret_cast<uint4*>(packed));
}

}  // namespace mfp8
