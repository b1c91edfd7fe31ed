// NVFP4 expert weights: load-time quantisation and packing for the decode-path GEMMs.
//
// Format (page "vllm.model_executor.layers.quantization.online.nvfp4", function
// _quantize_moe_weight_to_nvfp4): per expert, amax over the whole [N, K] weight (floored at
// 1e-8) and global_scale = (FLOAT4_E2M1_MAX * FLOAT8_E4M3_MAX) / amax = 2688 / amax; the
// weights times global_scale, rounded back to bf16, are quantised in blocks of 16 along K:
// block scale = e4m3(max|x| / 6), code = e2m1(x / block scale), two codes per byte (element 2i
// in the low nibble); the per-expert value stored for dequantisation is 1 / global_scale.
// Dequantised weight = e2m1(code) * block scale * (1 / global_scale).
//
// Packed layout read by the decode kernel: for every 16-row slab of an expert's [N, K] and
// every 128-wide K block, one 1152-byte unit = the slab's 16 rows x 64 code bytes, then its
// 16 rows x 8 block-scale bytes:  packed[e][N/16][K/128][1152].  A stage of the decode kernel
// then loads one contiguous run of units per slab, codes and scales together.
#include "kernels.cuh"

namespace mfp8 {

namespace {

constexpr float kFp4Max = 6.0f;
constexpr float kGlobalNumerator = 6.0f * 448.0f;   // FLOAT4_E2M1_MAX * FLOAT8_E4M3_MAX

// amax of |w| per expert, as float bits (non-negative floats order as unsigned integers)
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const uint16_t* __restrict__ w, int64_t per_expert,
                                                         uint32_t* __restrict__ amax_bits) {
    grid_dependency_wait();
    const int e = blockIdx.y;
    const uint4* src = reinterpret_cast<const uint4*>(w + static_cast<int64_t>(e) * per_expert);
    const int64_t n8 = per_expert / 8;
    float amax = 0.0f;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float f[8];
        unpack8(__ldg(src + i), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + e, __float_as_uint(amax));
}

__device__ __forceinline__ float global_scale_of(uint32_t amax_bits) {
    const float amax = fmaxf(__uint_as_float(amax_bits), 1e-8f);
    return __fdiv_rn(kGlobalNumerator, amax);
}

// e4m3 code of a non-negative fp32 value (nearest, ties to even, saturating) and its value
__device__ __forceinline__ uint32_t e4m3_code(float x) { return e4m3x2(x, 0.0f) & 0xFFu; }
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    float f;
    asm("{\n\t.reg .b16 t, lo, hi;\n\t.reg .b32 h;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 h, t;\n\t"
        "mov.b32 {lo, hi}, h;\n\tcvt.f32.f16 %0, lo;\n\t}"
        : "=f"(f)
        : "r"(code));
    return f;
}
// two e2m1 codes (nearest, ties to even, saturating at +-6): lo in bits 0-3, hi in bits 4-7
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// one thread per 16-element block: codes (8 bytes) and the block's scale
__global__ void __launch_bounds__(256) nvfp4_quant_kernel(const uint16_t* __restrict__ w, int E, int N, int K,
                                                          const uint32_t* __restrict__ amax_bits,
                                                          uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
    grid_dependency_wait();
    const int64_t per_expert = static_cast<int64_t>(N) * (K / 16);
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (blk >= static_cast<int64_t>(E) * per_expert) return;
    const int e = static_cast<int>(blk / per_expert);
    const float gsc = global_scale_of(amax_bits[e]);
    const uint4* src = reinterpret_cast<const uint4*>(w + blk * 16);
    float v[16];
    unpack8(__ldg(src), v);
    unpack8(__ldg(src + 1), v + 8);
    float vmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = bf16_bits_to_f32(bf16x2(__fmul_rn(v[i], gsc), 0.0f) & 0xFFFFu);   // product rounded to bf16
        vmax = fmaxf(vmax, fabsf(v[i]));
    }
    const uint32_t s = e4m3_code(__fdiv_rn(vmax, kFp4Max));
    const float sv = e4m3_value(s);
    uint32_t lo = 0, hi = 0;
    if (sv != 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo |= e2m1x2(__fdiv_rn(v[2 * i], sv), __fdiv_rn(v[2 * i + 1], sv)) << (8 * i);
            hi |= e2m1x2(__fdiv_rn(v[8 + 2 * i], sv), __fdiv_rn(v[8 + 2 * i + 1], sv)) << (8 * i);
        }
    }
    *reinterpret_cast<uint2*>(q + blk * 8) = make_uint2(lo, hi);
    sf[blk] = static_cast<uint8_t>(s);
}

// the stored per-expert value 1 / global_scale (after the quantiser has read the amax)
__global__ void nvfp4_global_kernel(int E, float* __restrict__ gs) {
    grid_dependency_wait();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < E) gs[e] = __fdiv_rn(1.0f, global_scale_of(__float_as_uint(gs[e])));
}

// one thread per 16 bytes of a packed unit: 64 code chunks (16 rows x 4), then 8 scale chunks
// (2 rows x 8 bytes each)
__global__ void __launch_bounds__(256) nvfp4_pack_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                                                         int64_t units, int KB, int K, uint8_t* __restrict__ packed) {
    grid_dependency_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= units * (kFp4UnitBytes / 16)) return;
    const int64_t unit = i / (kFp4UnitBytes / 16);
    const int c = static_cast<int>(i - unit * (kFp4UnitBytes / 16));
    const int64_t slab = unit / KB;
    const int kb = static_cast<int>(unit - slab * KB);
    uint4 v;
    if (c < 64) {
        const int64_t row = slab * 16 + c / 4;
        v = __ldg(reinterpret_cast<const uint4*>(q + row * (K / 2) + kb * 64 + (c % 4) * 16));
    } else {
        const int64_t row = slab * 16 + 2 * (c - 64);
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(sf + row * (K / 16) + kb * 8));
        const uint2 b = __ldg(reinterpret_cast<const uint2*>(sf + (row + 1) * (K / 16) + kb * 8));
        v = make_uint4(a.x, a.y, b.x, b.y);
    }
    reinterpret_cast<uint4*>(packed)[i] = v;
}

}  // namespace

cudaError_t launch_nvfp4_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, uint8_t* sf, float* gs,
                                      cudaStream_t stream) {
    if (E == 0 || N == 0 || K == 0) return cudaSuccess;
    // the amax bits go to gs first; the last kernel turns them into 1 / global_scale
    uint32_t* amax_bits = reinterpret_cast<uint32_t*>(gs);
    cudaError_t err = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t) * E, stream);
    if (err != cudaSuccess) return err;
    const int64_t per_expert = static_cast<int64_t>(N) * K;
    int64_t bx = (per_expert / 8 + 255) / 256;
    if (bx > 256) bx = 256;
    err = launch_pdl(nvfp4_amax_kernel, dim3(static_cast<unsigned>(bx), static_cast<unsigned>(E)), dim3(256), 0,
                     stream, w, per_expert, amax_bits);
    if (err != cudaSuccess) return err;
    const int64_t blocks = static_cast<int64_t>(E) * N * (K / 16);
    err = launch_pdl(nvfp4_quant_kernel, dim3(static_cast<unsigned>((blocks + 255) / 256)), dim3(256), 0, stream, w,
                     E, N, K, static_cast<const uint32_t*>(amax_bits), q, sf);
    if (err != cudaSuccess) return err;
    return launch_pdl(nvfp4_global_kernel, dim3((E + 255) / 256), dim3(256), 0, stream, E, gs);
}

size_t nvfp4_packed_bytes(int E, int N, int K) {
    return static_cast<size_t>(E) * (N / 16) * (K / 128) * kFp4UnitBytes;
}

cudaError_t launch_nvfp4_pack(const uint8_t* q, const uint8_t* sf, int E, int N, int K, uint8_t* packed,
                              cudaStream_t stream) {
    const int KB = K / 128;
    const int64_t units = static_cast<int64_t>(E) * (N / 16) * KB;
    if (units == 0) return cudaSuccess;
    const int64_t threads = units * (kFp4UnitBytes / 16);
    return launch_pdl(nvfp4_pack_kernel, dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256), 0, stream, q,
                      sf, units, KB, K, packed);
}

}  // namespace mfp8
