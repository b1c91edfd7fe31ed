// Shared device helpers for the sm_103a kernels of the block-FP8 MoE layer:
// mbarriers with bounded waits, TMA tile loads, tcgen05 (tensor memory + MMA)
// wrappers and the e4m3 conversion.  Every wait in this library is bounded in
// time: on expiry it reports MOE_STATUS_WAIT_TIMEOUT through the status word
// instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moefp8.h"

namespace mfp8 {

// Give up on a pipeline wait after this long (ns of %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void status_set(uint32_t* status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// Programmatic dependent launch: every kernel of this library is launched so that it
// may start while the previous kernel in the stream finishes; before it reads anything
// an earlier kernel wrote (or writes anything an earlier kernel reads) it waits here for
// the previous grid to complete and its memory to be visible.  Every kernel calls it on
// every path, so the wait also covers all grids before that one.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (after setting the timeout status bit and the CTA-wide abort flag) if it did
// not complete within kWaitLimitNs, or if another thread of the CTA already
// aborted.  `abort_flag` points to a shared int (may be null).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t outer = 0; outer < (1u << 26); ++outer) {
        for (int i = 0; i < 32; ++i)
            if (mbar_test(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
    if (abort_flag) *abort_flag = 1;
    status_set(status, MOE_STATUS_WAIT_TIMEOUT);
    return false;
}

// ---------------------------------------------------------------- TMA
// 2-D tiled bulk tensor load into shared memory, completion counted on `bar`
// in bytes.  x is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// 3-D and 4-D tiled loads (coordinates innermost first), completion on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            int32_t w, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_5d(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            int32_t w, int32_t v, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], "
        "[%7];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- cp.async (global -> shared)
__device__ __forceinline__ void cp_async_4(uint32_t smem_dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_16(uint32_t smem_dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed (the
// barrier's expected count must include this arrival).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 128 bytes long and stored with the 128-byte swizzle (the layout a TMA load
// with CU_TENSOR_MAP_SWIZZLE_128B writes): 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_k128_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);   // start address
    d |= static_cast<uint64_t>(0) << 16;                  // leading byte offset: unused here
    d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                  // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;                  // swizzle: 128 B
    return d;
}

// Instruction descriptor of a dense kind::f8f6f4 MMA: A and B e4m3, both
// K-major, fp32 accumulator, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
    return (1u << 4)                                     // D format: f32
           | (0u << 7) | (0u << 10)                      // A, B format: e4m3
           | (static_cast<uint32_t>(n >> 3) << 17)       // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);      // M / 16
}

// ---------------------------------------------------------------- block-scaled MMA (UE8M0)
// Packed UE8M0 scale factors ("UE8M0: packed UE8M0, 4 values per int32, Blackwell", page
// "Quantization and MoE Optimizations", section DeepGEMM Scale Formats).  The scales of 128 rows
// (or 128 weight columns) over 4 consecutive 128-wide K blocks form one 512-byte tile: 32 lines of
// 16 bytes, line l holding rows l, l+32, l+64, l+96 as four 32-bit words, byte b of a word the
// scale of K block 4q + b.  A tile goes to tensor memory as it is (tcgen05.cp 32x128b, copied to
// all four lane quarters): 4 columns, where row m's word sits in column m / 32 of every quarter,
// the layout the block-scaled MMA reads.
constexpr int kSfTileBytes = 512;

// Byte offset of (row r, K block kb) in a packed array of such tiles, tiles ordered
// [row / 128][kb / 4] with kb4 = ceil(K blocks / 4) tiles per 128 rows.
__host__ __device__ __forceinline__ int64_t packed_sf_offset(int64_t r, int kb, int kb4) {
    return ((r >> 7) * kb4 + (kb >> 2)) * kSfTileBytes + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

// UE8M0 byte of a power-of-two fp32 scale: its biased exponent (value 2^(byte - 127)).
__device__ __forceinline__ uint8_t ue8m0_byte(float s) {
    return static_cast<uint8_t>((__float_as_uint(s) >> 23) & 0xFFu);
}

// Shared-memory descriptor of a 32-row x 16-byte tile stored row after row (no swizzle): the
// source of tcgen05.cp 32x128b (8-row groups 128 bytes apart).
__device__ __forceinline__ uint64_t smem_desc_sf_tile(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);   // start address
    d |= static_cast<uint64_t>(128 >> 4) << 16;           // leading byte offset (one 16-byte column: unused)
    d |= static_cast<uint64_t>(128 >> 4) << 32;           // stride byte offset: 8 rows x 16 B
    d |= static_cast<uint64_t>(1) << 46;                  // descriptor version (sm_100 family)
    return d;                                             // swizzle field 0: none
}

// Copy a 512-byte scale-factor tile from shared memory into 4 tensor-memory columns of all four
// lane quarters (issued by one thread; ordered before the MMAs this thread issues after it).
__device__ __forceinline__ void tmem_copy_sf_tile(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor of a block-scaled kind::mxf8f6f4 MMA: A and B e4m3, both K-major,
// UE8M0 scale factors, fp32 accumulator, M = m, N = n; sf_id picks the byte of each 32-bit
// scale word (here: which of the 4 packed K blocks).
__host__ __device__ constexpr uint32_t idesc_e4m3_ue8m0(int m, int n, int sf_id) {
    return (static_cast<uint32_t>(sf_id & 3) << 4)          // B scale-factor byte
           | (0u << 7) | (0u << 10)                         // A, B format: e4m3
           | (static_cast<uint32_t>(n >> 3) << 17)          // N / 8
           | (1u << 23)                                     // scale-factor format: UE8M0
           | (static_cast<uint32_t>(m >> 4) << 24)          // M / 16
           | (static_cast<uint32_t>(sf_id & 3) << 29);      // A scale-factor byte
}

// D[tmem] (+)= (A * sfA)[smem] * (B * sfB)[smem]^T, 128 x N x 32 e4m3 with one UE8M0 scale per
// row of A and per column of B for these 32 K (scale factors in tensor memory), issued by one thread.
__device__ __forceinline__ void mma_e4m3_block_scaled(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                      uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                      uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
            "r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 1-D bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) into shared memory,
// completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t smem_dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, 128 x N x 32 e4m3, issued by one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Two 32-column fp32 loads of the warp's 32 TMEM lanes and the wait for both, in one
// asm statement so that no use of the results can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t taddr0, uint32_t taddr1, float* va, float* vb) {
    uint32_t a[32], b[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
          "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]),
          "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
          "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]),
          "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]),
          "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
        : "r"(taddr0), "r"(taddr1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        va[i] = __uint_as_float(a[i]);
        vb[i] = __uint_as_float(b[i]);
    }
}

// Register budget moves between warpgroups (all four warps of a warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- e4m3
// Two fp32 values to two e4m3fn bytes (round to nearest even, saturating):
// `lo` lands in the low byte, `hi` in the high byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 values to a packed bf16 pair (round to nearest even): `lo` in the low half.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// acc[0..1] += v[0..1] * s with one packed fp32x2 FMA (round to nearest)
__device__ __forceinline__ void ffma2(float* acc, const float* v, float s) {
    const float2 r = __ffma2_rn(make_float2(v[0], v[1]), make_float2(s, s), make_float2(acc[0], acc[1]));
    acc[0] = r.x;
    acc[1] = r.y;
}

// x / s rounded to nearest even, given r = 1/s rounded to nearest even: one product
// and one fused correction step (Markstein, "IA-64 and Elementary Functions", 2000:
// with r within half an ulp of 1/s and q within one ulp of x/s, q + (x - s*q)*r
// rounds to the correctly rounded quotient).  Holds while x/s is in the normal
// range; smaller quotients only ever map to e4m3 code 0 here.
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
    const float q = x * r;
    const float e = fmaf(-q, s, x);
    return fmaf(e, r, q);
}

// scale of a group from its amax: max(amax, 1e-8) / 448 with IEEE division
__device__ __forceinline__ float group_scale(float amax) {
    return __fdiv_rn(fmaxf(amax, 1e-8f), 448.0f);
}

// The same scale in format fmt: MOE_SCALE_F32 as is, MOE_SCALE_UE8M0 rounded up to a power
// of two (a positive normal float whose mantissa bits are not all zero goes to the next
// exponent), so that it is exactly an 8-bit exponent.
__device__ __forceinline__ float group_scale_fmt(float amax, int fmt) {
    const float t = group_scale(amax);
    if (fmt != MOE_SCALE_UE8M0) return t;
    const uint32_t b = __float_as_uint(t);
    return (b & 0x007FFFFFu) ? __uint_as_float((b & 0x7F800000u) + 0x00800000u) : t;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// ---------------------------------------------------------------- bf16 / e4m3 groups of 8
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    }
}

// codes of 8 values x / sc (correctly rounded quotient, see div_by_scale; rsc = 1/sc rounded)
__device__ __forceinline__ uint2 encode8(const float* f, float sc, float rsc) {
    uint32_t b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint16_t lo = e4m3x2(div_by_scale(f[2 * i], sc, rsc), div_by_scale(f[2 * i + 1], sc, rsc));
        b[i] = lo;
    }
    return make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}

// ---------------------------------------------------------------- block scan
// exclusive scan over the 1024 threads of the block
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int res = (warp ? warp_sums[warp - 1] : 0) + x - v;
    __syncthreads();
    return res;
}

}  // namespace mfp8
