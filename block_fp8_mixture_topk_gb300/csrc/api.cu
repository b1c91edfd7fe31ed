// C ABI of the block-FP8 MoE library: argument checks, workspace layout and the
// launch sequence of the whole layer.  See include/moefp8.h for the contract.
#include <mutex>

#include "kernels.cuh"
#include "route_select.cuh"

using namespace mfp8;

namespace {

// Device status word (MOE_STATUS_* bits), one per device that loads the library.
__device__ uint32_t g_status_word;

struct DeviceState {
    bool init = false;
    int rc = MOE_OK;
    int num_sms = 0;
    uint32_t* status = nullptr;  // device address of g_status_word on this device
};
constexpr int kMaxDevices = 128;
DeviceState g_devices[kMaxDevices];
std::mutex g_devices_mutex;

// Once per device (with that device current): check it is a GB300, look up the
// status word's device address and set the kernels' shared-memory limits.
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_devices_mutex);
    DeviceState& s = g_devices[dev];
    if (!s.init) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            return MOE_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            s.rc = MOE_ERR_DEVICE;
        } else {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || route_init_device() != cudaSuccess ||
                permute_init_device() != cudaSuccess || gemm_init_device() != cudaSuccess ||
                decode_init_device() != cudaSuccess) {
                cudaGetLastError();
                return MOE_ERR_CUDA;
            }
            s.status = static_cast<uint32_t*>(p);
            s.rc = MOE_OK;
        }
        s.init = true;
    }
    *out = &s;
    return s.rc;
}

inline int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int check_routing(int T, int E, int topk, const moe_routing_params* rp) {
    if (T < 0 || E < 1 || topk < 1) return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS || topk > E || topk > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!rp) return MOE_OK;
    if (rp->scoring != MOE_SCORING_SOFTMAX && rp->scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (rp->n_group < 1) return MOE_ERR_INVALID_ARG;
    if (rp->n_group > MOE_MAX_GROUPS || E % rp->n_group != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rp->bias && rp->scoring != MOE_SCORING_SIGMOID) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rp->n_group > 1) {
        const int G = E / rp->n_group;
        if (rp->scoring != MOE_SCORING_SIGMOID) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (rp->topk_group < 1 || rp->topk_group > rp->n_group) return MOE_ERR_INVALID_ARG;
        if (G < 2 || topk > rp->topk_group * G) return MOE_ERR_UNSUPPORTED_SHAPE;
    }
    return MOE_OK;
}

int64_t max_rows(int64_t P, int64_t E, int64_t bm) {
    const int64_t busy = P < E ? P : E;
    return P + busy * (bm - 1);
}

// bytes of the packed UE8M0 scale tiles of a [rows, K] operand (common.cuh, packed_sf_offset):
// one tile per 128 rows and 4 K blocks, or (MXFP8) per 128 rows and K block
int64_t packed_sf_bytes(int64_t rows, int K) {
    return (rows + 127) / 128 * ((K / 128 + 3) / 4) * kSfTileBytes;
}
int64_t mx_sf_bytes(int64_t rows, int K) { return (rows + 127) / 128 * (K / 128) * kSfTileBytes; }

struct ForwardLayout {
    size_t ids, wts, eoff, poff, sorted, pos, tile_e, tile_r, ntiles, counts, a1, a1s, a2, a2s, a1sf, a2sf, y, dh,
        dcnt, total;
    int64_t rows, tiles;
    int64_t dcnt_n;   // decode-path group counters (0: the step cannot take the decode path)
};

// Steps of up to this many tokens take the decode path by default (MOE_DECODE_AUTO).  Measured on
// GB300 with the DeepSeek-V3-shaped layer (E=256, top-8, tile-packed weights, CUDA-graph replay),
// ms per step, decode path against the tile GEMMs: two tokens 0.128 / 0.142, three 0.195 / 0.201,
// four 0.242 / 0.249, five 0.280 / 0.269, six 0.333 / 0.318.
constexpr int kDecodeAutoMaxTokens = 4;
// the w13 GEMM visits an expert's few tiles column by column when one expert's w13 has at least
// this many bytes (see GemmArgs::padded_offsets)
constexpr int64_t kColumnOrderMinExpertBytes = int64_t(16) << 20;
// the block-scaled w2 GEMM runs on the CTA-pair kernel (gemm.cu) when the routed rows average at
// least this many per expert: there the tensor pipe bounds it, and an expert's tiles pair up with
// little padding (with fewer rows most experts have one or two tiles).  Measured on GB300 with the
// Qwen3-30B-A3B-shaped skewed batch (16384 tokens, 1024 rows per expert), ms per layer: packed
// UE8M0 0.735 with the pair kernel for w2 against 0.754 without it; with it for w13 too, 0.779 (the
// w13 pair kernel, whose epilogue spills, ran 0.376 ms against 0.356 on the one-CTA kernel).
constexpr int64_t kPairMinRowsPerExpert = 512;

// Whether a step can take the decode-path GEMMs (decode.cu): at most 8 tokens (so at most 8
// rows per expert), a sort small enough for a CTA's shared memory (the decode kernel sorts the
// pairs itself), an expert's w13 under 2^31 bytes (the kernels' 32-bit row offsets) and tile
// records that fit a CTA's shared memory.
bool decode_possible(int T, int H, int I, int topk) {
    const int64_t P = static_cast<int64_t>(T) * topk;
    return T > 0 && decode_cols(T) > 0 && P <= kSmallPairs && static_cast<int64_t>(2) * I * H < (int64_t(1) << 31) &&
           static_cast<size_t>(P) <= decode_max_tiles();   // at most one tile per routed pair
}
bool use_decode(int T, int H, int I, int topk, int mode) {
    if (!decode_possible(T, H, I, topk) || mode == MOE_DECODE_OFF) return false;
    return mode == MOE_DECODE_ON || T <= kDecodeAutoMaxTokens;
}
// Copies of the token rows the decode prologue writes (into the a1 rows / a1s scales of the
// layout): 4, as the rows allow
int decode_x_copies(int T, int64_t rows) {
    const int64_t c = (rows - kDecodeCols) / T;
    return static_cast<int>(c < 1 ? 1 : (c > 4 ? 4 : c));
}
// Experts per lane with which the decode kernel routes the step in every CTA (the routing
// kernel's register-resident selection, up to 8 per lane: E <= 256), 0 when the step takes the
// routing kernel's ids instead
int decode_route_v(int E, int n_group) {
    const int v = reg_experts_per_lane(E, n_group);
    return v >= 1 && v <= 8 ? v : 0;
}

ForwardLayout forward_layout(int T, int H, int I, int E, int topk) {
    ForwardLayout L;
    const int64_t P = static_cast<int64_t>(T) * topk;
    // whole tiles, and a multiple of 4 so that each K block's row scales start 16-byte aligned
    L.rows = (max_rows(P, E, MOE_BLOCK_M) + MOE_BLOCK_M - 1) / MOE_BLOCK_M * MOE_BLOCK_M;
    L.tiles = L.rows / MOE_BLOCK_M;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align_up(bytes, 256);
        return o;
    };
    L.ids = take(P * 4);
    L.wts = take(P * 4);
    L.eoff = take((E + 1) * 4);
    L.poff = take((E + 1) * 4);
    L.sorted = take(L.rows * 4);
    L.pos = take(P * 4);
    L.tile_e = take(L.tiles * 4);
    L.tile_r = take(L.tiles * 4);
    L.ntiles = take(4);
    L.counts = take(permute_chunks(P) * E * 4);
    L.a1 = take(L.rows * H);
    L.a1s = take(static_cast<size_t>(H / 128) * L.rows * 4);
    L.a2 = take(L.rows * I);
    L.a2s = take(static_cast<size_t>(I / 128) * L.rows * 4);
    // packed scale tiles of A1 and A2 (MOE_SCALE_UE8M0_PACKED, MOE_SCALE_MXFP8: the larger)
    L.a1sf = take(mx_sf_bytes(L.rows, H));
    L.a2sf = take(mx_sf_bytes(L.rows, I));
    L.y = take(static_cast<size_t>(P) * H * 2);
    // decode path: h = silu(gate) * up by pair [P, I] fp32 and the counters (the decode path's
    // activations are copies of the token rows in a1 / a1s: decode_x_copies)
    L.dcnt_n = decode_possible(T, H, I, topk) ? decode_counters(static_cast<int>(L.tiles), I) : 0;
    L.dh = take(L.dcnt_n ? static_cast<size_t>(P) * I * 4 : 0);
    L.dcnt = take(static_cast<size_t>(L.dcnt_n) * 4);
    L.total = off;
    return L;
}

struct MaskedLayout {
    size_t row_map, pos, ones, tile_e, tile_r, ntiles, a1, a1s, a2, a2s, a1sf, a2sf, total;
    int64_t Mp, rows, tiles;
};

MaskedLayout masked_layout(int E, int M, int H, int I) {
    MaskedLayout L;
    L.Mp = (static_cast<int64_t>(M) + MOE_BLOCK_M - 1) / MOE_BLOCK_M * MOE_BLOCK_M;
    L.rows = static_cast<int64_t>(E) * L.Mp;
    L.tiles = L.rows / MOE_BLOCK_M;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align_up(bytes, 256);
        return o;
    };
    const size_t EM = static_cast<size_t>(E) * M;
    L.row_map = take(L.rows * 4);
    L.pos = take(EM * 4);
    L.ones = take(EM * 4);
    L.tile_e = take(L.tiles * 4);
    L.tile_r = take(L.tiles * 4);
    L.ntiles = take(4);
    L.a1 = take(L.rows * H);
    L.a1s = take(static_cast<size_t>(H / 128) * L.rows * 4);
    L.a2 = take(L.rows * I);
    L.a2s = take(static_cast<size_t>(I / 128) * L.rows * 4);
    L.a1sf = take(mx_sf_bytes(L.rows, H));
    L.a2sf = take(mx_sf_bytes(L.rows, I));
    L.total = off;
    return L;
}

inline bool known_scale_fmt(int f) {
    return f == MOE_SCALE_F32 || f == MOE_SCALE_UE8M0 || f == MOE_SCALE_UE8M0_PACKED || f == MOE_SCALE_MXFP8;
}
// formats whose GEMMs run on the block-scaled MMA: 1 = packed UE8M0, 2 = MXFP8, 0 = neither
inline int sf_mode(int f) { return f == MOE_SCALE_UE8M0_PACKED ? 1 : f == MOE_SCALE_MXFP8 ? 2 : 0; }

// Whether a step's block-scaled w2 GEMM qualifies for the CTA-pair kernel (besides the device's
// clusters): a packed scale format, a hidden size of whole 256-column items and at least
// kPairMinRowsPerExpert routed rows per expert on average (more than 32 tokens follows).
bool pair_shape(int T, int H, int E, int topk, bool packed) {
    return packed && H % 256 == 0 && static_cast<int64_t>(T) * topk >= kPairMinRowsPerExpert * E;
}

}  // namespace

namespace mfp8 {
// Device set-up and the status word's device address, for entry points in other files.
int device_status_word(uint32_t** status) {
    DeviceState* s = nullptr;
    const int rc = device_state(&s);
    if (rc == MOE_OK) *status = s->status;
    return rc;
}
}  // namespace mfp8

extern "C" {

int moe_device_supported(void) {
    DeviceState* s = nullptr;
    return device_state(&s) == MOE_OK ? 1 : 0;
}

const char* moe_error_string(int code) {
    switch (code) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
        default: return "MOE_ERR_UNKNOWN";
    }
}

int moe_get_device_status(uint32_t* status, int clear) {
    if (!status) return MOE_ERR_INVALID_ARG;
    DeviceState* s = nullptr;
    int rc = device_state(&s);
    if (rc != MOE_OK) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(status, s->status, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (clear && cudaMemset(s->status, 0, sizeof(uint32_t)) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_route_topk(const float* logits, int T, int E, int topk, int renormalize, const moe_routing_params* rp,
                   int32_t* topk_ids, float* topk_weights, void* stream) {
    int rc = check_routing(T, E, topk, rp);
    if (rc != MOE_OK) return rc;
    if (T > 0 && (!logits || !topk_ids || !topk_weights)) return MOE_ERR_INVALID_ARG;
    DeviceState* s = nullptr;
    if ((rc = device_state(&s)) != MOE_OK) return rc;
    const int scoring = rp ? rp->scoring : MOE_SCORING_SOFTMAX;
    const int n_group = rp ? rp->n_group : 1;
    const int topk_group = rp ? rp->topk_group : 1;
    const float scaling = rp ? rp->routed_scaling : 1.0f;
    const float* bias = rp ? rp->bias : nullptr;
    return cuda_rc(launch_route_topk(logits, T, E, topk, renormalize, scoring, n_group, topk_group, scaling, bias,
                                     topk_ids, topk_weights, static_cast<cudaStream_t>(stream)));
}

int64_t moe_max_padded_rows(int T, int topk, int E, int block_m) {
    if (T < 0 || topk < 1 || E < 1 || block_m < 1) return -1;
    return max_rows(static_cast<int64_t>(T) * topk, E, block_m);
}

int64_t moe_max_tiles(int T, int topk, int E, int block_m) {
    const int64_t r = moe_max_padded_rows(T, topk, E, block_m);
    return r < 0 ? -1 : r / block_m;
}

size_t moe_align_permute_workspace_size(int T, int topk, int E) {
    if (T < 0 || topk < 1 || E < 1) return 0;
    return align_up(static_cast<size_t>(permute_chunks(static_cast<int64_t>(T) * topk)) * E * 4, 256);
}

int moe_align_permute(const int32_t* topk_ids, int T, int topk, int E, int block_m, int32_t* expert_offsets,
                      int32_t* padded_offsets, int32_t* sorted_pair_ids, int32_t* pos, int32_t* tile_expert,
                      int32_t* tile_row0, int32_t* num_tiles, void* workspace, size_t workspace_bytes,
                      void* stream) {
    if (T < 0 || topk < 1 || E < 1 || block_m < 1) return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS || block_m > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t P = static_cast<int64_t>(T) * topk;
    if (max_rows(P, E, block_m) >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!expert_offsets || !padded_offsets || !num_tiles) return MOE_ERR_INVALID_ARG;
    if (P > 0 && (!topk_ids || !sorted_pair_ids || !pos || !tile_expert || !tile_row0)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < moe_align_permute_workspace_size(T, topk, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (P > 0 && !workspace) return MOE_ERR_INVALID_ARG;
    DeviceState* s = nullptr;
    int rc = device_state(&s);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_align_permute(topk_ids, P, E, block_m, expert_offsets, padded_offsets, sorted_pair_ids, pos,
                                        tile_expert, tile_row0, num_tiles, static_cast<int32_t*>(workspace),
                                        s->status, static_cast<cudaStream_t>(stream)));
}

int fp8_group_quant(const uint16_t* x, int rows, int cols, int ld, uint8_t* q, float* s, void* stream) {
    return fp8_group_quant_ex(x, rows, cols, ld, q, s, MOE_SCALE_F32, stream);
}

int fp8_group_quant_ex(const uint16_t* x, int rows, int cols, int ld, uint8_t* q, float* s, int scale_fmt,
                       void* stream) {
    if (rows < 0 || cols < 0 || ld < cols) return MOE_ERR_INVALID_ARG;
    if (!known_scale_fmt(scale_fmt)) return MOE_ERR_INVALID_ARG;
    if (cols % 128 != 0 || ld % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0 || cols == 0) return MOE_OK;
    if (!x || !q || !s) return MOE_ERR_INVALID_ARG;
    const bool packed = scale_fmt == MOE_SCALE_UE8M0_PACKED;
    const bool mx = scale_fmt == MOE_SCALE_MXFP8;
    if (!aligned(x, 16) || !aligned(q, 8) || (!packed && !mx && !aligned(s, 4))) return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    if (mx)
        return cuda_rc(launch_group_quant(x, rows, cols, ld, q, cols, nullptr, 0, 0, nullptr, 1, MOE_SCALE_MXFP8,
                                          static_cast<cudaStream_t>(stream), nullptr, reinterpret_cast<uint8_t*>(s)));
    if (packed)
        return cuda_rc(launch_group_quant(x, rows, cols, ld, q, cols, nullptr, 0, 0, nullptr, 1, MOE_SCALE_UE8M0,
                                          static_cast<cudaStream_t>(stream), reinterpret_cast<uint8_t*>(s)));
    return cuda_rc(launch_group_quant(x, rows, cols, ld, q, cols, s, cols / 128, 1, nullptr, 1, scale_fmt,
                                      static_cast<cudaStream_t>(stream)));
}

int fp8_block_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, float* s, void* stream) {
    return fp8_block_quant_weight_ex(w, E, N, K, q, s, MOE_SCALE_F32, stream);
}

int fp8_block_quant_weight_ex(const uint16_t* w, int E, int N, int K, uint8_t* q, float* s, int scale_fmt,
                              void* stream) {
    if (E < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (scale_fmt != MOE_SCALE_F32 && scale_fmt != MOE_SCALE_UE8M0) return MOE_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0 || K > (1 << 30)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (E == 0 || N == 0 || K == 0) return MOE_OK;
    if (E > 65535 || N / 128 > 65535) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!w || !q || !s || !aligned(w, 16) || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_block_quant_weight(w, E, N, K, q, s, scale_fmt, static_cast<cudaStream_t>(stream)));
}

int moe_fp8_block_pack_weights(const uint8_t* w, int E, int N, int K, uint8_t* packed, void* stream) {
    if (E < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(E) * N * (K / 128) >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (E == 0 || N == 0 || K == 0) return MOE_OK;
    if (!w || !packed || !aligned(w, 16) || !aligned(packed, 16)) return MOE_ERR_INVALID_ARG;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(w), b0 = reinterpret_cast<uintptr_t>(packed);
    const uintptr_t n = static_cast<uintptr_t>(E) * N * K;
    if (a0 < b0 + n && b0 < a0 + n) return MOE_ERR_INVALID_ARG;   // the conversion is not in place
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_pack_weights(w, E, N, K, packed, static_cast<cudaStream_t>(stream)));
}

size_t moe_packed_scale_bytes(int64_t rows, int K) {
    if (rows < 0 || K < 0 || K % 128 != 0) return 0;
    return static_cast<size_t>(packed_sf_bytes(rows, K));
}

int moe_fp8_block_pack_scales(const float* s, int E, int N, int K, uint8_t* out, void* stream) {
    if (E < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (E == 0 || N == 0 || K == 0) return MOE_OK;
    if (!s || !out || !aligned(s, 4) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_pack_scales(s, E, N, K, out, st->status, static_cast<cudaStream_t>(stream)));
}

size_t moe_mxfp8_packed_scale_bytes(int64_t rows, int K) {
    if (rows < 0 || K < 0 || K % 128 != 0) return 0;
    return static_cast<size_t>(mx_sf_bytes(rows, K));
}

int moe_mxfp8_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, uint8_t* s, void* stream) {
    if (E < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (K % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (E == 0 || N == 0 || K == 0) return MOE_OK;
    if (!w || !q || !s || !aligned(w, 16) || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    const int64_t rows = static_cast<int64_t>(E) * N;
    return cuda_rc(launch_group_quant(w, rows, K, K, q, K, nullptr, 0, 0, nullptr, 1, MOE_SCALE_MXFP8,
                                      static_cast<cudaStream_t>(stream), nullptr, s));
}

int moe_mxfp8_pack_scales(const uint8_t* s, int64_t rows, int K, uint8_t* out, void* stream) {
    if (rows < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (K % 128 != 0 || rows % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0 || K == 0) return MOE_OK;
    if (!s || !out || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_pack_scale_bytes(s, rows, K / 32, out, static_cast<cudaStream_t>(stream)));
}

int moe_nvfp4_quant_weight(const uint16_t* w, int E, int N, int K, uint8_t* q, uint8_t* block_scale,
                           float* global_scale, void* stream) {
    if (E < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (K % 16 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (E == 0 || N == 0 || K == 0) return MOE_OK;
    if (static_cast<int64_t>(E) * N * (K / 16) >= (int64_t(1) << 39)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!w || !q || !block_scale || !global_scale || !aligned(w, 16) || !aligned(q, 8) || !aligned(global_scale, 4))
        return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_nvfp4_quant_weight(w, E, N, K, q, block_scale, global_scale,
                                             static_cast<cudaStream_t>(stream)));
}

int moe_selftest_bounded_wait(int expire, void* stream) {
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_bounded_wait_check(expire, st->status, static_cast<cudaStream_t>(stream)));
}

size_t moe_nvfp4_packed_bytes(int E, int N, int K) {
    if (E < 0 || N < 0 || K < 0 || N % 16 != 0 || K % 128 != 0) return 0;
    return nvfp4_packed_bytes(E, N, K);
}

int moe_nvfp4_pack_weights(const uint8_t* q, const uint8_t* block_scale, int E, int N, int K, uint8_t* packed,
                           void* stream) {
    if (E < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (N % 16 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (E == 0 || N == 0 || K == 0) return MOE_OK;
    if (!q || !block_scale || !packed || !aligned(q, 16) || !aligned(block_scale, 8) || !aligned(packed, 16))
        return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_nvfp4_pack(q, block_scale, E, N, K, packed, static_cast<cudaStream_t>(stream)));
}

int fp8_block_grouped_gemm(const uint8_t* A, const float* a_scale, int64_t a_scale_row_stride,
                           int64_t a_scale_kb_stride, int64_t a_rows, const uint8_t* B, const float* b_scale, int N,
                           int K, int E, const int32_t* tile_expert, const int32_t* tile_row0,
                           const int32_t* num_tiles, int64_t max_tiles, const moe_gemm_epilogue* ep, void* stream) {
    if (!ep || N < 0 || K < 0 || E < 1 || max_tiles < 0 || a_rows < 0) return MOE_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0 || N == 0 || K == 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(E) * N >= (int64_t(1) << 31) || a_rows >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (ep->kind == MOE_EPI_SILU_MUL_QUANT && N % 256 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (max_tiles == 0) return MOE_OK;
    if (!A || !a_scale || !B || !b_scale || !tile_expert || !tile_row0 || !num_tiles) return MOE_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16)) return MOE_ERR_INVALID_ARG;
    if (ep->b_layout != MOE_WEIGHTS_NK && ep->b_layout != MOE_WEIGHTS_TILED) return MOE_ERR_INVALID_ARG;
    if (!known_scale_fmt(ep->scale_fmt)) return MOE_ERR_INVALID_ARG;
    const bool packed = sf_mode(ep->scale_fmt) != 0;
    if (packed) {
        if (ep->kind != MOE_EPI_STORE_F32 && ep->kind != MOE_EPI_SILU_MUL_QUANT &&
            ep->kind != MOE_EPI_WEIGHTED_PAIRS_BF16)
            return MOE_ERR_INVALID_ARG;
        if (!aligned(a_scale, 16) || !aligned(b_scale, 16)) return MOE_ERR_INVALID_ARG;
    }
    if (ep->b_layout == MOE_WEIGHTS_TILED && static_cast<int64_t>(E) * N * (K / 128) >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    switch (ep->kind) {
        case MOE_EPI_STORE_F32:
            if (!ep->out_f32 || !aligned(ep->out_f32, 16)) return MOE_ERR_INVALID_ARG;
            break;
        case MOE_EPI_SILU_MUL_QUANT:
            if (!ep->out_q || !ep->out_scale || !aligned(ep->out_q, 16)) return MOE_ERR_INVALID_ARG;
            break;
        case MOE_EPI_WEIGHTED_SCATTER:
        case MOE_EPI_WEIGHTED_ROWS:
            if (!ep->out_f32 || !aligned(ep->out_f32, 16) || !ep->sorted_pair_ids || !ep->topk_weights ||
                ep->topk < 1 || ep->num_pairs < 0)
                return MOE_ERR_INVALID_ARG;
            break;
        case MOE_EPI_WEIGHTED_PAIRS_BF16:
            if (!ep->out_bf16 || !aligned(ep->out_bf16, 16) || !ep->sorted_pair_ids || !ep->topk_weights ||
                ep->topk < 1 || ep->num_pairs < 0)
                return MOE_ERR_INVALID_ARG;
            break;
        default:
            return MOE_ERR_INVALID_ARG;
    }
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    GemmArgs g{};
    g.a_box_rows = 128;
    g.A = A;
    g.a_scale = a_scale;
    g.as_row_stride = a_scale_row_stride;
    g.as_kb_stride = a_scale_kb_stride;
    g.a_rows = a_rows;
    g.B = B;
    g.b_scale = b_scale;
    g.N = N;
    g.K = K;
    g.E = E;
    g.tile_expert = tile_expert;
    g.tile_row0 = tile_row0;
    g.num_tiles = num_tiles;
    g.max_tiles = max_tiles;
    g.epi = ep->kind;
    g.out_f32 = ep->out_f32;
    g.out_q = ep->out_q;
    g.out_scale = ep->out_scale;
    g.os_row_stride = ep->out_scale_row_stride;
    g.os_kb_stride = ep->out_scale_kb_stride;
    g.sorted_pair_ids = ep->sorted_pair_ids;
    g.topk_weights = ep->topk_weights;
    g.topk = ep->topk;
    g.num_pairs = ep->num_pairs;
    g.out_bf16 = ep->out_bf16;
    g.b_tiled = ep->b_layout == MOE_WEIGHTS_TILED;
    g.scale_fmt = packed ? MOE_SCALE_UE8M0 : ep->scale_fmt;
    if (packed) {
        g.sf_packed = sf_mode(ep->scale_fmt);
        g.a_sf = reinterpret_cast<const uint8_t*>(a_scale);
        g.b_sf = reinterpret_cast<const uint8_t*>(b_scale);
        g.out_sf = reinterpret_cast<uint8_t*>(ep->out_scale);
    }
    g.status = st->status;
    return cuda_rc(launch_grouped_gemm(g, st->num_sms, static_cast<cudaStream_t>(stream)));
}

int moe_unpermute_sum(const float* y, int64_t y_rows, const int32_t* pos, int T, int topk, int H, uint16_t* out,
                      void* stream) {
    if (T < 0 || topk < 1 || H < 0 || y_rows < 0) return MOE_ERR_INVALID_ARG;
    if (H % 4 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0 || H == 0) return MOE_OK;
    if (!y || !pos || !out || !aligned(y, 16) || !aligned(out, 8)) return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_unpermute_sum(y, y_rows, pos, T, topk, H, out, st->status,
                                        static_cast<cudaStream_t>(stream)));
}

int moe_combine_pairs(const uint16_t* y, const int32_t* pos, int T, int topk, int H, uint16_t* out, void* stream) {
    if (T < 0 || topk < 1 || H < 0) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0 || H == 0) return MOE_OK;
    if (!y || !pos || !out || !aligned(y, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return cuda_rc(launch_combine_pairs(y, pos, T, topk, H, out, static_cast<cudaStream_t>(stream)));
}

int moe_fp8_block_forward_kernel_count_ex(int T, int H, int I, int E, int topk, const moe_routing_params* rp,
                                          const moe_forward_options* opts) {
    if (T < 0 || H <= 0 || I <= 0 || E < 1 || topk < 1) return -1;
    if (T == 0) return 0;
    const int layout = opts ? opts->weight_layout : MOE_WEIGHTS_NK;
    const int fmt = opts ? opts->scale_fmt : MOE_SCALE_F32;
    const int mode = opts ? opts->decode_path : MOE_DECODE_AUTO;
    // the decode path: its prologue, the decode kernel and the weighted sum, after the routing
    // kernel when the decode kernel cannot route in every CTA
    const int decode_step = decode_route_v(E, rp ? rp->n_group : 1) > 0 ? 3 : 4;
    if (layout == MOE_WEIGHTS_NVFP4) return (T + kDecodeCols - 1) / kDecodeCols * decode_step;
    if (sf_mode(fmt) == 0 && use_decode(T, H, I, topk, mode)) return decode_step;
    const int64_t P = static_cast<int64_t>(T) * topk;
    return 1 + (P <= kSmallPairs ? 1 : 4) + 2 + 1;
}

int moe_fp8_block_forward_kernel_count(int T, int H, int I, int E, int topk) {
    return moe_fp8_block_forward_kernel_count_ex(T, H, I, E, topk, nullptr, nullptr);
}

int moe_fp8_block_pair_path(int T, int H, int E, int topk, int scale_fmt) {
    if (T < 0 || H < 0 || E < 1 || topk < 1 || !known_scale_fmt(scale_fmt)) return MOE_ERR_INVALID_ARG;
    if (!pair_shape(T, H, E, topk, sf_mode(scale_fmt) != 0)) return 0;
    DeviceState* st = nullptr;
    const int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    return gemm_pair_clusters();
}

int moe_fp8_block_decode_path(int T, int H, int I, int topk, int mode) {
    if (T < 0 || H < 0 || I < 0 || topk < 1) return -1;
    if (mode != MOE_DECODE_AUTO && mode != MOE_DECODE_OFF && mode != MOE_DECODE_ON) return -1;
    return use_decode(T, H, I, topk, mode) ? 1 : 0;
}

size_t moe_fp8_block_workspace_size(int T, int H, int I, int E, int topk) {
    if (T < 0 || H < 0 || I < 0 || E < 1 || topk < 1) return 0;
    return forward_layout(T, H, I, E, topk).total;
}

int moe_fp8_block_forward(const uint16_t* hidden, const float* router_logits, const uint8_t* w13,
                          const float* w13_scale, const uint8_t* w2, const float* w2_scale, int T, int H, int I, int E,
                          int topk, int renormalize, const moe_routing_params* rp, void* workspace,
                          size_t workspace_bytes, uint16_t* out, void* stream) {
    return moe_fp8_block_forward_ex(hidden, router_logits, w13, w13_scale, w2, w2_scale, T, H, I, E, topk,
                                    renormalize, rp, nullptr, workspace, workspace_bytes, out, stream, nullptr);
}

int moe_fp8_block_forward_packed(const uint16_t* hidden, const float* router_logits, const uint8_t* w13,
                                 const float* w13_scale, const uint8_t* w2, const float* w2_scale, int T, int H,
                                 int I, int E, int topk, int renormalize, const moe_routing_params* rp,
                                 void* workspace, size_t workspace_bytes, uint16_t* out, void* stream) {
    const moe_forward_options opts{MOE_WEIGHTS_TILED, MOE_SCALE_F32, MOE_DECODE_AUTO};
    return moe_fp8_block_forward_ex(hidden, router_logits, w13, w13_scale, w2, w2_scale, T, H, I, E, topk,
                                    renormalize, rp, &opts, workspace, workspace_bytes, out, stream, nullptr);
}

int moe_fp8_block_forward_ex(const uint16_t* hidden, const float* router_logits, const uint8_t* w13,
                             const float* w13_scale, const uint8_t* w2, const float* w2_scale, int T, int H, int I,
                             int E, int topk, int renormalize, const moe_routing_params* rp,
                             const moe_forward_options* opts, void* workspace, size_t workspace_bytes,
                             uint16_t* out, void* stream, void* const* events) {
    int rc = check_routing(T, E, topk, rp);
    if (rc != MOE_OK) return rc;
    const int weight_layout = opts ? opts->weight_layout : MOE_WEIGHTS_NK;
    const int scale_fmt = opts ? opts->scale_fmt : MOE_SCALE_F32;
    const int decode_mode = opts ? opts->decode_path : MOE_DECODE_AUTO;
    if (weight_layout != MOE_WEIGHTS_NK && weight_layout != MOE_WEIGHTS_TILED && weight_layout != MOE_WEIGHTS_NVFP4)
        return MOE_ERR_INVALID_ARG;
    if (!known_scale_fmt(scale_fmt)) return MOE_ERR_INVALID_ARG;
    if (decode_mode != MOE_DECODE_AUTO && decode_mode != MOE_DECODE_OFF && decode_mode != MOE_DECODE_ON)
        return MOE_ERR_INVALID_ARG;
    const bool fp4 = weight_layout == MOE_WEIGHTS_NVFP4;
    // packed UE8M0 scales: both GEMMs on the block-scaled MMA (tile kernels only)
    const int sfm = sf_mode(scale_fmt);
    const bool packed = sfm != 0;
    if (packed && (fp4 || decode_mode == MOE_DECODE_ON)) return MOE_ERR_INVALID_ARG;
    if (packed && (!aligned(w13_scale, 16) || !aligned(w2_scale, 16))) return MOE_ERR_INVALID_ARG;
    if (fp4 && T > kDecodeCols) {
        // NVFP4 weights run on the decode-path kernel only: steps of more tokens go through it
        // kDecodeCols tokens at a time (every token's rows are independent)
        if (H <= 0 || I <= 0 || !hidden || !router_logits || !out) return MOE_ERR_INVALID_ARG;
        if (H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
        // every check a pass of kDecodeCols tokens makes, before anything is enqueued (the last,
        // shorter pass needs no more than a full one)
        if (decode_mode == MOE_DECODE_OFF) return MOE_ERR_INVALID_ARG;
        if (static_cast<int64_t>(E) * 2 * I >= (int64_t(1) << 31) || static_cast<int64_t>(E) * H >= (int64_t(1) << 31))
            return MOE_ERR_UNSUPPORTED_SHAPE;
        if (!decode_possible(kDecodeCols, H, I, topk)) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (!w13 || !w13_scale || !w2 || !w2_scale || !workspace) return MOE_ERR_INVALID_ARG;
        if (!aligned(hidden, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) ||
            !aligned(workspace, 256))
            return MOE_ERR_INVALID_ARG;
        if (workspace_bytes < forward_layout(kDecodeCols, H, I, E, topk).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
        // stage events: the chunks' kernels interleave, so the whole step is recorded as the w13
        // stage (events 0-3 before the first chunk, 4-6 after the last)
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        for (int i = 0; events && i < 4; ++i)
            if (cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) != cudaSuccess) return MOE_ERR_CUDA;
        for (int t0 = 0; t0 < T; t0 += kDecodeCols) {
            const int n = T - t0 < kDecodeCols ? T - t0 : kDecodeCols;
            rc = moe_fp8_block_forward_ex(hidden + static_cast<int64_t>(t0) * H,
                                          router_logits + static_cast<int64_t>(t0) * E, w13, w13_scale, w2,
                                          w2_scale, n, H, I, E, topk, renormalize, rp, opts, workspace,
                                          workspace_bytes, out + static_cast<int64_t>(t0) * H, stream, nullptr);
            if (rc != MOE_OK) return rc;
        }
        for (int i = 4; events && i < MOE_FORWARD_NUM_EVENTS; ++i)
            if (cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (fp4 && decode_mode == MOE_DECODE_OFF) return MOE_ERR_INVALID_ARG;
    if (weight_layout == MOE_WEIGHTS_TILED &&
        static_cast<int64_t>(E) * 2 * I * (H / 128) >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(E) * 2 * I >= (int64_t(1) << 31) || static_cast<int64_t>(E) * H >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    const ForwardLayout L = forward_layout(T, H, I, E, topk);
    if (L.rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!hidden || !router_logits || !w13 || !w13_scale || !w2 || !w2_scale || !out || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(hidden, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) ||
        !aligned(workspace, 256))
        return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st)) != MOE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* ids = reinterpret_cast<int32_t*>(ws + L.ids);
    float* wts = reinterpret_cast<float*>(ws + L.wts);
    int32_t* sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
    int32_t* pos = reinterpret_cast<int32_t*>(ws + L.pos);
    int32_t* tile_e = reinterpret_cast<int32_t*>(ws + L.tile_e);
    int32_t* tile_r = reinterpret_cast<int32_t*>(ws + L.tile_r);
    int32_t* ntiles = reinterpret_cast<int32_t*>(ws + L.ntiles);
    uint8_t* a1 = ws + L.a1;
    float* a1s = reinterpret_cast<float*>(ws + L.a1s);
    uint8_t* a2 = ws + L.a2;
    float* a2s = reinterpret_cast<float*>(ws + L.a2s);
    uint16_t* ypairs = reinterpret_cast<uint16_t*>(ws + L.y);
    const int64_t P = static_cast<int64_t>(T) * topk;
    // an expert holds at most T rows: with T <= 32 only the first 32 rows of a tile can be
    // real, so the GEMMs load 32-row activation boxes
    const int a_box_rows = T <= 32 ? 32 : 128;
    const bool pair = pair_shape(T, H, E, topk, packed) && a_box_rows == 128 && gemm_pair_clusters() > 0;

    auto mark = [&](int i) {
        return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
    };
    const int scoring = rp ? rp->scoring : MOE_SCORING_SOFTMAX;
    const int n_group = rp ? rp->n_group : 1;
    const int topk_group = rp ? rp->topk_group : 1;
    const float routed_scaling = rp ? rp->routed_scaling : 1.0f;
    const float* bias = rp ? rp->bias : nullptr;
    if (fp4 && !decode_possible(T, H, I, topk)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const bool decode = fp4 || (!packed && use_decode(T, H, I, topk, decode_mode));
    cudaError_t e = mark(0);
    if (decode) {
        // Up to 8 tokens: the decode prologue (counters zeroed, tokens quantised token-major),
        // one kernel that routes and sorts the step in every CTA and runs both GEMMs with their
        // epilogues (decode.cu), and the weighted k-way sum; the routing kernel runs first only
        // for shapes the in-kernel selection does not take.  Stages: routing (that kernel or
        // empty), sort (empty), quantisation (the prologue), w13 (the decode kernel), w2 (empty),
        // the unpermute-sum.
        const int route_v = decode_route_v(E, n_group);
        if (e == cudaSuccess && route_v == 0)
            e = launch_route_topk(router_logits, T, E, topk, renormalize, scoring, n_group, topk_group,
                                  routed_scaling, bias, ids, wts, s);
        if (e == cudaSuccess) e = mark(1);
        if (e == cudaSuccess) e = mark(2);
        const int x_copies = decode_x_copies(T, L.rows);
        if (e == cudaSuccess)
            e = launch_decode_prologue(hidden, T, H, x_copies, a1, a1s, reinterpret_cast<int32_t*>(ws + L.dcnt),
                                       static_cast<int>(L.dcnt_n), scale_fmt, s);
        if (e == cudaSuccess) e = mark(3);
        DecodeMlpArgs d{};
        d.w13 = w13;
        d.w13_scale = w13_scale;
        d.w2 = w2;
        d.w2_scale = w2_scale;
        d.w_tiled = weight_layout == MOE_WEIGHTS_TILED;
        d.w_fp4 = fp4;
        d.H = H;
        d.I = I;
        d.E = E;
        d.T = T;
        d.topk = topk;
        d.route_v = route_v;
        d.logits = router_logits;
        d.bias = bias;
        d.renormalize = renormalize;
        d.scoring = scoring;
        d.n_group = n_group;
        d.topk_group = topk_group;
        d.vec_loads = route_v >= 4 && E == 32 * route_v && aligned(router_logits, 16);
        d.routed_scaling = routed_scaling;
        d.ids = ids;
        d.wts = wts;
        d.pos = pos;
        d.a1 = a1;
        d.a1s = a1s;
        d.x_copies = x_copies;
        d.a2 = a2;
        d.a2s = a2s;
        d.rows = L.rows;
        d.max_tiles = static_cast<int>(L.tiles);
        d.cols = decode_cols(T);
        d.h = reinterpret_cast<float*>(ws + L.dh);
        d.counters = reinterpret_cast<int32_t*>(ws + L.dcnt);
        d.scale_fmt = scale_fmt;
        d.y = ypairs;
        d.status = st->status;
        if (e == cudaSuccess) e = launch_decode_mlp(d, st->num_sms, s);
        if (e == cudaSuccess) e = mark(4);
        if (e == cudaSuccess) e = mark(5);
        if (e == cudaSuccess) e = launch_combine_pairs(ypairs, pos, T, topk, H, out, s);
        if (e == cudaSuccess) e = mark(6);
        return cuda_rc(e);
    }
    if (e == cudaSuccess)
        e = launch_route_topk(router_logits, T, E, topk, renormalize, scoring, n_group, topk_group, routed_scaling,
                              bias, ids, wts, s);
    if (e == cudaSuccess) e = mark(1);
    // a small batch is sorted and quantised by one block in one launch (the quantisation stage
    // is then empty); larger ones by the three sort kernels and the grid-wide quantiser
    const bool small = P <= kSmallPairs;
    uint8_t* a1sf = packed ? ws + L.a1sf : nullptr;
    uint8_t* a2sf = ws + L.a2sf;
    if (e == cudaSuccess && small)
        e = launch_sort_quant_small(ids, static_cast<int>(P), E, MOE_BLOCK_M, reinterpret_cast<int32_t*>(ws + L.eoff),
                                    reinterpret_cast<int32_t*>(ws + L.poff), sorted, pos, tile_e, tile_r, ntiles,
                                    st->status, hidden, T, H, topk, a1, H, packed ? nullptr : a1s, 1, L.rows,
                                    scale_fmt, s, a1sf);
    if (e == cudaSuccess && !small)
        e = launch_align_permute(ids, P, E, MOE_BLOCK_M, reinterpret_cast<int32_t*>(ws + L.eoff),
                                 reinterpret_cast<int32_t*>(ws + L.poff), sorted, pos, tile_e, tile_r, ntiles,
                                 reinterpret_cast<int32_t*>(ws + L.counts), st->status, s);
    // each token quantised once, its codes written to the sorted rows of its pairs (one
    // dense tile load per K block in the GEMM); the scales are stored transposed
    // ([H/128][rows]) for the GEMM's per-row reads
    if (e == cudaSuccess) e = mark(2);
    if (e == cudaSuccess && !small)
        e = launch_group_quant(hidden, T, H, H, a1, H, packed ? nullptr : a1s, 1, L.rows, pos, topk, scale_fmt, s,
                               a1sf);
    if (e == cudaSuccess) e = mark(3);
    if (e == cudaSuccess) {
        GemmArgs g{};
        g.a_box_rows = a_box_rows;
        g.A = a1;
        g.a_scale = a1s;
        g.as_row_stride = 1;
        g.as_kb_stride = L.rows;
        g.a_rows = L.rows;
        g.B = w13;
        g.b_tiled = weight_layout == MOE_WEIGHTS_TILED;
        g.b_scale = w13_scale;
        g.N = 2 * I;
        g.K = H;
        g.E = E;
        g.tile_expert = tile_e;
        g.tile_row0 = tile_r;
        g.num_tiles = ntiles;
        g.max_tiles = L.tiles;
        // column-by-column order for experts of a few tiles, where one expert's w13 is too large
        // to stay in L2 while a tile sweeps its columns (Mixtral-like 117 MB, DeepSeek-V3-like
        // 29 MB); experts of a few MB gain nothing from it and lost ~2% in measurement
        if (static_cast<int64_t>(2) * I * H >= kColumnOrderMinExpertBytes)
            g.padded_offsets = reinterpret_cast<const int32_t*>(ws + L.poff);
        g.epi = MOE_EPI_SILU_MUL_QUANT;
        g.scale_fmt = scale_fmt;
        g.sorted_pair_ids = sorted;
        g.row_offsets = reinterpret_cast<const int32_t*>(ws + L.eoff);
        g.row_padded = reinterpret_cast<const int32_t*>(ws + L.poff);
        g.out_q = a2;
        g.out_scale = a2s;
        g.os_row_stride = 1;
        g.os_kb_stride = L.rows;
        if (packed) {
            g.sf_packed = sfm;
            g.a_sf = a1sf;
            g.b_sf = reinterpret_cast<const uint8_t*>(w13_scale);
            g.out_sf = a2sf;
        }
        g.status = st->status;
        e = launch_grouped_gemm(g, st->num_sms, s);
        if (e == cudaSuccess) e = mark(4);
    }
    if (e == cudaSuccess) {
        GemmArgs g{};
        g.a_box_rows = a_box_rows;
        g.A = a2;
        g.a_scale = a2s;
        g.as_row_stride = 1;
        g.as_kb_stride = L.rows;
        g.a_rows = L.rows;
        g.B = w2;
        g.b_tiled = weight_layout == MOE_WEIGHTS_TILED;
        g.b_scale = w2_scale;
        g.N = H;
        g.K = I;
        g.E = E;
        g.tile_expert = tile_e;
        g.tile_row0 = tile_r;
        g.num_tiles = ntiles;
        g.max_tiles = L.tiles;
        g.epi = MOE_EPI_WEIGHTED_PAIRS_BF16;
        g.out_bf16 = ypairs;
        g.sorted_pair_ids = sorted;
        g.row_offsets = reinterpret_cast<const int32_t*>(ws + L.eoff);
        g.row_padded = reinterpret_cast<const int32_t*>(ws + L.poff);
        g.topk_weights = wts;
        g.topk = topk;
        g.num_pairs = P;
        if (packed) {
            g.sf_packed = sfm;
            g.a_sf = a2sf;
            g.b_sf = reinterpret_cast<const uint8_t*>(w2_scale);
            if (pair) g.pair_offsets = reinterpret_cast<const int32_t*>(ws + L.poff);
        }
        g.status = st->status;
        e = launch_grouped_gemm(g, st->num_sms, s);
        if (e == cudaSuccess) e = mark(5);
    }
    if (e == cudaSuccess) e = launch_combine_pairs(ypairs, pos, T, topk, H, out, s);
    if (e == cudaSuccess) e = mark(6);
    return cuda_rc(e);
}


size_t moe_fp8_block_masked_workspace_size(int E, int max_tokens, int H, int I) {
    if (E < 0 || max_tokens < 0 || H < 0 || I < 0) return 0;
    return masked_layout(E, max_tokens, H, I).total;
}

int moe_fp8_block_forward_masked(const uint16_t* hidden, const int32_t* counts, const uint8_t* w13,
                                 const float* w13_scale, const uint8_t* w2, const float* w2_scale, int E,
                                 int max_tokens, int H, int I, const moe_forward_options* opts, void* workspace,
                                 size_t workspace_bytes, uint16_t* out, void* stream) {
    if (E < 0 || max_tokens < 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    const int weight_layout = opts ? opts->weight_layout : MOE_WEIGHTS_NK;
    const int scale_fmt = opts ? opts->scale_fmt : MOE_SCALE_F32;
    if (weight_layout != MOE_WEIGHTS_NK && weight_layout != MOE_WEIGHTS_TILED) return MOE_ERR_INVALID_ARG;
    if (!known_scale_fmt(scale_fmt)) return MOE_ERR_INVALID_ARG;
    const int sfm = sf_mode(scale_fmt);
    const bool packed = sfm != 0;
    if (packed && (!aligned(w13_scale, 16) || !aligned(w2_scale, 16))) return MOE_ERR_INVALID_ARG;
    if (H % 128 != 0 || I % 128 != 0 || E > MOE_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (E == 0 || max_tokens == 0) return MOE_OK;
    const MaskedLayout L = masked_layout(E, max_tokens, H, I);
    if (L.rows >= (int64_t(1) << 31) || static_cast<int64_t>(E) * 2 * I * (H / 128) >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!hidden || !counts || !w13 || !w13_scale || !w2 || !w2_scale || !out || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(hidden, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) ||
        !aligned(workspace, 256))
        return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != MOE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* row_map = reinterpret_cast<int32_t*>(ws + L.row_map);
    int32_t* pos = reinterpret_cast<int32_t*>(ws + L.pos);
    float* ones = reinterpret_cast<float*>(ws + L.ones);
    int32_t* tile_e = reinterpret_cast<int32_t*>(ws + L.tile_e);
    int32_t* tile_r = reinterpret_cast<int32_t*>(ws + L.tile_r);
    int32_t* ntiles = reinterpret_cast<int32_t*>(ws + L.ntiles);
    uint8_t* a1 = ws + L.a1;
    float* a1s = reinterpret_cast<float*>(ws + L.a1s);
    uint8_t* a2 = ws + L.a2;
    float* a2s = reinterpret_cast<float*>(ws + L.a2s);
    const int64_t EM = static_cast<int64_t>(E) * max_tokens;

    uint8_t* a1sf = packed ? ws + L.a1sf : nullptr;
    uint8_t* a2sf = ws + L.a2sf;
    cudaError_t e = launch_masked_map(counts, E, max_tokens, static_cast<int>(L.Mp), row_map, pos, ones, tile_e,
                                      tile_r, ntiles, st->status, s);
    // valid rows quantised into their padded rows; scales transposed ([H/128][rows]), or packed
    if (e == cudaSuccess)
        e = launch_group_quant(hidden, EM, H, H, a1, H, packed ? nullptr : a1s, 1, L.rows, pos, 1, scale_fmt, s,
                               a1sf);
    if (e == cudaSuccess) {
        GemmArgs g{};
        g.a_box_rows = max_tokens <= 32 ? 32 : 128;   // no expert has more rows than max_tokens
        g.A = a1;
        g.a_scale = a1s;
        g.as_row_stride = 1;
        g.as_kb_stride = L.rows;
        g.a_rows = L.rows;
        g.B = w13;
        g.b_tiled = weight_layout == MOE_WEIGHTS_TILED;
        g.b_scale = w13_scale;
        g.N = 2 * I;
        g.K = H;
        g.E = E;
        g.tile_expert = tile_e;
        g.tile_row0 = tile_r;
        g.num_tiles = ntiles;
        g.max_tiles = L.tiles;
        g.epi = MOE_EPI_SILU_MUL_QUANT;
        g.scale_fmt = scale_fmt;
        g.sorted_pair_ids = row_map;
        g.out_q = a2;
        g.out_scale = a2s;
        g.os_row_stride = 1;
        g.os_kb_stride = L.rows;
        if (packed) {
            g.sf_packed = sfm;
            g.a_sf = a1sf;
            g.b_sf = reinterpret_cast<const uint8_t*>(w13_scale);
            g.out_sf = a2sf;
        }
        g.status = st->status;
        e = launch_grouped_gemm(g, st->num_sms, s);
    }
    if (e == cudaSuccess) {
        // one "pair" per input row: unit weight, written to the row's place in out
        GemmArgs g{};
        g.a_box_rows = max_tokens <= 32 ? 32 : 128;   // no expert has more rows than max_tokens
        g.A = a2;
        g.a_scale = a2s;
        g.as_row_stride = 1;
        g.as_kb_stride = L.rows;
        g.a_rows = L.rows;
        g.B = w2;
        g.b_tiled = weight_layout == MOE_WEIGHTS_TILED;
        g.b_scale = w2_scale;
        g.N = H;
        g.K = I;
        g.E = E;
        g.tile_expert = tile_e;
        g.tile_row0 = tile_r;
        g.num_tiles = ntiles;
        g.max_tiles = L.tiles;
        g.epi = MOE_EPI_WEIGHTED_PAIRS_BF16;
        g.out_bf16 = out;
        g.sorted_pair_ids = row_map;
        g.topk_weights = ones;
        g.topk = 1;
        g.num_pairs = EM;
        if (packed) {
            g.sf_packed = sfm;
            g.a_sf = a2sf;
            g.b_sf = reinterpret_cast<const uint8_t*>(w2_scale);
        }
        g.status = st->status;
        e = launch_grouped_gemm(g, st->num_sms, s);
    }
    return cuda_rc(e);
}

}  // extern "C"
