// Expert sort with no caller workspace: its scratch lives in a fixed array
// inside the library.
//
// Some callers cannot hand the library freshly allocated device memory: a
// plugin loaded into a host program that owns all device memory through its own
// pool, or a tight serving loop that must not call cudaMalloc (which may
// synchronise the device).  For them, moe_align_permute_noalloc does exactly
// what moe_align_permute does, but keeps its per-chunk histogram table in the
// file-scope array below instead of a workspace.  The caller still provides all
// inputs and outputs.
#include <mutex>

#include "kernels.cuh"

namespace {

// Scratch of the no-allocation sort: (chunks of 1024 pairs) x (experts) int32
// counts.  1 MiB, held by every GPU that loads the library until the process exits.
constexpr int64_t kScratchInts = MOE_NOALLOC_SORT_SCRATCH_INTS;
static __device__ __align__(256) int32_t g_sort_scratch[kScratchInts];

// Device address of g_sort_scratch on each device.  In host code the name
// g_sort_scratch is only a host-side handle, never a device pointer, so the
// address is looked up once per device, with that device current.
constexpr int kMaxDevices = 128;
int32_t* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

int scratch_for_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_sort_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_align_permute_noalloc(const int32_t* topk_ids, int T, int topk, int E, int block_m,
                                         int32_t* expert_offsets, int32_t* padded_offsets,
                                         int32_t* sorted_pair_ids, int32_t* pos, int32_t* tile_expert,
                                         int32_t* tile_row0, int32_t* num_tiles, void* stream) {
    if (T < 0 || topk < 1 || E < 1 || block_m < 1) return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS || block_m > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t P = static_cast<int64_t>(T) * topk;
    const int64_t busy = P < E ? P : E;
    if (P + busy * (block_m - 1) >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    // the fixed scratch must hold one count per (chunk, expert)
    if (mfp8::permute_chunks(P) * E > kScratchInts) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (!expert_offsets || !padded_offsets || !num_tiles) return MOE_ERR_INVALID_ARG;
    if (P > 0 && (!topk_ids || !sorted_pair_ids || !pos || !tile_expert || !tile_row0)) return MOE_ERR_INVALID_ARG;
    uint32_t* status = nullptr;
    int rc = mfp8::device_status_word(&status);
    if (rc != MOE_OK) return rc;
    int32_t* scratch = nullptr;
    if ((rc = scratch_for_current_device(&scratch)) != MOE_OK) return rc;
    // Every count the kernels read is first written by this call, so nothing in the
    // array has to start at zero and no clearing is needed between calls.
    const cudaError_t e = mfp8::launch_align_permute(topk_ids, P, E, block_m, expert_offsets, padded_offsets,
                                                     sorted_pair_ids, pos, tile_expert, tile_row0, num_tiles, scratch,
                                                     status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
