// ep_layout_noalloc: the routing layout with its scratch in a fixed array
// compiled into the library, for callers that cannot allocate device memory
// (their memory is owned by another allocator, or cudaMalloc's implicit
// device synchronisation is not acceptable where they run). Nothing here
// allocates: the same three layout kernels run with their per-chunk count
// table, per-block rank counts and state words placed in `g_scratch`.
#include <mutex>

#include "ep_internal.cuh"

namespace {

constexpr size_t kScratchBytes = EP_NOALLOC_SCRATCH_BYTES;
constexpr size_t kMetaSlot = 64;   // int32 words reserved for the state words (256 bytes)
constexpr int kMaxDevices = 64;

// One copy per device, alive while the library is loaded on that device.
static __device__ __align__(256) int32_t g_scratch[kScratchBytes / sizeof(int32_t)];

std::mutex g_mutex;
int32_t* g_scratch_dev[kMaxDevices] = {};   // device address of g_scratch, per device

// Device address of g_scratch on the current device. In host code the name
// g_scratch is only a stand-in symbol, so the address must come from the
// runtime, looked up once per device with that device current.
cudaError_t scratch_on_current_device(int32_t** out) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_dev[dev] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_dev[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_dev[dev];
    return cudaSuccess;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" ep_status_t ep_layout_noalloc(const int64_t* topk_idx, int T, int K, int E, int R,
                                         int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                         uint8_t* is_token_in_rank, int32_t* expert_offsets,
                                         int32_t* row_of_slot, int32_t* device_error, void* stream) {
    if (!num_tokens_per_expert || !num_tokens_per_rank || !expert_offsets) return EP_ERR_INVALID_ARG;
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS || R < 1 || R > EP_MAX_RANKS ||
        E % R != 0)
        return EP_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * K >= (int64_t{1} << 31)) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !is_token_in_rank || !row_of_slot)) return EP_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 8) || !aligned(num_tokens_per_expert, 4) || !aligned(num_tokens_per_rank, 4) ||
        !aligned(expert_offsets, 4) || !aligned(row_of_slot, 4) || !aligned(device_error, 4))
        return EP_ERR_INVALID_ARG;

    const ep::LayoutPlan plan = ep::make_layout_plan(T, K, E, R);
    const size_t cnt_words = static_cast<size_t>(E) * plan.num_chunks;
    const size_t rank_words = static_cast<size_t>(R) * plan.num_blocks;
    if ((kMetaSlot + cnt_words + rank_words) * sizeof(int32_t) > kScratchBytes) return EP_ERR_CAPACITY;

    int32_t* scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return EP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* meta = scratch;
    // the error accumulator must start at zero; the array keeps the last call's contents
    cudaError_t err = cudaMemsetAsync(meta, 0, sizeof(int32_t) * ep::kMetaWords, s);
    if (err == cudaSuccess) {
        if (T == 0) {
            err = cudaMemsetAsync(num_tokens_per_expert, 0, sizeof(int32_t) * E, s);
            if (err == cudaSuccess) err = cudaMemsetAsync(num_tokens_per_rank, 0, sizeof(int32_t) * R, s);
            if (err == cudaSuccess) err = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), s);
        } else {
            ep::LayoutArgs a{};
            a.topk_idx = topk_idx;
            a.num_tokens_per_expert = num_tokens_per_expert;
            a.num_tokens_per_rank = num_tokens_per_rank;
            a.is_token_in_rank = is_token_in_rank;
            a.expert_offsets = expert_offsets;
            a.row_of_slot = row_of_slot;
            a.chunk_cnt = scratch + kMetaSlot;
            a.block_rank = scratch + kMetaSlot + cnt_words;
            a.meta = meta;
            err = ep::launch_layout(plan, a, s);
        }
    }
    if (err == cudaSuccess && device_error)
        err = cudaMemcpyAsync(device_error, meta + ep::kMetaError, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    return err == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
