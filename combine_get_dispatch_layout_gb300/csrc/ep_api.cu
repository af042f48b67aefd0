// C ABI of libep.so: argument checks, handle lifecycle and kernel launches.
//
// The call set mirrors nccl_ep.cc (ncclEpCreateHandle -> ep_layout,
// ncclEpDispatch -> ep_dispatch, ncclEpCombine -> ep_combine,
// ncclEpHandleDestroy -> ep_handle_destroy, ncclEpHandleGetNumRecvTokens ->
// ep_handle_query). Where that file asserts on a bad argument, these calls
// return EP_ERR_INVALID_ARG before enqueuing anything. The handle owns one
// device block (slot -> row map, layout scratch, a few state words) allocated
// through the caller's hooks, and a pinned host mirror of the state words.
#include <cstdint>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "ep_internal.cuh"

struct ep_handle {
    int device = -1;
    ep_alloc_fn alloc_fn = nullptr;
    ep_free_fn free_fn = nullptr;
    // routing of the last ep_layout
    int T = 0, K = 0, E = 0, R = 0;   // E: the layout's key space (R for a non-expand layout)
    int routing_E = 0;          // the experts of the routing the last layout was given
    bool nonexpand = false;     // the last layout was ep_layout_nonexpand
    int align = 1;              // expert row alignment of the last layout
    int stride = 0;             // > 0: fixed rows per expert (strided layout)
    ep::LayoutPlan plan{};
    cudaStream_t layout_stream = nullptr;
    bool error_latched = false;
    bool meta_known = false;    // host_meta holds the last layout's state words
    bool captured = false;      // a layout was enqueued under stream capture: graph
                                // replays rerun it unseen, so nothing is cached
    int layout_kernels = 0;     // kernels the last ep_layout enqueued
    // capacities of the device block
    int64_t cap_slots = 0, cap_chunk_cells = 0, cap_rank_cells = 0, cap_experts = 0;
    void* dev_block = nullptr;
    int32_t* meta = nullptr;        // [ep::kMetaWords]
    int32_t* row_of_slot = nullptr; // [cap_slots]
    int32_t* chunk_cnt = nullptr;   // [cap_chunk_cells]
    int32_t* block_rank = nullptr;  // [cap_rank_cells]
    int32_t* counts = nullptr;      // [cap_experts] copy of num_tokens_per_expert
    int32_t* offsets = nullptr;     // [cap_experts + 1] copy of expert_offsets
    int64_t cap_keys = 0;
    int64_t* keys = nullptr;        // [cap_keys] derived (rank) keys of a non-expand layout
    int32_t* rank_scratch = nullptr;  // [cap_experts] second copy of the key counts
    int32_t* host_meta = nullptr;   // pinned [ep::kMetaWords]
};

namespace {

// A named NVTX range around each public call, so that profilers (ncu
// --nvtx-include, Nsight Systems) can attribute its kernels to it; with no
// tool attached a push is a pointer check.
struct ApiRange {
    explicit ApiRange(const char* name) { nvtxRangePushA(name); }
    ~ApiRange() { nvtxRangePop(); }
    ApiRange(const ApiRange&) = delete;
    ApiRange& operator=(const ApiRange&) = delete;
};

int default_alloc(void** p, size_t bytes) { return cudaMalloc(p, bytes) == cudaSuccess ? 0 : 1; }
int default_free(void* p) { return cudaFree(p) == cudaSuccess ? 0 : 1; }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

ep_status_t current_device_is(const ep_handle* h) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    return dev == h->device ? EP_OK : EP_ERR_INVALID_ARG;
}

void release_block(ep_handle* h) {
    if (h->dev_block) h->free_fn(h->dev_block);
    h->dev_block = nullptr;
    h->meta = h->row_of_slot = h->chunk_cnt = h->block_rank = h->counts = h->offsets = h->rank_scratch = nullptr;
    h->keys = nullptr;
    h->cap_slots = h->cap_chunk_cells = h->cap_rank_cells = h->cap_experts = h->cap_keys = 0;
}

bool capturing(cudaStream_t s);

// (Re)allocate the device block for at least the given sizes; zeroes the state
// words. Growing allocates and synchronises, which a stream capture forbids.
ep_status_t ensure_block(ep_handle* h, int64_t slots, int64_t chunk_cells, int64_t rank_cells,
                         int64_t experts, int64_t keys, cudaStream_t stream) {
    if (h->dev_block && slots <= h->cap_slots && chunk_cells <= h->cap_chunk_cells &&
        rank_cells <= h->cap_rank_cells && experts <= h->cap_experts && keys <= h->cap_keys)
        return EP_OK;
    if (capturing(stream)) return EP_ERR_INVALID_ARG;
    if (h->dev_block) {
        // work already enqueued may still read the old block
        if (cudaDeviceSynchronize() != cudaSuccess) return EP_ERR_CUDA;
        release_block(h);
    }
    const size_t a = 256;
    const size_t meta_b = round_up(sizeof(int32_t) * ep::kMetaWords, a);
    const size_t rows_b = round_up(sizeof(int32_t) * static_cast<size_t>(slots > 0 ? slots : 1), a);
    const size_t cnt_b = round_up(sizeof(int32_t) * static_cast<size_t>(chunk_cells > 0 ? chunk_cells : 1), a);
    const size_t rank_b = round_up(sizeof(int32_t) * static_cast<size_t>(rank_cells > 0 ? rank_cells : 1), a);
    const size_t exp_b = round_up(sizeof(int32_t) * static_cast<size_t>(3 * experts + 1), a);
    const size_t key_b = round_up(sizeof(int64_t) * static_cast<size_t>(keys > 0 ? keys : 1), a);
    void* block = nullptr;
    if (h->alloc_fn(&block, meta_b + rows_b + cnt_b + rank_b + exp_b + key_b) != 0 || block == nullptr)
        return EP_ERR_ALLOC;
    char* base = static_cast<char*>(block);
    h->dev_block = block;
    h->meta = reinterpret_cast<int32_t*>(base);
    h->row_of_slot = reinterpret_cast<int32_t*>(base + meta_b);
    h->chunk_cnt = reinterpret_cast<int32_t*>(base + meta_b + rows_b);
    h->block_rank = reinterpret_cast<int32_t*>(base + meta_b + rows_b + cnt_b);
    h->counts = reinterpret_cast<int32_t*>(base + meta_b + rows_b + cnt_b + rank_b);
    h->offsets = h->counts + experts;
    h->rank_scratch = h->offsets + experts + 1;
    h->keys = reinterpret_cast<int64_t*>(base + meta_b + rows_b + cnt_b + rank_b + exp_b);
    h->cap_keys = keys;
    h->cap_slots = slots;
    h->cap_chunk_cells = chunk_cells;
    h->cap_rank_cells = rank_cells;
    h->cap_experts = experts;
    // stream-ordered so the first layout on `stream` sees zeroed state words
    if (cudaMemsetAsync(h->meta, 0, meta_b, stream) != cudaSuccess) return EP_ERR_CUDA;
    return EP_OK;
}

bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
}

// Read the state words written by the last layout. Only layouts write them,
// so the first read after a layout synchronises its stream and later reads
// use the host copy until the next layout on this handle (always re-read
// for a handle whose layout a graph may replay). Not possible while the
// layout's stream is being captured.
ep_status_t read_meta(ep_handle* h, int64_t* rows, int32_t* err) {
    if (!h->meta_known || h->captured) {
        if (capturing(h->layout_stream)) return EP_ERR_INVALID_ARG;
        if (cudaMemcpyAsync(h->host_meta, h->meta, sizeof(int32_t) * ep::kMetaWords, cudaMemcpyDeviceToHost,
                            h->layout_stream) != cudaSuccess)
            return EP_ERR_CUDA;
        if (cudaStreamSynchronize(h->layout_stream) != cudaSuccess) return EP_ERR_CUDA;
        h->meta_known = true;
    }
    if (rows) *rows = h->host_meta[ep::kMetaRows];
    if (err) *err = h->host_meta[ep::kMetaError];
    // an invalid expert id blocks later calls; a strided overflow only drops slots
    h->error_latched = h->host_meta[ep::kMetaError] == EP_ERR_INVALID_EXPERT;
    return EP_OK;
}

// Most receive rows a routing can need: every slot valid, every expert padded;
// a strided layout always spans E * stride rows.
int64_t max_rows_of(int T, int K, int E, int align, int stride = 0) {
    if (stride > 0) return static_cast<int64_t>(E) * stride;
    return static_cast<int64_t>(T) * K + static_cast<int64_t>(E) * (align - 1);
}

// Rows that a consumer buffer must hold: skip the device read when the
// buffer holds the most a routing can produce.
ep_status_t check_rows(ep_handle* h, int64_t capacity, cudaStream_t stream) {
    // (a replayed layout may have cleared a latched error: graph handles
    // report it through ep_handle_query only)
    if (h->error_latched && !h->captured) return EP_ERR_INVALID_EXPERT;
    const int64_t max_rows = max_rows_of(h->T, h->K, h->E, h->align, h->stride);
    if (capacity >= max_rows) return EP_OK;
    if (h->stride > 0) return EP_ERR_CAPACITY;   // a strided buffer must span E * stride rows
    if (capturing(stream)) return EP_ERR_INVALID_ARG;   // N cannot be read inside a capture
    int64_t n = 0;
    int32_t err = 0;
    ep_status_t st = read_meta(h, &n, &err);
    if (st != EP_OK) return st;
    if (err == EP_ERR_INVALID_EXPERT) return EP_ERR_INVALID_EXPERT;
    return n > capacity ? EP_ERR_CAPACITY : EP_OK;
}

}  // namespace

namespace {

ep_status_t layout_impl(const int64_t* topk_idx, int T, int K, int E, int R, int align, int stride, bool nonexpand,
                        int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                        uint8_t* is_token_in_rank, int32_t* expert_offsets,
                        ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                        ep_handle_t* handle, void* stream) {
    if (!handle || !num_tokens_per_expert || !num_tokens_per_rank || !expert_offsets)
        return EP_ERR_INVALID_ARG;
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS || R < 1 || R > EP_MAX_RANKS ||
        E % R != 0)
        return EP_ERR_INVALID_ARG;
    if (align < 1 || align > EP_MAX_ALIGNMENT || stride < 0 || (stride > 0 && align != 1)) return EP_ERR_INVALID_ARG;
    if (max_rows_of(T, K, E, align) >= (int64_t{1} << 31)) return EP_ERR_INVALID_ARG;
    if (static_cast<int64_t>(E) * stride >= (int64_t{1} << 31)) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !is_token_in_rank)) return EP_ERR_INVALID_ARG;
    if ((alloc_fn == nullptr) != (free_fn == nullptr)) return EP_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 8) || !aligned(num_tokens_per_expert, 4) || !aligned(num_tokens_per_rank, 4) ||
        !aligned(expert_offsets, 4))
        return EP_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ep_handle* h = *handle;
    bool created = false;
    if (h == nullptr) {
        if (capturing(s)) return EP_ERR_INVALID_ARG;   // creating a handle allocates
        h = new (std::nothrow) ep_handle();
        if (!h) return EP_ERR_ALLOC;
        created = true;
        if (cudaGetDevice(&h->device) != cudaSuccess) { delete h; return EP_ERR_CUDA; }
        h->alloc_fn = alloc_fn ? alloc_fn : default_alloc;
        h->free_fn = free_fn ? free_fn : default_free;
        ep::prime_dispatch_launch_state();
        if (cudaMallocHost(reinterpret_cast<void**>(&h->host_meta), sizeof(int32_t) * ep::kMetaWords) !=
            cudaSuccess) {
            delete h;
            return EP_ERR_ALLOC;
        }
    } else {
        ep_status_t st = current_device_is(h);
        if (st != EP_OK) return st;
    }
    h->meta_known = false;   // this layout rewrites the state words
    if (capturing(static_cast<cudaStream_t>(stream))) h->captured = true;

    // a non-expand layout runs the expert layout over derived rank keys: the
    // key space is the R ranks (one "expert" per rank)
    const int KE = nonexpand ? R : E;
    ep::LayoutPlan plan = ep::make_layout_plan(T, K, KE, R);
    plan.align = align;
    plan.stride = stride;
    ep_status_t st = ensure_block(h, static_cast<int64_t>(T) * K,
                                  static_cast<int64_t>(KE) * plan.num_chunks,
                                  static_cast<int64_t>(R) * plan.num_blocks, KE,
                                  nonexpand ? static_cast<int64_t>(T) * K : 0, s);
    if (st != EP_OK) {
        if (created) {
            cudaFreeHost(h->host_meta);
            release_block(h);
            delete h;
        } else {
            h->T = 0;   // the old block is gone: later calls on this handle move nothing
            h->nonexpand = false;
        }
        return st;
    }
    h->T = T; h->K = K; h->E = KE; h->R = R;
    h->routing_E = E;
    h->nonexpand = nonexpand;
    h->align = align;
    h->stride = stride;
    h->plan = plan;
    h->layout_stream = s;
    h->error_latched = false;

    cudaError_t err;
    if (T == 0) {
        err = cudaMemsetAsync(num_tokens_per_expert, 0, sizeof(int32_t) * E, s);
        if (err == cudaSuccess) err = cudaMemsetAsync(num_tokens_per_rank, 0, sizeof(int32_t) * R, s);
        if (err == cudaSuccess) err = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (KE + 1), s);
        if (err == cudaSuccess) err = cudaMemsetAsync(h->meta, 0, sizeof(int32_t) * ep::kMetaWords, s);
        if (err == cudaSuccess) err = cudaMemsetAsync(h->counts, 0, sizeof(int32_t) * (2 * KE + 1), s);
        if (err == cudaSuccess && stride > 0)
            err = ep::launch_strided_empty(expert_offsets, h->offsets, h->meta, KE, stride, s);
    } else {
        ep::LayoutArgs a{};
        a.topk_idx = topk_idx;
        a.num_tokens_per_expert = num_tokens_per_expert;
        a.num_tokens_per_rank = num_tokens_per_rank;
        err = cudaSuccess;
        if (nonexpand) {
            // expert counts by the key pass; the key layout's per-key counts
            // are the per-rank token counts
            err = cudaMemsetAsync(num_tokens_per_expert, 0, sizeof(int32_t) * E, s);
            if (err == cudaSuccess)
                err = ep::launch_nonexpand_keys(topk_idx, T, K, E, R, h->keys, num_tokens_per_expert, s);
            a.topk_idx = h->keys;
            a.num_tokens_per_expert = num_tokens_per_rank;
            a.num_tokens_per_rank = h->rank_scratch;
        }
        a.is_token_in_rank = is_token_in_rank;
        a.expert_offsets = expert_offsets;
        a.row_of_slot = h->row_of_slot;
        a.chunk_cnt = h->chunk_cnt;
        a.block_rank = h->block_rank;
        a.meta = h->meta;
        a.h_counts = h->counts;
        a.h_offsets = h->offsets;
        if (err == cudaSuccess) err = ep::launch_layout(plan, a, s, &h->layout_kernels);
    }
    if (T == 0) h->layout_kernels = stride > 0 ? 1 : 0;
    *handle = h;
    return err == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

// The combine, and for the dispatch backward also the gather of the slot
// weights (row_weights non-null), in one kernel.
ep_status_t combine_impl(ep_handle* handle, const void* y, int64_t y_rows, int H, const float* topk_weights,
                         void* out, const float* row_weights, float* slot_weights, void* stream) {
    if (!handle) return EP_ERR_INVALID_ARG;
    if (H < 8 || H % 8 != 0 || y_rows < 0) return EP_ERR_INVALID_ARG;
    if (handle->T > 0 && !out) return EP_ERR_INVALID_ARG;
    if (y_rows > 0 && !y) return EP_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(topk_weights, 4)) return EP_ERR_INVALID_ARG;
    ep_status_t st = current_device_is(handle);
    if (st != EP_OK) return st;
    st = check_rows(handle, y_rows, static_cast<cudaStream_t>(stream));
    if (st != EP_OK) return st;

    ep::CombineArgs a{};
    a.y = y;
    a.row_of_slot = handle->row_of_slot;
    a.topk_weights = topk_weights;
    a.out = out;
    a.y_rows = y_rows;
    a.T = handle->T;
    a.K = handle->K;
    a.H = H;
    a.row_weights = row_weights;
    a.slot_weights = slot_weights;
    cudaError_t err = ep::launch_combine(a, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // namespace

extern "C" {

ep_status_t ep_layout(const int64_t* topk_idx, int T, int K, int E, int R,
                      int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                      uint8_t* is_token_in_rank, int32_t* expert_offsets,
                      ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                      ep_handle_t* handle, void* stream) {
    ApiRange range("ep_layout");
    return layout_impl(topk_idx, T, K, E, R, 1, 0, false, num_tokens_per_expert, num_tokens_per_rank, is_token_in_rank,
                       expert_offsets, alloc_fn, free_fn, handle, stream);
}

ep_status_t ep_layout_aligned(const int64_t* topk_idx, int T, int K, int E, int R, int expert_alignment,
                              int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                              uint8_t* is_token_in_rank, int32_t* expert_offsets,
                              ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                              ep_handle_t* handle, void* stream) {
    ApiRange range("ep_layout_aligned");
    return layout_impl(topk_idx, T, K, E, R, expert_alignment, 0, false, num_tokens_per_expert, num_tokens_per_rank,
                       is_token_in_rank, expert_offsets, alloc_fn, free_fn, handle, stream);
}

ep_status_t ep_layout_strided(const int64_t* topk_idx, int T, int K, int E, int R, int expert_capacity,
                              int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                              uint8_t* is_token_in_rank, int32_t* expert_offsets,
                              ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                              ep_handle_t* handle, void* stream) {
    ApiRange range("ep_layout_strided");
    if (expert_capacity < 1) return EP_ERR_INVALID_ARG;
    return layout_impl(topk_idx, T, K, E, R, 1, expert_capacity, false, num_tokens_per_expert, num_tokens_per_rank,
                       is_token_in_rank, expert_offsets, alloc_fn, free_fn, handle, stream);
}

ep_status_t ep_layout_nonexpand(const int64_t* topk_idx, int T, int K, int E, int R,
                                int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                uint8_t* is_token_in_rank, int32_t* rank_offsets,
                                ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                                ep_handle_t* handle, void* stream) {
    ApiRange range("ep_layout_nonexpand");
    return layout_impl(topk_idx, T, K, E, R, 1, 0, true, num_tokens_per_expert, num_tokens_per_rank,
                       is_token_in_rank, rank_offsets, alloc_fn, free_fn, handle, stream);
}

ep_status_t ep_nonexpand_recv_topk(ep_handle_t handle, const int64_t* topk_idx, const float* topk_weights, int E,
                                   int64_t* recv_topk_idx, float* recv_topk_weights, int64_t recv_capacity,
                                   void* stream) {
    ApiRange range("ep_nonexpand_recv_topk");
    if (!handle) return EP_ERR_INVALID_ARG;
    const int T = handle->T, K = handle->K, R = handle->R;
    // the rank-local ids come from E / R: only the E the layout itself was
    // given, on a non-expand layout's handle, gives the rows' true ids
    if (!handle->nonexpand || E != handle->routing_E) return EP_ERR_INVALID_ARG;
    if (E < 1 || E > EP_MAX_EXPERTS || E % R != 0 || recv_capacity < 0) return EP_ERR_INVALID_ARG;
    if (T > 0 && !topk_idx) return EP_ERR_INVALID_ARG;
    if (recv_capacity > 0 && !recv_topk_idx) return EP_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 8) || !aligned(recv_topk_idx, 8) || !aligned(topk_weights, 4) ||
        !aligned(recv_topk_weights, 4))
        return EP_ERR_INVALID_ARG;
    ep_status_t st = current_device_is(handle);
    if (st != EP_OK) return st;
    st = check_rows(handle, recv_capacity, static_cast<cudaStream_t>(stream));
    if (st != EP_OK) return st;
    return ep::launch_nonexpand_recv_topk(topk_idx, topk_weights, handle->row_of_slot, T, K, E, R, recv_topk_idx,
                                          recv_topk_weights, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? EP_OK
               : EP_ERR_CUDA;
}

ep_status_t ep_dispatch_ex(ep_handle_t handle, const void* x, const void* x_scales, int H,
                           const ep_dispatch_config_t* config, const float* topk_weights,
                           void* recv_x, void* recv_scales, int32_t* recv_src_token,
                           float* recv_weights, int64_t recv_capacity, void* stream) {
    ApiRange range("ep_dispatch_ex");
    if (!handle) return EP_ERR_INVALID_ARG;
    ep_dispatch_config_t cfg{};
    if (config) cfg = *config;
    const auto known = [](int d) {
        return d == EP_DTYPE_BF16 || d == EP_DTYPE_FP8_E4M3 || d == EP_DTYPE_FP8_E5M2;
    };
    if (!known(cfg.in_dtype) || !known(cfg.out_dtype)) return EP_ERR_INVALID_ARG;
    // fp8 input is moved unchanged, so it needs the same output type
    if (cfg.in_dtype != EP_DTYPE_BF16 && cfg.out_dtype != cfg.in_dtype) return EP_ERR_INVALID_ARG;
    if (cfg.scale_mode != EP_SCALE_FP32 && cfg.scale_mode != EP_SCALE_POW2 && cfg.scale_mode != EP_SCALE_UE8M0)
        return EP_ERR_INVALID_ARG;
    const bool fp8 = cfg.out_dtype != EP_DTYPE_BF16;
    const bool fp8_in = cfg.in_dtype != EP_DTYPE_BF16;
    if (H < 8 || H % 8 != 0 || recv_capacity < 0) return EP_ERR_INVALID_ARG;
    if (fp8 && H % 128 != 0) return EP_ERR_INVALID_ARG;
    const size_t scale_bytes = cfg.scale_mode == EP_SCALE_UE8M0 ? 1 : 4;
    if (fp8 && !aligned(recv_scales, scale_bytes)) return EP_ERR_INVALID_ARG;
    if (fp8 && cfg.scales_col_major && cfg.scales_ld < recv_capacity) return EP_ERR_INVALID_ARG;
    if (fp8_in && handle->T > 0 && (!x_scales || !aligned(x_scales, scale_bytes))) return EP_ERR_INVALID_ARG;
    if (recv_weights && !topk_weights && handle->T > 0) return EP_ERR_INVALID_ARG;
    if (handle->T > 0 && !x) return EP_ERR_INVALID_ARG;
    // zero-row receive buffers may be NULL; the capacity check below then
    // guarantees no row is written
    if (recv_capacity > 0 && (!recv_x || (fp8 && !recv_scales))) return EP_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv_x, 16) || !aligned(topk_weights, 4) || !aligned(recv_src_token, 4) ||
        !aligned(recv_weights, 4))
        return EP_ERR_INVALID_ARG;
    ep_status_t st = current_device_is(handle);
    if (st != EP_OK) return st;
    st = check_rows(handle, recv_capacity, static_cast<cudaStream_t>(stream));
    if (st != EP_OK) return st;

    ep::DispatchArgs a{};
    a.x = x;
    a.row_of_slot = handle->row_of_slot;
    a.topk_weights = topk_weights;
    a.recv_x = recv_x;
    a.recv_scales = recv_scales;
    a.recv_src_token = recv_src_token;
    a.recv_weights = recv_weights;
    a.recv_capacity = recv_capacity;
    a.T = handle->T;
    a.K = handle->K;
    a.H = H;
    a.scale_mode = cfg.scale_mode;
    a.fp8_format = cfg.out_dtype;
    a.scale_col_major = cfg.scales_col_major ? 1 : 0;
    a.scale_ld = cfg.scales_ld;
    a.x_scales = x_scales;
    a.overlap_layout = cfg.overlap_layout ? 1 : 0;
    if (a.overlap_layout && handle->T > 0) {
        // the L2 prefetch of x during the layout is for device memory only
        cudaPointerAttributes attr{};
        if (cudaPointerGetAttributes(&attr, x) == cudaSuccess && attr.type == cudaMemoryTypeDevice)
            a.prefetch_x = 1;
        cudaGetLastError();
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (handle->align > 1) {
        // the dispatch grid also zeroes the pad rows (at most align - 1 per expert)
        a.pad_counts = handle->counts;
        a.pad_offsets = handle->offsets;
        a.pad_experts = handle->E;
        a.pad_max = handle->align - 1;
        if (fp8) {
            a.pad_scales.ptr = recv_scales;
            a.pad_scales.nb = H / 128;
            a.pad_scales.bytes = static_cast<int>(scale_bytes);
            a.pad_scales.col_major = a.scale_col_major;
            a.pad_scales.ld = cfg.scales_ld;
        }
    }
    cudaError_t err = fp8_in ? ep::launch_dispatch_fp8_passthrough(a, s)
                      : fp8  ? ep::launch_dispatch_fp8(a, s)
                             : ep::launch_dispatch_bf16(a, s);
    return err == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

ep_status_t ep_dispatch(ep_handle_t handle, const void* x, int H, ep_dtype_t out_dtype,
                        const float* topk_weights,
                        void* recv_x, float* recv_scales, int32_t* recv_src_token,
                        float* recv_weights, int64_t recv_capacity, void* stream) {
    ApiRange range("ep_dispatch");
    ep_dispatch_config_t cfg{};
    cfg.in_dtype = EP_DTYPE_BF16;
    cfg.out_dtype = out_dtype;
    return ep_dispatch_ex(handle, x, nullptr, H, &cfg, topk_weights, recv_x, recv_scales, recv_src_token,
                          recv_weights, recv_capacity, stream);
}

ep_status_t ep_combine(ep_handle_t handle, const void* y, int64_t y_rows, int H,
                       const float* topk_weights, void* out, void* stream) {
    ApiRange range("ep_combine");
    return combine_impl(handle, y, y_rows, H, topk_weights, out, nullptr, nullptr, stream);
}

ep_status_t ep_combine_backward(ep_handle_t handle, const void* grad_out, const void* y, int64_t y_rows, int H,
                                const float* topk_weights, void* grad_y, int64_t grad_y_capacity,
                                float* grad_topk_weights, void* stream) {
    ApiRange range("ep_combine_backward");
    if (!handle) return EP_ERR_INVALID_ARG;
    if (H < 8 || H % 8 != 0 || y_rows < 0 || grad_y_capacity < 0) return EP_ERR_INVALID_ARG;
    if (handle->T > 0 && !grad_out) return EP_ERR_INVALID_ARG;
    if (grad_topk_weights && y_rows > 0 && !y) return EP_ERR_INVALID_ARG;
    if (grad_y_capacity > 0 && !grad_y) return EP_ERR_INVALID_ARG;
    if (!aligned(grad_out, 16) || !aligned(y, 16) || !aligned(grad_y, 16) || !aligned(topk_weights, 4) ||
        !aligned(grad_topk_weights, 4))
        return EP_ERR_INVALID_ARG;
    ep_status_t st = current_device_is(handle);
    if (st != EP_OK) return st;
    if (grad_y) {
        st = check_rows(handle, grad_y_capacity, static_cast<cudaStream_t>(stream));
        if (st != EP_OK) return st;
    }
    if (grad_topk_weights) {
        st = check_rows(handle, y_rows, static_cast<cudaStream_t>(stream));
        if (st != EP_OK) return st;
    }
    ep::CombineBackwardArgs a{};
    a.grad_out = grad_out;
    a.y = grad_topk_weights ? y : nullptr;
    a.row_of_slot = handle->row_of_slot;
    a.topk_weights = topk_weights;
    a.grad_y = grad_y;
    a.grad_w = grad_topk_weights;
    a.T = handle->T;
    a.K = handle->K;
    a.H = H;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = cudaSuccess;
    if (grad_y || grad_topk_weights) err = ep::launch_combine_backward(a, s);
    if (err == cudaSuccess && grad_y && handle->align > 1 && handle->T > 0)
        err = ep::launch_fill_pad_rows(handle->counts, handle->offsets, handle->E, static_cast<int64_t>(H) * 2,
                                       grad_y, ep::PadScales{}, nullptr, nullptr, s, handle->align - 1);
    return err == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

ep_status_t ep_dispatch_backward(ep_handle_t handle, const void* grad_recv, int64_t grad_rows, int H,
                                 const float* grad_recv_weights, void* grad_x, float* grad_topk_weights,
                                 void* stream) {
    ApiRange range("ep_dispatch_backward");
    if (!handle) return EP_ERR_INVALID_ARG;
    if (grad_topk_weights && !grad_recv_weights && grad_rows > 0) return EP_ERR_INVALID_ARG;
    if (!aligned(grad_recv_weights, 4) || !aligned(grad_topk_weights, 4)) return EP_ERR_INVALID_ARG;
    // the unweighted combine, which also gathers the weight gradients
    return combine_impl(handle, grad_recv, grad_rows, H, nullptr, grad_x,
                        grad_topk_weights ? grad_recv_weights : nullptr, grad_topk_weights, stream);
}

ep_status_t ep_topk_to_routing_map(const int64_t* topk_idx, const float* topk_weights, int T, int K, int E,
                                   uint8_t* routing_map, float* probs, int32_t* device_error, void* stream) {
    ApiRange range("ep_topk_to_routing_map");
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !routing_map)) return EP_ERR_INVALID_ARG;
    if (probs && !topk_weights && T > 0) return EP_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 8) || !aligned(topk_weights, 4) || !aligned(probs, 4) || !aligned(device_error, 4))
        return EP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = device_error ? cudaMemsetAsync(device_error, 0, sizeof(int32_t), s) : cudaSuccess;
    if (err == cudaSuccess)
        err = ep::launch_topk_to_routing_map(topk_idx, topk_weights, T, K, E, routing_map, probs, device_error, s);
    return err == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

ep_status_t ep_routing_map_to_topk(const uint8_t* routing_map, const float* probs, int T, int E, int K,
                                   int64_t* topk_idx, float* topk_weights, int32_t* device_error, void* stream) {
    ApiRange range("ep_routing_map_to_topk");
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !routing_map)) return EP_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 8) || !aligned(topk_weights, 4) || !aligned(probs, 4) || !aligned(device_error, 4))
        return EP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = device_error ? cudaMemsetAsync(device_error, 0, sizeof(int32_t), s) : cudaSuccess;
    if (err == cudaSuccess)
        err = ep::launch_routing_map_to_topk(routing_map, probs, T, E, K, topk_idx, topk_weights, device_error, s);
    return err == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

ep_status_t ep_handle_query(ep_handle_t handle, int64_t* num_recv_rows, int32_t* device_error) {
    ApiRange range("ep_handle_query");
    if (!handle) return EP_ERR_INVALID_ARG;
    ep_status_t st = current_device_is(handle);
    if (st != EP_OK) return st;
    int64_t n = 0;
    int32_t err = 0;
    st = read_meta(handle, &n, &err);
    if (st != EP_OK) return st;
    if (num_recv_rows) *num_recv_rows = n;
    if (device_error) *device_error = err;
    return err != 0 ? static_cast<ep_status_t>(err) : EP_OK;
}

ep_status_t ep_handle_copy_row_of_slot(ep_handle_t handle, int32_t* dst, void* stream) {
    if (!handle) return EP_ERR_INVALID_ARG;
    const size_t bytes = sizeof(int32_t) * static_cast<size_t>(handle->T) * handle->K;
    if (bytes == 0) return EP_OK;
    if (!dst || !aligned(dst, 4)) return EP_ERR_INVALID_ARG;
    ep_status_t st = current_device_is(handle);
    if (st != EP_OK) return st;
    return cudaMemcpyAsync(dst, handle->row_of_slot, bytes, cudaMemcpyDeviceToDevice,
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? EP_OK
               : EP_ERR_CUDA;
}

ep_status_t ep_handle_destroy(ep_handle_t handle) {
    if (!handle) return EP_OK;
    int prev = -1;
    cudaGetDevice(&prev);
    const bool switch_dev = prev != handle->device;
    if (switch_dev && cudaSetDevice(handle->device) != cudaSuccess) return EP_ERR_CUDA;
    ep_status_t st = cudaDeviceSynchronize() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
    release_block(handle);
    if (handle->host_meta) cudaFreeHost(handle->host_meta);
    delete handle;
    if (switch_dev) cudaSetDevice(prev);
    return st;
}

int ep_handle_layout_kernels(ep_handle_t handle) { return handle ? handle->layout_kernels : -1; }

const char* ep_status_string(ep_status_t status) {
    switch (status) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
        case EP_ERR_INVALID_EXPERT: return "EP_ERR_INVALID_EXPERT";
        case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY";
        case EP_ERR_CUDA: return "EP_ERR_CUDA";
        case EP_ERR_ALLOC: return "EP_ERR_ALLOC";
    }
    return "EP_ERR_UNKNOWN";
}

int ep_layout_cluster_ctas(int T, int K, int E, int R) {
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS || R < 1 || R > EP_MAX_RANKS || E % R != 0)
        return -1;
    if (static_cast<int64_t>(T) * K >= (int64_t{1} << 31)) return -1;
    if (T == 0) return 0;
    return ep::layout_cluster_ctas(ep::make_layout_plan(T, K, E, R));
}

}  // extern "C"
