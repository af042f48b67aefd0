// Internal declarations shared by the translation units of libep.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ep.h"

namespace ep {

constexpr unsigned kFullMask = 0xffffffffu;

// Every kernel of the library is launched as a programmatic dependent of the
// work before it on the stream (launch_dependent below, or the layout's and
// dispatch's own launchers): its blocks may be scheduled while the preceding
// grid drains. This is the first statement of such a kernel: wait for that
// grid (and so for all earlier work) before any global memory access, then
// let this grid's own dependent be scheduled. Releasing only after the wait
// keeps the chain's guarantee: when a kernel starts, all work before its
// immediate predecessor is complete. Both instructions are no-ops when the
// launch serialised anyway (an event or a copy in between).
__device__ __forceinline__ void dependent_entry() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
}

// Launch `kernel` as a programmatic dependent of the preceding work on `stream`.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Layout of the handle's small device word block.
enum MetaWord : int {
    kMetaRows = 0,        // N = number of valid slots
    kMetaError = 1,       // EP_ERR_INVALID_EXPERT once an id outside [-1, E) was seen
    kMetaErrorAccum = 2,  // set by any block that sees a bad id; folded into kMetaError
    kMetaWords = 4,
};

// Chunking of the routing table for the layout kernels: each warp owns a
// chunk of `chunk_tokens` consecutive tokens; `warps_per_block` warps form a block.
struct LayoutPlan {
    int T, K, E, R, L;
    int key_bits;            // bits of (expert id + 1)
    int align;               // expert row alignment (1 = packed)
    int stride;              // > 0: expert e's rows start at e * stride (fixed capacity)
    int chunk_tokens;
    int num_chunks;
    int warps_per_block;
    int num_blocks;
    size_t smem_count;       // dynamic shared memory of the count kernel
    size_t smem_assign;      // dynamic shared memory of the assign kernel
    // single-kernel path: one thread-block cluster of cl_ctas CTAs x cl_warps
    // warps; chosen at launch when the routing is small enough
    int cl_ctas;
    int cl_warps;
    int cl_chunk_tokens;
    unsigned l_magic;        // ceil(2^32 / L): rank = umulhi(expert, l_magic)
    int itr_words;           // is_token_in_rank rows can be written as 32-bit words
    size_t smem_cluster;
};

LayoutPlan make_layout_plan(int T, int K, int E, int R);

struct LayoutArgs {
    const int64_t* topk_idx;
    int32_t* num_tokens_per_expert;
    int32_t* num_tokens_per_rank;
    uint8_t* is_token_in_rank;
    int32_t* expert_offsets;
    int32_t* row_of_slot;      // [T*K]
    int32_t* chunk_cnt;        // [E][num_chunks]: counts, then exclusive bases
    int32_t* block_rank;       // [R][num_blocks]: per-block tokens per rank
    int32_t* meta;             // [kMetaWords]
    int32_t* h_counts;         // [E] handle copy of the counts (or null)
    int32_t* h_offsets;        // [E+1] handle copy of the offsets (or null)
};

// Launches the layout; *kernels (if not null) receives the number of kernels
// enqueued (1 on the single-cluster path, 3 on the multi-block path).
cudaError_t launch_layout(const LayoutPlan& p, const LayoutArgs& a, cudaStream_t stream, int* kernels = nullptr);
// CTAs per cluster of the single-launch layout of `p` on the current device;
// 0 when the routing takes the three-kernel path, -1 on a CUDA error.
int layout_cluster_ctas(const LayoutPlan& p);
// The offsets and row count of a strided layout with no tokens (after the
// outputs and state words have been zeroed): offsets[e] = e * stride, N = E * stride.
cudaError_t launch_strided_empty(int32_t* expert_offsets, int32_t* h_offsets, int32_t* meta, int E, int stride,
                                 cudaStream_t stream);

// The fp8 scales of pad rows, zeroed with them.
struct PadScales {
    void* ptr = nullptr;       // null: no scales
    int nb = 0;                // blocks per row
    int bytes = 4;             // 4 (fp32) or 1 (UE8M0)
    int col_major = 0;
    int64_t ld = 0;
};
struct DispatchArgs {
    const void* x;             // bf16 [T, H]
    const int32_t* row_of_slot;
    const float* topk_weights; // [T, K] or null
    void* recv_x;
    void* recv_scales;         // fp32, or uint8 exponents in UE8M0 mode
    int32_t* recv_src_token;
    float* recv_weights;
    int64_t recv_capacity;
    int T, K, H;
    int scale_mode;            // EP_SCALE_FP32 / EP_SCALE_POW2 / EP_SCALE_UE8M0
    int fp8_format;            // EP_DTYPE_FP8_E4M3 / EP_DTYPE_FP8_E5M2 (fp8 output)
    int scale_col_major;       // 0: scales [rows, H/128]; 1: [H/128, scale_ld]
    int64_t scale_ld;
    const void* x_scales;      // fp8 input: [T, H/128] fp32 (uint8 in UE8M0 mode)
    int overlap_layout;        // launch as the preceding layout's programmatic dependent
    int prefetch_x;            // overlap_layout with x in device memory: prefetch x into L2
    // aligned layouts: the grid's first pad_blocks blocks zero the pad rows
    // (one warp per (expert, pad row), at most pad_max pad rows per expert)
    int64_t pad_blocks;
    const int32_t* pad_counts;
    const int32_t* pad_offsets;
    int pad_experts;
    int pad_max;
    PadScales pad_scales;
};

cudaError_t launch_dispatch_bf16(const DispatchArgs& a, cudaStream_t stream);
// Look up, for the current device, what the dispatch launchers query once
// (the resident warps that pick the item size), so that the first dispatch
// never makes that query inside a stream capture. Called at handle creation.
void prime_dispatch_launch_state();
cudaError_t launch_dispatch_fp8(const DispatchArgs& a, cudaStream_t stream);
// fp8 input: codes [T, H] bytes and scale rows moved unchanged to every slot's row
cudaError_t launch_dispatch_fp8_passthrough(const DispatchArgs& a, cudaStream_t stream);

// Zero the pad rows of an aligned layout: for each expert e the rows from
// offsets[e] + counts[e] up to offsets[e+1] (at most max_pad of them) get
// zero bytes (row_bytes each, a multiple of 16), zero scales (if any, in their
// layout), source -1 (if src) and weight 0 (if weights). The dispatch does
// this inside its own grid (DispatchArgs::pad_blocks); this launch serves the
// other producers of receive-shaped rows (the combine backward's grad_y).
cudaError_t launch_fill_pad_rows(const int32_t* counts, const int32_t* offsets, int E, int64_t row_bytes,
                                 void* recv, const PadScales& scales, int32_t* src, float* weights,
                                 cudaStream_t stream, int max_pad);

struct CombineArgs {
    const void* y;             // bf16 [y_rows, H]
    const int32_t* row_of_slot;
    const float* topk_weights; // [T, K] or null (all ones)
    void* out;                 // bf16 [T, H]
    int64_t y_rows;
    int T, K, H;
    // optional (dispatch backward): slot_weights[t, k] = row_weights[row(t, k)],
    // 0 for an unused slot, written by the warp of each token's first segment
    const float* row_weights;
    float* slot_weights;
};

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

struct CombineBackwardArgs {
    const void* grad_out;      // bf16 [T, H]
    const void* y;             // bf16 [rows, H] forward expert outputs
    const int32_t* row_of_slot;
    const float* topk_weights; // [T, K] or null (all ones)
    void* grad_y;              // bf16 [rows, H] or null
    float* grad_w;             // [T, K] or null
    int T, K, H;
};

cudaError_t launch_combine_backward(const CombineBackwardArgs& a, cudaStream_t stream);


cudaError_t launch_topk_to_routing_map(const int64_t* topk_idx, const float* w, int T, int K, int E,
                                       uint8_t* routing_map, float* probs, int32_t* device_error,
                                       cudaStream_t stream);
cudaError_t launch_nonexpand_keys(const int64_t* topk_idx, int T, int K, int E, int R, int64_t* keys,
                                  int32_t* expert_counts, cudaStream_t stream);
cudaError_t launch_nonexpand_recv_topk(const int64_t* topk_idx, const float* w, const int32_t* row_of_slot, int T,
                                       int K, int E, int R, int64_t* recv_topk_idx, float* recv_topk_weights,
                                       cudaStream_t stream);
cudaError_t launch_routing_map_to_topk(const uint8_t* routing_map, const float* probs, int T, int E, int K,
                                       int64_t* topk_idx, float* topk_weights, int32_t* device_error,
                                       cudaStream_t stream);

}  // namespace ep
