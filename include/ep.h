/*
 * ep.h -- C ABI of the GB300 MoE token dispatch / combine library (libep.so).
 *
 * One GPU, one process. The R "ranks" of expert parallelism are logical
 * slabs of one receive buffer in this GPU's memory: expert e belongs to
 * rank e / (E / R), and rank r's slab is receive rows
 * [expert_offsets[r*E/R], expert_offsets[(r+1)*E/R]).
 *
 * Calls and the passages they follow (page title, then section):
 *   ep_layout          nccl_ep.cc, ncclEpCreateHandle (handle built from
 *                      topk_idx) and struct ncclEpHandle (is_token_in_rank,
 *                      num_tokens_for_experts, sparse_to_dense_map);
 *                      DeepEP API docs, "Prefix Sum Interpretation for Expert
 *                      Token Counts" and "Computing with Handle Metadata".
 *   ep_dispatch        nccl_ep.cc, ncclEpDispatch; DeepEP API docs,
 *                      "dispatch()" with do_expand (one row per (token,
 *                      expert) pair).
 *   ep_combine         nccl_ep.cc, ncclEpCombine (low-latency branch:
 *                      weighted by topk_weights); NeMo fused_a2a,
 *                      HybridEPCombine.forward (rows back in token order).
 *   ep_handle_destroy  nccl_ep.cc, ncclEpHandleDestroy.
 *   ep_handle_query    nccl_ep.cc, ncclEpHandleGetNumRecvTokens.
 *
 * Conventions for every call:
 *  - Pointers named as device pointers must be memory the current GPU can
 *    address: its device memory, managed memory, or pinned host memory
 *    mapped into the unified address space (cudaHostAlloc / cudaHostRegister;
 *    on GB300 the kernels then stream it over NVLink-C2C, which is how a
 *    caller with host-resident tokens avoids a separate copy). The caller
 *    owns them; the library never frees caller memory. The library sees
 *    addresses and sizes only: every buffer must hold at least the elements
 *    its call documents (rows x row length for the sizes passed), in the
 *    stated element type, or kernels read or write past it. Alignment is
 *    checked (EP_ERR_INVALID_ARG); lengths cannot be. The Python binding
 *    checks both against the tensors it is given.
 *  - All device work is enqueued on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and is asynchronous, except where a call says it
 *    synchronises.
 *  - Every kernel of the library is launched as a programmatic dependent of
 *    the kernel before it on the stream: its blocks may be scheduled while
 *    that kernel finishes, but wait for it before their first global memory
 *    access (the one exception is the dispatch's early read of x with
 *    overlap_layout, below), so stream order holds as for ordinary launches.
 *    Every kernel here releases its dependents only after that wait, so when
 *    one starts, all work before its immediate predecessor is complete.
 *  - N (the receive rows of the last layout) and the device error word are
 *    read from the device at most once per layout: the first call that needs
 *    them (ep_handle_query, or a dispatch / combine whose buffer is smaller
 *    than the most rows the routing can need) synchronises the layout's
 *    stream; later calls use the host copy until the next layout on the
 *    handle.
 *  - Stream capture (CUDA graphs): ep_layout*, ep_dispatch*, ep_combine* and
 *    the backward calls can be captured when the handle already exists with
 *    room for the routing and every buffer holds the most rows the routing
 *    can need (T*K, plus E*(A-1) when aligned). Inside a capture, a call
 *    that would allocate (creating or growing a handle) or need N from the
 *    device (a smaller buffer, ep_handle_query) returns EP_ERR_INVALID_ARG
 *    and enqueues nothing. A replay reruns the captured layout unseen by the
 *    host, so a handle whose layout was captured keeps no host copy of N or
 *    of the error word: ep_handle_query re-reads them after every replay,
 *    and dispatch / combine on it report an invalid expert id only through
 *    that query.
 *  - Arguments are checked on the host first. A failed check returns
 *    EP_ERR_INVALID_ARG and enqueues nothing.
 *  - Row buffers (x, recv_x, y, out) must be 16-byte aligned.
 *  - An array with no elements may be passed as NULL, and an input is only
 *    required when something would be read from it (T = 0, or no receive
 *    rows, needs no token, weight or row data).
 *  - A handle may be used from one host thread at a time.
 */
#ifndef EP_GB300_EP_H
#define EP_GB300_EP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or dtype       */
    EP_ERR_INVALID_EXPERT = 2, /* a topk_idx entry outside [-1, E) was seen   */
    EP_ERR_CAPACITY = 3,       /* receive buffer smaller than the valid rows  */
    EP_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed        */
    EP_ERR_ALLOC = 5           /* the allocation hook (or cudaMalloc) failed  */
} ep_status_t;

typedef enum {
    EP_DTYPE_BF16 = 0,         /* receive rows are the bf16 token rows        */
    EP_DTYPE_FP8_E4M3 = 1,     /* receive rows are e4m3 bytes + fp32 scales   */
    EP_DTYPE_FP8_E5M2 = 2      /* receive rows are e5m2 bytes + fp32 scales   */
} ep_dtype_t;

/* How fp8 block scales are formed and stored (one per 128 channels). F is the
 * largest finite value of the output format: 448 for e4m3, 57344 for e5m2. */
typedef enum {
    EP_SCALE_FP32 = 0,  /* scale = amax / F (IEEE fp32 division), stored as fp32          */
    EP_SCALE_POW2 = 1,  /* smallest power of two >= amax / F, stored as fp32            */
    EP_SCALE_UE8M0 = 2  /* that power (at least 2^-127) stored as its biased exponent
                           byte b, value 2^(b - 127)                                    */
} ep_scale_mode_t;

/* Options of ep_dispatch_ex; an all-zero struct means bf16 in, bf16 out. */
typedef struct {
    int in_dtype;          /* EP_DTYPE_BF16: x is bf16 [T, H]; EP_DTYPE_FP8_E4M3 or _E5M2:
                              x is fp8 codes [T, H] with x_scales, moved unchanged
                              (needs out_dtype == in_dtype)                          */
    int out_dtype;         /* EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3 or EP_DTYPE_FP8_E5M2      */
    int scale_mode;        /* ep_scale_mode_t for fp8 output (and the x_scales type)      */
    int scales_col_major;  /* 0: recv_scales [cap, H/128]; 1: [H/128, scales_ld]          */
    int64_t scales_ld;     /* rows of the column-major scale matrix (>= recv_capacity)    */
    int overlap_layout;    /* 1: the caller enqueues this dispatch directly after the
                              ep_layout* call that built the handle, on the same stream,
                              with x complete before that layout was enqueued; the
                              dispatch's blocks, scheduled on the SMs the layout leaves
                              idle, then load x while the layout runs instead of after
                              it; if x is device memory its first blocks also prefetch
                              later rows of x into L2 meanwhile.
                              0: every access waits for the preceding kernel.         */
} ep_dispatch_config_t;

/* Opaque routing handle: owns the slot -> row map [T*K] int32, the layout
 * scratch and a small pinned host mirror. Keeps no pointer to topk_idx. */
typedef struct ep_handle* ep_handle_t;

/* Device-memory hooks (return 0 on success). NULL = cudaMalloc / cudaFree. */
typedef int (*ep_alloc_fn)(void** ptr, size_t bytes);
typedef int (*ep_free_fn)(void* ptr);

/* Limits checked on the host. */
#define EP_MAX_EXPERTS 4096
#define EP_MAX_RANKS 1024
#define EP_MAX_TOPK 32
#define EP_MAX_ALIGNMENT 1024

/*
 * ep_layout -- routing layout of topk_idx (the "get dispatch layout" step).
 *
 *  topk_idx               device, int64 [T, K] row-major. Entry e in [0, E)
 *                         routes the slot to expert e; -1 marks an unused
 *                         (dropped) slot. Any other value is an invalid
 *                         expert: that slot is treated as unused and the
 *                         handle latches EP_ERR_INVALID_EXPERT (see
 *                         ep_handle_query).
 *  T, K, E, R             tokens, top-k, experts, logical ranks.
 *                         1 <= K <= EP_MAX_TOPK, 1 <= E <= EP_MAX_EXPERTS,
 *                         1 <= R <= EP_MAX_RANKS, E % R == 0, T >= 0,
 *                         T*K < 2^31.
 *  num_tokens_per_expert  device, int32 [E]: slots routed to each expert.
 *  num_tokens_per_rank    device, int32 [R]: tokens with at least one slot
 *                         on the rank (a token counts once per rank).
 *  is_token_in_rank       device, uint8 [T, R]: 1 if token t has a slot on
 *                         rank r, else 0.
 *  expert_offsets         device, int32 [E + 1]: exclusive prefix sum of
 *                         num_tokens_per_expert; expert_offsets[E] = N, the
 *                         number of valid slots. Expert e owns receive rows
 *                         [expert_offsets[e], expert_offsets[e+1]), filled in
 *                         ascending (token, k) order.
 *  alloc_fn, free_fn      device-memory hooks for a new handle (may be NULL).
 *  handle                 in/out. If *handle is NULL a new handle is created
 *                         (allocates device memory, pinned host memory and
 *                         synchronises the device once). If *handle is an
 *                         existing handle it is reused; it grows (after a
 *                         stream synchronise) only if T*K or the chunking
 *                         outgrows it. Reuse is stream-ordered: earlier work
 *                         that reads the handle must be on `stream` or
 *                         finished.
 * Writes every element of the four outputs; needs no zeroed memory.
 * One kernel (a single thread-block cluster) for routings up to 2^18 slots
 * whose plan fits its shared memory, else three (count, scan, assign);
 * ep_handle_layout_kernels says which. No host synchronisation except on
 * creation or growth.
 */
EP_API ep_status_t ep_layout(const int64_t* topk_idx, int T, int K, int E, int R,
                      int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                      uint8_t* is_token_in_rank, int32_t* expert_offsets,
                      ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                      ep_handle_t* handle, void* stream);

/*
 * ep_layout_aligned -- ep_layout with every expert's receive rows starting on
 * a multiple of expert_alignment (DeepEP API docs, "dispatch()"
 * expert_alignment, and "Prefix Sum Interpretation for Expert Token Counts":
 * in expand mode an expert's range starts at the previous expert's end
 * rounded up to the alignment), for consumers such as grouped GEMMs that
 * want tile-aligned expert blocks.
 *
 *  expert_alignment       1 <= A <= EP_MAX_ALIGNMENT; A = 1 is ep_layout.
 *  num_tokens_per_expert  real slots per expert (unpadded).
 *  expert_offsets         expert_offsets[e] = sum over e' < e of
 *                         roundup(num_tokens_per_expert[e'], A);
 *                         expert_offsets[E] = padded row total. Expert e's
 *                         real rows are expert_offsets[e] + 0 .. count - 1
 *                         in (token, k) order; the rest of its range, up to
 *                         expert_offsets[e+1], are pad rows.
 * Later ep_dispatch calls on the handle also zero the pad rows (zero bytes,
 * scale 0, recv_src_token -1, recv_weights 0), and receive / combine-input
 * buffers must hold the padded total (at most T*K + E*(A-1) rows).
 * Other arguments, outputs and errors as ep_layout; T*K + E*(A-1) < 2^31.
 */
EP_API ep_status_t ep_layout_aligned(const int64_t* topk_idx, int T, int K, int E, int R,
                                     int expert_alignment,
                                     int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                     uint8_t* is_token_in_rank, int32_t* expert_offsets,
                                     ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                                     ep_handle_t* handle, void* stream);

/*
 * ep_layout_strided -- ep_layout for the padded 3-D receive buffer of the
 * low-latency path (nccl_ep.cc, ncclEpDispatch low-latency branch: recv_x
 * [num_local_experts, num_ranks * max_tokens_per_rank, hidden] with
 * per-expert receive counts): expert e owns the fixed row block
 * [e * expert_capacity, (e + 1) * expert_capacity), its slots taking the first
 * rows in (token, k) order; num_tokens_per_expert says how many are valid.
 * expert_offsets[e] = e * expert_capacity and expert_offsets[E] = E *
 * expert_capacity, the rows every receive / expert-output buffer must hold.
 * Rows past an expert's count are never written. Reading: a slot whose rank
 * inside its expert reaches the capacity is dropped (row -1, skipped by
 * dispatch and combine) and ep_handle_query then returns EP_ERR_CAPACITY;
 * later calls on the handle still run. E * expert_capacity < 2^31.
 */
EP_API ep_status_t ep_layout_strided(const int64_t* topk_idx, int T, int K, int E, int R,
                                     int expert_capacity,
                                     int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                     uint8_t* is_token_in_rank, int32_t* expert_offsets,
                                     ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                                     ep_handle_t* handle, void* stream);

/*
 * ep_layout_nonexpand -- layout with one receive row per (token, rank) pair
 * instead of per (token, expert) (DeepEP API docs, "Prefix Sum Interpretation
 * for Expert Token Counts", non-expand mode; nccl_ep.cc, struct ncclEpHandle:
 * sparse_to_dense_map [tokens, ranks], -1 = not routed). Rows are grouped by
 * rank, tokens ascending inside a rank; rank r owns rows
 * [rank_offsets[r], rank_offsets[r+1]) (int32 [R + 1], the exclusive scan of
 * num_tokens_per_rank). In the handle, a token's row for rank r belongs to its
 * first slot on r (lowest k); its other slots on r hold -1. So ep_dispatch
 * writes each token once per rank it reaches, and ep_combine with NULL
 * weights sums one expert-side row per rank (the expert side applies the
 * per-expert weights, see ep_nonexpand_recv_topk). num_tokens_per_expert,
 * num_tokens_per_rank and is_token_in_rank are those of ep_layout. Other
 * arguments and errors as ep_layout.
 */
EP_API ep_status_t ep_layout_nonexpand(const int64_t* topk_idx, int T, int K, int E, int R,
                                       int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                       uint8_t* is_token_in_rank, int32_t* rank_offsets,
                                       ep_alloc_fn alloc_fn, ep_free_fn free_fn,
                                       ep_handle_t* handle, void* stream);

/*
 * ep_nonexpand_recv_topk -- what each non-expand receive row carries for its
 * rank's experts (DeepEP API docs, "dispatch()": recv_topk_idx and
 * recv_topk_weights): for the row of (t, r), entry k is the rank-local expert
 * id e - r * (E/R) if slot k of token t names an expert e of rank r, else -1;
 * the weight is topk_weights[t, k] there, else 0. topk_idx / topk_weights are
 * the ones given to ep_layout_nonexpand (weights may be NULL);
 * recv_topk_idx int64 [cap, K], recv_topk_weights fp32 [cap, K] or NULL.
 * Rows >= N are not written. Returns EP_ERR_INVALID_ARG, enqueuing nothing,
 * when the handle's last layout was not ep_layout_nonexpand or when E differs
 * from the E that layout was given (the rank-local ids depend on it).
 */
EP_API ep_status_t ep_nonexpand_recv_topk(ep_handle_t handle, const int64_t* topk_idx, const float* topk_weights,
                                          int E, int64_t* recv_topk_idx, float* recv_topk_weights,
                                          int64_t recv_capacity, void* stream);

/*
 * ep_dispatch -- stable expert-major permute of the token rows.
 *
 * For every valid slot (t, k) with receive row n = row_of_slot[t, k]:
 *   EP_DTYPE_BF16:     recv_x[n, :] = x[t, :]                 (bf16 [cap, H])
 *   EP_DTYPE_FP8_E4M3: per 128-channel block b of token t,
 *                      amax = max |x[t, 128b : 128b+128]|,
 *                      scale = amax / 448 (fp32, IEEE division),
 *                      recv_x[n, c] = e4m3 satfinite RNE of x[t, c] / scale
 *                      (uint8 [cap, H]), recv_scales[n, b] = scale
 *                      (fp32 [cap, H/128] row-major). An all-zero block has
 *                      scale 0 and zero bytes.
 *   EP_DTYPE_FP8_E5M2: the same with scale = amax / 57344 and e5m2 codes
 *                      (OCP E5M2: bias 15, 2 mantissa bits, largest finite
 *                      57344; satfinite RNE). nccl_ep.cc (ncclTypeSize,
 *                      ncclEpDispatch) lists e5m2 beside e4m3 as a one-byte
 *                      fp8 token type; the scale rule is e4m3's with the
 *                      format's largest finite value in place of 448.
 *   recv_src_token[n] = t          (optional, int32 [cap], NULL = skip)
 *   recv_weights[n] = topk_weights[t, k]  (optional, fp32 [cap]; needs
 *                                  topk_weights; NULL = skip)
 * x is bf16 [T, H] (device); H % 8 == 0, and H % 128 == 0 for fp8.
 * recv_x (and recv_scales for fp8) may be NULL only when recv_capacity is 0.
 * After an aligned layout (ep_layout_aligned) the pad rows are written too:
 * zero bytes, scale 0, recv_src_token -1, recv_weights 0.
 * Rows >= N (the padded total after an aligned layout) are not written.
 * recv_capacity is the number of rows the receive buffers hold. If it is
 * below the most the routing can need (T*K, plus E*(A-1) when aligned) the
 * call needs N (read once per layout, see above) and returns
 * EP_ERR_CAPACITY, enqueuing nothing, when N > recv_capacity.
 * Returns EP_ERR_INVALID_EXPERT if the handle is known to have seen an
 * invalid expert id.
 */
EP_API ep_status_t ep_dispatch(ep_handle_t handle, const void* x, int H, ep_dtype_t out_dtype,
                        const float* topk_weights,
                        void* recv_x, float* recv_scales, int32_t* recv_src_token,
                        float* recv_weights, int64_t recv_capacity, void* stream);

/*
 * ep_dispatch_ex -- ep_dispatch with the fp8 options of the pages: power-of-two
 * and UE8M0 scales (nccl_ep.cc, ncclEpDispatch: round_scales; DeepEP API docs,
 * "dispatch()": use_ue8m0), a column-major scale layout (DeepEP
 * "dispatch()": use_tma_aligned_col_major_sf), and fp8 input pass-through
 * (DeepEP "dispatch()": x as an (fp8 data, scales) tuple; nccl_ep.cc: fp8
 * tokens with their scales in the high-throughput path), for e4m3 and e5m2
 * (nccl_ep.cc, ncclEpDispatch: fp8 input is either type).
 *
 * With in_dtype = EP_DTYPE_BF16 and fp8 output, each 128-channel block of
 * token t gets s = amax / F (F = 448 for e4m3, 57344 for e5m2 output) and,
 * by scale_mode: FP32 -> scale = s;
 * POW2 -> the smallest power of two >= s; UE8M0 -> that power raised to at
 * least 2^-127 and stored as its exponent byte. Codes are the output
 * format's rne_satfinite(x / scale). An all-zero block has zero codes and
 * scale 0 (UE8M0 byte 0). With fp8 in_dtype (out_dtype must match), x holds
 * codes [T, H] (bytes) and x_scales [T, H/128] (fp32, or bytes in UE8M0
 * mode); both are copied to every slot's row. recv_scales is fp32 (bytes in
 * UE8M0 mode), [cap, H/128] row-major or, with scales_col_major, element
 * (row n, block b) at n + b * scales_ld. Other arguments and errors as ep_dispatch; config may
 * be NULL (bf16 in and out).
 */
EP_API ep_status_t ep_dispatch_ex(ep_handle_t handle, const void* x, const void* x_scales, int H,
                                  const ep_dispatch_config_t* config, const float* topk_weights,
                                  void* recv_x, void* recv_scales, int32_t* recv_src_token,
                                  float* recv_weights, int64_t recv_capacity, void* stream);

/*
 * ep_combine -- weighted top-k gather-reduce back to token order.
 *
 *   out[t, h] = bf16_rne( sum over k = 0..K-1 with row_of_slot[t,k] >= 0 of
 *                         w[t,k] * y[row_of_slot[t,k], h] )
 * accumulated in fp32 with fused multiply-adds in ascending k from +0, and
 * rounded once. topk_weights is fp32 [T, K] (device) or NULL for all-ones.
 * y is bf16 [y_rows, H] (device), out is bf16 [T, H] (device), H % 8 == 0.
 * A token with no valid slot gets +0. If y_rows < T*K the call needs N
 * (read once per layout) and returns EP_ERR_CAPACITY when N > y_rows.
 */
EP_API ep_status_t ep_combine(ep_handle_t handle, const void* y, int64_t y_rows, int H,
                       const float* topk_weights, void* out, void* stream);

/*
 * ep_combine_backward -- gradients of ep_combine (DeepEP API docs, README
 * training snippet: the backward of combine is a dispatch; nccl_ep.cc,
 * ncclEpCombine: its backward mode also reduces the probabilities).
 *
 *   grad_y[row(t,k), h]  = bf16_rne( w[t,k] * grad_out[t, h] )  (fp32 product)
 *   grad_topk_weights[t,k] = sum over h of grad_out[t,h] * y[row(t,k), h]
 *                          (fp32; 0 for dropped slots; a fixed reduction
 *                          order, so repeated calls give the same bits)
 * grad_out is bf16 [T, H]; y is the forward expert output bf16 [y_rows, H]
 * (needed only for grad_topk_weights); topk_weights fp32 [T, K] or NULL (all
 * ones); grad_y bf16 [grad_y_capacity, H] or NULL; grad_topk_weights fp32
 * [T, K] or NULL. After an aligned layout the pad rows of grad_y are zeroed.
 * Buffers smaller than the most rows the routing can need need N (read once
 * per layout) and give EP_ERR_CAPACITY if they hold fewer than N rows.
 */
EP_API ep_status_t ep_combine_backward(ep_handle_t handle, const void* grad_out, const void* y, int64_t y_rows,
                                       int H, const float* topk_weights, void* grad_y,
                                       int64_t grad_y_capacity, float* grad_topk_weights, void* stream);

/*
 * ep_dispatch_backward -- gradients of ep_dispatch (bf16 path): the
 * unweighted combine of the row gradients (DeepEP API docs, README training
 * snippet: the backward of dispatch is a combine),
 *   grad_x[t] = bf16_rne( sum over valid k, ascending, of grad_recv[row(t,k)] ),
 * and, if grad_recv_weights (fp32 [rows], the gradient of recv_weights) is
 * given, grad_topk_weights[t,k] = grad_recv_weights[row(t,k)] (0 if dropped).
 * grad_recv is bf16 [grad_rows, H]; grad_x is bf16 [T, H]. Errors as ep_combine.
 */
EP_API ep_status_t ep_dispatch_backward(ep_handle_t handle, const void* grad_recv, int64_t grad_rows, int H,
                                        const float* grad_recv_weights, void* grad_x, float* grad_topk_weights,
                                        void* stream);

/*
 * ep_topk_to_routing_map -- sparse top-k routing to a dense routing map
 * (nccl_ep.cc: convert_topk_to_routing_map and sparse_to_dense_prob; NeMo
 * fused_a2a, HybridEPDispatch: routing_map [T, E] and probs [T, E]).
 *   routing_map[t, e] = 1 if some slot of token t names expert e, else 0
 *   probs[t, e]       = fp32 sum in ascending k of those slots' weights, else 0
 * topk_idx int64 [T, K] (-1 = unused), topk_weights fp32 [T, K] (needed for
 * probs), routing_map uint8 [T, E], probs fp32 [T, E] or NULL. Every element
 * of the outputs is written. device_error (int32 [1] or NULL) is set to 0, or
 * EP_ERR_INVALID_EXPERT if an id outside [-1, E) was seen (and skipped).
 */
EP_API ep_status_t ep_topk_to_routing_map(const int64_t* topk_idx, const float* topk_weights, int T, int K,
                                          int E, uint8_t* routing_map, float* probs, int32_t* device_error,
                                          void* stream);

/*
 * ep_routing_map_to_topk -- dense routing map to sparse top-k (nccl_ep.cc:
 * dense_to_sparse_prob). The experts e with routing_map[t, e] != 0, in
 * ascending e, fill slots 0, 1, ... of token t; the rest are -1 with weight 0.
 * topk_weights takes probs[t, e] (1 if probs is NULL). device_error (int32
 * [1] or NULL) is set to 0, or EP_ERR_CAPACITY if a token has more than K
 * experts (the first K are kept). The result feeds ep_layout directly.
 */
EP_API ep_status_t ep_routing_map_to_topk(const uint8_t* routing_map, const float* probs, int T, int E, int K,
                                          int64_t* topk_idx, float* topk_weights, int32_t* device_error,
                                          void* stream);

/*
 * ep_handle_query -- synchronous read of the handle's device state after the
 * last layout call: N (receive rows: valid slots, the padded total after
 * ep_layout_aligned, E * capacity after ep_layout_strided) and the device
 * error word (0, EP_ERR_INVALID_EXPERT, or EP_ERR_CAPACITY when a strided
 * layout dropped slots). Synchronises the layout stream on the first read
 * after a layout; later queries return the host copy. Returns the error
 * word's code if it is set (outputs still filled). Either output pointer may
 * be NULL.
 */
EP_API ep_status_t ep_handle_query(ep_handle_t handle, int64_t* num_recv_rows, int32_t* device_error);

/*
 * ep_handle_copy_row_of_slot -- copy the handle's slot -> row map
 * (int32 [T, K], -1 for unused slots) into dst (device, caller-owned),
 * enqueued on stream.
 */
EP_API ep_status_t ep_handle_copy_row_of_slot(ep_handle_t handle, int32_t* dst, void* stream);

/*
 * ep_handle_destroy -- free the handle's device and pinned memory (with its
 * own free hook). Synchronises the device first so no enqueued work still
 * reads it. NULL is a no-op.
 */
EP_API ep_status_t ep_handle_destroy(ep_handle_t handle);

/*
 * ep_handle_layout_kernels -- number of kernels the last ep_layout on this
 * handle enqueued: 1 on the single-cluster path, 3 on the multi-block path,
 * 0 for T = 0 (1 for a strided layout, which still writes its offsets);
 * -1 for a NULL handle. For launch accounting only.
 */
EP_API int ep_handle_layout_kernels(ep_handle_t handle);

/*
 * ep_layout_cluster_ctas -- which path ep_layout (and ep_layout_noalloc)
 * takes for a routing of T tokens, top-K, E experts and R ranks on the
 * current device: the number of CTAs in the thread-block cluster of the
 * single-launch path (up to 16 where the GPU co-schedules 16, else up to 8;
 * small routings take fewer, at least 4, so that each warp holds at most
 * one 32-slot round), or 0 when
 * the routing takes the three-kernel path (more than 2^18 slots, a plan
 * beyond the cluster's shared memory, or more slots per warp than the
 * cluster kernel holds). -1 for invalid arguments or a CUDA error. Enqueues
 * nothing. For tests and launch accounting.
 */
EP_API int ep_layout_cluster_ctas(int T, int K, int E, int R);

/*
 * ep_layout_noalloc -- the routing layout of ep_layout, for callers that
 * cannot allocate device memory.
 *
 * No counterpart on the pages this library follows: it exists for callers
 * whose device memory is all owned by someone else -- for example a serving
 * engine that reserves the GPU's memory for its own pool at start-up and
 * hands out no allocation hook -- or that must not pay cudaMalloc's
 * implicit device synchronisation inside a latency-critical loop. It calls
 * no cudaMalloc, cudaFree, cudaMallocHost or other allocating routine.
 *
 * Instead of a handle it uses one fixed scratch array compiled into the
 * library, EP_NOALLOC_SCRATCH_BYTES (2 MiB) of device memory that every GPU
 * which loads the library keeps until the process exits. The limit is that
 * of the three-kernel layout path, whose tables live there: E * C + R * B +
 * 64 int32 words, where C <= 256 is the number of token chunks and B the
 * number of count blocks (B = C/8 when E <= 2730), so roughly (E + R) * 256
 * words. The single-cluster path uses only the 64 state words, but which
 * path runs is decided at launch from what the GPU can co-schedule, so the
 * check is applied to every routing: one that would need more is rejected
 * with EP_ERR_CAPACITY before anything is enqueued.
 *
 * Arguments and outputs are those of ep_layout, plus:
 *  row_of_slot    device, int32 [T, K]: receive row of each slot, -1 if
 *                 unused (what ep_handle_copy_row_of_slot returns for a
 *                 handle); the caller owns it.
 *  device_error   device, int32 [1] or NULL: set to 0, or to
 *                 EP_ERR_INVALID_EXPERT if an id outside [-1, E) was seen
 *                 (those slots are treated as unused). It is filled by a
 *                 4-byte device-to-device copy enqueued after the layout
 *                 kernels, so a kernel launched next on the stream as a
 *                 programmatic dependent starts after that copy rather than
 *                 overlapping the layout's last wave; pass NULL when that
 *                 overlap matters more than the error word.
 *
 * Calls share the one scratch array, which keeps the last call's contents;
 * each call clears the words that must start at zero. Calls whose work
 * overlaps on the GPU (different streams, or several host threads) race on
 * that array and give wrong results: order them on one stream.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 */
#define EP_NOALLOC_SCRATCH_BYTES (2u << 20)
EP_API ep_status_t ep_layout_noalloc(const int64_t* topk_idx, int T, int K, int E, int R,
                                     int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                     uint8_t* is_token_in_rank, int32_t* expert_offsets,
                                     int32_t* row_of_slot, int32_t* device_error, void* stream);

/* Human-readable name of a status code (static storage). */
EP_API const char* ep_status_string(ep_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_EP_H */
