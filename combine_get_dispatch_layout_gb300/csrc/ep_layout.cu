// Routing layout: expert histogram, is_token_in_rank, per-rank token counts,
// exclusive expert offsets and the stable slot -> receive-row map.
//
// What is computed follows nccl_ep.cc (struct ncclEpHandle: is_token_in_rank
// as the outbound [token, rank] mask; num_tokens_for_experts counting a token
// once per destination; -1 for "not routed") and the DeepEP API docs ("Prefix
// Sum Interpretation for Expert Token Counts": expert i owns a contiguous row
// range given by a prefix sum of counts; "dispatch()" with do_expand: one row
// per (token, expert) pair). Rows inside an expert are in ascending (token, k)
// order, which makes the permutation deterministic.
//
// GPU design (two launches, no host sync, no memset):
//   count  : each warp owns a chunk of consecutive tokens and builds its
//            chunk's expert histogram with warp-aggregated updates
//            (__match_any_sync; one leader lane per distinct expert adds the
//            popcount), writes is_token_in_rank for its tokens and adds per-rank
//            token counts into a block accumulator. The last block to finish
//            (atomic ticket, no waiting) scans the [E][chunks] count table
//            per expert with warp shuffles, scans the expert totals across the
//            block, and writes counts, offsets, per-rank totals and N.
//   assign : each warp walks its chunk again in (token, k) order; a slot's row
//            is its expert's running base plus the number of earlier lanes in
//            the same round with the same expert (popc of the match mask below
//            the lane).
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kRoundsInFlight = 4;   // 32-slot rounds whose loads are issued together

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Classify a slot: expert id in [0, E) -> id, -1 or out of range -> -1.
__device__ __forceinline__ int slot_key(int64_t e, int E, bool& bad) {
    bad = (e < -1) || (e >= E);
    return (e >= 0 && e < E) ? static_cast<int>(e) : -1;
}

// Exclusive scan of `n` ints held in shared memory, by the whole block
// (blockDim.x multiple of 32). Returns the total. `warp_tmp` holds >= 32 ints.
__device__ int block_exclusive_scan(int* data, int n, int* warp_tmp) {
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
    const int per = (n + nthreads - 1) / nthreads;
    const int beg = min(n, tid * per), end = min(n, beg + per);
    int local = 0;
    for (int i = beg; i < end; ++i) local += data[i];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int v = __shfl_up_sync(kFullMask, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) warp_tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < nwarps ? warp_tmp[lane] : 0;
        int s = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int u = __shfl_up_sync(kFullMask, s, d);
            if (lane >= d) s += u;
        }
        if (lane < nwarps) warp_tmp[lane] = s - v;   // exclusive warp bases
        if (lane == 31) warp_tmp[32] = s;           // block total
    }
    __syncthreads();
    int run = warp_tmp[warp] + incl - local;
    for (int i = beg; i < end; ++i) {
        int v = data[i];
        data[i] = run;
        run += v;
    }
    int total = warp_tmp[32];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(256)
layout_count_kernel(LayoutPlan p, LayoutArgs a) {
    extern __shared__ int smem[];
    const int wpb = p.warps_per_block;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int* hist = smem + warp * p.E;                 // this warp's chunk histogram
    int* rank_acc = smem + wpb * p.E;              // [R] block's tokens per rank
    int* warp_tmp = rank_acc + p.R;                // [33] scan scratch
    __shared__ int s_is_last;

    for (int e = lane; e < p.E; e += 32) hist[e] = 0;
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) rank_acc[r] = 0;
    __syncthreads();

    const int chunk = blockIdx.x * wpb + warp;
    if (chunk < p.num_chunks) {
        const int t0 = chunk * p.chunk_tokens;
        const int t1 = min(p.T, t0 + p.chunk_tokens);
        const int64_t s0 = static_cast<int64_t>(t0) * p.K, s1 = static_cast<int64_t>(t1) * p.K;
        bool any_bad = false;
        for (int64_t base = s0; base < s1; base += 32 * kRoundsInFlight) {
            int64_t e_r[kRoundsInFlight];
#pragma unroll
            for (int j = 0; j < kRoundsInFlight; ++j) {
                const int64_t s = base + j * 32 + lane;
                e_r[j] = s < s1 ? __ldg(a.topk_idx + s) : -1;
            }
#pragma unroll
            for (int j = 0; j < kRoundsInFlight; ++j) {
                bool bad;
                const int key = slot_key(e_r[j], p.E, bad);
                any_bad |= bad;
                const unsigned peers = __match_any_sync(kFullMask, key);
                if (key >= 0 && lane == __ffs(peers) - 1) hist[key] += __popc(peers);
                __syncwarp();
            }
        }
        if (__any_sync(kFullMask, any_bad) && lane == 0) atomicOr(a.meta + kMetaErrorAccum, 1);

        // expert counts of this chunk -> [E][num_chunks] table
        for (int e = lane; e < p.E; e += 32) a.chunk_cnt[static_cast<int64_t>(e) * p.num_chunks + chunk] = hist[e];

        // is_token_in_rank for the chunk's tokens: pair i = (token, rank), lanes
        // cover consecutive pairs so the byte stores are contiguous.
        const int pairs = (t1 - t0) * p.R;
        for (int i = lane; i < pairs; i += 32) {
            const int tl = i / p.R, r = i - tl * p.R;
            const int64_t* row = a.topk_idx + static_cast<int64_t>(t0 + tl) * p.K;
            const int e_lo = r * p.L, e_hi = e_lo + p.L;
            uint8_t hit = 0;
            for (int k = 0; k < p.K; ++k) {
                const int64_t e = __ldg(row + k);
                hit |= (e >= e_lo && e < e_hi) ? 1 : 0;
            }
            a.is_token_in_rank[static_cast<int64_t>(t0) * p.R + i] = hit;
            if (hit) atomicAdd(rank_acc + r, 1);
        }
    }
    __syncthreads();
    for (int r = threadIdx.x; r < p.R; r += blockDim.x)
        a.block_rank[static_cast<int64_t>(r) * p.num_blocks + blockIdx.x] = rank_acc[r];

    // ---- last block to finish turns the tables into offsets (no waiting) ----
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int ticket = atomicAdd(a.meta + kMetaDone, 1);
        s_is_last = (ticket == p.num_blocks - 1);
    }
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();

    int* tot = smem;   // reuse the histogram area: [E] expert totals
    const int nwarps = blockDim.x >> 5;
    for (int e = warp; e < p.E; e += nwarps) {
        int* col = a.chunk_cnt + static_cast<int64_t>(e) * p.num_chunks;
        int carry = 0;
        for (int c0 = 0; c0 < p.num_chunks; c0 += 128) {
            int v[4];
            int local = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = c0 + lane * 4 + i;
                v[i] = c < p.num_chunks ? __ldcg(col + c) : 0;
                local += v[i];
            }
            int incl = local;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int u = __shfl_up_sync(kFullMask, incl, d);
                if (lane >= d) incl += u;
            }
            int run = carry + incl - local;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = c0 + lane * 4 + i;
                if (c < p.num_chunks) col[c] = run;
                run += v[i];
            }
            carry += __shfl_sync(kFullMask, incl, 31);
        }
        if (lane == 0) tot[e] = carry;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) a.num_tokens_per_expert[e] = tot[e];
    __syncthreads();
    const int n_rows = block_exclusive_scan(tot, p.E, warp_tmp);
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) a.expert_offsets[e] = tot[e];
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
        int s = 0;
        const int32_t* col = a.block_rank + static_cast<int64_t>(r) * p.num_blocks;
        for (int b = 0; b < p.num_blocks; ++b) s += __ldcg(col + b);
        a.num_tokens_per_rank[r] = s;
    }
    if (threadIdx.x == 0) {
        a.expert_offsets[p.E] = n_rows;
        a.meta[kMetaRows] = n_rows;
        a.meta[kMetaError] = atomicExch(a.meta + kMetaErrorAccum, 0) ? EP_ERR_INVALID_EXPERT : 0;
        a.meta[kMetaDone] = 0;   // ready for the next call on this handle
    }
}

__global__ void __launch_bounds__(256)
layout_assign_kernel(LayoutPlan p, LayoutArgs a) {
    extern __shared__ int smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunk = blockIdx.x * p.warps_per_block + warp;
    if (chunk >= p.num_chunks) return;
    int* run = smem + warp * p.E;
    for (int e = lane; e < p.E; e += 32)
        run[e] = __ldcg(a.expert_offsets + e) +
                 __ldcg(a.chunk_cnt + static_cast<int64_t>(e) * p.num_chunks + chunk);
    __syncwarp();

    const int t0 = chunk * p.chunk_tokens;
    const int t1 = min(p.T, t0 + p.chunk_tokens);
    const int64_t s0 = static_cast<int64_t>(t0) * p.K, s1 = static_cast<int64_t>(t1) * p.K;
    const unsigned lt = lanemask_lt();
    for (int64_t base = s0; base < s1; base += 32 * kRoundsInFlight) {
        int64_t e_r[kRoundsInFlight];
#pragma unroll
        for (int j = 0; j < kRoundsInFlight; ++j) {
            const int64_t s = base + j * 32 + lane;
            e_r[j] = s < s1 ? __ldg(a.topk_idx + s) : -1;
        }
#pragma unroll
        for (int j = 0; j < kRoundsInFlight; ++j) {
            bool bad;
            const int key = slot_key(e_r[j], p.E, bad);
            const unsigned peers = __match_any_sync(kFullMask, key);
            int row = -1;
            if (key >= 0) row = run[key] + __popc(peers & lt);
            __syncwarp();
            if (key >= 0 && lane == __ffs(peers) - 1) run[key] += __popc(peers);
            __syncwarp();
            const int64_t s = base + j * 32 + lane;
            if (s < s1) a.row_of_slot[s] = row;
        }
    }
}

}  // namespace

LayoutPlan make_layout_plan(int T, int K, int E, int R) {
    LayoutPlan p{};
    p.T = T; p.K = K; p.E = E; p.R = R; p.L = E / R;
    // About 256 warp-chunks: enough parallelism for a latency-bound pass while
    // keeping the [E][chunks] table the last block scans small.
    int ct = (T + 255) / 256;
    if (ct < 1) ct = 1;
    p.chunk_tokens = ct;
    p.num_chunks = T > 0 ? (T + ct - 1) / ct : 0;
    int wpb = 8;
    while (wpb > 1 && static_cast<size_t>(wpb) * E * sizeof(int) > 96 * 1024) wpb >>= 1;
    p.warps_per_block = wpb;
    p.num_blocks = p.num_chunks > 0 ? (p.num_chunks + wpb - 1) / wpb : 0;
    p.mask_words = (R + 31) / 32;
    p.smem_count = (static_cast<size_t>(wpb) * E + R + 33) * sizeof(int);
    p.smem_assign = static_cast<size_t>(wpb) * E * sizeof(int);
    return p;
}

cudaError_t launch_layout(const LayoutPlan& p, const LayoutArgs& a, cudaStream_t stream) {
    // the shared-memory opt-in is per device
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t derr = cudaGetDevice(&dev);
    if (derr != cudaSuccess) return derr;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e1 = cudaFuncSetAttribute(layout_count_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        cudaError_t e2 = cudaFuncSetAttribute(layout_assign_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e1 != cudaSuccess) return e1;
        if (e2 != cudaSuccess) return e2;
        attr_set[dev] = true;
    }
    if (p.num_blocks == 0) return cudaSuccess;
    const int threads = p.warps_per_block * 32;
    layout_count_kernel<<<p.num_blocks, threads, p.smem_count, stream>>>(p, a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    layout_assign_kernel<<<p.num_blocks, threads, p.smem_assign, stream>>>(p, a);
    return cudaGetLastError();
}

}  // namespace ep
