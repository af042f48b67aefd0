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
// GPU design (three short launches, no host sync, no memset):
//   count  : each warp owns a chunk of consecutive tokens and builds its
//            chunk's expert histogram with warp-aggregated updates
//            (__match_any_sync; one leader lane per distinct expert adds the
//            popcount), writes is_token_in_rank for its tokens and adds per-rank
//            token counts into a block accumulator.
//   scan   : one warp per expert scans that expert's per-chunk counts into
//            per-chunk bases (coalesced loads, warp shuffles) and writes the
//            expert total; extra warps reduce the per-rank counts. Spreading
//            the scan over many SMs keeps it from serialising on L2 latency.
//   assign : every block rebuilds the E expert offsets from the totals with a
//            block scan; each warp then walks its chunk again in (token, k)
//            order, and a slot's row is its expert's running base plus the
//            number of earlier lanes in the same round with the same expert
//            (popc of the match mask below the lane).
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
// (blockDim.x a multiple of 32, at most 32 warps). Returns the total.
// `warp_tmp` holds 33 ints.
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
        const int v = __shfl_up_sync(kFullMask, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) warp_tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < nwarps ? warp_tmp[lane] : 0;
        int s = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int u = __shfl_up_sync(kFullMask, s, d);
            if (lane >= d) s += u;
        }
        if (lane < nwarps) warp_tmp[lane] = s - v;   // exclusive warp bases
        if (lane == 31) warp_tmp[32] = s;           // block total
    }
    __syncthreads();
    int run = warp_tmp[warp] + incl - local;
    for (int i = beg; i < end; ++i) {
        const int v = data[i];
        data[i] = run;
        run += v;
    }
    const int total = warp_tmp[32];
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
        for (int e = lane; e < p.E; e += 32)
            a.chunk_cnt[static_cast<int64_t>(e) * p.num_chunks + chunk] = hist[e];

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
}

// Warps [0, E): exclusive scan (in place) of expert e's per-chunk counts and
// its total. Warps [E, E+R): per-rank token totals. Warp E+R: error word.
__global__ void __launch_bounds__(256)
layout_scan_kernel(LayoutPlan p, LayoutArgs a) {
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw < p.E) {
        int* col = a.chunk_cnt + static_cast<int64_t>(gw) * p.num_chunks;
        int carry = 0;
        for (int c0 = 0; c0 < p.num_chunks; c0 += 128) {
            int v[4];
            int local = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = c0 + lane * 4 + i;
                v[i] = c < p.num_chunks ? col[c] : 0;
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
        if (lane == 0) a.num_tokens_per_expert[gw] = carry;
    } else if (gw < p.E + p.R) {
        const int r = gw - p.E;
        const int32_t* col = a.block_rank + static_cast<int64_t>(r) * p.num_blocks;
        int s = 0;
        for (int b = lane; b < p.num_blocks; b += 32) s += col[b];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) s += __shfl_xor_sync(kFullMask, s, d);
        if (lane == 0) a.num_tokens_per_rank[r] = s;
    } else if (gw == p.E + p.R && lane == 0) {
        // every count block has finished (stream order): publish, then clear
        a.meta[kMetaError] = atomicExch(a.meta + kMetaErrorAccum, 0) ? EP_ERR_INVALID_EXPERT : 0;
    }
}

__global__ void __launch_bounds__(256)
layout_assign_kernel(LayoutPlan p, LayoutArgs a) {
    extern __shared__ int smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int* offs = smem;                                  // [E] exclusive expert offsets
    int* warp_tmp = smem + p.E;                        // [33]
    int* run = smem + p.E + 33 + warp * p.E;           // this warp's running rows
    // every block rebuilds the E offsets from the totals (E <= 4096 values)
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) offs[e] = a.num_tokens_per_expert[e];
    __syncthreads();
    const int n_rows = block_exclusive_scan(offs, p.E, warp_tmp);
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) a.expert_offsets[e] = offs[e];
        if (threadIdx.x == 0) {
            a.expert_offsets[p.E] = n_rows;
            a.meta[kMetaRows] = n_rows;
        }
    }
    const int chunk = blockIdx.x * p.warps_per_block + warp;
    if (chunk >= p.num_chunks) return;
    for (int e = lane; e < p.E; e += 32)
        run[e] = offs[e] + a.chunk_cnt[static_cast<int64_t>(e) * p.num_chunks + chunk];
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
    // keeping the [E][chunks] table small.
    int ct = (T + 255) / 256;
    if (ct < 1) ct = 1;
    p.chunk_tokens = ct;
    p.num_chunks = T > 0 ? (T + ct - 1) / ct : 0;
    int wpb = 8;
    while (wpb > 1 && static_cast<size_t>(wpb + 1) * E * sizeof(int) > 96 * 1024) wpb >>= 1;
    p.warps_per_block = wpb;
    p.num_blocks = p.num_chunks > 0 ? (p.num_chunks + wpb - 1) / wpb : 0;
    p.smem_count = (static_cast<size_t>(wpb) * E + R) * sizeof(int);
    p.smem_assign = (static_cast<size_t>(wpb + 1) * E + 33) * sizeof(int);
    return p;
}

cudaError_t launch_layout(const LayoutPlan& p, const LayoutArgs& a, cudaStream_t stream) {
    // the shared-memory opt-in is per device
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        err = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(layout_assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    if (p.num_blocks == 0) return cudaSuccess;
    const int threads = p.warps_per_block * 32;
    layout_count_kernel<<<p.num_blocks, threads, p.smem_count, stream>>>(p, a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int scan_warps = p.E + p.R + 1;
    layout_scan_kernel<<<(scan_warps + 7) / 8, 256, 0, stream>>>(p, a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    layout_assign_kernel<<<p.num_blocks, threads, p.smem_assign, stream>>>(p, a);
    return cudaGetLastError();
}

}  // namespace ep
