// Routing layout: expert histogram, is_token_in_rank, per-rank token counts,
// exclusive expert offsets and the stable slot -> receive-row map.
//
// What is computed follows nccl_ep.cc (struct ncclEpHandle: is_token_in_rank
// as the outbound [token, rank] mask; num_tokens_for_experts counting a token
// once per destination; -1 for "not routed") and the DeepEP API docs ("Prefix
// Sum Interpretation for Expert Token Counts": expert i owns a contiguous row
// range given by a prefix sum of counts; "dispatch()" with do_expand: one row
// per (token, expert) pair; expert_alignment: each expert's rows start on a
// multiple of the alignment, its real rows first and pad rows after). Rows
// inside an expert are in ascending (token, k) order, which makes the
// permutation deterministic.
//
// GPU design for large routings (three short launches, each a programmatic
// dependent of the one before; no host sync, no memset):
//   count  : each warp owns a chunk of consecutive tokens and builds its
//            chunk's expert histogram with warp-aggregated updates
//            (lanes with the same expert found with one ballot per key bit;
//            one leader lane per distinct expert adds the popcount), writes is_token_in_rank for its tokens and adds per-rank
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
// Small routings (the usual case) take a single-launch path instead: one
// thread-block cluster of up to 16 CTAs runs the same three phases with the
// per-warp histograms in shared memory, exchanges the per-CTA expert totals
// through distributed shared memory, and separates the phases with hardware
// cluster barriers. That needs no global scratch and replaces three
// dependent launches with one.
#include <algorithm>

#include <cooperative_groups.h>

#include <map>
#include <mutex>
#include <utility>

#include "ep_internal.cuh"

namespace cg = cooperative_groups;

namespace ep {

namespace {

constexpr int kRoundsInFlight = 4;   // 32-slot rounds whose loads are issued together
constexpr int kMaxKeyBits = 13;      // E + 1 <= 4097 distinct keys (EP_MAX_EXPERTS = 4096)
constexpr size_t kClusterSmemBudget = 200 * 1024;
constexpr int kMaxClusterCtas = 16;
constexpr int kMaxRounds = 16;       // cluster path: slots per warp <= 16 * 32
constexpr int kSmallRounds = 8;      // up to this many rounds keys and ranks stay unpacked
constexpr int64_t kClusterMaxSlots = int64_t{1} << 18;   // larger routings use the multi-block path

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Lanes whose key equals this lane's key (key in [-1, 2^nbits - 1)), built
// from one ballot per key bit: a lane is a peer if it agrees on every bit.
// In a one-CTA timing of the layout this was about 20% faster than
// __match_any_sync.
__device__ __forceinline__ unsigned peer_mask(int key, int nbits) {
    const unsigned k = static_cast<unsigned>(key + 1);   // 0 = unused slot
    unsigned peers = kFullMask;
#pragma unroll
    for (int b = 0; b < kMaxKeyBits; ++b) {
        if (b < nbits) {
            const bool bit = (k >> b) & 1u;
            const unsigned bal = __ballot_sync(kFullMask, bit);
            peers &= bit ? bal : ~bal;
        }
    }
    return peers;
}

__device__ __forceinline__ int round_up_to(int v, int a) { return (v + a - 1) / a * a; }

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
    dependent_entry();
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
            const int nr = static_cast<int>(min(static_cast<int64_t>(kRoundsInFlight), (s1 - base + 31) / 32));
#pragma unroll
            for (int j = 0; j < kRoundsInFlight; ++j) {
                if (j >= nr) break;   // uniform: rounds past the chunk end hold no slots
                bool bad;
                const int key = slot_key(e_r[j], p.E, bad);
                any_bad |= bad;
                const unsigned peers = peer_mask(key, p.key_bits);
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
#pragma unroll 8
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
    dependent_entry();
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
    dependent_entry();
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ int smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int* offs = smem;                                  // [E] exclusive expert offsets
    int* warp_tmp = smem + p.E;                        // [33]
    int* run = smem + p.E + 33 + warp * p.E;           // this warp's running rows
    // every block rebuilds the E offsets from the totals (E <= 4096 values)
    __shared__ int s_over;
    if (threadIdx.x == 0) s_over = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        const int c = a.num_tokens_per_expert[e];
        offs[e] = p.stride > 0 ? c : round_up_to(c, p.align);
        if (p.stride > 0 && c > p.stride) s_over = 1;
        if (blockIdx.x == 0 && a.h_counts) a.h_counts[e] = c;
    }
    __syncthreads();
    int n_rows = block_exclusive_scan(offs, p.E, warp_tmp);
    if (p.stride > 0) {
        // fixed stride: expert e's block starts at e * stride
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) offs[e] = e * p.stride;
        n_rows = p.E * p.stride;
        __syncthreads();
        // the scan kernel wrote the invalid-id word; a capacity overflow adds to it
        if (blockIdx.x == 0 && threadIdx.x == 0 && s_over && a.meta[kMetaError] == 0)
            a.meta[kMetaError] = EP_ERR_CAPACITY;
    }
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
            a.expert_offsets[e] = offs[e];
            if (a.h_offsets) a.h_offsets[e] = offs[e];
        }
        if (threadIdx.x == 0) {
            a.expert_offsets[p.E] = n_rows;
            if (a.h_offsets) a.h_offsets[p.E] = n_rows;
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
        const int nr = static_cast<int>(min(static_cast<int64_t>(kRoundsInFlight), (s1 - base + 31) / 32));
#pragma unroll
        for (int j = 0; j < kRoundsInFlight; ++j) {
            if (j >= nr) break;
            bool bad;
            const int key = slot_key(e_r[j], p.E, bad);
            const unsigned peers = peer_mask(key, p.key_bits);
            int row = -1;
            if (key >= 0) {
                row = run[key] + __popc(peers & lt);
                if (p.stride > 0 && row - key * p.stride >= p.stride) row = -1;   // past the expert's capacity
            }
            __syncwarp();
            if (key >= 0 && lane == __ffs(peers) - 1) run[key] += __popc(peers);
            __syncwarp();
            const int64_t s = base + j * 32 + lane;
            if (s < s1) a.row_of_slot[s] = row;
        }
    }
}

// Exclusive scan of n ints in shared memory by one warp (lane l owns a
// contiguous run). Returns the total to every lane.
__device__ int warp_exclusive_scan(int* data, int n, int lane) {
    const int per = (n + 31) / 32;
    const int beg = min(n, lane * per), end = min(n, beg + per);
    int local = 0;
    for (int i = beg; i < end; ++i) local += data[i];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(kFullMask, incl, d);
        if (lane >= d) incl += v;
    }
    int run = incl - local;
    for (int i = beg; i < end; ++i) {
        const int v = data[i];
        data[i] = run;
        run += v;
    }
    return __shfl_sync(kFullMask, incl, 31);
}

// Rank of expert e (e / L) by multiply-high with magic = ceil(2^32 / L);
// exact for e * L < 2^32, far beyond EP_MAX_EXPERTS.
__device__ __forceinline__ unsigned rank_of(unsigned e, const LayoutPlan& p) {
    return p.L == 1 ? e : __umulhi(e, p.l_magic);
}

// Single-launch layout by one cluster of p.cl_ctas CTAs, p.cl_warps warps each.
// Warp g (CTA-major) owns tokens [g*ct, (g+1)*ct), at most kRounds rounds
// of 32 slots, whose keys and stable local ranks stay in registers: as two
// arrays for up to kSmallRounds rounds, else packed one per round as
// (key + 1) | (local rank << 13) (keys take 13 bits for E <= 4096, local
// ranks 9 for at most 512 slots a warp), which fits 16 rounds in the same
// registers.
// Shared memory (ints, sized for 16 CTAs): hist[W][E] | all_tot[16][E] |
// all_rank[16][R] | all_bad[16] | tail[max(W * ct_cap, 2E)], where the tail
// holds the token rank masks (R <= 32) and later the offsets and CTA bases.
// With E no larger than the CTA's thread count (and no fixed stride) each
// thread owns one expert in the offset scan, which then runs in registers.
template <int kRounds>
__global__ void __launch_bounds__(1024, 1)
layout_cluster_kernel(LayoutPlan p, LayoutArgs a) {
    constexpr bool kPacked = kRounds > kSmallRounds;
    // Launched as the preceding kernel's programmatic dependent: it zeroes
    // its own shared memory, then waits for that kernel (and so for all
    // earlier work) before touching global memory; only then may a dispatch
    // launched as this grid's dependent start on idle SMs (it reads the slot
    // map only after this grid has finished).
    extern __shared__ int smem[];
    __shared__ int s_over;
    __shared__ int s_scan[32];
    cg::cluster_group cluster = cg::this_cluster();
    const int cta = static_cast<int>(cluster.block_rank());
    const int C = p.cl_ctas, W = p.cl_warps, E = p.E, R = p.R, ct = p.cl_chunk_tokens;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int* hist = smem;                              // counts, then the warp's base in the CTA
    int* all_tot = hist + W * E;                   // [C][E] every CTA's expert totals (pushed)
    int* all_rank = all_tot + C * E;               // [C][R] every CTA's tokens per rank
    int* all_bad = all_rank + C * R;               // [C] every CTA's invalid-id flag
    int* tail = all_bad + kMaxClusterCtas;
    unsigned* tokmask = reinterpret_cast<unsigned*>(tail);   // [W][ct] token rank bitmasks
    int* mine = hist + warp * E;
    unsigned* my_mask = tokmask + warp * ct;
    const bool small_r = R <= 32;

    // Peers write into this CTA's shared memory later; that is only allowed
    // once every CTA of the cluster runs, so arrive now and wait before the
    // first remote store (by then every CTA has long started).
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // this CTA's own shared state, zeroed before the wait for the preceding
    // kernel (nothing here is memory that kernel could write)
    int* rank_acc = all_rank + cta * R;   // this CTA's tokens per rank until the push
    for (int e = lane; e < E; e += 32) mine[e] = 0;
    if (small_r)
        for (int i = lane; i < ct; i += 32) my_mask[i] = 0u;
    for (int r = threadIdx.x; r < R; r += blockDim.x) rank_acc[r] = 0;
    if (threadIdx.x == 0) {
        all_bad[cta] = 0;   // own entry only: peers write their own
        s_over = 0;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    // ---- phase 1: stable local ranks, the warp's histogram, token rank masks
    const int g = cta * W + warp;
    const int t0 = min(p.T, g * ct);
    const int t1 = min(p.T, t0 + ct);
    const int64_t s0 = static_cast<int64_t>(t0) * p.K, s1 = static_cast<int64_t>(t1) * p.K;
    const int nr = static_cast<int>((s1 - s0 + 31) / 32);   // <= kRounds (host check)
    const unsigned lt = lanemask_lt();
    int key_r[kPacked ? 1 : kRounds], loc_r[kPacked ? 1 : kRounds];
    unsigned kl_r[kPacked ? kRounds : 1];
    bool any_bad = false;
#pragma unroll
    for (int j0 = 0; j0 < kRounds; j0 += kRoundsInFlight) {
        if (j0 >= nr) break;
        int64_t e_r[kRoundsInFlight];
#pragma unroll
        for (int j = 0; j < kRoundsInFlight; ++j) {
            const int64_t s = s0 + (j0 + j) * 32 + lane;
            e_r[j] = s < s1 ? __ldg(a.topk_idx + s) : -1;
        }
#pragma unroll
        for (int j = 0; j < kRoundsInFlight; ++j) {
            if (j0 + j >= nr) break;
            bool bad;
            const int key = slot_key(e_r[j], E, bad);
            any_bad |= bad;
            const unsigned peers = peer_mask(key, p.key_bits);
            int loc = -1;
            if (key >= 0) {
                loc = mine[key] + __popc(peers & lt);
                if (small_r) {
                    // (a butterfly OR over each token's lane group measured slower)
                    const int tl = static_cast<int>((s0 + (j0 + j) * 32 + lane) / p.K) - t0;
                    atomicOr(my_mask + tl, 1u << rank_of(static_cast<unsigned>(key), p));
                }
            }
            __syncwarp();
            if (key >= 0 && lane == __ffs(peers) - 1) mine[key] += __popc(peers);
            __syncwarp();
            if constexpr (kPacked) {
                kl_r[j0 + j] = key >= 0 ? (static_cast<unsigned>(key + 1) | (static_cast<unsigned>(loc) << 13)) : 0u;
            } else {
                key_r[j0 + j] = key;
                loc_r[j0 + j] = loc;
            }
        }
    }
    const bool warp_bad = __any_sync(kFullMask, any_bad);

    // is_token_in_rank and this warp's tokens per rank (lane r counts rank r)
    int my_rank_cnt = 0;
    if (small_r) {
        for (int tb = 0; tb < t1 - t0; tb += 32) {
            const int tl = tb + lane;
            const unsigned mask = tl < t1 - t0 ? my_mask[tl] : 0u;
            if (tl < t1 - t0) {
                uint8_t* dst = a.is_token_in_rank + static_cast<int64_t>(t0 + tl) * R;
                if (p.itr_words) {
                    for (int w = 0; w < R / 4; ++w) {
                        const unsigned m4 = mask >> (4 * w);
                        reinterpret_cast<unsigned*>(dst)[w] =
                            (m4 & 1u) | ((m4 >> 1 & 1u) << 8) | ((m4 >> 2 & 1u) << 16) | ((m4 >> 3 & 1u) << 24);
                    }
                } else {
                    for (int r = 0; r < R; ++r) dst[r] = (mask >> r) & 1u;
                }
            }
            for (int r = 0; r < R; ++r) {
                const int c = __popc(__ballot_sync(kFullMask, (mask >> r) & 1u));
                if (lane == r) my_rank_cnt += c;
            }
        }
    }
    if (small_r) {
        if (lane < R && my_rank_cnt) atomicAdd(rank_acc + lane, my_rank_cnt);
    } else {
        const int pairs = (t1 - t0) * R;
        for (int i = lane; i < pairs; i += 32) {
            const int tl = i / R, r = i - tl * R;
            const int64_t* row = a.topk_idx + static_cast<int64_t>(t0 + tl) * p.K;
            const int e_lo = r * p.L, e_hi = e_lo + p.L;
            uint8_t hit = 0;
#pragma unroll 8
            for (int k = 0; k < p.K; ++k) {
                const int64_t e = __ldg(row + k);
                hit |= (e >= e_lo && e < e_hi) ? 1 : 0;
            }
            a.is_token_in_rank[static_cast<int64_t>(t0) * R + i] = hit;
            if (hit) atomicAdd(rank_acc + r, 1);
        }
    }
    if (warp_bad && lane == 0) all_bad[cta] = 1;   // only ever set: peers read after the barrier
    __syncthreads();

    // ---- phase 2: per-warp bases inside the CTA; push this CTA's totals,
    // rank counts and error flag into every CTA of the cluster
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // all CTAs have started
    int* own_tot = all_tot + cta * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int w0 = 0; w0 < W; w0 += 8) {   // W is a multiple of 8
            int c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = hist[(w0 + i) * E + e];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                hist[(w0 + i) * E + e] = run;
                run += c[i];
            }
        }
        own_tot[e] = run;
    }
    __syncthreads();
    // push this CTA's row of totals into every peer: one remote store per
    // (piece, peer), 16-byte pieces when E % 4 == 0
    if (E % 4 == 0) {
        const int pieces = E / 4;
        for (int i = threadIdx.x; i < pieces * C; i += blockDim.x) {
            const int c = i / pieces, q = i - c * pieces;
            if (c == cta) continue;
            const int4 v = reinterpret_cast<const int4*>(own_tot)[q];
            *reinterpret_cast<int4*>(cluster.map_shared_rank(own_tot + 4 * q, c)) = v;
        }
    } else {
        for (int i = threadIdx.x; i < E * C; i += blockDim.x) {
            const int c = i / E, e = i - c * E;
            if (c != cta) *cluster.map_shared_rank(own_tot + e, c) = own_tot[e];
        }
    }
    for (int i = threadIdx.x; i < (R + 1) * C; i += blockDim.x) {
        const int c = i / (R + 1), k = i - c * (R + 1);
        if (c == cta) continue;
        if (k < R) *cluster.map_shared_rank(all_rank + cta * R + k, c) = rank_acc[k];
        else *cluster.map_shared_rank(all_bad + cta, c) = all_bad[cta];
    }
    // Every push lands before any CTA passes this barrier (release/acquire at
    // cluster scope), and nothing touches another CTA's shared memory after
    // it, so CTAs may finish independently.
    cluster.sync();

    // ---- phase 3 (local): expert totals, this CTA's base per expert and the
    // expert offsets
    int* offs = tail;          // the token masks are consumed: reuse the tail
    int* cta_base = tail + E;
    // the last CTA takes the rank totals and the error word, CTA 0 the
    // counts and offsets, so that no CTA carries both
    if (cta == C - 1)
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            int total = 0;
            for (int c = 0; c < C; ++c) total += all_rank[c * R + r];
            a.num_tokens_per_rank[r] = total;
        }
    if (p.stride == 0 && E <= static_cast<int>(blockDim.x)) {
        // one expert per thread: its padded row count is scanned in registers
        // (shuffles inside each warp, then the warp sums), no serial pass
        const int e = threadIdx.x;
        int v = 0;
        if (e < E) {
            int below = 0, total = 0;
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) {
                const int x = c < C ? all_tot[c * E + e] : 0;
                below += c < cta ? x : 0;
                total += x;
            }
            cta_base[e] = below;
            v = round_up_to(total, p.align);
            if (cta == 0) {
                a.num_tokens_per_expert[e] = total;
                if (a.h_counts) a.h_counts[e] = total;
            }
        }
        int incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int u = __shfl_up_sync(kFullMask, incl, d);
            if (lane >= d) incl += u;
        }
        if (lane == 31) s_scan[warp] = incl;
        __syncthreads();
        const int nw = static_cast<int>(blockDim.x >> 5);
        const int ws = lane < nw ? s_scan[lane] : 0;
        int wincl = ws;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int u = __shfl_up_sync(kFullMask, wincl, d);
            if (lane >= d) wincl += u;
        }
        const int wbase = __shfl_sync(kFullMask, wincl - ws, warp);
        const int n_rows = __shfl_sync(kFullMask, wincl, nw - 1);
        if (e < E) {
            const int o = wbase + incl - v;
            offs[e] = o;
            if (cta == 0) {
                a.expert_offsets[e] = o;
                if (a.h_offsets) a.h_offsets[e] = o;
            }
        }
        if (threadIdx.x == 0) {
            if (cta == 0) {
                a.expert_offsets[E] = n_rows;
                if (a.h_offsets) a.h_offsets[E] = n_rows;
                a.meta[kMetaRows] = n_rows;
            }
            if (cta == C - 1) {
                int bad = 0;
                for (int c = 0; c < C; ++c) bad |= all_bad[c];
                a.meta[kMetaError] = bad ? EP_ERR_INVALID_EXPERT : 0;
            }
        }
        __syncthreads();
    } else {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int below = 0, total = 0;
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) {
                const int v = c < C ? all_tot[c * E + e] : 0;
                below += c < cta ? v : 0;
                total += v;
            }
            cta_base[e] = below;
            offs[e] = p.stride > 0 ? e * p.stride : round_up_to(total, p.align);
            if (p.stride > 0 && total > p.stride) s_over = 1;
            if (cta == 0) {
                a.num_tokens_per_expert[e] = total;
                if (a.h_counts) a.h_counts[e] = total;
            }
        }
        __syncthreads();
        if (cta == C - 1 && threadIdx.x == 0) {
            int bad = 0;
            for (int c = 0; c < C; ++c) bad |= all_bad[c];
            a.meta[kMetaError] = bad ? EP_ERR_INVALID_EXPERT : (s_over ? EP_ERR_CAPACITY : 0);
        }
        if (p.stride > 0) {
            if (cta == 0 && threadIdx.x == 0) {
                a.expert_offsets[E] = E * p.stride;
                if (a.h_offsets) a.h_offsets[E] = E * p.stride;
                a.meta[kMetaRows] = E * p.stride;
            }
        } else if (warp == 0) {
            const int n_rows = warp_exclusive_scan(offs, E, lane);
            if (cta == 0 && lane == 0) {
                a.expert_offsets[E] = n_rows;
                if (a.h_offsets) a.h_offsets[E] = n_rows;
                a.meta[kMetaRows] = n_rows;
            }
        }
        __syncthreads();
        if (cta == 0)
            for (int e = threadIdx.x; e < E; e += blockDim.x) {
                a.expert_offsets[e] = offs[e];
                if (a.h_offsets) a.h_offsets[e] = offs[e];
            }
    }

    // ---- phase 4: row = expert offset + rows in lower CTAs + rows in lower
    // warps of this CTA + the slot's local rank
#pragma unroll
    for (int j = 0; j < kRounds; ++j) {
        if (j >= nr) break;
        const int64_t s = s0 + j * 32 + lane;
        int key, loc;
        if constexpr (kPacked) {
            key = static_cast<int>(kl_r[j] & 0x1fffu) - 1;
            loc = static_cast<int>(kl_r[j] >> 13);
        } else {
            key = key_r[j];
            loc = loc_r[j];
        }
        int row = -1;
        if (key >= 0) {
            const int local = cta_base[key] + mine[key] + loc;   // rank inside the expert
            row = (p.stride > 0 && local >= p.stride) ? -1 : offs[key] + local;
        }
        if (s < s1) a.row_of_slot[s] = row;
    }
}

}  // namespace

// A strided layout of no tokens still spans E * stride rows: expert e's rows
// start at e * stride (the counts are zero, the error word stays clear).
__global__ void strided_empty_kernel(int32_t* expert_offsets, int32_t* h_offsets, int32_t* meta, int E,
                                     int stride) {
    dependent_entry();
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e <= E; e += gridDim.x * blockDim.x) {
        expert_offsets[e] = e * stride;
        if (h_offsets) h_offsets[e] = e * stride;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) meta[kMetaRows] = E * stride;
}

cudaError_t launch_strided_empty(int32_t* expert_offsets, int32_t* h_offsets, int32_t* meta, int E, int stride,
                                 cudaStream_t stream) {
    return launch_dependent(strided_empty_kernel, dim3((E + 256) / 256), dim3(256), 0, stream, expert_offsets,
                            h_offsets, meta, E, stride);
}

LayoutPlan make_layout_plan(int T, int K, int E, int R) {
    LayoutPlan p{};
    p.T = T; p.K = K; p.E = E; p.R = R; p.L = E / R;
    p.align = 1;
    p.stride = 0;
    p.key_bits = 1;
    while ((1 << p.key_bits) < E + 1) ++p.key_bits;   // keys -1..E-1 shift to 0..E
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
    // single-cluster geometry (CTA count fixed at launch), warps per CTA
    // counted on a 16-CTA cluster: 8 while that gives each warp at most one
    // 32-slot round, else 16, doubling (to 32) while a warp would have more
    // than about four rounds; fewer if shared memory does not fit, and
    // smem_cluster = 0 disables the path. Graph-chained layouts (top-8): 16
    // warps beat 8 at T=1024 and 2048 by 0.3 and 0.7 us, 8 stay best below,
    // 32 at 2^16 slots.
    const int64_t slots = static_cast<int64_t>(T) * K;
    int cw = slots > static_cast<int64_t>(16) * 8 * 32 ? 16 : 8;
    while (cw < 32 && slots > static_cast<int64_t>(16) * cw * 32 * kRoundsInFlight) cw <<= 1;
    auto cluster_smem = [&](int w) {
        const size_t ct_cap = static_cast<size_t>(kMaxRounds * 32 / K);
        const size_t tail = std::max(static_cast<size_t>(w) * ct_cap, static_cast<size_t>(2 * E));
        return (static_cast<size_t>(w + kMaxClusterCtas) * E + kMaxClusterCtas * (R + 1) + tail) * sizeof(int);
    };
    while (cw > 8 && cluster_smem(cw) > kClusterSmemBudget) cw >>= 1;
    p.cl_warps = cw;
    p.cl_ctas = 0;
    p.cl_chunk_tokens = 0;
    p.smem_cluster = cluster_smem(cw) <= kClusterSmemBudget ? cluster_smem(cw) : 0;
    p.l_magic = p.L > 1 ? static_cast<unsigned>(((uint64_t{1} << 32) + p.L - 1) / p.L) : 0u;
    p.itr_words = 0;
    return p;
}

namespace {

// Per-device launch state, shared by every handle and host thread.
struct DeviceLaunchState {
    bool attrs_set = false;
    std::map<std::pair<int, size_t>, int> cluster_ctas;   // (warps, smem) -> CTAs, 0 = none
};
std::mutex g_launch_mu;
DeviceLaunchState g_launch_state[64];

// Opt-ins the layout kernels need, set once per device (the current one):
// dynamic shared memory up to the largest any plan uses, and cluster sizes
// above the portable 8.
cudaError_t set_kernel_attributes(DeviceLaunchState& st) {
    if (st.attrs_set) return cudaSuccess;
    const int budget = static_cast<int>(kClusterSmemBudget);
    cudaError_t err = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, budget);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(layout_assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, budget);
    for (auto kernel : {layout_cluster_kernel<kSmallRounds>, layout_cluster_kernel<kMaxRounds>}) {
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, budget);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    if (err == cudaSuccess) st.attrs_set = true;
    return err;
}

// Largest cluster (16, else 8) that the device can co-schedule for the
// single-launch kernel with the given block; 0 if none. Cached.
int cluster_ctas_for(DeviceLaunchState& st, int warps, size_t smem) {
    const auto key = std::make_pair(warps, smem);
    const auto it = st.cluster_ctas.find(key);
    if (it != st.cluster_ctas.end()) return it->second;
    int found = 0;
    for (int c : {16, 8}) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c);
        cfg.blockDim = dim3(warps * 32);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = c;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, layout_cluster_kernel<kMaxRounds>, &cfg) == cudaSuccess && n > 0) {
            found = c;
            break;
        }
    }
    cudaGetLastError();   // a refused probe must not leak into the caller's error state
    st.cluster_ctas[key] = found;
    return found;
}

// The single-launch geometry for `plan` on the current device: CTAs per
// cluster (0 = the routing takes the three-kernel path) and tokens per warp.
cudaError_t choose_cluster(const LayoutPlan& plan, int* ctas_out, int* chunk_tokens_out) {
    *ctas_out = 0;
    *chunk_tokens_out = 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int ctas = 0;
    const int64_t slots = static_cast<int64_t>(plan.T) * plan.K;
    const bool try_cluster = slots <= kClusterMaxSlots && plan.smem_cluster > 0;
    {
        std::lock_guard<std::mutex> lock(g_launch_mu);
        DeviceLaunchState& st = g_launch_state[dev];
        err = set_kernel_attributes(st);
        if (err != cudaSuccess) return err;
        if (try_cluster && plan.num_blocks > 0) ctas = cluster_ctas_for(st, plan.cl_warps, plan.smem_cluster);
    }
    if (!try_cluster || ctas == 0) return cudaSuccess;
    // A small routing takes fewer CTAs: the smallest power of two (at least
    // 4) that gives each warp at most one 32-slot round. Fewer CTAs mean
    // fewer shared-memory pushes to wait for at the cluster barrier.
    // Graph-chained layout / warm step, E=256 top-8: at T=256 (2048 slots)
    // 8 CTAs took 3.90 / 12.59 us against 4.43 / 13.65 with 16; at T=64,
    // 4 CTAs 3.69 / 8.30 against 4.00 / 8.81; 1024 tokens and more stay at 16.
    {
        const int64_t per_cta = static_cast<int64_t>(plan.cl_warps) * 32;
        int want = 4;
        while (want < ctas && static_cast<int64_t>(want) * per_cta < slots) want <<= 1;
        if (want < ctas) ctas = want;
    }
    const int warps = ctas * plan.cl_warps;
    const int ct = (plan.T + warps - 1) / warps;
    // each warp's chunk must fit kMaxRounds rounds (and the token-mask area)
    if (static_cast<int64_t>(ct) * plan.K > kMaxRounds * 32) return cudaSuccess;
    *ctas_out = ctas;
    *chunk_tokens_out = ct;
    return cudaSuccess;
}

}  // namespace

int layout_cluster_ctas(const LayoutPlan& plan) {
    int ctas = 0, ct = 0;
    return choose_cluster(plan, &ctas, &ct) == cudaSuccess ? ctas : -1;
}

cudaError_t launch_layout(const LayoutPlan& plan, const LayoutArgs& a, cudaStream_t stream, int* kernels) {
    if (kernels) *kernels = 0;
    int ctas = 0, ct = 0;
    cudaError_t err = choose_cluster(plan, &ctas, &ct);
    if (err != cudaSuccess) return err;
    if (plan.num_blocks == 0) return cudaSuccess;

    if (ctas > 0) {
        LayoutPlan p = plan;
        p.cl_ctas = ctas;
        p.cl_chunk_tokens = ct;
        p.itr_words = (p.R % 4 == 0 && reinterpret_cast<uintptr_t>(a.is_token_in_rank) % 4 == 0) ? 1 : 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(ctas);
        cfg.blockDim = dim3(p.cl_warps * 32);
        cfg.dynamicSmemBytes = p.smem_cluster;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = ctas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        // may be scheduled while the preceding kernel drains; it waits for
        // that kernel before its first memory access
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        if (kernels) *kernels = 1;
        // the unpacked instance while each warp needs at most kSmallRounds rounds
        if (static_cast<int64_t>(ct) * plan.K <= kSmallRounds * 32)
            return cudaLaunchKernelEx(&cfg, layout_cluster_kernel<kSmallRounds>, p, a);
        return cudaLaunchKernelEx(&cfg, layout_cluster_kernel<kMaxRounds>, p, a);
    }

    const int threads = plan.warps_per_block * 32;
    if (kernels) *kernels = 3;
    err = launch_dependent(layout_count_kernel, dim3(plan.num_blocks), dim3(threads), plan.smem_count, stream, plan, a);
    if (err != cudaSuccess) return err;
    const int scan_warps = plan.E + plan.R + 1;
    err = launch_dependent(layout_scan_kernel, dim3((scan_warps + 7) / 8), dim3(256), 0, stream, plan, a);
    if (err != cudaSuccess) return err;
    return launch_dependent(layout_assign_kernel, dim3(plan.num_blocks), dim3(threads), plan.smem_assign, stream, plan,
                            a);
}

}  // namespace ep
