// Conversions between sparse top-k routing (topk_idx / topk_weights [T, K])
// and a dense routing map with probabilities (routing_map / probs [T, E]).
//
// nccl_ep.cc converts top-k indices to a per-token routing map
// (convert_topk_to_routing_map) and probabilities between the two forms
// (sparse_to_dense_prob, dense_to_sparse_prob); NeMo fused_a2a's
// HybridEPDispatch takes routing_map [T, E] bool and probs [T, E]. Reading:
// the dense-to-sparse direction lists a token's experts in ascending id, and
// a dense probability is the fp32 sum, in ascending k, of the weights of the
// slots naming that expert.
//
// GPU design (scalar forms): one warp per token. topk -> map: lane k holds slot k, every
// lane owns experts lane, lane + 32, ... and tests them against the K
// broadcast slots, so the byte and fp32 rows are written coalesced.
// map -> topk: each 32-expert chunk is one ballot; a set bit's slot is the
// count of set bits before it.
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kConvWarps = 8;

// log2 of the lanes serving one token in the vector forms: the power of two
// >= E / 8, at most 32.
inline int lanes_per_token_log2(int E) {
    int gs = 0;
    while (gs < 5 && (8 << gs) < E) ++gs;
    return gs;
}

// Vector forms (E % 8 == 0, map rows 8-byte and probs rows 16-byte aligned):
// a token is served by G lanes (G = the power of two >= E / 8, at most 32;
// a warp serves 32 / G tokens), lane g owning experts 8g .. 8g+7 of each
// block of 8G experts. topk -> map: the K slots are broadcast within the
// group by width-G shuffles (lanes read them themselves when K > G), and a
// lane writes one 8-byte map store and two 16-byte probs stores per block. map -> topk: a
// lane loads its 8 map bytes and 8 probs together, and the routed experts
// are placed by a G-wide prefix scan. Same arithmetic as the scalar forms
// below (which serve the other shapes): probabilities are summed from +0 in
// ascending k; experts are listed in ascending id.
__global__ void __launch_bounds__(kConvWarps * 32)
topk_to_routing_map_vec_kernel(const int64_t* topk_idx, const float* w, int T, int K, int E, int gs,
                               uint8_t* routing_map, float* probs, int32_t* device_error) {
    dependent_entry();
    const int G = 1 << gs;   // lanes per token
    const int lane = threadIdx.x & 31, gl = lane & (G - 1);
    const int t = ((blockIdx.x * kConvWarps + (threadIdx.x >> 5)) << (5 - gs)) + (lane >> gs);
    const bool active = t < T;   // inactive lanes still take part in the shuffles
    const int64_t* ids = topk_idx + static_cast<int64_t>(t) * K;
    const float* wts = w ? w + static_cast<int64_t>(t) * K : nullptr;
    // K <= G: lane g of the group holds slot g and broadcasts it (width-G
    // shuffles); otherwise every lane reads the K slots itself
    const bool bcast = K <= G;
    int my_key = -1;
    float my_w = 0.0f;
    if (active && bcast && gl < K) {
        const int64_t e = __ldg(ids + gl);
        if (e < -1 || e >= E) {
            if (device_error) atomicExch(device_error, EP_ERR_INVALID_EXPERT);
        } else {
            my_key = static_cast<int>(e);
        }
        if (wts) my_w = __ldg(wts + gl);
    }
    if (active && !bcast && gl == 0 && device_error) {
        bool bad = false;
        for (int k = 0; k < K; ++k) {
            const int64_t e = __ldg(ids + k);
            bad |= e < -1 || e >= E;
        }
        if (bad) atomicExch(device_error, EP_ERR_INVALID_EXPERT);
    }
    for (int e0 = 0; e0 < E; e0 += 8 * G) {
        const int eb = e0 + 8 * gl;
        const bool mine = active && eb < E;
        unsigned lo = 0u, hi = 0u;
        float p[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) p[q] = 0.0f;
        for (int k = 0; k < K; ++k) {
            int ek;
            float wk;
            if (bcast) {
                ek = __shfl_sync(kFullMask, my_key, k, G);
                wk = __shfl_sync(kFullMask, my_w, k, G);
            } else {
                const int64_t e = mine ? __ldg(ids + k) : -1;
                ek = (e >= 0 && e < E) ? static_cast<int>(e) : -1;
                wk = (mine && wts) ? __ldg(wts + k) : 0.0f;
            }
            const int j = ek - eb;
            if (mine && ek >= 0 && j >= 0 && j < 8) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q == j) p[q] = p[q] + wk;
                if (j < 4) lo |= 1u << (8 * j);
                else hi |= 1u << (8 * (j - 4));
            }
        }
        if (mine) {
            const int64_t o = static_cast<int64_t>(t) * E + eb;
            *reinterpret_cast<uint2*>(routing_map + o) = make_uint2(lo, hi);
            if (probs) {
                reinterpret_cast<float4*>(probs + o)[0] = make_float4(p[0], p[1], p[2], p[3]);
                reinterpret_cast<float4*>(probs + o)[1] = make_float4(p[4], p[5], p[6], p[7]);
            }
        }
    }
}

__global__ void __launch_bounds__(kConvWarps * 32)
routing_map_to_topk_vec_kernel(const uint8_t* routing_map, const float* probs, int T, int E, int K, int gs,
                               int64_t* topk_idx, float* topk_weights, int32_t* device_error) {
    dependent_entry();
    const int G = 1 << gs;   // lanes per token
    const int lane = threadIdx.x & 31, gl = lane & (G - 1);
    const int t = ((blockIdx.x * kConvWarps + (threadIdx.x >> 5)) << (5 - gs)) + (lane >> gs);
    const bool active = t < T;   // inactive lanes still take part in the shuffles
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 8 * G) {
        const int eb = e0 + 8 * gl;
        const bool mine = active && eb < E;
        const int64_t o = static_cast<int64_t>(t) * E + eb;
        uint2 m = make_uint2(0u, 0u);
        float4 pa = make_float4(1.0f, 1.0f, 1.0f, 1.0f), pb = pa;
        if (mine) {
            m = __ldg(reinterpret_cast<const uint2*>(routing_map + o));
            if (probs) {
                pa = __ldg(reinterpret_cast<const float4*>(probs + o));
                pb = __ldg(reinterpret_cast<const float4*>(probs + o) + 1);
            }
        }
        unsigned on = 0u;   // bit q: expert eb + q is routed
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            on |= ((m.x >> (8 * q)) & 0xffu) ? (1u << q) : 0u;
            on |= ((m.y >> (8 * q)) & 0xffu) ? (1u << (q + 4)) : 0u;
        }
        const int c = __popc(on);
        int incl = c;
        for (int d = 1; d < G; d <<= 1) {
            const int v = __shfl_up_sync(kFullMask, incl, d, G);
            if (gl >= d) incl += v;
        }
        const int total = __shfl_sync(kFullMask, incl, G - 1, G);
        if (on) {
            const float pv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
            int pos = base + incl - c;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (!((on >> q) & 1u)) continue;
                if (pos < K) {
                    topk_idx[static_cast<int64_t>(t) * K + pos] = eb + q;
                    if (topk_weights) topk_weights[static_cast<int64_t>(t) * K + pos] = pv[q];
                }
                ++pos;
            }
        }
        base += total;
    }
    if (!active) return;
    for (int k = base + gl; k < K; k += G) {
        topk_idx[static_cast<int64_t>(t) * K + k] = -1;
        if (topk_weights) topk_weights[static_cast<int64_t>(t) * K + k] = 0.0f;
    }
    if (base > K && gl == 0 && device_error) atomicExch(device_error, EP_ERR_CAPACITY);
}

__global__ void __launch_bounds__(kConvWarps * 32)
topk_to_routing_map_kernel(const int64_t* topk_idx, const float* w, int T, int K, int E, uint8_t* routing_map,
                           float* probs, int32_t* device_error) {
    dependent_entry();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kConvWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int64_t my_e = -1;
    float my_w = 0.0f;
    if (lane < K) {
        my_e = topk_idx[static_cast<int64_t>(t) * K + lane];
        if (w) my_w = w[static_cast<int64_t>(t) * K + lane];
    }
    const bool bad = my_e < -1 || my_e >= E;
    if (__any_sync(kFullMask, bad) && lane == 0 && device_error) atomicExch(device_error, EP_ERR_INVALID_EXPERT);
    const int key = (my_e >= 0 && my_e < E) ? static_cast<int>(my_e) : -1;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        uint8_t hit = 0;
        float p = 0.0f;
        for (int k = 0; k < K; ++k) {
            const int ek = __shfl_sync(kFullMask, key, k);
            const float wk = __shfl_sync(kFullMask, my_w, k);
            if (ek == e) {
                hit = 1;
                p = p + wk;
            }
        }
        if (e < E) {
            routing_map[static_cast<int64_t>(t) * E + e] = hit;
            if (probs) probs[static_cast<int64_t>(t) * E + e] = p;
        }
    }
}

__global__ void __launch_bounds__(kConvWarps * 32)
routing_map_to_topk_kernel(const uint8_t* routing_map, const float* probs, int T, int E, int K, int64_t* topk_idx,
                           float* topk_weights, int32_t* device_error) {
    dependent_entry();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kConvWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const unsigned lt = (1u << lane) - 1u;
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool on = e < E && routing_map[static_cast<int64_t>(t) * E + e] != 0;
        const unsigned m = __ballot_sync(kFullMask, on);
        const int pos = base + __popc(m & lt);
        if (on && pos < K) {
            topk_idx[static_cast<int64_t>(t) * K + pos] = e;
            if (topk_weights) topk_weights[static_cast<int64_t>(t) * K + pos] = probs ? probs[static_cast<int64_t>(t) * E + e] : 1.0f;
        }
        base += __popc(m);
    }
    for (int k = base + lane; k < K; k += 32) {
        topk_idx[static_cast<int64_t>(t) * K + k] = -1;
        if (topk_weights) topk_weights[static_cast<int64_t>(t) * K + k] = 0.0f;
    }
    if (base > K && lane == 0 && device_error) atomicExch(device_error, EP_ERR_CAPACITY);
}

}  // namespace

cudaError_t launch_topk_to_routing_map(const int64_t* topk_idx, const float* w, int T, int K, int E,
                                       uint8_t* routing_map, float* probs, int32_t* device_error,
                                       cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((T + kConvWarps - 1) / kConvWarps);
    if (E % 8 == 0 && reinterpret_cast<uintptr_t>(routing_map) % 8 == 0 &&
        reinterpret_cast<uintptr_t>(probs) % 16 == 0) {
        const int gs = lanes_per_token_log2(E);
        const int per_block = kConvWarps << (5 - gs);
        return launch_dependent(topk_to_routing_map_vec_kernel, dim3((T + per_block - 1) / per_block),
                                dim3(kConvWarps * 32), 0, stream, topk_idx, w, T, K, E, gs, routing_map, probs,
                                device_error);
    }
    return launch_dependent(topk_to_routing_map_kernel, dim3(blocks), dim3(kConvWarps * 32), 0, stream, topk_idx, w,
                            T, K, E, routing_map, probs, device_error);
}

cudaError_t launch_routing_map_to_topk(const uint8_t* routing_map, const float* probs, int T, int E, int K,
                                       int64_t* topk_idx, float* topk_weights, int32_t* device_error,
                                       cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((T + kConvWarps - 1) / kConvWarps);
    if (E % 8 == 0 && reinterpret_cast<uintptr_t>(routing_map) % 8 == 0 &&
        reinterpret_cast<uintptr_t>(probs) % 16 == 0) {
        const int gs = lanes_per_token_log2(E);
        const int per_block = kConvWarps << (5 - gs);
        return launch_dependent(routing_map_to_topk_vec_kernel, dim3((T + per_block - 1) / per_block),
                                dim3(kConvWarps * 32), 0, stream, routing_map, probs, T, E, K, gs, topk_idx,
                                topk_weights, device_error);
    }
    return launch_dependent(routing_map_to_topk_kernel, dim3(blocks), dim3(kConvWarps * 32), 0, stream, routing_map,
                            probs, T, E, K, topk_idx, topk_weights, device_error);
}

}  // namespace ep

// ---------------------------------------------------------------- non-expand

namespace ep {

namespace {

// One thread per token: key[t, k] = rank of slot k's expert if it is the
// token's first slot on that rank, -1 otherwise (repeats, unused slots), -2
// for an id outside [-1, E) so the layout that follows reports it. Valid
// slots are counted per expert in a shared-memory histogram that each block
// adds to the global counts once per non-empty bin (integer adds: exact in
// any order). Ranks seen so far live in a register mask when R <= 32.
__global__ void __launch_bounds__(256)
nonexpand_keys_kernel(const int64_t* topk_idx, int T, int K, int E, int R, int L, int64_t* keys,
                      int32_t* expert_counts) {
    dependent_entry();
    extern __shared__ int hist[];                  // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < T) {
        const int64_t* row = topk_idx + static_cast<int64_t>(t) * K;
        int64_t* out = keys + static_cast<int64_t>(t) * K;
        unsigned seen_small = 0u;
        for (int k = 0; k < K; ++k) {
            const int64_t e = row[k];
            int64_t key = -1;
            if (e < -1 || e >= E) {
                key = -2;
            } else if (e >= 0) {
                atomicAdd(hist + e, 1);
                const int r = static_cast<int>(e / L);
                bool first;
                if (R <= 32) {
                    first = !(seen_small & (1u << r));
                    seen_small |= 1u << r;
                } else {
                    first = true;
                    for (int j = 0; j < k; ++j) {
                        const int64_t ej = row[j];
                        if (ej >= 0 && ej < E && ej / L == r) { first = false; break; }
                    }
                }
                if (first) key = r;
            }
            out[k] = key;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (hist[e]) atomicAdd(expert_counts + e, hist[e]);
}

// One warp per token: for each slot that owns a (token, rank) row, write that
// row's K entries: rank-local expert id (and weight) for the token's slots on
// the rank, -1 (and 0) for the others.
__global__ void __launch_bounds__(kConvWarps * 32)
nonexpand_recv_topk_kernel(const int64_t* topk_idx, const float* w, const int32_t* row_of_slot, int T, int K,
                           int E, int L, int64_t* recv_topk_idx, float* recv_topk_weights) {
    dependent_entry();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kConvWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int64_t e = -1;
    float wk = 0.0f;
    int row = -1;
    if (lane < K) {
        e = topk_idx[static_cast<int64_t>(t) * K + lane];
        if (w) wk = w[static_cast<int64_t>(t) * K + lane];
        row = row_of_slot[static_cast<int64_t>(t) * K + lane];
    }
    const int rank = (e >= 0 && e < E) ? static_cast<int>(e / L) : -1;
    for (int j = 0; j < K; ++j) {
        const int rj = __shfl_sync(kFullMask, row, j);
        const int rkj = __shfl_sync(kFullMask, rank, j);
        if (rj < 0) continue;
        if (lane < K) {
            const bool on = rank == rkj;
            recv_topk_idx[static_cast<int64_t>(rj) * K + lane] = on ? e - static_cast<int64_t>(rkj) * L : -1;
            if (recv_topk_weights) recv_topk_weights[static_cast<int64_t>(rj) * K + lane] = on ? wk : 0.0f;
        }
    }
}

}  // namespace

cudaError_t launch_nonexpand_keys(const int64_t* topk_idx, int T, int K, int E, int R, int64_t* keys,
                                  int32_t* expert_counts, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    return launch_dependent(nonexpand_keys_kernel, dim3((T + 255) / 256), dim3(256), static_cast<size_t>(E) * sizeof(int),
                            stream, topk_idx, T, K, E, R, E / R, keys, expert_counts);
}

cudaError_t launch_nonexpand_recv_topk(const int64_t* topk_idx, const float* w, const int32_t* row_of_slot, int T,
                                       int K, int E, int R, int64_t* recv_topk_idx, float* recv_topk_weights,
                                       cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    return launch_dependent(nonexpand_recv_topk_kernel, dim3((T + kConvWarps - 1) / kConvWarps), dim3(kConvWarps * 32),
                            0, stream, topk_idx, w, row_of_slot, T, K, E, E / R, recv_topk_idx, recv_topk_weights);
}

}  // namespace ep
