// Combine: weighted top-k gather-reduce of expert outputs back to token order,
//   out[t, :] = bf16( sum_k w[t,k] * y[row_of_slot[t,k], :] ).
//
// What is computed follows nccl_ep.cc, ncclEpCombine (low-latency branch:
// expert outputs are combined with the fp32 topk_weights [T, K] into
// out [T, hidden] of the input dtype) and NeMo fused_a2a,
// HybridEPCombine.forward (rows come back in the original token order).
// Reading where the pages are silent: fp32 fused multiply-adds in ascending k
// starting from +0, skipping unused slots, then one round to nearest-even.
//
// GPU design: the work item is (token, column segment), one warp per item.
// The warp compacts the token's used slots (ballot + popc) into shared memory
// in ascending k, then for its two 16-byte column vectors issues the loads of
// a group of slots at once before accumulating them in k order. Items are
// 512 channels and blocks are 2 warps. The group is K split into the fewest
// round trips of at most 6 slots, in equal parts: 4 + 4 for top-8, one trip
// of 6 for top-6 (groups of 4 there cost 5% on a 4 + 2 split; groups of 8
// for top-8 cost 2% in occupancy). Vectors per lane, A/B on one box, three
// interleaved rounds: two instead of one took the skewed step (top-6) from
// 298.2 to 292.4 us, the decode step (T=256) from 14.08 to 13.72 us warm and
// the prefill step from 314.4 to 313.5 us; four lost on all three (the top-6
// instance then needs 152 registers); 1 or 4 warps per block lost to 2.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kWarpsPerBlock = 2;   // small blocks: fine-grained scheduling
constexpr int kUnroll = 2;      // 16-byte column vectors per lane per item
constexpr int kMaxGroup = 6;    // most slots whose loads are issued together

__device__ __forceinline__ int4 ld_stream(const int4* p) {
    int4 v;
    asm volatile("ld.global.nc.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void fma8(float* acc, float w, const int4& v) {
    const unsigned u[4] = {static_cast<unsigned>(v.x), static_cast<unsigned>(v.y),
                           static_cast<unsigned>(v.z), static_cast<unsigned>(v.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(w, __uint_as_float(u[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(u[i] & 0xffff0000u), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
    const unsigned short l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const unsigned short h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return static_cast<unsigned>(l) | (static_cast<unsigned>(h) << 16);
}

template <int kGroup>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
combine_kernel(CombineArgs a, int64_t num_items, int num_segments) {
    // launched as the preceding kernel's programmatic dependent: nothing is
    // read or written before that kernel has finished
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ int s_row[kWarpsPerBlock][32];
    __shared__ float s_w[kWarpsPerBlock][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
    if (item >= num_items) return;
    const int t = static_cast<int>(item / num_segments);
    const int seg = static_cast<int>(item - static_cast<int64_t>(t) * num_segments);
    const int H16 = a.H / 8;

    int row = -1;
    float w = 1.0f;
    if (lane < a.K) {
        row = __ldg(a.row_of_slot + static_cast<int64_t>(t) * a.K + lane);
        if (a.topk_weights) w = __ldg(a.topk_weights + static_cast<int64_t>(t) * a.K + lane);
    }
    if (a.slot_weights && seg == 0 && lane < a.K)
        a.slot_weights[static_cast<int64_t>(t) * a.K + lane] = row >= 0 ? __ldg(a.row_weights + row) : 0.0f;
    const unsigned used = __ballot_sync(kFullMask, row >= 0);
    const int n_used = __popc(used);
    if (row >= 0) {
        const int pos = __popc(used & ((1u << lane) - 1u));   // ascending k order
        s_row[warp][pos] = row;
        s_w[warp][pos] = w;
    }
    __syncwarp();

    const int4* y = reinterpret_cast<const int4*>(a.y);
    int4* out = reinterpret_cast<int4*>(a.out) + static_cast<int64_t>(t) * H16;
    const int j0 = seg * (32 * kUnroll) + lane;

    float acc[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;

    for (int g = 0; g < n_used; g += kGroup) {
        int4 v[kUnroll][kGroup];
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
            if (g + i < n_used) {
                const int4* yr = y + static_cast<int64_t>(s_row[warp][g + i]) * H16;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int j = j0 + u * 32;
                    if (j < H16) v[u][i] = ld_stream(yr + j);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
            if (g + i < n_used) {
                const float wk = s_w[warp][g + i];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) fma8(acc[u], wk, v[u][i]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int j = j0 + u * 32;
        if (j < H16) {
            int4 o;
            o.x = static_cast<int>(pack_bf16x2(acc[u][0], acc[u][1]));
            o.y = static_cast<int>(pack_bf16x2(acc[u][2], acc[u][3]));
            o.z = static_cast<int>(pack_bf16x2(acc[u][4], acc[u][5]));
            o.w = static_cast<int>(pack_bf16x2(acc[u][6], acc[u][7]));
            out[j] = o;
        }
    }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
    const int H16 = a.H / 8;
    const int per_item = 32 * kUnroll;
    const int segs = (H16 + per_item - 1) / per_item;
    const int64_t items = static_cast<int64_t>(a.T) * segs;
    if (items == 0) return cudaSuccess;
    const int64_t blocks = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int trips = (a.K + kMaxGroup - 1) / kMaxGroup;
    const int group = (a.K + trips - 1) / trips;      // 1..6
    // a programmatic dependent of whatever kernel precedes it on the stream:
    // its blocks may be scheduled while that kernel's last wave runs, and wait
    // for it to finish before touching memory
    cudaLaunchConfig_t cfg = {};
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;   // beyond the grid limit: refuse
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (group <= 4) return cudaLaunchKernelEx(&cfg, combine_kernel<4>, a, items, segs);
    return cudaLaunchKernelEx(&cfg, combine_kernel<kMaxGroup>, a, items, segs);
}

}  // namespace ep
