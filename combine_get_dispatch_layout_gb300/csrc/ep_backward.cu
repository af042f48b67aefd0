// Backward passes of dispatch and combine.
//
// DeepEP API docs (README training snippet): the backward of dispatch is a
// combine and the backward of combine is a dispatch; nccl_ep.cc, ncclEpCombine:
// the high-throughput backward mode also reduces the probabilities. With the
// weighted forward combine out[t] = sum_k w[t,k] * y[row(t,k)]:
//   combine backward:  grad_y[row(t,k)] = bf16(w[t,k] * grad_out[t])   (fp32 product, one round)
//                      grad_w[t,k]      = sum_h grad_out[t,h] * y[row(t,k),h]   (fp32)
//   dispatch backward: grad_x[t] = bf16(sum_k grad_recv[row(t,k)])     (the unweighted combine)
//                      grad_topk_weights[t,k] = grad_recv_weights[row(t,k)]  (0 if dropped)
// The dispatch backward runs as the combine kernel (ep_combine.cu) with null
// weights, whose warps for each token's first column segment also write the
// token's weight gradients.
//
// GPU design (combine backward): one 4-warp block per token. Each thread owns
// a stride of 16-byte column vectors; for each vector it loads grad_out once,
// the vectors of up to 4 slots at a time, writes the scaled gradient rows with
// streaming stores, and adds the 8-channel products to a per-(slot, thread)
// fp32 partial in shared memory. The partials are reduced per slot by a fixed
// shuffle tree, so the weight gradient is deterministic.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdGroup = 4;

__device__ __forceinline__ int4 ld_nc(const int4* p) {
    int4 v;
    asm volatile("ld.global.nc.v4.s32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void unpack8(const int4& v, float* f) {
    const unsigned u[4] = {static_cast<unsigned>(v.x), static_cast<unsigned>(v.y), static_cast<unsigned>(v.z),
                           static_cast<unsigned>(v.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ unsigned bf16x2(float lo, float hi) {
    return static_cast<unsigned>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<unsigned>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

__global__ void __launch_bounds__(kBwdThreads)
combine_backward_kernel(CombineBackwardArgs a) {
    dependent_entry();
    __shared__ int s_row[EP_MAX_TOPK];
    __shared__ float s_w[EP_MAX_TOPK];
    __shared__ int s_k[EP_MAX_TOPK];
    __shared__ int s_n;
    __shared__ float s_part[EP_MAX_TOPK * kBwdThreads];
    __shared__ float s_warp[EP_MAX_TOPK][kBwdThreads / 32];
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H16 = a.H / 8;

    if (warp == 0) {
        int row = -1;
        float w = 1.0f;
        if (lane < a.K) {
            row = a.row_of_slot[static_cast<int64_t>(t) * a.K + lane];
            if (a.topk_weights) w = a.topk_weights[static_cast<int64_t>(t) * a.K + lane];
        }
        const unsigned used = __ballot_sync(kFullMask, row >= 0);
        if (row >= 0) {
            const int pos = __popc(used & ((1u << lane) - 1u));
            s_row[pos] = row;
            s_w[pos] = w;
            s_k[pos] = lane;
        }
        if (lane == 0) s_n = __popc(used);
    }
    __syncthreads();
    const int n = s_n;
    for (int i = 0; i < n; ++i) s_part[i * kBwdThreads + tid] = 0.0f;

    const int4* g_row = reinterpret_cast<const int4*>(a.grad_out) + static_cast<int64_t>(t) * H16;
    const int4* y = reinterpret_cast<const int4*>(a.y);
    int4* gy = reinterpret_cast<int4*>(a.grad_y);
    for (int j = tid; j < H16; j += kBwdThreads) {
        float g[8];
        unpack8(ld_nc(g_row + j), g);
        for (int i0 = 0; i0 < n; i0 += kBwdGroup) {
            int4 v[kBwdGroup];
#pragma unroll
            for (int i = 0; i < kBwdGroup; ++i)
                if (i0 + i < n) v[i] = ld_nc(y + static_cast<int64_t>(s_row[i0 + i]) * H16 + j);
#pragma unroll
            for (int i = 0; i < kBwdGroup; ++i) {
                if (i0 + i < n) {
                    float f[8];
                    unpack8(v[i], f);
                    float p = s_part[(i0 + i) * kBwdThreads + tid];
#pragma unroll
                    for (int c = 0; c < 8; ++c) p = __fmaf_rn(g[c], f[c], p);
                    s_part[(i0 + i) * kBwdThreads + tid] = p;
                    if (gy) {
                        const float wk = s_w[i0 + i];
                        int4 o;
                        o.x = static_cast<int>(bf16x2(__fmul_rn(wk, g[0]), __fmul_rn(wk, g[1])));
                        o.y = static_cast<int>(bf16x2(__fmul_rn(wk, g[2]), __fmul_rn(wk, g[3])));
                        o.z = static_cast<int>(bf16x2(__fmul_rn(wk, g[4]), __fmul_rn(wk, g[5])));
                        o.w = static_cast<int>(bf16x2(__fmul_rn(wk, g[6]), __fmul_rn(wk, g[7])));
                        __stcs(gy + static_cast<int64_t>(s_row[i0 + i]) * H16 + j, o);
                    }
                }
            }
        }
    }
    if (!a.grad_w) return;
    // fixed-order reduction of each slot's 128 partials
    for (int i = 0; i < n; ++i) {
        float p = s_part[i * kBwdThreads + tid];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) p += __shfl_xor_sync(kFullMask, p, d);
        if (lane == 0) s_warp[i][warp] = p;
    }
    __syncthreads();
    if (tid < a.K) {
        float gw = 0.0f;   // dropped slots get 0
        for (int i = 0; i < n; ++i) {
            if (s_k[i] == tid) {
                float s = 0.0f;
#pragma unroll
                for (int w = 0; w < kBwdThreads / 32; ++w) s += s_warp[i][w];
                gw = s;
            }
        }
        a.grad_w[static_cast<int64_t>(t) * a.K + tid] = gw;
    }
}

}  // namespace

cudaError_t launch_combine_backward(const CombineBackwardArgs& a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    return launch_dependent(combine_backward_kernel, dim3(a.T), dim3(kBwdThreads), 0, stream, a);
}

}  // namespace ep
