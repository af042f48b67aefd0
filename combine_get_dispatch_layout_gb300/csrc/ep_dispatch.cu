// Dispatch: stable expert-major permute of token rows into the receive buffer,
// optionally quantised to fp8 (e4m3 or e5m2) with one scale per 128 channels.
//
// What is computed follows nccl_ep.cc, ncclEpDispatch (tokens are bf16 rows;
// the fp8 path writes fp32 scales shaped [rows, hidden/128]) and the DeepEP
// API docs, "dispatch()" (do_expand: every (token, expert) pair gets its own
// received row). Readings where the pages are silent: scale = amax / 448 with
// IEEE division, q = e4m3(x / scale) rounded to nearest-even and saturated to
// +-448, and an all-zero block gives scale 0 and zero bytes. nccl_ep.cc
// (ncclTypeSize, ncclEpDispatch) also takes e5m2 as a one-byte fp8 token
// type; its quantiser here is the same rule with e5m2's largest finite value,
// 57344, in place of 448.
//
// GPU design: the work item is (token, column segment), one warp per item.
// The warp reads its slice of the token row once with 16-byte loads and
// writes it to each of the token's K receive rows with 16-byte streaming
// stores, so x is read once although it is written K times. For fp8, a lane
// holds 16 channels (two 16-byte loads, one 16-byte code store per copy),
// 8 lanes one 128-channel block; the block amax is a 3-step xor-shuffle max,
// and the scale and codes are computed once per token and reused for all K
// copies. Item sizes won sweeps on the prefill shape: 2 vectors per lane for
// bf16 (of 1 to 8), one 512-channel group per item for fp8 (16 channels per
// lane beat 8 by 6-11%); small items shorten the last wave. A bf16 grid of
// less than one wave (the decode shapes) takes one vector per lane instead,
// so twice as many warps share the stores: 0.4 us off the T=256 step, none
// lost at the prefill shape, which keeps two.
// The slot map is read only after griddepcontrol.wait: launched as the
// layout's programmatic dependent, a block loads (and quantises) its x slice
// on an SM the layout leaves idle, then waits for the layout to finish.
#include <atomic>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kBf16Unroll = 2;     // 16-byte vectors per lane per item
constexpr int kFp8Unroll = 1;      // 512-channel groups per item (16 channels per lane)

__device__ __forceinline__ int4 ld_stream(const int4* p) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Wait for the preceding grid (normally the layout that wrote row_of_slot)
// and so for all earlier work; the dispatch is always launched as that
// grid's programmatic dependent, and the wait is a no-op when the launch had
// to serialise anyway (an event or a copy in between). Then
// let a kernel launched as this grid's dependent (a combine) be scheduled on
// SMs that this grid's last wave leaves free: it waits for this grid to
// finish before its first memory access. Triggering only after the wait keeps
// the chain's guarantee: when a kernel starts, all work before its immediate
// predecessor is complete.
__device__ __forceinline__ void wait_for_layout() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
}

// Zero pad row `item` of an aligned layout (item = expert * max_pad + i, one
// warp each): row offsets[e] + counts[e] + i if it is below offsets[e + 1].
__device__ __forceinline__ void zero_pad_row(const int32_t* counts, const int32_t* offsets, int E, int max_pad,
                                             int64_t item, int64_t row_bytes, char* recv, const PadScales& sc,
                                             int32_t* src, float* weights, int lane) {
    const int e = static_cast<int>(item / max_pad);
    const int i = static_cast<int>(item - static_cast<int64_t>(e) * max_pad);
    if (e >= E) return;
    const int64_t row = static_cast<int64_t>(offsets[e]) + counts[e] + i;
    if (row >= offsets[e + 1]) return;
    int4* d = reinterpret_cast<int4*>(recv + row * row_bytes);   // row_bytes % 16 == 0
    for (int64_t j = lane; j < row_bytes / 16; j += 32) d[j] = make_int4(0, 0, 0, 0);
    if (sc.ptr)
        for (int b = lane; b < sc.nb; b += 32) {
            const int64_t si = sc.col_major ? static_cast<int64_t>(b) * sc.ld + row : row * sc.nb + b;
            if (sc.bytes == 1) static_cast<uint8_t*>(sc.ptr)[si] = 0;
            else static_cast<float*>(sc.ptr)[si] = 0.0f;
        }
    if (lane == 0) {
        if (src) src[row] = -1;
        if (weights) weights[row] = 0.0f;
    }
}

// The grid's first a.pad_blocks blocks zero the pad rows of an aligned layout
// and return true; the others return false and dispatch, their block index
// counted from the end of the pad blocks. Pad rows are disjoint from the rows
// the dispatch writes, so both share the grid (and HBM) from the first wave;
// the pad counts come from the layout, hence the same wait.
__device__ __forceinline__ bool pad_block(const DispatchArgs& a, int64_t row_bytes, int64_t& block) {
    block = static_cast<int64_t>(blockIdx.x) - a.pad_blocks;
    if (block >= 0) return false;
    wait_for_layout();
    const int64_t item = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    zero_pad_row(a.pad_counts, a.pad_offsets, a.pad_experts, a.pad_max, item, row_bytes,
                 static_cast<char*>(a.recv_x), a.pad_scales, a.recv_src_token, a.recv_weights, threadIdx.x & 31);
    return true;
}

constexpr int kPrefetchCtas = 1024;                   // blocks that issue the x prefetch
constexpr int64_t kPrefetchWindow = int64_t{96} << 20;   // bytes of x prefetched past theirs

// HBM is idle while the layout runs. In a dispatch launched as the layout's
// programmatic dependent, the first kPrefetchCtas blocks (resident from the
// layout's start) ask the L2 to fetch up to kPrefetchWindow bytes of x past
// the rows they read themselves: one bulk L2 prefetch each, holding no
// registers or shared memory. Later blocks then find their rows in L2 (the
// receive stores are evict-first, so the prefetched lines survive until
// read), which takes those bytes off the dispatch's critical path. A hint
// only: results do not depend on it. Prefill step (300 chained steps):
// 321.6 us without it; a 96 MB window from 512 blocks 315.9 us, from 1024
// blocks 314.3 us. Windows of 24 / 48 / 64 / 128 MB from 512 blocks gave
// 317.9 / 317.4 / 316.9 / 315.5 us, and 2048 or 4096 blocks 320-322 us (the
// blocks past the first wave start only after the layout, so their prefetch
// competes with the dispatch itself). Part of the prefetched x is evicted
// and read again before use, but fetching it while HBM is otherwise idle
// still wins. An evict-last cache policy was slower (and kept x in L2 past
// the dispatch).
__device__ __forceinline__ void prefetch_x_during_layout(const DispatchArgs& a, int num_segments,
                                                         int64_t row_bytes, int64_t block) {
    if (!a.prefetch_x || block >= kPrefetchCtas || threadIdx.x != 0) return;
    // tokens the prefetching blocks read themselves (row_bytes % 16 == 0)
    const int64_t own = (static_cast<int64_t>(kPrefetchCtas) * kWarpsPerBlock + num_segments - 1) / num_segments;
    const int64_t lo0 = own * row_bytes;
    const int64_t end = min(static_cast<int64_t>(a.T) * row_bytes, lo0 + kPrefetchWindow);
    if (end <= lo0) return;
    const int64_t per = ((end - lo0 + kPrefetchCtas - 1) / kPrefetchCtas + 15) / 16 * 16;
    const int64_t lo = lo0 + block * per;
    const int64_t hi = min(lo + per, end);
    if (lo >= hi) return;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                 :: "l"(static_cast<const char*>(a.x) + lo), "r"(static_cast<unsigned>(hi - lo)) : "memory");
}

// Row of each slot of token t, lane k holds slot k (K <= 32); -1 if unused.
__device__ __forceinline__ int slot_row(const int32_t* row_of_slot, int t, int K, int lane) {
    return lane < K ? __ldg(row_of_slot + static_cast<int64_t>(t) * K + lane) : -1;
}

__device__ __forceinline__ void write_side_outputs(const DispatchArgs& a, int t, int lane, int row) {
    if (lane < a.K && row >= 0) {
        if (a.recv_src_token) a.recv_src_token[row] = t;
        if (a.recv_weights) a.recv_weights[row] = __ldg(a.topk_weights + static_cast<int64_t>(t) * a.K + lane);
    }
}

template <int kUnroll>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
dispatch_bf16_kernel(DispatchArgs a, int64_t num_items, int num_segments) {
    const int lane = threadIdx.x & 31;
    int64_t block;
    if (pad_block(a, static_cast<int64_t>(a.H) * 2, block)) return;
    const int64_t item = block * kWarpsPerBlock + (threadIdx.x >> 5);
    if (item >= num_items) return;
    const int t = static_cast<int>(item / num_segments);
    const int seg = static_cast<int>(item - static_cast<int64_t>(t) * num_segments);
    const int H16 = a.H / 8;                          // 16-byte vectors per row

    const int4* src = reinterpret_cast<const int4*>(a.x) + static_cast<int64_t>(t) * H16;
    int4* dst = reinterpret_cast<int4*>(a.recv_x);
    const int j0 = seg * (32 * kUnroll) + lane;
    if (!a.overlap_layout) wait_for_layout();
    int4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int j = j0 + u * 32;
        if (j < H16) v[u] = ld_stream(src + j);
    }
    if (a.overlap_layout) {
        // x is ready before the layout starts; the slot map only after it ends
        prefetch_x_during_layout(a, num_segments, static_cast<int64_t>(a.H) * 2, block);
        wait_for_layout();
    }
    const int row = slot_row(a.row_of_slot, t, a.K, lane);
    if (seg == 0) write_side_outputs(a, t, lane, row);
    for (int k = 0; k < a.K; ++k) {
        const int r = __shfl_sync(kFullMask, row, k);
        if (r < 0) continue;
        int4* d = dst + static_cast<int64_t>(r) * H16;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = j0 + u * 32;
            if (j < H16) __stcs(d + j, v[u]);
        }
    }
}

// Two fp32 values -> two codes of the fp8 format kFmt (EP_DTYPE_FP8_E4M3 or
// EP_DTYPE_FP8_E5M2; RNE, satfinite); `lo` goes to the low byte.
template <int kFmt>
__device__ __forceinline__ unsigned short fp8x2(float lo, float hi) {
    unsigned short d;
    if (kFmt == EP_DTYPE_FP8_E5M2)
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Largest finite value of the fp8 format; a block's amax maps onto it.
template <int kFmt>
__host__ __device__ constexpr float fp8_max() {
    return kFmt == EP_DTYPE_FP8_E5M2 ? 57344.0f : 448.0f;
}

__device__ __forceinline__ float bf16_lo(unsigned u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(unsigned u) { return __uint_as_float(u & 0xffff0000u); }

// Smallest power of two >= s (s > 0, finite), from the bit pattern: a
// normal s with a zero mantissa is already a power of two, otherwise the next
// exponent; a subnormal s (value f * 2^-149) rounds its mantissa f up to a
// power of two, which is itself the bit pattern of the result (2^23 being the
// smallest normal).
__device__ __forceinline__ float pow2_ceil(float s) {
    const unsigned u = __float_as_uint(s);
    const unsigned e = u >> 23, f = u & 0x7fffffu;
    if (e == 0) return __uint_as_float((f & (f - 1u)) == 0u ? f : (1u << (32 - __clz(f))));
    return f == 0u ? s : __uint_as_float((e + 1u) << 23);
}

// Where block b of receive row r keeps its scale.
template <bool kColMajor>
__device__ __forceinline__ int64_t scale_index(const DispatchArgs& a, int64_t r, int b, int nb) {
    return kColMajor ? static_cast<int64_t>(b) * a.scale_ld + r : r * nb + b;
}

// kMode: EP_SCALE_FP32 (scale = amax/F), EP_SCALE_POW2 (smallest power of
// two >= amax/F, stored as fp32) or EP_SCALE_UE8M0 (that power, at least
// 2^-127, stored as its biased exponent byte); F = fp8_max<kFmt>().
template <int kMode, bool kColMajor, int kFmt>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
dispatch_fp8_kernel(DispatchArgs a, int64_t num_items, int num_segments) {
    const int lane = threadIdx.x & 31;
    int64_t block;
    if (pad_block(a, a.H, block)) return;
    const int64_t item = block * kWarpsPerBlock + (threadIdx.x >> 5);
    if (item >= num_items) return;
    const int t = static_cast<int>(item / num_segments);
    const int seg = static_cast<int>(item - static_cast<int64_t>(t) * num_segments);
    const int G = a.H / 16;                           // 16-channel groups per row (lane units)
    const int nb = a.H / 128;
    const int4* src = reinterpret_cast<const int4*>(a.x) + static_cast<int64_t>(t) * (a.H / 8);
    uint4 q[kFp8Unroll];
    float scale[kFp8Unroll];
    const int g0 = seg * (32 * kFp8Unroll) + lane;
    if (!a.overlap_layout) wait_for_layout();
#pragma unroll
    for (int u = 0; u < kFp8Unroll; ++u) {
        const int g = g0 + u * 32;
        int4 v0 = make_int4(0, 0, 0, 0), v1 = make_int4(0, 0, 0, 0);
        if (g < G) {
            v0 = ld_stream(src + 2 * g);
            v1 = ld_stream(src + 2 * g + 1);
        }
        float f[16] = {bf16_lo(v0.x), bf16_hi(v0.x), bf16_lo(v0.y), bf16_hi(v0.y),
                       bf16_lo(v0.z), bf16_hi(v0.z), bf16_lo(v0.w), bf16_hi(v0.w),
                       bf16_lo(v1.x), bf16_hi(v1.x), bf16_lo(v1.y), bf16_hi(v1.y),
                       bf16_lo(v1.z), bf16_hi(v1.z), bf16_lo(v1.w), bf16_hi(v1.w)};
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(f[i]));
#pragma unroll
        for (int d = 4; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, d));
        // m is now the amax of this lane's 128-channel block (8 lanes)
        if (m == 0.0f) {
            scale[u] = 0.0f;
            q[u] = make_uint4(0u, 0u, 0u, 0u);
        } else {
            float s = __fdiv_rn(m, fp8_max<kFmt>());
            if (kMode != EP_SCALE_FP32) s = pow2_ceil(s);
            if (kMode == EP_SCALE_UE8M0) s = fmaxf(s, __uint_as_float(0x00400000u));   // 2^-127
            scale[u] = s;
            unsigned w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = fp8x2<kFmt>(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s));
            q[u] = make_uint4(w[0] | (w[1] << 16), w[2] | (w[3] << 16), w[4] | (w[5] << 16), w[6] | (w[7] << 16));
        }
    }
    if (a.overlap_layout) {
        prefetch_x_during_layout(a, num_segments, static_cast<int64_t>(a.H) * 2, block);
        wait_for_layout();
    }
    const int row = slot_row(a.row_of_slot, t, a.K, lane);
    if (seg == 0) write_side_outputs(a, t, lane, row);
    uint4* dst = reinterpret_cast<uint4*>(a.recv_x);
    for (int k = 0; k < a.K; ++k) {
        const int r = __shfl_sync(kFullMask, row, k);
        if (r < 0) continue;
        uint4* d = dst + static_cast<int64_t>(r) * G;
#pragma unroll
        for (int u = 0; u < kFp8Unroll; ++u) {
            const int g = g0 + u * 32;
            if (g < G) {
                __stcs(d + g, q[u]);
                if ((lane & 7) == 0) {
                    const int64_t si = scale_index<kColMajor>(a, r, g / 8, nb);
                    if (kMode == EP_SCALE_UE8M0) {
                        // a power of two >= 2^-127: normal -> exponent field, 2^-127 -> 0
                        const unsigned bits = __float_as_uint(scale[u]);
                        static_cast<uint8_t*>(a.recv_scales)[si] = static_cast<uint8_t>(bits >> 23);
                    } else {
                        __stcs(static_cast<float*>(a.recv_scales) + si, scale[u]);
                    }
                }
            }
        }
    }
}

// fp8 input pass-through: one warp per (token, column segment) copies the
// token's fp8 codes (e4m3 or e5m2: bytes either way) to each of its K rows with 16-byte vectors; the warp of
// segment 0 also copies the token's scale row (fp32, or bytes in UE8M0 mode)
// into every receive row's scales, in the requested layout.
template <bool kColMajor>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
dispatch_fp8_passthrough_kernel(DispatchArgs a, int64_t num_items, int num_segments) {
    const int lane = threadIdx.x & 31;
    int64_t block;
    if (pad_block(a, a.H, block)) return;
    const int64_t item = block * kWarpsPerBlock + (threadIdx.x >> 5);
    if (item >= num_items) return;
    const int t = static_cast<int>(item / num_segments);
    const int seg = static_cast<int>(item - static_cast<int64_t>(t) * num_segments);
    const int V = a.H / 16;                           // 16-byte vectors of codes per row
    const int nb = a.H / 128;
    const int4* src = reinterpret_cast<const int4*>(a.x) + static_cast<int64_t>(t) * V;
    int4* dst = reinterpret_cast<int4*>(a.recv_x);
    const int j0 = seg * (32 * kBf16Unroll) + lane;
    if (!a.overlap_layout) wait_for_layout();
    int4 v[kBf16Unroll];
#pragma unroll
    for (int u = 0; u < kBf16Unroll; ++u) {
        const int j = j0 + u * 32;
        if (j < V) v[u] = ld_stream(src + j);
    }
    const bool ue = a.scale_mode == EP_SCALE_UE8M0;
    if (a.overlap_layout) {
        prefetch_x_during_layout(a, num_segments, a.H, block);
        wait_for_layout();
    }
    const int row = slot_row(a.row_of_slot, t, a.K, lane);
    if (seg == 0) write_side_outputs(a, t, lane, row);
    for (int k = 0; k < a.K; ++k) {
        const int r = __shfl_sync(kFullMask, row, k);
        if (r < 0) continue;
        int4* d = dst + static_cast<int64_t>(r) * V;
#pragma unroll
        for (int u = 0; u < kBf16Unroll; ++u) {
            const int j = j0 + u * 32;
            if (j < V) __stcs(d + j, v[u]);
        }
        if (seg == 0) {
            for (int b = lane; b < nb; b += 32) {
                const int64_t si = scale_index<kColMajor>(a, r, b, nb);
                if (ue)
                    static_cast<uint8_t*>(a.recv_scales)[si] =
                        static_cast<const uint8_t*>(a.x_scales)[static_cast<int64_t>(t) * nb + b];
                else
                    static_cast<float*>(a.recv_scales)[si] =
                        __ldg(static_cast<const float*>(a.x_scales) + static_cast<int64_t>(t) * nb + b);
            }
        }
    }
}

// One warp per (expert, pad row): zero a pad row of an aligned layout.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
fill_pad_rows_kernel(const int32_t* counts, const int32_t* offsets, int E, int max_pad, int64_t row_bytes,
                     char* recv, PadScales sc, int32_t* src, float* weights) {
    dependent_entry();
    const int64_t item = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    zero_pad_row(counts, offsets, E, max_pad, item, row_bytes, recv, sc, src, weights, threadIdx.x & 31);
}

// Launch as a programmatic dependent of the preceding grid: the blocks may be
// scheduled while that grid drains. Each waits for it before touching global
// memory, except that with overlap_layout it first loads (and quantises) its
// slice of x, which the caller guarantees was written before the layout.
template <typename... Params, typename... Args>
cudaError_t launch_dispatch_kernel(void (*kernel)(Params...), int64_t blocks, cudaStream_t stream, Args... args) {
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;   // beyond the grid limit: refuse
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The arguments with pad_blocks set: enough blocks, one warp per (expert,
// pad row), to zero the pad rows of an aligned layout (0 without padding).
DispatchArgs with_pad_blocks(const DispatchArgs& a) {
    DispatchArgs b = a;
    b.pad_blocks = a.pad_max > 0
                       ? (static_cast<int64_t>(a.pad_experts) * a.pad_max + kWarpsPerBlock - 1) / kWarpsPerBlock
                       : 0;
    return b;
}

// Warps the GPU holds at once for the bf16 dispatch (SMs x resident blocks x
// warps per block), per device, looked up once (any thread may store it:
// every lookup gives the same value).
int64_t resident_dispatch_warps() {
    static std::atomic<int64_t> warps[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int64_t w = warps[dev].load(std::memory_order_relaxed);
    if (w == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_bf16_kernel<kBf16Unroll>,
                                                          kWarpsPerBlock * 32, 0) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        w = static_cast<int64_t>(sms) * per_sm * kWarpsPerBlock;
        warps[dev].store(w, std::memory_order_relaxed);
    }
    return w;
}

}  // namespace

void prime_dispatch_launch_state() { resident_dispatch_warps(); }

cudaError_t launch_dispatch_bf16(const DispatchArgs& args, cudaStream_t stream) {
    const DispatchArgs a = with_pad_blocks(args);
    const int H16 = a.H / 8;
    const int per_item = 32 * kBf16Unroll;
    const int segs = (H16 + per_item - 1) / per_item;
    const int64_t items = static_cast<int64_t>(a.T) * segs;
    if (items == 0) return cudaSuccess;
    // a grid of less than one wave leaves SMs short of warps: halve the items
    // (one 16-byte vector per lane) so twice as many warps share the stores
    if (items < resident_dispatch_warps()) {
        const int segs1 = (H16 + 31) / 32;
        const int64_t items1 = static_cast<int64_t>(a.T) * segs1;
        const int64_t blocks1 = (items1 + kWarpsPerBlock - 1) / kWarpsPerBlock + a.pad_blocks;
        return launch_dispatch_kernel(dispatch_bf16_kernel<1>, blocks1, stream, a, items1, segs1);
    }
    const int64_t blocks = (items + kWarpsPerBlock - 1) / kWarpsPerBlock + a.pad_blocks;
    return launch_dispatch_kernel(dispatch_bf16_kernel<kBf16Unroll>, blocks, stream, a, items, segs);
}

cudaError_t launch_fill_pad_rows(const int32_t* counts, const int32_t* offsets, int E, int64_t row_bytes,
                                 void* recv, const PadScales& scales, int32_t* src, float* weights,
                                 cudaStream_t stream, int max_pad) {
    if (E == 0 || max_pad <= 0) return cudaSuccess;
    const int64_t items = static_cast<int64_t>(E) * max_pad;
    const int64_t blocks = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_dependent(fill_pad_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kWarpsPerBlock * 32), 0,
                            stream, counts, offsets, E, max_pad, row_bytes, static_cast<char*>(recv), scales, src,
                            weights);
}

cudaError_t launch_dispatch_fp8_passthrough(const DispatchArgs& args, cudaStream_t stream) {
    const DispatchArgs a = with_pad_blocks(args);
    const int V = a.H / 16;
    const int per_item = 32 * kBf16Unroll;
    const int segs = (V + per_item - 1) / per_item;
    const int64_t items = static_cast<int64_t>(a.T) * segs;
    if (items == 0) return cudaSuccess;
    const int64_t g = (items + kWarpsPerBlock - 1) / kWarpsPerBlock + a.pad_blocks;
    if (a.scale_col_major)
        return launch_dispatch_kernel(dispatch_fp8_passthrough_kernel<true>, g, stream, a, items, segs);
    return launch_dispatch_kernel(dispatch_fp8_passthrough_kernel<false>, g, stream, a, items, segs);
}

namespace {

template <int kMode, int kFmt>
cudaError_t launch_fp8_variant(const DispatchArgs& a, int64_t g, cudaStream_t stream, int64_t items, int segs) {
    if (a.scale_col_major)
        return launch_dispatch_kernel(dispatch_fp8_kernel<kMode, true, kFmt>, g, stream, a, items, segs);
    return launch_dispatch_kernel(dispatch_fp8_kernel<kMode, false, kFmt>, g, stream, a, items, segs);
}

template <int kFmt>
cudaError_t launch_fp8_format(const DispatchArgs& a, int64_t g, cudaStream_t stream, int64_t items, int segs) {
    if (a.scale_mode == EP_SCALE_POW2) return launch_fp8_variant<EP_SCALE_POW2, kFmt>(a, g, stream, items, segs);
    if (a.scale_mode == EP_SCALE_UE8M0) return launch_fp8_variant<EP_SCALE_UE8M0, kFmt>(a, g, stream, items, segs);
    return launch_fp8_variant<EP_SCALE_FP32, kFmt>(a, g, stream, items, segs);
}

}  // namespace

cudaError_t launch_dispatch_fp8(const DispatchArgs& args, cudaStream_t stream) {
    const DispatchArgs a = with_pad_blocks(args);
    const int G = a.H / 16;                           // 16-channel groups per row
    const int per_item = 32 * kFp8Unroll;
    const int segs = (G + per_item - 1) / per_item;
    const int64_t items = static_cast<int64_t>(a.T) * segs;
    if (items == 0) return cudaSuccess;
    const int64_t g = (items + kWarpsPerBlock - 1) / kWarpsPerBlock + a.pad_blocks;
    if (a.fp8_format == EP_DTYPE_FP8_E5M2) return launch_fp8_format<EP_DTYPE_FP8_E5M2>(a, g, stream, items, segs);
    return launch_fp8_format<EP_DTYPE_FP8_E4M3>(a, g, stream, items, segs);
}

}  // namespace ep
