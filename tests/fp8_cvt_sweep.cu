// Test-only kernel: every fp32 bit pattern in [lo, lo + n) through the
// hardware conversions the fp8 dispatch uses (cvt.rn.satfinite.e4m3x2.f32 and
// cvt.rn.satfinite.e5m2x2.f32), so that the oracle's encoders can be checked
// against them over all 2^32 inputs. Built by the test that uses it; not part
// of the library.
#include <cstdint>

#include <cuda_runtime.h>

namespace {

__global__ void cvt_sweep_kernel(uint32_t lo, uint32_t n, uint8_t* q4, uint8_t* q5) {
    // each thread converts one pair of consecutive patterns (n is even)
    const uint32_t i = (blockIdx.x * blockDim.x + threadIdx.x) * 2u;
    if (i >= n) return;
    const float a = __uint_as_float(lo + i);
    const float b = __uint_as_float(lo + i + 1u);
    unsigned short d4, d5;
    // the first source operand goes to the high byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d4) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d5) : "f"(b), "f"(a));
    q4[i] = static_cast<uint8_t>(d4 & 0xffu);
    q4[i + 1u] = static_cast<uint8_t>(d4 >> 8);
    q5[i] = static_cast<uint8_t>(d5 & 0xffu);
    q5[i + 1u] = static_cast<uint8_t>(d5 >> 8);
}

}  // namespace

// q4 and q5 are device buffers of n bytes; n even, lo + n <= 2^32.
extern "C" int fp8_cvt_sweep(uint32_t lo, uint32_t n, uint8_t* q4, uint8_t* q5, void* stream) {
    if (n == 0) return 0;
    if ((n & 1u) != 0u || q4 == nullptr || q5 == nullptr) return 1;
    if (static_cast<uint64_t>(lo) + n > (uint64_t{1} << 32)) return 1;
    const uint32_t pairs = n / 2u;
    const unsigned threads = 256;
    const unsigned blocks = (pairs + threads - 1u) / threads;
    cvt_sweep_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(lo, n, q4, q5);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
