// Measurement helpers.  First: sustained throughput of the warp-level INT8 tensor
// instruction (mma.sync m16n8k32, s8 x s8 -> s32) on this GPU.  It is the
// measured denominator for "fraction of dense INT8 peak"; it is not part of
// the Linear.  Each warp keeps 8 independent accumulators so the tensor pipe,
// not instruction latency, bounds the loop.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace w8a8 {
namespace {

constexpr int kAcc = 8;

static __device__ int g_sink;

__global__ void __launch_bounds__(256) imma_peak_kernel(int iters) {
    uint32_t a0 = 0x01010101u * (threadIdx.x & 7), a1 = a0 ^ 0x02020202u, a2 = a0 + 0x01000100u, a3 = ~a0 & 0x3F3F3F3Fu;
    uint32_t b0 = 0x01020304u + threadIdx.x, b1 = b0 ^ 0x05050505u;
    int32_t c[kAcc][4];
#pragma unroll
    for (int j = 0; j < kAcc; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kAcc; ++j) {
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                "{%0, %1, %2, %3};"
                : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < kAcc; ++j) s += c[j][0] ^ c[j][1] ^ c[j][2] ^ c[j][3];
    if (s == 0x7FFFFFFF) g_sink = s;  // keeps the loop live; practically never taken
}

// Measurement helper: the memory traffic of an activation quantization --
// read 2 bytes, write 1 byte per element -- as a plain grid-stride stream of
// 16-byte loads and 8-byte stores with no arithmetic to speak of (each
// output byte is the high byte of its input element).  Timed under the same
// conditions as the quantization, it is the floor a streaming kernel of that
// size reaches on this memory system.
__global__ void __launch_bounds__(256) stream_floor_kernel(const uint4* __restrict__ src, int64_t n16,
                                                           uint2* __restrict__ dst) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint4 v = __ldcs(src + i);
        __stcs(dst + i, make_uint2(__byte_perm(v.x, v.y, 0x7531), __byte_perm(v.z, v.w, 0x7531)));
    }
}

}  // namespace

cudaError_t launch_stream_floor(const void* src, int64_t n, void* dst, int num_sms, cudaStream_t st) {
    const int64_t n16 = n >> 3;  // 8 elements per 16-byte load
    int64_t grid = (n16 + 255) / 256;
    if (grid > static_cast<int64_t>(num_sms) * 8) grid = static_cast<int64_t>(num_sms) * 8;
    if (grid < 1) grid = 1;
    stream_floor_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<const uint4*>(src), n16,
                                                                     static_cast<uint2*>(dst));
    return cudaGetLastError();
}

cudaError_t measure_imma_peak(double* tops, int num_sms, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    const int blocks = num_sms * 4, threads = 256;
    const int iters = 4096;
    imma_peak_kernel<<<blocks, threads, 0, st>>>(64);  // warm-up
    cudaEvent_t t0, t1;
    cudaEventCreate(&t0);
    cudaEventCreate(&t1);
    cudaEventRecord(t0, st);
    imma_peak_kernel<<<blocks, threads, 0, st>>>(iters);
    cudaEventRecord(t1, st);
    e = cudaEventSynchronize(t1);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t0, t1);
    cudaEventDestroy(t0);
    cudaEventDestroy(t1);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    const double warps = static_cast<double>(blocks) * threads / 32.0;
    const double ops = warps * iters * kAcc * (2.0 * 16 * 8 * 32);
    *tops = ops / (ms * 1e-3) / 1e12;
    return e;
}

}  // namespace w8a8
