// Quantization kernels of the W8A8 Linear ("TurboDiffusion Integration Notes",
// section "Reused Components", W8A8 Linear: weights quantized to INT8 once,
// activations quantized dynamically before each Linear), and the exact
// int8 -> bf16 image the tensor-core GEMM consumes.
//
// Quantizer: s = absmax / 127 (IEEE fp32 division); q = clamp(rne(x / s),
// -127, 127) with x / s an IEEE fp32 division; absmax 0 gives s = 0, q = 0.
//
// The per-element division is evaluated as t = x * (1/s), where 1/s is the
// correctly rounded reciprocal.  Error bound: with u = 2^-24, t and the
// correctly rounded quotient fl(x/s) both lie within 3u*|x/s| <= 3u*127.01
// (< 2.3e-5) of each other, so they round to the same integer unless one of
// them is within that distance of a half-integer.  Elements whose t lies
// within 2^-14 (6.1e-5) of a half-integer take the exact path (IEEE division
// and round-half-even); every other element provably gets the same q.
//
// Rounding uses the 1.5 * 2^23 constant: for |t| < 2^22, fl(t + 1.5*2^23)
// rounds t to the nearest integer with ties to even, and the low byte of its
// bit pattern is that integer in two's complement.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace w8a8 {

namespace {

constexpr float kQMax = 127.0f;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kTieGuard = 6.103515625e-05f;  // 2^-14

struct RowScale {
    float s;    // stored scale
    float inv;  // correctly rounded 1/s (0 when s == 0)
};

__device__ __forceinline__ RowScale make_scale(float amax) {
    RowScale r;
    r.s = __fdiv_rn(amax, kQMax);
    r.inv = (r.s > 0.0f) ? __frcp_rn(r.s) : 0.0f;
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Exact path: IEEE quotient, round half to even, clamp.
__device__ __noinline__ int quant_exact(float x, float s) {
    if (s == 0.0f) return 0;
    float r = rintf(__fdiv_rn(x, s));
    r = fminf(fmaxf(r, -kQMax), kQMax);
    return static_cast<int>(r);
}

// Quantize one value; returns the int8 code in the low byte.
__device__ __forceinline__ uint32_t quant_one(float x, const RowScale& sc) {
    const float t = __fmul_rn(x, sc.inv);
    const float big = __fadd_rn(t, kRoundMagic);
    const float r = __fsub_rn(big, kRoundMagic);
    const float dist = fabsf(__fsub_rn(t, r));  // exact: |t - rne(t)| <= 0.5
    // Near-ties take the exact path; so does a NaN distance, which arises only
    // when 1/s overflowed (s below 2^-128) and must not be trusted.
    if (!(dist <= 0.5f - kTieGuard)) return static_cast<uint32_t>(quant_exact(x, sc.s)) & 0xFFu;
    // |t| <= 127.01, so r is within [-127, 127] except through rounding slop
    // at the boundary; clamp on the biased value keeps the byte extraction valid.
    const float lo = kRoundMagic - kQMax, hi = kRoundMagic + kQMax;
    const float c = fminf(fmaxf(big, lo), hi);
    return __float_as_uint(c) & 0xFFu;
}

// absmax of the 8 bf16 values in a 16-byte chunk, as a non-negative float.
__device__ __forceinline__ float chunk_absmax(const uint4& v) {
    // Clearing the sign bits gives |x| for each bf16 half; bf16x2 max of
    // non-negative finite values is exact.
    const uint32_t m = 0x7FFF7FFFu;
    uint32_t w[4] = {v.x & m, v.y & m, v.z & m, v.w & m};
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&w[0]);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&w[1]);
    __nv_bfloat162 c = *reinterpret_cast<__nv_bfloat162*>(&w[2]);
    __nv_bfloat162 d = *reinterpret_cast<__nv_bfloat162*>(&w[3]);
    __nv_bfloat162 x = __hmax2(__hmax2(a, b), __hmax2(c, d));
    const uint32_t xb = *reinterpret_cast<uint32_t*>(&x);
    return fmaxf(bf16_lo(xb), bf16_hi(xb));
}

__device__ __forceinline__ uint32_t quant_word(uint32_t w, const RowScale& sc) {
    uint32_t q0 = quant_one(bf16_lo(w), sc);
    uint32_t q1 = quant_one(bf16_hi(w), sc);
    return q0 | (q1 << 8);
}

// 8 bf16 -> 8 int8 packed into a uint2.
__device__ __forceinline__ uint2 quant_chunk(const uint4& v, const RowScale& sc) {
    uint2 o;
    o.x = quant_word(v.x, sc) | (quant_word(v.y, sc) << 16);
    o.y = quant_word(v.z, sc) | (quant_word(v.w, sc) << 16);
    return o;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    const int nw = blockDim.x >> 5;
    float r = (lane < nw) ? red[lane] : 0.0f;
    r = warp_max(r);
    __syncthreads();  // red[] may be reused by the caller
    return r;
}

// One CTA per row of A[R,K]; the row stays in registers (CPT 16-byte chunks
// per thread) between the absmax pass and the quantize pass.
template <int CPT>
__global__ void __launch_bounds__(256) quant_rows_reg_kernel(const uint4* __restrict__ A, int64_t R, int64_t K,
                                                             uint2* __restrict__ Aq, float* __restrict__ s) {
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    if (row >= R) return;
    const int64_t chunks = K >> 3;
    const uint4* a = A + row * chunks;
    uint4 v[CPT];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * blockDim.x;
        if (c < chunks) {
            v[i] = __ldcs(a + c);
            amax = fmaxf(amax, chunk_absmax(v[i]));
        }
    }
    amax = block_max(amax, red);
    const RowScale sc = make_scale(amax);
    if (threadIdx.x == 0) s[row] = sc.s;
    uint2* q = Aq + row * chunks;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * blockDim.x;
        if (c < chunks) __stcs(q + c, quant_chunk(v[i], sc));
    }
}

// Rows too long to keep in registers: absmax pass, then a second read.
__global__ void __launch_bounds__(256) quant_rows_2pass_kernel(const uint4* __restrict__ A, int64_t R, int64_t K,
                                                               uint2* __restrict__ Aq, float* __restrict__ s) {
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    if (row >= R) return;
    const int64_t chunks = K >> 3;
    const uint4* a = A + row * chunks;
    float amax = 0.0f;
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) amax = fmaxf(amax, chunk_absmax(a[c]));
    amax = block_max(amax, red);
    const RowScale sc = make_scale(amax);
    if (threadIdx.x == 0) s[row] = sc.s;
    uint2* q = Aq + row * chunks;
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) __stcs(q + c, quant_chunk(__ldcs(a + c), sc));
}

// 1x128 activation blocks: 16 lanes own one block (8 bf16 each).  Each warp
// handles two blocks per step and UNROLL steps per iteration of a grid-stride
// loop, with all loads of an iteration issued before any arithmetic.
template <int UNROLL>
__global__ void __launch_bounds__(256) quant_act_block_kernel(const uint4* __restrict__ X, int64_t n_blocks,
                                                              uint2* __restrict__ Xq, float* __restrict__ sx) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, sub = lane & 15;
    const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps_total = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp_global * 2 * UNROLL; base < n_blocks; base += warps_total * 2 * UNROLL) {
        uint4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            if (blk < n_blocks) v[u] = __ldcs(X + blk * 16 + sub);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            float m = (blk < n_blocks) ? chunk_absmax(v[u]) : 0.0f;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const RowScale sc = make_scale(m);
            if (blk < n_blocks) {
                __stcs(Xq + blk * 16 + sub, quant_chunk(v[u], sc));
                if (sub == 0) sx[blk] = sc.s;
            }
        }
    }
}

// 128x128 weight blocks: one CTA (256 threads) per block; 8 chunks each.
__global__ void __launch_bounds__(256) quant_weight_block_kernel(const uint4* __restrict__ W, int64_t N, int64_t K,
                                                                 uint2* __restrict__ Wq, float* __restrict__ sw) {
    __shared__ float red[32];
    const int64_t kb = blockIdx.x, nb = blockIdx.y;
    const int64_t kbs = K >> 7;
    const int64_t chunks_per_row = K >> 3;
    // chunk c of the block: row nb*128 + c/16, 16-byte column chunk kb*16 + c%16
    uint4 v[8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = threadIdx.x + i * 256;
        const int64_t n = nb * 128 + (c >> 4);
        if (n < N) {
            v[i] = W[n * chunks_per_row + kb * 16 + (c & 15)];
            amax = fmaxf(amax, chunk_absmax(v[i]));
        }
    }
    amax = block_max(amax, red);
    const RowScale sc = make_scale(amax);
    if (threadIdx.x == 0) sw[nb * kbs + kb] = sc.s;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = threadIdx.x + i * 256;
        const int64_t n = nb * 128 + (c >> 4);
        if (n < N) Wq[n * chunks_per_row + kb * 16 + (c & 15)] = quant_chunk(v[i], sc);
    }
}

// int8 -> bf16, exact.  For a byte b holding x in two's complement,
// bits 0x4B000000 | (b ^ 0x80) encode 2^23 + x + 128, and subtracting
// 2^23 + 128 gives x exactly; bf16 holds every integer in [-128, 127].
__device__ __forceinline__ uint32_t s8x2_to_bf16x2(uint32_t w, int first) {
    const float k = 8388736.0f;  // 2^23 + 128
    const uint32_t flipped = w ^ 0x80808080u;
    const float f0 = __fsub_rn(__uint_as_float(0x4B000000u | ((flipped >> (8 * first)) & 0xFFu)), k);
    const float f1 = __fsub_rn(__uint_as_float(0x4B000000u | ((flipped >> (8 * first + 8)) & 0xFFu)), k);
    __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(256) expand_s8_bf16_kernel(const uint4* __restrict__ src, int64_t n16,
                                                             uint4* __restrict__ dst) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint4 v = __ldcs(src + i);
        uint4 o0, o1;
        o0.x = s8x2_to_bf16x2(v.x, 0);
        o0.y = s8x2_to_bf16x2(v.x, 2);
        o0.z = s8x2_to_bf16x2(v.y, 0);
        o0.w = s8x2_to_bf16x2(v.y, 2);
        o1.x = s8x2_to_bf16x2(v.z, 0);
        o1.y = s8x2_to_bf16x2(v.z, 2);
        o1.z = s8x2_to_bf16x2(v.w, 0);
        o1.w = s8x2_to_bf16x2(v.w, 2);
        dst[2 * i] = o0;
        dst[2 * i + 1] = o1;
    }
}

}  // namespace

cudaError_t launch_quant_rows(const void* A, int64_t R, int64_t K, int8_t* Aq, float* s, cudaStream_t st) {
    const int64_t chunks = K >> 3;
    const uint4* a = static_cast<const uint4*>(A);
    uint2* q = reinterpret_cast<uint2*>(Aq);
    const dim3 grid(static_cast<unsigned>(R));
    if (chunks <= 256)
        quant_rows_reg_kernel<1><<<grid, chunks <= 128 ? 128 : 256, 0, st>>>(a, R, K, q, s);
    else if (chunks <= 512)
        quant_rows_reg_kernel<2><<<grid, 256, 0, st>>>(a, R, K, q, s);
    else if (chunks <= 1024)
        quant_rows_reg_kernel<4><<<grid, 256, 0, st>>>(a, R, K, q, s);
    else if (chunks <= 2048)
        quant_rows_reg_kernel<8><<<grid, 256, 0, st>>>(a, R, K, q, s);
    else
        quant_rows_2pass_kernel<<<grid, 256, 0, st>>>(a, R, K, q, s);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_block(const void* X, int64_t M, int64_t K, int8_t* Xq, float* sx, int num_sms,
                                   cudaStream_t st) {
    const int64_t n_blocks = M * (K >> 7);
    constexpr int kUnroll = 4;
    const int64_t warps_needed = (n_blocks + 2 * kUnroll - 1) / (2 * kUnroll);
    int64_t grid = (warps_needed + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    quant_act_block_kernel<kUnroll><<<static_cast<unsigned>(grid), 256, 0, st>>>(
        static_cast<const uint4*>(X), n_blocks, reinterpret_cast<uint2*>(Xq), sx);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight_block(const void* W, int64_t N, int64_t K, int8_t* Wq, float* sw,
                                      cudaStream_t st) {
    const dim3 grid(static_cast<unsigned>(K >> 7), static_cast<unsigned>((N + 127) >> 7));
    quant_weight_block_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(W), N, K,
                                                    reinterpret_cast<uint2*>(Wq), sw);
    return cudaGetLastError();
}

cudaError_t launch_expand_s8_bf16(const int8_t* src, int64_t n, void* dst, int num_sms, cudaStream_t st) {
    const int64_t n16 = n >> 4;
    int64_t grid = (n16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    expand_s8_bf16_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(reinterpret_cast<const uint4*>(src), n16,
                                                                       static_cast<uint4*>(dst));
    return cudaGetLastError();
}

}  // namespace w8a8
