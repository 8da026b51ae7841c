// Quantization kernels of the W8A8 Linear ("TurboDiffusion Integration Notes",
// section "Reused Components", W8A8 Linear: weights quantized to INT8 once,
// activations quantized dynamically before each Linear), and the exact
// int8 -> bf16 image the tensor-core GEMM consumes.
//
// Quantizer: s = absmax / 127 (IEEE fp32 division); q = clamp(rne(x / s),
// -127, 127) with x / s an IEEE fp32 division; absmax 0 gives s = 0, q = 0.
//
// Scales without division.  absmax is a bf16 value, M * 2^k with an 8-bit
// significand M in [128, 255].  Scaling by a power of two commutes with
// rounding while the result stays normal, so fl(absmax / 127) =
// fl(M / 127) * 2^k and fl(1 / s) = fl(1 / fl(M / 127)) * 2^-k.  The two
// 128-entry tables fl(M/127) and fl(1/fl(M/127)) are compile-time constants
// in device memory; a scale is then a table read plus an exponent add.  (An
// exhaustive host check over every bf16 value confirms the identity for
// exponent fields 7..254; the tables are used for 8..250 and every other
// nonzero absmax takes IEEE division.)
//
// Quantizing one value x with P = x * (1/s) (the exact product):
//   big = fma(x, 1/s, 1.5*2^23): for |P| < 2^22 this rounds P to the nearest
//         integer with ties to even, and the low byte of its bit pattern is
//         that integer in two's complement;
//   d   = fma(x, 1/s, -(big - 1.5*2^23)) = P - rne(P), rounded once.
// Error bound: with u = 2^-24, |P - x/s| <= u|x/s| and the IEEE quotient
// fl(x/s) is within u|x/s| of x/s, so P and fl(x/s) are within
// 2u * 127.01 < 1.6e-5 of each other.  They round to different integers only
// if a half-integer lies between them, and then |d| >= 0.5 - 1.6e-5 - 2^-25.
// Any chunk holding a value with |d| > 0.5 - 2^-14 (6.1e-5) takes the exact
// path (IEEE division, round half to even, clamp) for those values; every
// other value provably gets round_half_even(fl(x/s)).
//
// No clamp is needed on the fast path: |x| <= absmax and s >= (absmax/127)
// (1-u), so |P| <= 127 (1+u)^2 < 127.5 and rne(P) lies in [-127, 127].  That
// bound needs a normal s; a group whose scale is subnormal takes the exact
// path for every element, which clamps.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gelu.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "quant_core.cuh"

namespace w8a8 {

namespace {

// fl(M / 127) and fl(1 / fl(M / 127)) for M = 128 + i, i in [0, 128): built
// at compile time (the host compiler folds IEEE single-precision division
// with round to nearest) and placed in device global memory, where the
// per-block lookups of the 1x128 and 128x128 kernels hit L1.
struct ScaleTables {
    float T[128];
    float R[128];
};

constexpr ScaleTables make_scale_tables() {
    ScaleTables t{};
    for (int i = 0; i < 128; ++i) {
        t.T[i] = static_cast<float>(128 + i) / 127.0f;
        t.R[i] = 1.0f / t.T[i];
    }
    return t;
}

__device__ const ScaleTables kScaleTables = make_scale_tables();

__device__ __forceinline__ RowScale make_scale(float amax, const ScaleTables& t = kScaleTables) {
    RowScale r;
    const uint32_t b = __float_as_uint(amax);  // a bf16 value: low 16 bits are zero
    const int ef = static_cast<int>(b >> 23);
    if (ef >= 8 && ef <= 250) {
        const int f = static_cast<int>((b >> 16) & 0x7Fu);
        const int k = ef - 134;
        r.s = __uint_as_float(__float_as_uint(__ldg(&t.T[f])) + (k << 23));
        r.inv = __uint_as_float(__float_as_uint(__ldg(&t.R[f])) - (k << 23));
        r.exact = false;
    } else {
        r.s = __fdiv_rn(amax, kQMax);
        r.inv = (r.s > 0.0f) ? __frcp_rn(r.s) : 0.0f;
        r.exact = r.s > 0.0f && r.s < kMinNormal;
    }
    return r;
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

// One CTA of T threads per row of A[R,K]; the row stays in registers (CPT
// 16-byte chunks per thread) between the absmax pass and the quantize pass,
// so it is read from memory once.  MINB CTAs per SM bound the registers
// (65536 / (T * MINB) per thread); with many rows, small CTAs and many of them
// per SM keep the most bytes in flight (one 64-thread CTA per 5120-wide row,
// 16 per SM: 160 KB of loads in flight per SM).
template <int CPT, int T, int MINB, int OUT>
__global__ void __launch_bounds__(T, MINB) quant_rows_reg_kernel(const uint4* __restrict__ A, int64_t R, int64_t K,
                                                                 uint2* __restrict__ Aq, uint4* __restrict__ img,
                                                                 float* __restrict__ s) {
    grid_launch_dependents();
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    if (row >= R) return;
    const int64_t chunks = K >> 3;
    const uint4* a = A + row * chunks;
    uint4 v[CPT];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * T;
        if (c < chunks) v[i] = __ldcs(a + c);
    }
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * T;
        if (c < chunks) amax = fmaxf(amax, chunk_absmax(v[i]));
    }
    amax = T > 32 ? block_max(amax, red) : warp_max(amax);
    const RowScale sc = make_scale_div(amax);
    if (threadIdx.x == 0) s[row] = sc.s;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * T;
        if (c < chunks) emit_chunk<OUT>(Aq, img, row * chunks + c, v[i], sc);
    }
}

// 8 int8 codes -> their 8 exact fp16 values: the byte b ^ 0x80 under the
// exponent of 1024 (0x64xx is 1024 + (b ^ 0x80)), less 1152.
__device__ __forceinline__ uint4 s8x8_to_f16x8(uint2 c) {
    const __half2 k1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const uint32_t w0 = c.x ^ 0x80808080u, w1 = c.y ^ 0x80808080u;
    uint32_t p[4] = {__byte_perm(w0, 0x64646464u, 0x4140), __byte_perm(w0, 0x64646464u, 0x4342),
                     __byte_perm(w1, 0x64646464u, 0x4140), __byte_perm(w1, 0x64646464u, 0x4342)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&p[i]), k1152);
        p[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(p[0], p[1], p[2], p[3]);
}

// Per-token quantization feeding the few-token GEMM on int8 weight codes: one
// CTA per row (kept in registers, as quant_rows_reg_kernel) writes the row's
// scale, its codes when Aq is given, and the fp16 image of its codes (the
// GEMM's token operand), and zeroes its share of the GEMM's split-K sums and
// counters (nz16 16-byte words at zero).
template <int CPT, int T>
__global__ void __launch_bounds__(T) quant_tokens_f16_kernel(const uint4* __restrict__ A, int64_t R, int64_t K,
                                                             uint2* __restrict__ Aq, uint4* __restrict__ img16,
                                                             float* __restrict__ s, uint4* __restrict__ zero,
                                                             int64_t nz16) {
    grid_launch_dependents();
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    if (row >= R) return;
    {
        const int64_t per = (nz16 + R - 1) / R;
        const int64_t z0 = row * per;
        const int64_t z1 = z0 + per < nz16 ? z0 + per : nz16;
        for (int64_t i = z0 + threadIdx.x; i < z1; i += T) zero[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    const int64_t chunks = K >> 3;
    const uint4* a = A + row * chunks;
    uint4 v[CPT];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * T;
        if (c < chunks) v[i] = __ldcs(a + c);
    }
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * T;
        if (c < chunks) amax = fmaxf(amax, chunk_absmax(v[i]));
    }
    amax = block_max(amax, red);
    const RowScale sc = make_scale_div(amax);
    if (threadIdx.x == 0) s[row] = sc.s;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * T;
        if (c < chunks) {
            const uint2 code = quant_chunk(v[i], sc);
            if (Aq) __stcs(Aq + row * chunks + c, code);
            img16[row * chunks + c] = s8x8_to_f16x8(code);
        }
    }
}

// One warp per row, two passes: the absmax pass streams the row with U
// 16-byte loads per lane in flight, the quantize pass reads it again (from
// L2, where the first pass left it) and writes the codes.  Few registers, so
// many rows are in flight per SM.
template <int U>
__global__ void __launch_bounds__(256, 4) quant_rows_warp2_kernel(const uint4* __restrict__ A, int64_t R, int64_t K,
                                                                  uint2* __restrict__ Aq, uint4* __restrict__ img,
                                                                  float* __restrict__ s) {
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= R) return;
    const int chunks = static_cast<int>(K >> 3);
    const uint4* a = A + row * chunks;
    float amax = 0.0f;
    for (int c0 = 0; c0 < chunks; c0 += 32 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + lane + 32 * u;
            if (c < chunks) v[u] = a[c];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + lane + 32 * u;
            if (c < chunks) amax = fmaxf(amax, chunk_absmax(v[u]));
        }
    }
    amax = warp_max(amax);
    const RowScale sc = make_scale_div(amax);
    if (lane == 0) s[row] = sc.s;
    for (int c0 = 0; c0 < chunks; c0 += 32 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + lane + 32 * u;
            if (c < chunks) v[u] = __ldcs(a + c);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + lane + 32 * u;
            if (c < chunks) put_codes(Aq, img, row * chunks + c, quant_chunk(v[u], sc));
        }
    }
}

// Rows too long to keep in registers: absmax pass, then a second read.
__global__ void __launch_bounds__(256) quant_rows_2pass_kernel(const uint4* __restrict__ A, int64_t R, int64_t K,
                                                               uint2* __restrict__ Aq, uint4* __restrict__ img,
                                                               float* __restrict__ s) {
    grid_launch_dependents();
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    if (row >= R) return;
    const int64_t chunks = K >> 3;
    const uint4* a = A + row * chunks;
    float amax = 0.0f;
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) amax = fmaxf(amax, chunk_absmax(a[c]));
    amax = block_max(amax, red);
    const RowScale sc = make_scale_div(amax);
    if (threadIdx.x == 0) s[row] = sc.s;
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x)
        put_codes(Aq, img, row * chunks + c, quant_chunk(__ldcs(a + c), sc));
}

// 1x128 activation blocks: 4 lanes own one block (4 chunks of 8 bf16 each),
// so a warp handles 8 blocks per step.  For chunk i of its block, lane l reads
// 16 bytes at offset 16 * ((l & 3) + 4 i) of block (l >> 2): each load
// instruction of the warp covers 8 runs of 64 contiguous bytes.  A grid-stride
// loop with UNROLL steps per iteration keeps 64 * UNROLL bytes per lane in
// flight.
template <int UNROLL>
__global__ void __launch_bounds__(256) quant_act_block_kernel(const uint4* __restrict__ X, int64_t n_blocks,
                                                              uint2* __restrict__ Xq, uint4* __restrict__ img,
                                                              float* __restrict__ sx) {
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int sub = lane & 3, bl = lane >> 2;
    const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps_total = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp_global * 8 * UNROLL; base < n_blocks; base += warps_total * 8 * UNROLL) {
        uint4 v[UNROLL][4];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 8 * u + bl;
            if (blk < n_blocks) {
#pragma unroll
                for (int i = 0; i < 4; ++i) v[u][i] = __ldcs(X + blk * 16 + sub + 4 * i);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 8 * u + bl;
            float m = 0.0f;
            if (blk < n_blocks) {
#pragma unroll
                for (int i = 0; i < 4; ++i) m = fmaxf(m, chunk_absmax(v[u][i]));
            }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const RowScale sc = make_scale(m);
            if (blk < n_blocks) {
#pragma unroll
                for (int i = 0; i < 4; ++i) put_codes(Xq, img, blk * 16 + sub + 4 * i, quant_chunk(v[u][i], sc));
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

__global__ void __launch_bounds__(256) expand_s8_bf16_kernel(const uint4* __restrict__ src, int64_t n16,
                                                             uint4* __restrict__ dst) {
    grid_launch_dependents();
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

// Test export of the FFN up-projection's activation: G[i] = bf16(gelu(Y[i]))
// with the epilogue's own device function (gelu.cuh), 8 values per thread.
__global__ void __launch_bounds__(256) gelu_bf16_kernel(const uint4* __restrict__ y, int64_t n8,
                                                        uint4* __restrict__ g) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const uint4 v = y[i];
        uint4 o;
        o.x = gelu_bf16x2(bf16_lo(v.x), bf16_hi(v.x));
        o.y = gelu_bf16x2(bf16_lo(v.y), bf16_hi(v.y));
        o.z = gelu_bf16x2(bf16_lo(v.z), bf16_hi(v.z));
        o.w = gelu_bf16x2(bf16_lo(v.w), bf16_hi(v.w));
        g[i] = o;
    }
}

}  // namespace

cudaError_t launch_quant_rows(const void* A, int64_t R, int64_t K, int8_t* Aq, void* img, float* s, int num_sms,
                              cudaStream_t st) {
    const int64_t chunks = K >> 3;
    const uint4* a = static_cast<const uint4*>(A);
    uint2* q = reinterpret_cast<uint2*>(Aq);
    uint4* im = static_cast<uint4*>(img);
    const dim3 grid(static_cast<unsigned>(R));
    // Many rows (at least 16 per SM): CTAs sized for bytes in flight.  Fewer
    // rows: 128- or 256-thread CTAs, so that each row's loads spread over
    // more threads and the few rows finish sooner.
    const bool many = R >= static_cast<int64_t>(num_sms) * 16;
    const int out = (q ? kOutCodes : 0) | (im ? kOutImage : 0);
    auto reg = [&](auto kern, int threads) { kern<<<grid, threads, 0, st>>>(a, R, K, q, im, s); };
#define W8A8_ROWS(CPT, T, MINB)                                                       \
    (out == kOutCodes   ? reg(quant_rows_reg_kernel<CPT, T, MINB, kOutCodes>, T)      \
     : out == kOutImage ? reg(quant_rows_reg_kernel<CPT, T, MINB, kOutImage>, T)      \
                        : reg(quant_rows_reg_kernel<CPT, T, MINB, kOutBoth>, T))
    if (chunks <= 128)
        W8A8_ROWS(1, 128, 8);
    else if (chunks <= 256)
        W8A8_ROWS(2, 128, 8);
    else if (chunks <= 512)
        W8A8_ROWS(4, 128, 8);
    else if (many && chunks <= 640)
        W8A8_ROWS(10, 64, 16);
    else if (many && chunks <= 1024)
        W8A8_ROWS(8, 128, 8);
    else if (chunks <= 1024)
        W8A8_ROWS(4, 256, 1);
    else if (chunks <= 2048)
        W8A8_ROWS(8, 256, 4);
#undef W8A8_ROWS
    else if (chunks <= 16384)
        quant_rows_warp2_kernel<8><<<static_cast<unsigned>((R + 7) / 8), 256, 0, st>>>(a, R, K, q, im, s);
    else
        quant_rows_2pass_kernel<<<grid, 256, 0, st>>>(a, R, K, q, im, s);
    return cudaGetLastError();
}

bool quant_tokens_f16_takes(int64_t K) { return (K >> 3) <= 2048; }

cudaError_t launch_quant_tokens_f16(const void* X, int64_t M, int64_t K, int8_t* Xq, void* img16, float* sx,
                                    void* zero, size_t zero_bytes, cudaStream_t st) {
    const int64_t chunks = K >> 3;
    if (chunks > 2048) return cudaErrorInvalidValue;
    const uint4* a = static_cast<const uint4*>(X);
    uint2* q = reinterpret_cast<uint2*>(Xq);
    uint4* im = static_cast<uint4*>(img16);
    uint4* z = static_cast<uint4*>(zero);
    const int64_t nz16 = static_cast<int64_t>(zero_bytes / 16);
    const dim3 grid(static_cast<unsigned>(M));
    if (chunks <= 128)
        quant_tokens_f16_kernel<1, 128><<<grid, 128, 0, st>>>(a, M, K, q, im, sx, z, nz16);
    else if (chunks <= 256)
        quant_tokens_f16_kernel<2, 128><<<grid, 128, 0, st>>>(a, M, K, q, im, sx, z, nz16);
    else if (chunks <= 512)
        quant_tokens_f16_kernel<4, 128><<<grid, 128, 0, st>>>(a, M, K, q, im, sx, z, nz16);
    else if (chunks <= 1024)
        quant_tokens_f16_kernel<4, 256><<<grid, 256, 0, st>>>(a, M, K, q, im, sx, z, nz16);
    else
        quant_tokens_f16_kernel<8, 256><<<grid, 256, 0, st>>>(a, M, K, q, im, sx, z, nz16);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_block(const void* X, int64_t M, int64_t K, int8_t* Xq, void* img, float* sx,
                                   int num_sms, cudaStream_t st) {
    const int64_t n_blocks = M * (K >> 7);
    constexpr int kUnroll = 2;
    const int64_t warps_needed = (n_blocks + 8 * kUnroll - 1) / (8 * kUnroll);
    int64_t grid = (warps_needed + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    quant_act_block_kernel<kUnroll><<<static_cast<unsigned>(grid), 256, 0, st>>>(
        static_cast<const uint4*>(X), n_blocks, reinterpret_cast<uint2*>(Xq), static_cast<uint4*>(img), sx);
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

cudaError_t launch_gelu_bf16(const void* Y, int64_t n, void* G, int num_sms, cudaStream_t st) {
    const int64_t n8 = n >> 3;
    int64_t grid = (n8 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    gelu_bf16_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<const uint4*>(Y), n8,
                                                                  static_cast<uint4*>(G));
    return cudaGetLastError();
}

cudaError_t quant_read_device_error(unsigned int* code) {
    unsigned int v = 0, z = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_device_error, &z, sizeof z);
    *code = v;
    return e;
}

}  // namespace w8a8
