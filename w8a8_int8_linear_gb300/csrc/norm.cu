// RMSNorm / LayerNorm fused with per-token activation quantization
// ("TurboDiffusion Integration Notes", section "Reused Components": FastNorm
// replaces RMSNorm/LayerNorm with fused implementations; W8A8 + FastNorm is
// the one combined stage of section "End-to-End Result").  One read of each
// row; it leaves as int8 codes (and/or their bf16 image for the GEMM) plus the
// per-token scale, and optionally as the normalized bf16 row.
//
//   RMSNorm:   r = 1 / sqrt(S(x*x) / K + eps),  y = bf16((x * r) * gamma)
//   LayerNorm: mu = S(x) / K, d = x - mu, r = 1 / sqrt(S(d*d) / K + eps),
//              y = bf16(((d * r) * gamma) + beta)
// then s = absmax(y) / 127, q = clamp(rne(y / s), -127, 127).  A missing
// gamma or beta skips that operation; every operation is IEEE binary32,
// rounded on its own.
//
// S() has a fixed order that does not depend on the launch shape: chunks of 8
// consecutive elements summed left to right, then the chunk sums, zero-padded
// to P = the next power of two of K/8, added pairwise level by level.  A CTA
// of T threads gives thread t the C consecutive chunks [tC, (t+1)C) with
// T*C = P (or T = 32 and only the first P/C threads holding chunks when
// P/C < 32); the first log2(C) levels of the tree are inside a thread, the
// next ones XOR shuffles between lanes (lane t and t^o hold adjacent subtrees;
// IEEE addition is commutative, so both get the same sum), the last ones the
// same butterfly over the per-warp sums.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "quant_core.cuh"

namespace w8a8 {

namespace {

// Pairwise tree over the block's per-thread subtree sums (threads [0, tree)
// hold subtrees in chunk order; tree is a power of two).  Every thread gets
// the total.
__device__ __forceinline__ float tree_sum_block(float v, int tree, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int lanes = tree < 32 ? tree : 32;
    for (int o = 1; o < lanes; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (tree <= 32) return __shfl_sync(0xffffffffu, v, 0);
    const int W = tree >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = (lane < W) ? red[lane] : 0.0f;
    for (int o = 1; o < W; o <<= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
    t = __shfl_sync(0xffffffffu, t, 0);
    __syncthreads();  // red[] is reused by the next reduction
    return t;
}

__device__ __forceinline__ float block_absmax(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = (lane < nw) ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
    __syncthreads();
    return t;
}

// Pairwise tree over this thread's C chunk sums (C a power of two).
template <int C>
__device__ __forceinline__ float tree_sum_local(float (&s)[C]) {
#pragma unroll
    for (int w = C; w > 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w / 2; ++i) s[i] = __fadd_rn(s[2 * i], s[2 * i + 1]);
    }
    return s[0];
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf16_lo(w[i]);
        f[2 * i + 1] = bf16_hi(w[i]);
    }
}

template <int C>
__global__ void __launch_bounds__(512) norm_quant_kernel(const uint4* __restrict__ X, const uint4* __restrict__ gamma,
                                                         const uint4* __restrict__ beta, float eps, int layer,
                                                         int K, int tree, uint4* __restrict__ Y,
                                                         uint2* __restrict__ Xq, uint4* __restrict__ img,
                                                         float* __restrict__ sx) {
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int chunks = K >> 3;
    const uint4* x = X + row * chunks;
    const int c0 = threadIdx.x * C;
    uint4 v[C];
#pragma unroll
    for (int i = 0; i < C; ++i) v[i] = (c0 + i < chunks) ? __ldcs(x + c0 + i) : make_uint4(0, 0, 0, 0);
    const float Kf = static_cast<float>(K);
    float mu = 0.0f;
    if (layer) {
        float s[C];
#pragma unroll
        for (int i = 0; i < C; ++i) {
            float f[8];
            unpack8(v[i], f);
            float a = f[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) a = __fadd_rn(a, f[j]);
            s[i] = (c0 + i < chunks) ? a : 0.0f;
        }
        mu = __fdiv_rn(tree_sum_block(tree_sum_local(s), tree, red), Kf);
    }
    float s[C];
#pragma unroll
    for (int i = 0; i < C; ++i) {
        float f[8];
        unpack8(v[i], f);
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float d = layer ? __fsub_rn(f[j], mu) : f[j];
            const float t = __fmul_rn(d, d);
            a = (j == 0) ? t : __fadd_rn(a, t);
        }
        s[i] = (c0 + i < chunks) ? a : 0.0f;
    }
    const float var = __fdiv_rn(tree_sum_block(tree_sum_local(s), tree, red), Kf);
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(var, eps)));
    uint4 yv[C];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < C; ++i) {
        const int c = c0 + i;
        if (c >= chunks) {
            yv[i] = make_uint4(0, 0, 0, 0);
            continue;
        }
        float f[8], g[8], b[8];
        unpack8(v[i], f);
        if (gamma) unpack8(__ldg(gamma + c), g);
        if (layer && beta) unpack8(__ldg(beta + c), b);
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            float y0 = __fmul_rn(layer ? __fsub_rn(f[j], mu) : f[j], r);
            float y1 = __fmul_rn(layer ? __fsub_rn(f[j + 1], mu) : f[j + 1], r);
            if (gamma) {
                y0 = __fmul_rn(y0, g[j]);
                y1 = __fmul_rn(y1, g[j + 1]);
            }
            if (layer && beta) {
                y0 = __fadd_rn(y0, b[j]);
                y1 = __fadd_rn(y1, b[j + 1]);
            }
            __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
            o[j >> 1] = *reinterpret_cast<uint32_t*>(&h);
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(o[j >> 1])), fabsf(bf16_hi(o[j >> 1]))));
        }
        yv[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    amax = block_absmax(amax, red);
    const RowScale sc = make_scale_div(amax);
    if (threadIdx.x == 0) sx[row] = sc.s;
#pragma unroll
    for (int i = 0; i < C; ++i) {
        const int c = c0 + i;
        if (c >= chunks) continue;
        if (Y) Y[row * chunks + c] = yv[i];
        if (Xq || img) put_codes(Xq, img, row * chunks + c, quant_chunk(yv[i], sc));
    }
}

}  // namespace

cudaError_t launch_norm_quant(const void* X, const void* gamma, const void* beta, float eps, int layer, int64_t M,
                              int64_t K, void* Y, int8_t* Xq, void* img, float* sx, cudaStream_t st) {
    const int chunks = static_cast<int>(K >> 3);
    int P = 1;
    while (P < chunks) P <<= 1;
    const dim3 grid(static_cast<unsigned>(M));
    const uint4* x = static_cast<const uint4*>(X);
    const uint4* g = static_cast<const uint4*>(gamma);
    const uint4* b = static_cast<const uint4*>(beta);
    uint4* y = static_cast<uint4*>(Y);
    uint2* q = reinterpret_cast<uint2*>(Xq);
    uint4* im = static_cast<uint4*>(img);
    if (P <= 32) {
        norm_quant_kernel<1><<<grid, 32, 0, st>>>(x, g, b, eps, layer, static_cast<int>(K), P, y, q, im, sx);
    } else if (P <= 512) {
        const int T = P / 4 < 32 ? 32 : P / 4;
        norm_quant_kernel<4><<<grid, T, 0, st>>>(x, g, b, eps, layer, static_cast<int>(K), P / 4, y, q, im, sx);
    } else {
        norm_quant_kernel<8><<<grid, P / 8, 0, st>>>(x, g, b, eps, layer, static_cast<int>(K), P / 8, y, q, im, sx);
    }
    return cudaGetLastError();
}

}  // namespace w8a8
