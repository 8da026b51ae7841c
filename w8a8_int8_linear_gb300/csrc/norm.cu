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
// to P = the next power of two of K/8, added pairwise level by level.  Thread
// t of a row's CTA owns the C consecutive chunks [tC, (t+1)C), so the tree
// spans P/C threads; only the warps that hold real chunks are launched (the
// others would hold padding, whose subtree sums are +0 and enter the tree as
// such).  The first log2(C) levels of the tree are inside a thread, the next
// ones XOR shuffles between lanes (lane t and t^o hold adjacent subtrees; IEEE
// addition is commutative, so both get the same sum), the last ones the same
// butterfly over the per-warp sums.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "quant_core.cuh"

namespace w8a8 {

namespace {

// Pairwise tree over the per-thread subtree sums of `tree` threads (a power
// of two) in chunk order.  Threads the launch leaves out (the warps from
// blockDim.x / 32 up to tree / 32) would hold only padding; their subtree
// sums are +0, which is what enters the tree in their place.  Every thread
// gets the total.  `red` is this reduction's own scratch, so one barrier
// suffices.
__device__ __forceinline__ float tree_sum_block(float v, int tree, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int lanes = tree < 32 ? tree : 32;
    for (int o = 1; o < lanes; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (tree <= 32) return __shfl_sync(0xffffffffu, v, 0);
    const int W = tree >> 5;
    const int launched = static_cast<int>(blockDim.x >> 5);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = (lane < W && lane < launched) ? red[lane] : 0.0f;
    for (int o = 1; o < W; o <<= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
    return __shfl_sync(0xffffffffu, t, 0);
}

__device__ __forceinline__ float block_absmax(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (nw == 1) return v;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = (lane < nw) ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
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

// The normalized bf16 values of one chunk, packed.  d = x - mu, d * r and
// (d * r) * gamma run two values at a time on the packed fp32 pipe (a
// subtraction feeding a multiplication and products feeding products, which
// are never contracted); the beta addition is scalar with explicit rounding.
// layer / use_gamma / add_beta are compile-time constants in the specialized
// kernels, so the unrolled chunk code carries no branches on them.
__device__ __forceinline__ uint4 normalize_chunk(const uint4& v, const uint4* __restrict__ gamma,
                                                 const uint4* __restrict__ beta, bool layer, bool use_gamma,
                                                 bool add_beta, int c, float mu, float r) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t gw[4] = {0, 0, 0, 0}, bw[4] = {0, 0, 0, 0};
    if (use_gamma) {
        const uint4 t = __ldg(gamma + c);
        gw[0] = t.x; gw[1] = t.y; gw[2] = t.z; gw[3] = t.w;
    }
    if (add_beta) {
        const uint4 t = __ldg(beta + c);
        bw[0] = t.x; bw[1] = t.y; bw[2] = t.z; bw[3] = t.w;
    }
    const uint64_t r2 = f2_pack(r, r);
    const uint64_t mu2 = f2_pack(mu, mu);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint64_t d = f2_pack(bf16_lo(w[i]), bf16_hi(w[i]));
        if (layer) d = f2_sub(d, mu2);
        float y0, y1;
        uint64_t t = f2_mul(d, r2);
        if (use_gamma) t = f2_mul(t, f2_pack(bf16_lo(gw[i]), bf16_hi(gw[i])));
        f2_unpack(t, y0, y1);
        if (add_beta) {
            y0 = __fadd_rn(y0, bf16_lo(bw[i]));
            y1 = __fadd_rn(y1, bf16_hi(bw[i]));
        }
        __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
        o[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Kernel forms: the generic one tests every option at run time; the two
// common ones (gamma, and for LayerNorm beta; only the code image and the
// scales written) have them fixed at compile time.
enum NormForm : int { kNormGeneric = 0, kNormRmsImage = 1, kNormLayerImage = 2 };

// One row's statistics, normalization and scale.  v holds this thread's
// chunks [c0, c0 + C) of the row as bf16 on entry and their normalized
// values y on exit.  Every chunk slot is normalized without a branch; a slot
// past the row (zeros, gamma and beta read at chunk 0) is left out of the
// absmax by a select.  Each reduction has its own slot of `red`, so one
// barrier per reduction suffices, also from one row to the next.
template <int C>
__device__ __forceinline__ RowScale norm_row(uint4 (&v)[C], const uint4* __restrict__ gamma,
                                             const uint4* __restrict__ beta, float eps, bool layer, bool use_gamma,
                                             bool add_beta, int K, int c0, int tree, float (*red)[32]) {
    const int chunks = K >> 3;
    const float Kf = static_cast<float>(K);
    float mu = 0.0f;
    if (layer) {
        float s[C];
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            float a = bf16_lo(w[0]);
            a = __fadd_rn(a, bf16_hi(w[0]));
#pragma unroll
            for (int j = 1; j < 4; ++j) {
                a = __fadd_rn(a, bf16_lo(w[j]));
                a = __fadd_rn(a, bf16_hi(w[j]));
            }
            s[i] = (c0 + i < chunks) ? a : 0.0f;
        }
        mu = __fdiv_rn(tree_sum_block(tree_sum_local(s), tree, red[0]), Kf);
    }
    // d = x - mu and d * d two values at a time on the packed fp32 pipe (a
    // subtraction feeding a multiplication, a product feeding nothing packed);
    // the sum stays a scalar chain with explicit rounding.
    const uint64_t mu2 = f2_pack(mu, mu);
    float s[C];
#pragma unroll
    for (int i = 0; i < C; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint64_t d = f2_pack(bf16_lo(w[j]), bf16_hi(w[j]));
            if (layer) d = f2_sub(d, mu2);
            float t0, t1;
            f2_unpack(f2_mul(d, d), t0, t1);
            a = (j == 0) ? t0 : __fadd_rn(a, t0);
            a = __fadd_rn(a, t1);
        }
        s[i] = (c0 + i < chunks) ? a : 0.0f;
    }
    const float var = __fdiv_rn(tree_sum_block(tree_sum_local(s), tree, red[1]), Kf);
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(var, eps)));
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < C; ++i) {
        const int c = c0 + i;
        const bool in = c < chunks;
        v[i] = normalize_chunk(v[i], gamma, beta, layer, use_gamma, add_beta, in ? c : 0, mu, r);  // v holds y
        const float ca = chunk_absmax(v[i]);
        amax = in ? fmaxf(amax, ca) : amax;
    }
    return make_scale_div(block_absmax(amax, red[2]));
}

// The code image of this thread's chunks (the specialized forms).  The row's
// path (exact for a subnormal scale) is chosen once, not per chunk.
template <int C>
__device__ __forceinline__ void store_image(const uint4 (&v)[C], const RowScale& sc, uint4* __restrict__ img_row,
                                            int c0, int chunks) {
    auto store = [&](const RowScale& scl) {
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const int c = c0 + i;
            const uint4 q = quant_chunk_img(v[i], scl);
            if (c < chunks) img_row[c] = q;
        }
    };
    RowScale fixed = sc;
    if (sc.exact) {
        fixed.exact = true;
        store(fixed);
    } else {
        fixed.exact = false;
        store(fixed);
    }
}

// One CTA per row; thread t owns chunks [tC, (t+1)C).  The row stays in
// registers as bf16, and so do its normalized values between the absmax and
// the quantization.
template <int C, int TMAX, int MINB, int FORM>
__global__ void __launch_bounds__(TMAX, MINB) norm_quant_kernel(const uint4* __restrict__ X,
                                                                const uint4* __restrict__ gamma,
                                                                const uint4* __restrict__ beta, float eps,
                                                                int layer_arg, int K, int tree,
                                                                uint4* __restrict__ Y, uint2* __restrict__ Xq,
                                                                uint4* __restrict__ img, float* __restrict__ sx) {
    grid_launch_dependents();
    constexpr bool kFixed = FORM != kNormGeneric;
    const bool layer = kFixed ? FORM == kNormLayerImage : layer_arg != 0;
    const bool use_gamma = kFixed ? true : gamma != nullptr;
    const bool add_beta = kFixed ? FORM == kNormLayerImage : (layer && beta != nullptr);
    __shared__ float red[3][32];
    const int64_t row = blockIdx.x;
    const int chunks = K >> 3;
    const uint4* x = X + row * chunks;
    const int c0 = threadIdx.x * C;
    uint4 v[C];
#pragma unroll
    for (int i = 0; i < C; ++i) v[i] = (c0 + i < chunks) ? __ldg(x + c0 + i) : make_uint4(0, 0, 0, 0);
    const RowScale sc = norm_row<C>(v, gamma, beta, eps, layer, use_gamma, add_beta, K, c0, tree, red);
    if (threadIdx.x == 0) sx[row] = sc.s;
    if constexpr (kFixed) {
        store_image<C>(v, sc, img + row * chunks, c0, chunks);
    } else {
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const int c = c0 + i;
            if (c >= chunks) continue;
            const int64_t o = row * chunks + c;
            if (Y) Y[o] = v[i];
            if (img) img[o] = quant_chunk_img(v[i], sc);
            if (Xq) __stcs(Xq + o, quant_chunk(v[i], sc));
        }
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
    // C chunks per thread; only the warps that hold real chunks are
    // launched, the tree still spans P / C threads.
    const int k = static_cast<int>(K);
    auto warps_for = [&](int C) { return ((chunks + C - 1) / C + 31) / 32; };
    // the specialized forms (rows of 257..8192 elements): gamma (and beta
    // exactly for LayerNorm), only the code image and the scales written;
    // held to 64 registers (4 CTAs of 256 threads, 6 rows of 5120 per SM)
    const bool image_only = im && !y && !q && g;
    const int form = (image_only && !layer && !b) ? kNormRmsImage
                     : (image_only && layer && b) ? kNormLayerImage
                                                  : kNormGeneric;
    auto launch = [&](auto kern, int threads, int tree) {
        kern<<<grid, threads, 0, st>>>(x, g, b, eps, layer, k, tree, y, q, im, sx);
    };
    if (P <= 32) {
        launch(norm_quant_kernel<1, 32, 16, kNormGeneric>, 32, P);
    } else if (P <= 1024) {
        const int t = 32 * warps_for(4);
        if (form == kNormRmsImage) launch(norm_quant_kernel<4, 256, 4, kNormRmsImage>, t, P / 4);
        else if (form == kNormLayerImage) launch(norm_quant_kernel<4, 256, 4, kNormLayerImage>, t, P / 4);
        else launch(norm_quant_kernel<4, 256, 3, kNormGeneric>, t, P / 4);
    } else {
        // rows over 8192 elements: the specialized forms would need 124-130
        // registers here (85 generic), one CTA per SM instead of three
        launch(norm_quant_kernel<8, 256, 1, kNormGeneric>, 32 * warps_for(8), P / 8);
    }
    return cudaGetLastError();
}

}  // namespace w8a8
