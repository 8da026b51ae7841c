// Few-token post-scale W8A8 GEMM as a GEMV on the CUDA cores.
//
// With a handful of tokens the post-scale Linear ("Differences From
// TurboDiffusion": INT8 accumulation continuous over K, activation and weight
// scales applied in the epilogue) is a stream of the weight codes, each byte
// used M <= 4 times: no contraction dense enough for a tensor-core tile.  This
// kernel streams the int8 codes once and forms the dot products with dp4a
// (four int8 products summed into an int32).  The int32 sums are exact in any
// order: |acc| <= 127 * 127 * K < 2^31 for K <= 131072.
//
// Work layout: a persistent grid of 8-warp CTAs.  Each CTA first stages the
// M x K activation codes in shared memory: one bulk copy from Xq, or (the fused
// Linear with one or two tokens) quantized from the bf16 rows of X by the CTA
// itself, with the per-token quantizer's arithmetic, so one kernel does the
// whole Linear.
// Each warp owns a contiguous range of row groups (R weight rows each),
// balanced to within one group, and walks it in steps of U 512-byte slices
// per row (each lane reads 16 bytes of a slice: coalesced), issuing the next
// step's weight loads before it consumes the current step; its first loads
// go out before the activations are staged.  Each activation read from
// shared memory serves the R rows of the group.  At the end of a group the
// lane sums are reduced across the warp and the epilogue is the tensor-core
// GEMM's:
//   y = bf16(((float(acc) * sx[m]) * sw[n]) + bias[n]), each operation rounded
// on its own (the bias add is skipped when there is no bias).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemv.h"
#include "kernels.h"
#include "ptx.cuh"
#include "quant_core.cuh"

namespace w8a8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSiteGemvStage = 40;  // the bounded wait for the staged activation codes
constexpr size_t kSmemPerSm = 228 * 1024;  // shared memory of one SM, for the CTAs-per-SM estimate

struct GemvParams {
    const void* x;         // Xq int8 [M,K], or X bf16 [M,K] when the kernel quantizes
    float* sx;             // [M]: read, or written by CTA 0 when the kernel quantizes
    int8_t* xq_out;        // quantizing: codes [M,K] written by CTA 0, or null
    const int8_t* wq;      // [N,K]
    const float* sw;       // [N]
    const __nv_bfloat16* bias;  // [N] or null
    void* out;             // Y bf16 [M,N] or acc int32 [M,N]
    int M, N, K;
    int settled;           // Wq complete before the kernel this one depends on started
};

// 16 bytes of a stream that is read once: no L1 allocation, 256-byte L2 fetch.
__device__ __forceinline__ int4 ld_stream16(const int8_t* p) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// c + the dot product of 16 int8 pairs.
__device__ __forceinline__ int dot16(const int4& a, const int4& b, int c) {
    c = __dp4a(a.x, b.x, c);
    c = __dp4a(a.y, b.y, c);
    c = __dp4a(a.z, b.z, c);
    return __dp4a(a.w, b.w, c);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Per-token quantization of the M rows of X into the CTA's shared memory:
// s = absmax / 127 and the codes of quant_chunk, as the activation quantizer
// computes them.  Every CTA keeps its own scales in shared memory (sxs) for
// its epilogue; CTA 0 also stores them and, if asked, the codes to global
// memory, which no other CTA reads.
template <int MT>
__device__ __forceinline__ void stage_quantized(const GemvParams& p, int4* xs4, float (*red)[MT], float* sxs) {
    const uint4* X = static_cast<const uint4*>(p.x);  // 8 bf16 per 16-byte chunk
    const int k8 = p.K >> 3;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        amax[m] = 0.0f;
        if (m < p.M)
            for (int c = threadIdx.x; c < k8; c += kThreads)
                amax[m] = fmaxf(amax[m], chunk_absmax(__ldg(X + static_cast<int64_t>(m) * k8 + c)));
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float v = warp_max(amax[m]);
        if (lane == 0) red[warp][m] = v;
    }
    __syncthreads();
    const bool first = blockIdx.x == 0;
    uint2* xs2 = reinterpret_cast<uint2*>(xs4);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < p.M) {
            float a = red[0][m];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) a = fmaxf(a, red[w][m]);
            const RowScale sc = make_scale_div(a);
            if (threadIdx.x == 0) {
                sxs[m] = sc.s;
                if (first) p.sx[m] = sc.s;
            }
            for (int c = threadIdx.x; c < k8; c += kThreads) {
                const int64_t i = static_cast<int64_t>(m) * k8 + c;
                const uint2 q = quant_chunk(__ldg(X + i), sc);
                xs2[i] = q;
                if (first && p.xq_out) reinterpret_cast<uint2*>(p.xq_out)[i] = q;
            }
        }
    }
}

// MT: tokens the accumulators cover (M <= MT); R: weight rows per group;
// U: 512-byte slices per row and step; MINB: CTAs per SM the registers allow;
// QUANT: the CTA quantizes X itself.
template <int MT, int R, int U, int MINB, int EPI, bool QUANT>
__global__ void __launch_bounds__(kThreads, MINB) gemv_s8_kernel(const __grid_constant__ GemvParams p) {
    extern __shared__ int4 xs4[];  // the M x K activation codes, row-major
    __shared__ float red[kWarps][MT];
    __shared__ float sxs[MT];      // this CTA's activation scales (quantizing kernel)
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int M = p.M, N = p.N, K = p.K;
    const int kq = K >> 4;                         // 16-byte slices per row
    const int spr = (kq + 32 * U - 1) / (32 * U);  // steps per group
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int64_t groups = (static_cast<int64_t>(N) + R - 1) / R;
    const int64_t g_end = groups * (wid + 1) / nwarps;
    int64_t g = groups * wid / nwarps;
    const bool busy = g < g_end;
    const int8_t* __restrict__ Wq = p.wq;

    auto load = [&](int64_t grp, int step, int4(&w)[U][R]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = (step * U + u) * 32 + lane;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = grp * R + r;
                if (c < kq && row < N)
                    w[u][r] = ld_stream16(Wq + row * K + static_cast<int64_t>(c) * 16);
                else
                    w[u][r] = make_int4(0, 0, 0, 0);
            }
        }
    };

    // The first weight loads are in flight while the activations are staged;
    // settled weights are read before the dependency wait.
    int4 cur[U][R], nxt[U][R];
    if (p.settled && busy) load(g, 0, cur);
    grid_dependency_wait();
    if (!p.settled && busy) load(g, 0, cur);
    if constexpr (QUANT) {
        stage_quantized<MT>(p, xs4, red, sxs);
        __syncthreads();
    } else {
        // The M x K codes arrive in one bulk copy (Xq is 16-byte aligned and
        // M * K a multiple of 16), instead of a loop of dependent 16-byte
        // loads per thread.  Every thread waits on the copy's barrier; a wait
        // that runs out (2 s) is recorded as 0x100 + kSiteGemvStage and ends
        // the CTA on every thread alike.
        __shared__ uint64_t staged;
        if (threadIdx.x == 0) {
            mbar_init(&staged, 1);
            fence_mbarrier_init();
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(M) * static_cast<uint32_t>(K);
            mbar_arrive_expect_tx(&staged, bytes);
            bulk_load(xs4, p.x, bytes, &staged);
        }
        const bool ok = mbar_wait(&staged, 0, kSiteGemvStage);
        if (__syncthreads_or(!ok)) {
            // the copy may still be on its way: one more bounded wait for it
            // before this CTA's shared memory is released
            if (threadIdx.x == 0) mbar_wait(&staged, 0, kSiteGemvStage);
            return;
        }
    }
    if (!busy) return;

    int32_t acc[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0;
    int j = 0;
    while (true) {
        int64_t gn = g;
        int jn = j + 1;
        if (jn == spr) {
            jn = 0;
            ++gn;
        }
        const bool more = gn < g_end;
        if (more) load(gn, jn, nxt);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = (j * U + u) * 32 + lane;
            if (c < kq) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < M) {
                        const int4 x = xs4[m * kq + c];
#pragma unroll
                        for (int r = 0; r < R; ++r) acc[r][m] = dot16(cur[u][r], x, acc[r][m]);
                    }
                }
            }
        }
        if (jn == 0) {
            // group g is complete: warp sums, then lane r * MT + m writes (row g*R + r, token m)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = g * R + r;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    int v = acc[r][m];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    acc[r][m] = 0;
                    if (lane == r * MT + m && m < M && row < N) {
                        const int64_t o = static_cast<int64_t>(m) * N + row;
                        if constexpr (EPI == kEpiPostscaleS32) {
                            static_cast<int32_t*>(p.out)[o] = v;
                        } else {
                            const float sxm = QUANT ? sxs[m] : p.sx[m];
                            float y = __fmul_rn(__fmul_rn(__int2float_rn(v), sxm), __ldg(p.sw + row));
                            if (p.bias) y = __fadd_rn(y, __bfloat162float(p.bias[row]));
                            static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(y);
                        }
                    }
                }
            }
        }
        if (!more) break;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int r = 0; r < R; ++r) cur[u][r] = nxt[u][r];
        g = gn;
        j = jn;
    }
}

template <int MT, int R, int EPI, bool QUANT>
cudaError_t launch_mt(const GemvParams& p, int num_sms, cudaStream_t st) {
    constexpr int U = 4 / R;  // 4 x 16 bytes of weights per lane and step
    // CTAs per SM: 4 (64 registers) unless the staging's scales next to the
    // first weight loads need more
    constexpr int MINB = (QUANT && MT >= 2) ? 3 : 4;
    static_assert(!QUANT || MT <= kGemvFusedMaxTokens, "the fused quantization is built for few tokens");
    static_assert(R * MT <= 32, "one writing lane per output of a group");
    auto kern = gemv_s8_kernel<MT, R, U, MINB, EPI, QUANT>;
    const size_t smem = static_cast<size_t>(p.M) * static_cast<size_t>(p.K);
    cudaError_t e;
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
            cudaSuccess)
        return e;
    int per_sm = MINB;
    const int by_smem = static_cast<int>(kSmemPerSm / (smem + 1024 + sizeof(float) * kWarps * MT));
    if (by_smem < per_sm) per_sm = by_smem < 1 ? 1 : by_smem;
    const int64_t groups = (static_cast<int64_t>(p.N) + R - 1) / R;
    int64_t grid = (groups + kWarps - 1) / kWarps;
    if (grid > static_cast<int64_t>(num_sms) * per_sm) grid = static_cast<int64_t>(num_sms) * per_sm;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// Rows sharing each activation read: one for one or two tokens, and for 3..4
// while N <= kOneRowMaxN (one row per warp is then within a wave of warps
// and the GEMV is bound by load latency: more warps, fewer steps each; at
// N = 3072 the GEMM went from 8.8 to 7.1 us); else two, which halves the
// shared-memory reads per weight byte (faster from N = 5120 on).
constexpr int kOneRowMaxN = 4096;

template <int EPI, bool QUANT>
cudaError_t launch_tokens(const GemvParams& p, int num_sms, cudaStream_t st) {
    if (p.M <= 1) return launch_mt<1, 1, EPI, QUANT>(p, num_sms, st);
    if constexpr (QUANT) {
        return launch_mt<2, 1, EPI, QUANT>(p, num_sms, st);
    } else {
        if (p.M <= 2) return launch_mt<2, 1, EPI, QUANT>(p, num_sms, st);
        return p.N <= kOneRowMaxN ? launch_mt<4, 1, EPI, QUANT>(p, num_sms, st)
                                  : launch_mt<4, 2, EPI, QUANT>(p, num_sms, st);
    }
}

bool shape_ok(int64_t M, int64_t N, int64_t K) {
    return gemv_takes(M, K) && N > 0 && N <= INT32_MAX && K > 0 && K % 16 == 0;
}

GemvParams make_params(const void* x, float* sx, int8_t* xq_out, const int8_t* Wq, const float* sw,
                       const void* bias, void* out, int64_t M, int64_t N, int64_t K, bool settled) {
    GemvParams p;
    p.x = x;
    p.sx = sx;
    p.xq_out = xq_out;
    p.wq = Wq;
    p.sw = sw;
    p.bias = static_cast<const __nv_bfloat16*>(bias);
    p.out = out;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.settled = settled ? 1 : 0;
    return p;
}

}  // namespace

cudaError_t launch_gemv_s8(int epilogue, const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                           const void* bias, void* out, int64_t M, int64_t N, int64_t K, bool weights_settled,
                           int num_sms, cudaStream_t st) {
    if (!shape_ok(M, N, K)) return cudaErrorInvalidValue;
    const GemvParams p = make_params(Xq, const_cast<float*>(sx), nullptr, Wq, sw, bias, out, M, N, K, weights_settled);
    switch (epilogue) {
        case kEpiPostscaleBf16: return launch_tokens<kEpiPostscaleBf16, false>(p, num_sms, st);
        case kEpiPostscaleS32: return launch_tokens<kEpiPostscaleS32, false>(p, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv_s8_quant(const void* X, float* sx, int8_t* Xq, const int8_t* Wq, const float* sw,
                                 const void* bias, void* Y, int64_t M, int64_t N, int64_t K, int num_sms,
                                 cudaStream_t st) {
    if (!shape_ok(M, N, K) || M > kGemvFusedMaxTokens) return cudaErrorInvalidValue;
    return launch_tokens<kEpiPostscaleBf16, true>(make_params(X, sx, Xq, Wq, sw, bias, Y, M, N, K, false), num_sms,
                                                  st);
}

}  // namespace w8a8
