// Few-token post-scale GEMM on the CUDA cores (gemv.cu): launchers shared
// with the C-ABI layer.  Arguments are validated by the caller.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace w8a8 {

// Token counts up to this take the CUDA-core GEMV instead of the tensor cores
// (from 5 tokens on, the int8-operand tensor-core kernel is faster),
constexpr int64_t kGemvMaxTokens = 4;
// ... when the M x K activation codes fit in one CTA's shared memory.
constexpr int64_t kGemvMaxCodeBytes = 131072;

inline bool gemv_takes(int64_t M, int64_t K) {
    return M >= 1 && M <= kGemvMaxTokens && M * K <= kGemvMaxCodeBytes;
}

// Every CTA of the fused kernel quantizes all M rows of X; that pays for the
// saved launch up to this many tokens.
constexpr int64_t kGemvFusedMaxTokens = 2;

// Post-scale GEMM on int8 codes Xq [M,K], Wq [N,K] (16-byte aligned,
// K % 16 == 0, gemv_takes(M, K)), int32 sums exact.  epilogue
// kEpiPostscaleBf16 writes Y [M,N] bf16 = bf16(((acc * sx) * sw) + bias)
// (bias may be null); kEpiPostscaleS32 writes acc [M,N] int32 (sx, sw and
// bias unused).  weights_settled: Wq was complete before the previous kernel
// in the stream started, so the first weight reads may precede the kernel's
// dependency wait on that kernel.
cudaError_t launch_gemv_s8(int epilogue, const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                           const void* bias, void* out, int64_t M, int64_t N, int64_t K, bool weights_settled,
                           int num_sms, cudaStream_t st);

// The same GEMM with the per-token quantization of X [M,K] bf16 folded in,
// for M <= kGemvFusedMaxTokens: every CTA quantizes the M rows into its
// shared memory; the first CTA also writes the scales sx [M] and, when Xq is
// not null, the codes Xq [M,K].  Codes and scales are those of the per-token
// activation quantizer.
cudaError_t launch_gemv_s8_quant(const void* X, float* sx, int8_t* Xq, const int8_t* Wq, const float* sw,
                                 const void* bias, void* Y, int64_t M, int64_t N, int64_t K, int num_sms,
                                 cudaStream_t st);

}  // namespace w8a8
