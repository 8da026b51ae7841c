// Internal launchers shared by the C-ABI layer (api.cu) and the kernel
// translation units.  Arguments are validated by the caller.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace w8a8 {

// Per-row quantization of A[R,K] (bf16): one scale per row (per token for
// activations, per output channel for weights).  Writes the int8 codes to Aq
// and/or their exact bf16 image to img (either may be null, not both).
cudaError_t launch_quant_rows(const void* A, int64_t R, int64_t K, int8_t* Aq, void* img, float* s, int num_sms,
                              cudaStream_t st);
// 1x128-block activation quantization, sx[M][K/128]; outputs as above.
cudaError_t launch_quant_act_block(const void* X, int64_t M, int64_t K, int8_t* Xq, void* img, float* sx,
                                   int num_sms, cudaStream_t st);
// 128x128-block weight quantization, sw[ceil(N/128)][K/128].
cudaError_t launch_quant_weight_block(const void* W, int64_t N, int64_t K, int8_t* Wq, float* sw,
                                      cudaStream_t st);
// Exact int8 -> bf16 image of n values (n % 16 == 0).
cudaError_t launch_expand_s8_bf16(const int8_t* src, int64_t n, void* dst, int num_sms, cudaStream_t st);

// Per-token quantization of X [M,K] bf16 for the few-token GEMM on int8
// weight codes: scales sx [M], codes Xq [M,K] (may be null), the fp16 image
// of the codes img16 [M,K] (the GEMM's token operand, in the GEMM's scratch),
// and zero_bytes (a multiple of 16) of zeros at zero (the GEMM's split-K sums
// and counters).  For K <= 16384 (quant_tokens_f16_takes).
bool quant_tokens_f16_takes(int64_t K);
cudaError_t launch_quant_tokens_f16(const void* X, int64_t M, int64_t K, int8_t* Xq, void* img16, float* sx,
                                    void* zero, size_t zero_bytes, cudaStream_t st);

// Test export of the FFN up-projection's activation: G[i] = bf16(gelu(Y[i]))
// for n bf16 values (n % 8 == 0), with the GEMM epilogue's device function.
cudaError_t launch_gelu_bf16(const void* Y, int64_t n, void* G, int num_sms, cudaStream_t st);

// RMSNorm (layer = 0) or LayerNorm (layer = 1) of bf16 X[M,K] fused with
// per-token quantization; K % 8 == 0, K <= 16384.  gamma / beta (bf16 [K]) and
// the outputs Y (normalized bf16), Xq (int8), img (bf16 image of Xq) may be null.
cudaError_t launch_norm_quant(const void* X, const void* gamma, const void* beta, float eps, int layer, int64_t M,
                              int64_t K, void* Y, int8_t* Xq, void* img, float* sx, cudaStream_t st);

enum GemmEpilogue : int {
    kEpiPostscaleBf16 = 0,  // Y = bf16(((acc * sx) * sw) + bias)
    kEpiPostscaleS32 = 1,   // acc int32
    kEpiBlockwiseBf16 = 2,  // Y = bf16(acc_f32 + bias)
    kEpiBlockwiseF32 = 3,   // acc fp32
    kEpiGeluQuant = 4,      // FFN up: bf16 image of the 1x128 codes of bf16(gelu(post-scale Y)), scales to sg
};

struct GemmArgs {
    const float* sx;
    const float* sw;
    const void* bias;  // bf16 [N] or nullptr
    void* out;         // Y bf16 / acc int32 / acc fp32, [M,N]
    int64_t M, N, K;
    int32_t* partial;  // split-K partial sums, splitk_partial_bytes(M,N,K) bytes (unused when that is 0);
                       // with int8_operands, the scratch of s8_workspace_bytes(M,N,K) bytes (256-byte aligned)
    float* sg;         // kEpiGeluQuant: 1x128 block scales of the GELU output [M][N/128]
    bool weights_settled;  // Bb was complete before the previous kernel in the stream started
    bool int8_operands;    // Ab / Bb are the int8 codes themselves (gemm_takes_int8 shapes only)
    bool tokens_widened;   // int8_operands: the scratch already holds the tokens' fp16 image and
                           // zeroed split-K sums and counters (s8_scratch_zero), written by the
                           // kernel just before this one
};

// Whether launch_gemm takes int8 codes directly (instead of bf16 images) for
// this epilogue and M: the few-token post-scale GEMM streams int8 operands.
bool gemm_takes_int8(int epilogue, int64_t M);

// Split K for few-token post-scale GEMMs: the number of K splits (1: none)
// and, through split_stages, the 64-wide K stages each split covers.
int splitk_plan(bool blockwise, int64_t M, int64_t N, int64_t K, int* split_stages);
// Bytes of int32 partial sums a post-scale GEMM of this shape needs (0 without split).
size_t splitk_partial_bytes(int64_t M, int64_t N, int64_t K);
// Scratch bytes of the GEMM on int8 operands (gemm_takes_int8 shapes): the
// fp16 image of the tokens' codes and, when the shape may split K, int32 sums
// [M][N] and arrival counters.
size_t s8_workspace_bytes(int64_t M, int64_t N, int64_t K);
// The part of that scratch a launch on num_sms SMs needs zeroed (its split-K
// sums and counters): bytes from offset, 0 bytes when K is not split.
void s8_scratch_zero(int64_t M, int64_t N, int64_t K, int num_sms, size_t* offset, size_t* bytes);

// Tensor-core GEMM on the bf16 images (Ab [M,K], Bb [N,K]) of the int8
// operands.  `encode` is the driver's cuTensorMapEncodeTiled.
// On failure, a one-line description is written to `detail` (size `n`).
cudaError_t launch_gemm(int epilogue, const void* Ab, const void* Bb, const GemmArgs& args, int num_sms,
                        void* encode_fn, cudaStream_t st, char* detail, size_t n);

// The int8-operand GEMM (gemm_s8.cu) that launch_gemm routes
// args.int8_operands calls to: Xq [M,K] and Wq [N,K] int8 codes, post-scale
// epilogues only, args.partial its scratch of s8_workspace_bytes(M,N,K).
cudaError_t launch_gemm_s8(int epilogue, const void* Xq, const void* Wq, const GemmArgs& args, int num_sms,
                           void* encode_fn, cudaStream_t st, char* detail, size_t n);

// Device error codes at or above this value mean a bounded wait ran out.
constexpr unsigned int kDeviceErrorTimeoutBase = 0x100;

// Read and clear the device error words of the GEMM and quantization
// translation units.
cudaError_t gemm_read_device_error(unsigned int* code);
cudaError_t gemm_s8_read_device_error(unsigned int* code);
// One CTA whose bounded mbarrier wait runs out (nothing arrives): records a
// timeout in the GEMM translation unit's device error word and returns.
cudaError_t launch_wait_timeout_probe(cudaStream_t st);
cudaError_t quant_read_device_error(unsigned int* code);

// Throughput kernel of warp-level INT8 MMAs; returns tera-ops per second.
cudaError_t measure_imma_peak(double* tops, int num_sms, cudaStream_t st);

// Streaming copy with the traffic of an activation quantization (n bf16 in,
// n bytes out; n % 8 == 0), for the quantization's memory floor.
cudaError_t launch_stream_floor(const void* src, int64_t n, void* dst, int num_sms, cudaStream_t st);

}  // namespace w8a8
