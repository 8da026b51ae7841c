// C ABI of the W8A8 INT8 Linear library (declared in include/w8a8.h):
// argument checks, device checks, workspace carving and kernel launches.
// Every check runs before anything is enqueued, so a rejected call leaves
// all outputs untouched.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdint>
#include <mutex>

#include "../../include/w8a8.h"
#include "gemv.h"
#include "kernels.h"

namespace {

constexpr int64_t kMaxK = 131072;  // 127 * 127 * K must stay below 2^31
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ok;
    int num_sms;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::atomic<bool> g_dev_known[kMaxDevices];
void* g_encode = nullptr;
thread_local char t_detail[256] = "";
thread_local cudaEvent_t t_gemm_start = nullptr;
thread_local cudaEvent_t t_gemm_end = nullptr;

void set_detail(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_detail, sizeof t_detail, fmt, ap);
    va_end(ap);
}

w8a8_status cuda_fail(const char* what, cudaError_t e) {
    set_detail("%s: %s", what, cudaGetErrorString(e));
    return W8A8_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace of the GEMM on bf16 operand images: the images of Xq and Wq and
// the int32 partial sums of the K splits.
size_t image_gemm_need(int64_t M, int64_t N, int64_t K) {
    return align256(static_cast<size_t>(M) * K * 2) + align256(static_cast<size_t>(N) * K * 2) +
           align256(w8a8::splitk_partial_bytes(M, N, K));
}

// Current device must be compute capability 10.3.
w8a8_status current_device(DeviceInfo* out) {
    int dev = 0;
    cudaError_t ge = cudaGetDevice(&dev);
    if (ge != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("cudaGetDevice", ge);
    }
    if (dev < 0 || dev >= kMaxDevices) return W8A8_ERR_UNSUPPORTED_DEVICE;
    if (!g_dev_known[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_dev_known[dev].load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
                cudaGetLastError();
                set_detail("cudaDeviceGetAttribute failed on device %d", dev);
                return W8A8_ERR_CUDA;
            }
            g_dev[dev].ok = (major == 10 && minor == 3);
            g_dev[dev].num_sms = sms;
            g_dev_known[dev].store(true, std::memory_order_release);
        }
    }
    *out = g_dev[dev];
    return out->ok ? W8A8_OK : W8A8_ERR_UNSUPPORTED_DEVICE;
}

void* encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn) {
            g_encode = fn;
        } else {
            cudaGetLastError();
            set_detail("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled): %s, query result %d",
                       cudaGetErrorString(e), (int)q);
        }
    }
    return g_encode;
}

w8a8_status from_cuda(cudaError_t e, const char* what = "kernel launch") {
    return e == cudaSuccess ? W8A8_OK : cuda_fail(what, e);
}

w8a8_status check_k(int64_t K, bool block) {
    if (K <= 0) return W8A8_ERR_INVALID_ARG;
    if (K % 16 != 0 || K > kMaxK) return W8A8_ERR_SHAPE;
    if (block && K % 128 != 0) return W8A8_ERR_SHAPE;
    return W8A8_OK;
}

// Workspace bytes the post-scale GEMM (int8 codes in) uses for this shape:
// none for the few-token GEMV; when the GEMM streams the int8 codes itself
// (M <= 288), the fp16 image of Xq and, where K may be split, int32 sums and
// counters; else the bf16 images of Xq and Wq plus the partial sums of the
// K splits.  M, N, K > 0.
size_t postscale_gemm_need(int64_t M, int64_t N, int64_t K) {
    if (w8a8::gemv_takes(M, K)) return 0;
    if (w8a8::gemm_takes_int8(w8a8::kEpiPostscaleBf16, M)) return w8a8::s8_workspace_bytes(M, N, K);
    return image_gemm_need(M, N, K);
}

// Shared checks of the GEMM entry points.  need_sx/need_sw: scale pointers
// used by this variant.
w8a8_status check_gemm(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw, const void* bias,
                       const void* out, int64_t M, int64_t N, int64_t K, bool block, bool need_scales,
                       const void* ws, size_t ws_bytes, DeviceInfo* dev, bool* nothing_to_do) {
    *nothing_to_do = false;
    if (M < 0 || N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, block);
    if (s != W8A8_OK) return s;
    if (M > INT32_MAX || N > INT32_MAX) return W8A8_ERR_SHAPE;
    if (M == 0 || N == 0) {
        *nothing_to_do = true;
        return W8A8_OK;
    }
    if (!Xq || !Wq || !out || (need_scales && (!sx || !sw))) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(Xq) || !aligned16(Wq) || !aligned16(out) || (sx && !aligned16(sx)) ||
        (sw && !aligned16(sw)) || (bias && !aligned16(bias)))
        return W8A8_ERR_ALIGNMENT;
    const size_t need = block ? w8a8_gemm_workspace_size(M, N, K) : postscale_gemm_need(M, N, K);
    if (need && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need)) return W8A8_ERR_WORKSPACE;
    return current_device(dev);
}

// GEMM on bf16 operand images, with the timing hook around the launch.
w8a8_status run_gemm_images(int epi, const void* Ab, const void* Bb, const float* sx, const float* sw,
                            const void* bias, void* out, int64_t M, int64_t N, int64_t K, void* partial,
                            const DeviceInfo& dev, cudaStream_t st, float* sg = nullptr,
                            bool weights_settled = false, bool int8_operands = false,
                            bool tokens_widened = false) {
    void* enc = encode_fn();
    if (!enc) return W8A8_ERR_CUDA;
    w8a8::GemmArgs a;
    a.sx = sx;
    a.sw = sw;
    a.bias = bias;
    a.out = out;
    a.M = M;
    a.N = N;
    a.K = K;
    a.partial = static_cast<int32_t*>(partial);
    a.sg = sg;
    a.weights_settled = weights_settled;
    a.int8_operands = int8_operands;
    a.tokens_widened = tokens_widened;
    cudaError_t e;
    if (t_gemm_start && (e = cudaEventRecord(t_gemm_start, st)) != cudaSuccess) return cuda_fail("event", e);
    e = w8a8::launch_gemm(epi, Ab, Bb, a, dev.num_sms, enc, st, t_detail, sizeof t_detail);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W8A8_ERR_CUDA;
    }
    if (t_gemm_end && (e = cudaEventRecord(t_gemm_end, st)) != cudaSuccess) return cuda_fail("event", e);
    return W8A8_OK;
}

// Checks and launches of the fused Linear entry points.
w8a8_status run_linear(bool block, const void* X, const void* Wimg, const float* sw, const void* bias, void* Y,
                       int64_t M, int64_t N, int64_t K, float* sx, int8_t* Xq, void* ws, size_t ws_bytes,
                       cudaStream_t st) {
    if (M < 0 || N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, block);
    if (s != W8A8_OK) return s;
    if (M > INT32_MAX || N > INT32_MAX) return W8A8_ERR_SHAPE;
    if (M == 0 || N == 0) return W8A8_OK;
    if (!X || !Wimg || !sw || !Y || !sx) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Wimg) || !aligned16(sw) || !aligned16(Y) || !aligned16(sx) ||
        (Xq && !aligned16(Xq)) || (bias && !aligned16(bias)))
        return W8A8_ERR_ALIGNMENT;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < w8a8_linear_workspace_size(M, N, K))
        return W8A8_ERR_WORKSPACE;
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    cudaError_t e = block ? w8a8::launch_quant_act_block(X, M, K, Xq, ws, sx, dev.num_sms, st)
                          : w8a8::launch_quant_rows(X, M, K, Xq, ws, sx, dev.num_sms, st);
    if (e != cudaSuccess) return cuda_fail("activation quant launch", e);
    void* partial = static_cast<uint8_t*>(ws) + align256(static_cast<size_t>(M) * K * 2);
    // Wimg predates the quantization kernel just launched (which waited for
    // all earlier work), so the GEMM may start reading it before that kernel ends.
    return run_gemm_images(block ? w8a8::kEpiBlockwiseBf16 : w8a8::kEpiPostscaleBf16, ws, Wimg, sx, sw, bias, Y, M,
                           N, K, partial, dev, st, nullptr, true);
}

// Checks and launches of the fused FFN up-projection (quant, GEMM with the
// GELU + 1x128 quantization epilogue).
w8a8_status run_linear_gelu_quant(const void* X, const void* Wimg, const float* sw, const void* bias, void* Gimg,
                                  float* sg, int64_t M, int64_t N, int64_t K, float* sx, int8_t* Xq, void* ws,
                                  size_t ws_bytes, cudaStream_t st) {
    if (M < 0 || N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, false);
    if (s != W8A8_OK) return s;
    if (M > INT32_MAX || N > INT32_MAX || N % 128 != 0) return W8A8_ERR_SHAPE;
    if (M == 0 || N == 0) return W8A8_OK;
    if (!X || !Wimg || !sw || !Gimg || !sg || !sx) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Wimg) || !aligned16(sw) || !aligned16(Gimg) || !aligned16(sg) ||
        !aligned16(sx) || (Xq && !aligned16(Xq)) || (bias && !aligned16(bias)))
        return W8A8_ERR_ALIGNMENT;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < w8a8_linear_workspace_size(M, N, K))
        return W8A8_ERR_WORKSPACE;
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    cudaError_t e = w8a8::launch_quant_rows(X, M, K, Xq, ws, sx, dev.num_sms, st);
    if (e != cudaSuccess) return cuda_fail("activation quant launch", e);
    return run_gemm_images(w8a8::kEpiGeluQuant, ws, Wimg, sx, sw, bias, Gimg, M, N, K, nullptr, dev, st, sg, true);
}

// Few-token post-scale GEMM on the CUDA cores (with the per-token
// quantization folded in when X is given instead of Xq), with the timing hook
// around the launch.
w8a8_status run_gemv(int epi, const void* X, const int8_t* Xq, float* sx, int8_t* Xq_out, const int8_t* Wq,
                     const float* sw, const void* bias, void* out, int64_t M, int64_t N, int64_t K,
                     bool weights_settled, const DeviceInfo& dev, cudaStream_t st) {
    cudaError_t e;
    if (t_gemm_start && (e = cudaEventRecord(t_gemm_start, st)) != cudaSuccess) return cuda_fail("event", e);
    e = X ? w8a8::launch_gemv_s8_quant(X, sx, Xq_out, Wq, sw, bias, out, M, N, K, dev.num_sms, st)
          : w8a8::launch_gemv_s8(epi, Xq, sx, Wq, sw, bias, out, M, N, K, weights_settled, dev.num_sms, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("few-token GEMV launch", e);
    }
    if (t_gemm_end && (e = cudaEventRecord(t_gemm_end, st)) != cudaSuccess) return cuda_fail("event", e);
    return W8A8_OK;
}

bool takes_gemv(int epi, int64_t M, int64_t K) {
    return (epi == w8a8::kEpiPostscaleBf16 || epi == w8a8::kEpiPostscaleS32) && w8a8::gemv_takes(M, K);
}

w8a8_status run_gemm(int epi, const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                     const void* bias, void* out, int64_t M, int64_t N, int64_t K, void* ws, const DeviceInfo& dev,
                     cudaStream_t st, bool weights_settled = false) {
    // a handful of tokens: a GEMV streaming the int8 weight codes
    if (takes_gemv(epi, M, K))
        return run_gemv(epi, nullptr, Xq, const_cast<float*>(sx), nullptr, Wq, sw, bias, out, M, N, K,
                        weights_settled, dev, st);
    void* enc = encode_fn();
    if (!enc) return W8A8_ERR_CUDA;
    uint8_t* w = static_cast<uint8_t*>(ws);
    if (w8a8::gemm_takes_int8(epi, M)) {
        // few tokens: the GEMM streams the int8 codes itself, no images
        return run_gemm_images(epi, Xq, Wq, sx, sw, bias, out, M, N, K, w, dev, st, nullptr, weights_settled, true);
    }
    void* Ab = w;
    void* Bb = w + align256(static_cast<size_t>(M) * K * 2);
    void* partial = static_cast<uint8_t*>(Bb) + align256(static_cast<size_t>(N) * K * 2);
    cudaError_t e = w8a8::launch_expand_s8_bf16(Xq, M * K, Ab, dev.num_sms, st);
    if (e != cudaSuccess) return cuda_fail("expand Xq launch", e);
    e = w8a8::launch_expand_s8_bf16(Wq, N * K, Bb, dev.num_sms, st);
    if (e != cudaSuccess) return cuda_fail("expand Wq launch", e);
    return run_gemm_images(epi, Ab, Bb, sx, sw, bias, out, M, N, K, partial, dev, st);
}

bool linear_codes_fused(int64_t M, int64_t K) { return w8a8::gemv_takes(M, K) && M <= w8a8::kGemvFusedMaxTokens; }

// The one-kernel GEMV path needs no workspace; otherwise the codes of X, plus
// the GEMM's workspace unless the GEMM is the GEMV.
size_t linear_codes_workspace(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || linear_codes_fused(M, K)) return 0;
    return align256(static_cast<size_t>(M) * K) + postscale_gemm_need(M, N, K);
}

// Checks and launches of the fused Linear on int8 weight codes: per-token
// quantization of X, then the post-scale GEMM on the codes.
w8a8_status run_linear_codes(const void* X, const int8_t* Wq, const float* sw, const void* bias, void* Y, int64_t M,
                             int64_t N, int64_t K, float* sx, int8_t* Xq, void* ws, size_t ws_bytes,
                             cudaStream_t st) {
    if (M < 0 || N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, false);
    if (s != W8A8_OK) return s;
    if (M > INT32_MAX || N > INT32_MAX) return W8A8_ERR_SHAPE;
    if (M == 0 || N == 0) return W8A8_OK;
    if (!X || !Wq || !sw || !Y || !sx) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(sw) || !aligned16(Y) || !aligned16(sx) ||
        (Xq && !aligned16(Xq)) || (bias && !aligned16(bias)))
        return W8A8_ERR_ALIGNMENT;
    const size_t need = linear_codes_workspace(M, N, K);
    if (need && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need))
        return W8A8_ERR_WORKSPACE;
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    // one or two tokens: one kernel quantizes X in every CTA and streams the weight codes
    if (linear_codes_fused(M, K))
        return run_gemv(w8a8::kEpiPostscaleBf16, X, nullptr, sx, Xq, Wq, sw, bias, Y, M, N, K, false, dev, st);
    int8_t* q = Xq ? Xq : static_cast<int8_t*>(ws);
    uint8_t* rest = static_cast<uint8_t*>(ws) + align256(static_cast<size_t>(M) * K);
    if (!w8a8::gemv_takes(M, K) && w8a8::gemm_takes_int8(w8a8::kEpiPostscaleBf16, M) &&
        w8a8::quant_tokens_f16_takes(K)) {
        // few tokens on the int8-operand GEMM: the quantization kernel also
        // writes the GEMM's fp16 token image and zeroes its split-K sums
        size_t zoff = 0, zbytes = 0;
        w8a8::s8_scratch_zero(M, N, K, dev.num_sms, &zoff, &zbytes);
        cudaError_t e = w8a8::launch_quant_tokens_f16(X, M, K, Xq, rest, sx, rest + zoff, zbytes, st);
        if (e != cudaSuccess) return cuda_fail("activation quant launch", e);
        return run_gemm_images(w8a8::kEpiPostscaleBf16, Xq, Wq, sx, sw, bias, Y, M, N, K, rest, dev, st, nullptr,
                               true, true, true);
    }
    cudaError_t e = w8a8::launch_quant_rows(X, M, K, q, nullptr, sx, dev.num_sms, st);
    if (e != cudaSuccess) return cuda_fail("activation quant launch", e);
    // Wq predates the quantization kernel just launched (which waited for all
    // earlier work), so the GEMM may start reading it before that kernel ends.
    return run_gemm(w8a8::kEpiPostscaleBf16, q, sx, Wq, sw, bias, Y, M, N, K, rest, dev, st, true);
}

// Scratch of the allocation-free GEMM entry point: a fixed device array,
// loaded with the library on every device that uses it and held until the
// process exits.  The name is a host-side stand-in; its device address comes
// from cudaGetSymbolAddress, taken once per device with that device current.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
void* g_noalloc_ptr[kMaxDevices];
std::atomic<bool> g_noalloc_ready[kMaxDevices];

w8a8_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("cudaGetDevice", e);
    }
    if (dev < 0 || dev >= kMaxDevices) return W8A8_ERR_UNSUPPORTED_DEVICE;
    if (!g_noalloc_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_noalloc_ready[dev].load(std::memory_order_relaxed)) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return cuda_fail("cudaGetSymbolAddress(no-alloc scratch)", e);
            }
            g_noalloc_ptr[dev] = p;
            g_noalloc_ready[dev].store(true, std::memory_order_release);
        }
    }
    *out = g_noalloc_ptr[dev];
    return W8A8_OK;
}

}  // namespace

extern "C" {

const char* w8a8_status_string(w8a8_status s) {
    switch (s) {
        case W8A8_OK: return "W8A8_OK";
        case W8A8_ERR_INVALID_ARG: return "W8A8_ERR_INVALID_ARG: null pointer, bad mode or negative size";
        case W8A8_ERR_ALIGNMENT: return "W8A8_ERR_ALIGNMENT: a pointer is not 16-byte aligned";
        case W8A8_ERR_SHAPE: return "W8A8_ERR_SHAPE: K must be a positive multiple of 16 (128 for blocks), <= 131072";
        case W8A8_ERR_UNSUPPORTED_DEVICE: return "W8A8_ERR_UNSUPPORTED_DEVICE: current device is not sm_103";
        case W8A8_ERR_CUDA: return "W8A8_ERR_CUDA: a CUDA call failed";
        case W8A8_ERR_TIMEOUT: return "W8A8_ERR_TIMEOUT: a device-side bounded wait ran out";
        case W8A8_ERR_WORKSPACE: return "W8A8_ERR_WORKSPACE: workspace missing, unaligned or too small";
    }
    return "unknown w8a8_status";
}

w8a8_status w8a8_quantize_weight(const void* W, int64_t N, int64_t K, w8a8_scale_mode mode, int8_t* Wq,
                                 float* sw, void* stream) {
    if (mode != W8A8_SCALE_PER_ROW && mode != W8A8_SCALE_BLOCK) return W8A8_ERR_INVALID_ARG;
    if (N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, mode == W8A8_SCALE_BLOCK);
    if (s != W8A8_OK) return s;
    if (N > INT32_MAX) return W8A8_ERR_SHAPE;
    if (N == 0) return W8A8_OK;
    if (!W || !Wq || !sw) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(Wq) || !aligned16(sw)) return W8A8_ERR_ALIGNMENT;
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (mode == W8A8_SCALE_PER_ROW) return from_cuda(w8a8::launch_quant_rows(W, N, K, Wq, nullptr, sw, dev.num_sms, st));
    if ((N + 127) / 128 > 65535) return W8A8_ERR_SHAPE;
    return from_cuda(w8a8::launch_quant_weight_block(W, N, K, Wq, sw, st));
}

w8a8_status w8a8_quantize_act(const void* X, int64_t M, int64_t K, w8a8_scale_mode mode, int8_t* Xq, float* sx,
                              void* stream) {
    if (mode != W8A8_SCALE_PER_ROW && mode != W8A8_SCALE_BLOCK) return W8A8_ERR_INVALID_ARG;
    if (M < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, mode == W8A8_SCALE_BLOCK);
    if (s != W8A8_OK) return s;
    if (M > INT32_MAX) return W8A8_ERR_SHAPE;
    if (M == 0) return W8A8_OK;
    if (!X || !Xq || !sx) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Xq) || !aligned16(sx)) return W8A8_ERR_ALIGNMENT;
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (mode == W8A8_SCALE_PER_ROW) return from_cuda(w8a8::launch_quant_rows(X, M, K, Xq, nullptr, sx, dev.num_sms, st));
    return from_cuda(w8a8::launch_quant_act_block(X, M, K, Xq, nullptr, sx, dev.num_sms, st));
}

w8a8_status w8a8_pack_weight(const int8_t* Wq, int64_t N, int64_t K, void* Wimg, void* stream) {
    if (N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, false);
    if (s != W8A8_OK) return s;
    if (N == 0) return W8A8_OK;
    if (!Wq || !Wimg) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(Wq) || !aligned16(Wimg)) return W8A8_ERR_ALIGNMENT;
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    return from_cuda(w8a8::launch_expand_s8_bf16(Wq, N * K, Wimg, dev.num_sms, static_cast<cudaStream_t>(stream)));
}

size_t w8a8_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return align256(static_cast<size_t>(M) * K * 2) + align256(w8a8::splitk_partial_bytes(M, N, K));
}

w8a8_status w8a8_linear_postscale(const void* X, const void* Wimg, const float* sw, const void* bias, void* Y,
                                  int64_t M, int64_t N, int64_t K, float* sx, int8_t* Xq, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    return run_linear(false, X, Wimg, sw, bias, Y, M, N, K, sx, Xq, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream));
}

size_t w8a8_linear_codes_workspace_size(int64_t M, int64_t N, int64_t K) { return linear_codes_workspace(M, N, K); }

w8a8_status w8a8_linear_postscale_codes(const void* X, const int8_t* Wq, const float* sw, const void* bias, void* Y,
                                        int64_t M, int64_t N, int64_t K, float* sx, int8_t* Xq, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    return run_linear_codes(X, Wq, sw, bias, Y, M, N, K, sx, Xq, workspace, workspace_bytes,
                            static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_linear_blockwise(const void* X, const void* Wimg, const float* sw, const void* bias, void* Y,
                                  int64_t M, int64_t N, int64_t K, float* sx, int8_t* Xq, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    return run_linear(true, X, Wimg, sw, bias, Y, M, N, K, sx, Xq, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_linear_postscale_gelu_quant(const void* X, const void* Wimg, const float* sw, const void* bias,
                                             void* Gimg, float* sg, int64_t M, int64_t N, int64_t K, float* sx,
                                             int8_t* Xq, void* workspace, size_t workspace_bytes, void* stream) {
    return run_linear_gelu_quant(X, Wimg, sw, bias, Gimg, sg, M, N, K, sx, Xq, workspace, workspace_bytes,
                                 static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_gemm_blockwise_images(const void* Ximg, const float* sx, const void* Wimg, const float* sw,
                                       const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* stream) {
    if (M < 0 || N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, true);
    if (s != W8A8_OK) return s;
    if (M > INT32_MAX || N > INT32_MAX) return W8A8_ERR_SHAPE;
    if (M == 0 || N == 0) return W8A8_OK;
    if (!Ximg || !sx || !Wimg || !sw || !Y) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(Ximg) || !aligned16(sx) || !aligned16(Wimg) || !aligned16(sw) || !aligned16(Y) ||
        (bias && !aligned16(bias)))
        return W8A8_ERR_ALIGNMENT;
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    return run_gemm_images(w8a8::kEpiBlockwiseBf16, Ximg, Wimg, sx, sw, bias, Y, M, N, K, nullptr, dev,
                           static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_norm_quant(const void* X, const void* gamma, const void* beta, float eps, w8a8_norm_kind kind,
                            int64_t M, int64_t K, void* Y, int8_t* Xq, void* Ximg, float* sx, void* stream) {
    if (M < 0 || K <= 0) return W8A8_ERR_INVALID_ARG;
    if (kind != W8A8_NORM_RMS && kind != W8A8_NORM_LAYER) return W8A8_ERR_INVALID_ARG;
    if (K % 8 != 0 || K > 16384 || M > INT32_MAX) return W8A8_ERR_SHAPE;
    if (M == 0) return W8A8_OK;
    if (!X || !sx) return W8A8_ERR_INVALID_ARG;
    if (!(eps >= 0.0f)) return W8A8_ERR_INVALID_ARG;  // also rejects NaN
    if (!aligned16(X) || !aligned16(sx) || (gamma && !aligned16(gamma)) || (beta && !aligned16(beta)) ||
        (Y && !aligned16(Y)) || (Xq && !aligned16(Xq)) || (Ximg && !aligned16(Ximg)))
        return W8A8_ERR_ALIGNMENT;
    DeviceInfo dev;
    w8a8_status s = current_device(&dev);
    if (s != W8A8_OK) return s;
    return from_cuda(w8a8::launch_norm_quant(X, gamma, beta, eps, kind == W8A8_NORM_LAYER ? 1 : 0, M, K, Y, Xq, Ximg,
                                             sx, static_cast<cudaStream_t>(stream)));
}

size_t w8a8_splitk_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return align256(w8a8::splitk_partial_bytes(M, N, K));
}

w8a8_status w8a8_gemm_postscale_images(const void* Ximg, const float* sx, const void* Wimg, const float* sw,
                                       const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    if (M < 0 || N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, false);
    if (s != W8A8_OK) return s;
    if (M > INT32_MAX || N > INT32_MAX) return W8A8_ERR_SHAPE;
    if (M == 0 || N == 0) return W8A8_OK;
    if (!Ximg || !sx || !Wimg || !sw || !Y) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(Ximg) || !aligned16(sx) || !aligned16(Wimg) || !aligned16(sw) || !aligned16(Y) ||
        (bias && !aligned16(bias)))
        return W8A8_ERR_ALIGNMENT;
    const size_t need = w8a8_splitk_workspace_size(M, N, K);
    if (need && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need))
        return W8A8_ERR_WORKSPACE;
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    return run_gemm_images(w8a8::kEpiPostscaleBf16, Ximg, Wimg, sx, sw, bias, Y, M, N, K, workspace, dev,
                           static_cast<cudaStream_t>(stream));
}

size_t w8a8_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const size_t img = image_gemm_need(M, N, K);
    const size_t s8 = w8a8::gemm_takes_int8(w8a8::kEpiPostscaleBf16, M) ? w8a8::s8_workspace_bytes(M, N, K) : 0;
    return img > s8 ? img : s8;
}

w8a8_status w8a8_gemm_postscale(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                                const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* workspace,
                                size_t workspace_bytes, void* stream) {
    DeviceInfo dev;
    bool none;
    w8a8_status s =
        check_gemm(Xq, sx, Wq, sw, bias, Y, M, N, K, false, true, workspace, workspace_bytes, &dev, &none);
    if (s != W8A8_OK || none) return s;
    return run_gemm(w8a8::kEpiPostscaleBf16, Xq, sx, Wq, sw, bias, Y, M, N, K, workspace, dev,
                    static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_gemm_blockwise(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                                const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* workspace,
                                size_t workspace_bytes, void* stream) {
    DeviceInfo dev;
    bool none;
    w8a8_status s =
        check_gemm(Xq, sx, Wq, sw, bias, Y, M, N, K, true, true, workspace, workspace_bytes, &dev, &none);
    if (s != W8A8_OK || none) return s;
    return run_gemm(w8a8::kEpiBlockwiseBf16, Xq, sx, Wq, sw, bias, Y, M, N, K, workspace, dev,
                    static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_gemm_postscale_noalloc(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                                        const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* stream) {
    if (M < 0 || N < 0) return W8A8_ERR_INVALID_ARG;
    w8a8_status s = check_k(K, false);
    if (s != W8A8_OK) return s;
    if (M > INT32_MAX || N > INT32_MAX) return W8A8_ERR_SHAPE;
    if (M == 0 || N == 0) return W8A8_OK;
    const size_t need = postscale_gemm_need(M, N, K);
    if (need > kNoAllocScratchBytes) {
        set_detail("shape %lld x %lld x %lld needs %zu bytes of scratch; the fixed no-alloc scratch holds %zu",
                   (long long)M, (long long)N, (long long)K, need, kNoAllocScratchBytes);
        return W8A8_ERR_WORKSPACE;
    }
    DeviceInfo dev;
    if ((s = current_device(&dev)) != W8A8_OK) return s;
    void* scratch = nullptr;
    if ((s = noalloc_scratch(&scratch)) != W8A8_OK) return s;
    bool none;
    s = check_gemm(Xq, sx, Wq, sw, bias, Y, M, N, K, false, true, scratch, kNoAllocScratchBytes, &dev, &none);
    if (s != W8A8_OK || none) return s;
    return run_gemm(w8a8::kEpiPostscaleBf16, Xq, sx, Wq, sw, bias, Y, M, N, K, scratch, dev,
                    static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_gemm_postscale_s32(const int8_t* Xq, const int8_t* Wq, int32_t* acc, int64_t M, int64_t N,
                                    int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    DeviceInfo dev;
    bool none;
    w8a8_status s = check_gemm(Xq, nullptr, Wq, nullptr, nullptr, acc, M, N, K, false, false, workspace,
                               workspace_bytes, &dev, &none);
    if (s != W8A8_OK || none) return s;
    return run_gemm(w8a8::kEpiPostscaleS32, Xq, nullptr, Wq, nullptr, nullptr, acc, M, N, K, workspace, dev,
                    static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_gemm_blockwise_f32(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                                    float* acc, int64_t M, int64_t N, int64_t K, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    DeviceInfo dev;
    bool none;
    w8a8_status s = check_gemm(Xq, sx, Wq, sw, nullptr, acc, M, N, K, true, true, workspace, workspace_bytes,
                               &dev, &none);
    if (s != W8A8_OK || none) return s;
    return run_gemm(w8a8::kEpiBlockwiseF32, Xq, sx, Wq, sw, nullptr, acc, M, N, K, workspace, dev,
                    static_cast<cudaStream_t>(stream));
}

w8a8_status w8a8_gelu_bf16(const void* Y, int64_t n, void* G, void* stream) {
    if (n < 0) return W8A8_ERR_INVALID_ARG;
    if (n % 8 != 0) return W8A8_ERR_SHAPE;
    if (n == 0) return W8A8_OK;
    if (!Y || !G) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(Y) || !aligned16(G)) return W8A8_ERR_ALIGNMENT;
    DeviceInfo dev;
    w8a8_status s = current_device(&dev);
    if (s != W8A8_OK) return s;
    return from_cuda(w8a8::launch_gelu_bf16(Y, n, G, dev.num_sms, static_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_get_device_error(int* code) {
    if (!code) return W8A8_ERR_INVALID_ARG;
    *code = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return W8A8_ERR_CUDA;
    }
    unsigned int v = 0, vs = 0, vq = 0;
    if (w8a8::gemm_read_device_error(&v) != cudaSuccess) return W8A8_ERR_CUDA;
    if (w8a8::gemm_s8_read_device_error(&vs) != cudaSuccess) return W8A8_ERR_CUDA;
    if (w8a8::quant_read_device_error(&vq) != cudaSuccess) return W8A8_ERR_CUDA;
    if (v == 0) v = vs;
    if (v == 0) v = vq;
    *code = static_cast<int>(v);
    if (v >= w8a8::kDeviceErrorTimeoutBase) return W8A8_ERR_TIMEOUT;
    return v ? W8A8_ERR_CUDA : W8A8_OK;
}

w8a8_status w8a8_probe_wait_timeout(void* stream) {
    DeviceInfo dev;
    w8a8_status s = current_device(&dev);
    if (s != W8A8_OK) return s;
    return from_cuda(w8a8::launch_wait_timeout_probe(static_cast<cudaStream_t>(stream)));
}

const char* w8a8_last_error_detail(void) { return t_detail; }

w8a8_status w8a8_set_gemm_timing_events(void* start, void* end) {
    if ((start == nullptr) != (end == nullptr)) return W8A8_ERR_INVALID_ARG;
    t_gemm_start = static_cast<cudaEvent_t>(start);
    t_gemm_end = static_cast<cudaEvent_t>(end);
    return W8A8_OK;
}

w8a8_status w8a8_measure_imma_peak(double* tops, void* stream) {
    if (!tops) return W8A8_ERR_INVALID_ARG;
    DeviceInfo dev;
    w8a8_status s = current_device(&dev);
    if (s != W8A8_OK) return s;
    return from_cuda(w8a8::measure_imma_peak(tops, dev.num_sms, static_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_stream_floor(const void* src, int64_t n, void* dst, void* stream) {
    if (n < 0) return W8A8_ERR_INVALID_ARG;
    if (n % 8 != 0) return W8A8_ERR_SHAPE;
    if (n == 0) return W8A8_OK;
    if (!src || !dst) return W8A8_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return W8A8_ERR_ALIGNMENT;
    DeviceInfo dev;
    w8a8_status s = current_device(&dev);
    if (s != W8A8_OK) return s;
    return from_cuda(w8a8::launch_stream_floor(src, n, dst, dev.num_sms, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
