// Quantizer core shared by the quantization kernels and the GEMM's fused
// GELU + 1x128 quantization epilogue (one definition, so both produce the
// same codes).  The method and its error analysis are stated at the top of
// quant.cu: s = absmax / 127 (IEEE division), q = clamp(rne(x / s), -127, 127),
// computed as rne(x * (1/s)) with a proven tie guard and an exact fallback.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace w8a8 {
namespace {

constexpr float kQMax = 127.0f;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kTieGuard = 6.103515625e-05f;  // 2^-14

struct RowScale {
    float s;     // stored scale
    float inv;   // correctly rounded 1/s (0 when s == 0)
    bool exact;  // subnormal, nonzero scale: every element takes the exact path
};

constexpr float kMinNormal = 1.17549435e-38f;  // 2^-126

// The scale of one row by IEEE division, once per row: the same values as
// the table path below (s = fl(amax / 127); 1/s scales by powers of two
// exactly), without a memory access in the row kernels' dependency chain.
__device__ __forceinline__ RowScale make_scale_div(float amax) {
    RowScale r;
    r.s = __fdiv_rn(amax, kQMax);
    r.inv = (r.s > 0.0f) ? __frcp_rn(r.s) : 0.0f;
    r.exact = r.s > 0.0f && r.s < kMinNormal;
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

// Exact-path code of one value, as a byte.
__device__ __forceinline__ uint32_t quant_byte_exact(float x, float s) {
    return static_cast<uint32_t>(quant_exact(x, s)) & 0xFFu;
}

// 8 bf16 -> 8 int8 packed into a uint2.  Two values per packed fp32
// operation; a chunk holding a value within 2^-14 of a rounding boundary
// re-derives those values on the exact path.
__device__ __forceinline__ uint2 quant_chunk(const uint4& v, const RowScale& sc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (sc.exact) {
        uint32_t b[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            b[2 * i] = quant_byte_exact(bf16_lo(w[i]), sc.s);
            b[2 * i + 1] = quant_byte_exact(bf16_hi(w[i]), sc.s);
        }
        return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                          b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
    }
    const uint64_t inv2 = f2_pack(sc.inv, sc.inv);
    const uint64_t magic2 = f2_pack(kRoundMagic, kRoundMagic);
    uint32_t big[8];
    float dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint64_t x2 = f2_pack(bf16_lo(w[i]), bf16_hi(w[i]));
        const uint64_t bg = f2_fma(x2, inv2, magic2);     // rne(P) + 1.5*2^23
        const uint64_t nr = f2_sub(magic2, bg);           // -rne(P), exact
        const uint64_t d = f2_fma(x2, inv2, nr);          // P - rne(P), rounded once
        float b0, b1, d0, d1;
        f2_unpack(bg, b0, b1);
        f2_unpack(d, d0, d1);
        big[2 * i] = __float_as_uint(b0);
        big[2 * i + 1] = __float_as_uint(b1);
        dmax = fmaxf(dmax, fmaxf(fabsf(d0), fabsf(d1)));
    }
    if (!(dmax <= 0.5f - kTieGuard)) {
        // rare: recompute each remainder (the same operations give the same
        // values) rather than keep all eight live on the common path
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t x2 = f2_pack(bf16_lo(w[i]), bf16_hi(w[i]));
            const uint64_t bg = f2_fma(x2, inv2, magic2);
            float d0, d1;
            f2_unpack(f2_fma(x2, inv2, f2_sub(magic2, bg)), d0, d1);
            if (!(fabsf(d0) <= 0.5f - kTieGuard)) big[2 * i] = quant_byte_exact(bf16_lo(w[i]), sc.s);
            if (!(fabsf(d1) <= 0.5f - kTieGuard)) big[2 * i + 1] = quant_byte_exact(bf16_hi(w[i]), sc.s);
        }
    }
    // low byte of each value, four to a word
    const uint32_t lo01 = __byte_perm(big[0], big[1], 0x0040);
    const uint32_t lo23 = __byte_perm(big[2], big[3], 0x0040);
    const uint32_t lo45 = __byte_perm(big[4], big[5], 0x0040);
    const uint32_t lo67 = __byte_perm(big[6], big[7], 0x0040);
    return make_uint2(__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo45, lo67, 0x5410));
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

// Write one chunk of 8 codes: as int8 to q[i] (when q is given) and as the
// exact bf16 image of the codes to img[i] (when img is given).
// Like quant_chunk, but returns the codes as their exact bf16 values (the
// image the tensor-core GEMM reads): the rounded quotient rne(P) =
// big - 1.5*2^23 is an integer in [-127, 127] held exactly in fp32, so it is
// packed to bf16 directly.  -0 from the exact path is turned into +0, the
// bf16 image of the code 0.
__device__ __forceinline__ uint4 quant_chunk_img(const uint4& v, const RowScale& sc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float q[8];
    if (sc.exact) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[2 * i] = __fadd_rn(static_cast<float>(quant_exact(bf16_lo(w[i]), sc.s)), 0.0f);
            q[2 * i + 1] = __fadd_rn(static_cast<float>(quant_exact(bf16_hi(w[i]), sc.s)), 0.0f);
        }
    } else {
        const uint64_t inv2 = f2_pack(sc.inv, sc.inv);
        const uint64_t magic2 = f2_pack(kRoundMagic, kRoundMagic);
        float dmax = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t x2 = f2_pack(bf16_lo(w[i]), bf16_hi(w[i]));
            const uint64_t bg = f2_fma(x2, inv2, magic2);  // rne(P) + 1.5*2^23
            const uint64_t nr = f2_sub(magic2, bg);        // -rne(P), exact
            const uint64_t d = f2_fma(x2, inv2, nr);       // P - rne(P), rounded once
            float d0, d1;
            f2_unpack(f2_sub(bg, magic2), q[2 * i], q[2 * i + 1]);  // rne(P), exact (+0 for 0)
            f2_unpack(d, d0, d1);
            dmax = fmaxf(dmax, fmaxf(fabsf(d0), fabsf(d1)));
        }
        if (!(dmax <= 0.5f - kTieGuard)) {
            // rare: recompute each remainder instead of keeping all eight live
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint64_t x2 = f2_pack(bf16_lo(w[i]), bf16_hi(w[i]));
                const uint64_t bg = f2_fma(x2, inv2, magic2);
                float d0, d1;
                f2_unpack(f2_fma(x2, inv2, f2_sub(magic2, bg)), d0, d1);
                if (!(fabsf(d0) <= 0.5f - kTieGuard))
                    q[2 * i] = __fadd_rn(static_cast<float>(quant_exact(bf16_lo(w[i]), sc.s)), 0.0f);
                if (!(fabsf(d1) <= 0.5f - kTieGuard))
                    q[2 * i + 1] = __fadd_rn(static_cast<float>(quant_exact(bf16_hi(w[i]), sc.s)), 0.0f);
            }
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(q[2 * i], q[2 * i + 1]);
        o[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Outputs of a quantization kernel, fixed at compile time.
enum QuantOut : int { kOutCodes = 1, kOutImage = 2, kOutBoth = 3 };

// Quantize chunk i of 8 values and write the int8 codes to q[i] and/or their
// exact bf16 image to img[i], as OUT says.
template <int OUT>
__device__ __forceinline__ void emit_chunk(uint2* __restrict__ q, uint4* __restrict__ img, int64_t i, const uint4& v,
                                           const RowScale& sc) {
    if constexpr (OUT == kOutImage) {
        img[i] = quant_chunk_img(v, sc);
    } else {
        const uint2 c = quant_chunk(v, sc);
        __stcs(q + i, c);
        if constexpr (OUT == kOutBoth) {
            uint4 o;
            o.x = s8x2_to_bf16x2(c.x, 0);
            o.y = s8x2_to_bf16x2(c.x, 2);
            o.z = s8x2_to_bf16x2(c.y, 0);
            o.w = s8x2_to_bf16x2(c.y, 2);
            img[i] = o;
        }
    }
}

__device__ __forceinline__ void put_codes(uint2* __restrict__ q, uint4* __restrict__ img, int64_t i, uint2 c) {
    if (q) __stcs(q + i, c);
    if (img) {
        uint4 o;
        o.x = s8x2_to_bf16x2(c.x, 0);
        o.y = s8x2_to_bf16x2(c.x, 2);
        o.z = s8x2_to_bf16x2(c.y, 0);
        o.w = s8x2_to_bf16x2(c.y, 2);
        img[i] = o;
    }
}

}  // namespace
}  // namespace w8a8
