// GELU of the FFN up-projection, in its erf form: gelu(x) = x * Phi(x),
// Phi(x) = (1 + erf(x / sqrt 2)) / 2, the bf16 result of a bf16 input.
//
// Phi is evaluated through the complementary error function, which keeps its
// relative accuracy in the negative tail:
//   Phi(-|x|) = erfc(z) / 2,  Phi(|x|) = 1 - erfc(z) / 2,  z = |x| / sqrt 2,
// with erfc from the Chebyshev-fitted formula of Press, Teukolsky, Vetterling
// and Flannery, Numerical Recipes in C, 2nd ed., section 6.2:
//   erfc(z) = t * exp(-z^2 + P(t)),  t = 1 / (1 + z / 2),
//   P(t) = -1.26551223 + t (1.00002368 + t (0.37409196 + ... + t 0.17087277)),
// whose fractional error is below 1.2e-7 for every z >= 0.
//
// Binary32 evaluation, two values at a time on the packed fp32 pipe:
//   t = rcp(fma(z, 1/2, 1)), P by Horner (fused multiply-adds),
//   A = fma(-z, z, P), e = 2^(fma(A, log2 e, 64)) (ex2), h = (t / 2) * e,
// so h = Phi(-|x|) * 2^64, which stays a normal number down to the far tail;
//   x >= 0:  g = x * (1 - h * 2^-64),     x < 0:  g = (x * h) * 2^-64,
// the last multiplication rounding a tiny result into the subnormal range
// once.  rcp.approx and ex2.approx are within 1 ulp and 2^-22 of exact.  The
// relative error of g is below 1e-6 for |x| < 4 and below 7e-6 anywhere (the
// roundings of z^2 and of A * log2 e in the far tail); bf16 keeps 8
// significant bits, so the bf16 result is within 1 ulp of the bf16 of the
// exact GELU everywhere, and equal to it except where the exact value lies
// within that error of a bf16 rounding boundary.  Large |x| needs no special
// case: z^2 overflows to infinity, e to 0, and g to x (x > 0) or -0 (x < 0).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace w8a8 {
namespace {

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ uint64_t f2_splat(float v) { return f2_pack(v, v); }

// bf16(gelu(x0)), bf16(gelu(x1)) packed (x0 in the low half).
__device__ __forceinline__ uint32_t gelu_bf16x2(float x0, float x1) {
    constexpr float kRsqrt2 = 0.70710678118654752f;
    constexpr float kLog2e = 1.44269504088896341f;
    constexpr float kTwoM64 = 5.42101086242752217e-20f;  // 2^-64
    const uint64_t z = f2_mul(f2_pack(fabsf(x0), fabsf(x1)), f2_splat(kRsqrt2));
    const uint64_t nz = f2_mul(f2_pack(-fabsf(x0), -fabsf(x1)), f2_splat(kRsqrt2));  // -z, exactly
    float d0, d1;
    f2_unpack(f2_fma(z, f2_splat(0.5f), f2_splat(1.0f)), d0, d1);
    const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
    uint64_t p = f2_splat(0.17087277f);
    p = f2_fma(t, p, f2_splat(-0.82215223f));
    p = f2_fma(t, p, f2_splat(1.48851587f));
    p = f2_fma(t, p, f2_splat(-1.13520398f));
    p = f2_fma(t, p, f2_splat(0.27886807f));
    p = f2_fma(t, p, f2_splat(-0.18628806f));
    p = f2_fma(t, p, f2_splat(0.09678418f));
    p = f2_fma(t, p, f2_splat(0.37409196f));
    p = f2_fma(t, p, f2_splat(1.00002368f));
    p = f2_fma(t, p, f2_splat(-1.26551223f));
    const uint64_t a = f2_fma(nz, z, p);                                  // -z^2 + P(t)
    float e0, e1;
    f2_unpack(f2_fma(a, f2_splat(kLog2e), f2_splat(64.0f)), e0, e1);
    const uint64_t h = f2_mul(f2_mul(t, f2_splat(0.5f)), f2_pack(ex2_approx(e0), ex2_approx(e1)));  // Phi(-|x|) 2^64
    const uint64_t x = f2_pack(x0, x1);
    const uint64_t gp = f2_mul(x, f2_sub(f2_splat(1.0f), f2_mul(h, f2_splat(kTwoM64))));
    const uint64_t gn = f2_mul(f2_mul(x, h), f2_splat(kTwoM64));
    float p0, p1, n0, n1;
    f2_unpack(gp, p0, p1);
    f2_unpack(gn, n0, n1);
    __nv_bfloat162 r = __floats2bfloat162_rn(x0 >= 0.0f ? p0 : n0, x1 >= 0.0f ? p1 : n1);
    return *reinterpret_cast<uint32_t*>(&r);
}

}  // namespace
}  // namespace w8a8
