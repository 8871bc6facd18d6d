// GELU epilogue arithmetic shared by the library's kernels (device code only).
//
// GELU(v) = v * Phi(v) = v * (1 + erf(v / sqrt 2)) / 2, the erf form.  erf comes from
// Abramowitz & Stegun, Handbook of Mathematical Functions, eq. 7.1.28 (after Hastings):
// erf(z) = 1 - (1 + a1 z + ... + a6 z^6)^-16 for z >= 0, |error| <= 3e-7.  Since v * erf(v/sqrt2)
// = |v| erf(|v|/sqrt2), GELU(v) = max(v, 0) - |v| (1 - erf(|v|/sqrt2)) / 2 = max(v, 0) - |v| / (2 y^16)
// for either sign, y = 1 + a1 z + ... with z = |v|/sqrt2: one reciprocal, one fused
// multiply-add and no exponential or select per value.  Evaluated in fp32 over [-8, 8], with the
// reciprocal anywhere within one unit in the last place, the GELU error stays below 9.5e-7 |v|
// (1.4e-7 |v| in exact arithmetic; the rest is mostly the rounding of y near 1, raised to the
// 16th power), far below both output bounds (bf16 rounding; fp32: 1e-5 of the sum of |x w|).
#pragma once
#include <stdint.h>

namespace convfwd {

// Reciprocal on the special-function unit (rcp.approx: within one unit in the last place; 0
// for arguments above 2^126, which flush to zero).
__device__ __forceinline__ float rcp_approx(float y) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

__device__ __forceinline__ float gelu(float v) {
    const float z = fabsf(v) * 0.70710678118654752f;
    float y = fmaf(z, 0.0000430638f, 0.0002765672f);
    y = fmaf(z, y, 0.0001520143f);
    y = fmaf(z, y, 0.0092705272f);
    y = fmaf(z, y, 0.0422820123f);
    y = fmaf(z, y, 0.0705230784f);
    y = fmaf(z, y, 1.0f);
    y = y * y; y = y * y; y = y * y; y = y * y;         // (.)^16
    return fmaf(-0.5f * fabsf(v), rcp_approx(y), fmaxf(v, 0.0f));   // y overflowing gives max(v, 0)
}

// Two fp32 values in one 64-bit register pair, for the packed f32x2 arithmetic of sm_100+
// (one instruction computes both lanes, each rounded exactly as the scalar operation).
__device__ __forceinline__ uint64_t f2pk(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2up(uint64_t r, float& a, float& b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r)); }
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// a += b, b2 for two fp32 values in place
__device__ __forceinline__ void add2(float& a, float& b, float ba, float bb) { f2up(f2add(f2pk(a, b), f2pk(ba, bb)), a, b); }

// gelu on two values at once, for bf16 outputs: the same A&S 7.1.28 form with the argument
// scale 1/sqrt(2) and the factor 1/2 folded into the coefficients, y'(|v|) = 2^(1/16) *
// (1 + a1 |v|/sqrt2 + ... + a6 (|v|/sqrt2)^6), so that y'^16 = 2 y^16 and GELU(v) = max(v, 0) -
// |v| / y'^16.  The polynomial runs in u = -|v| with the odd coefficients negated (Horner's
// steps then carry the same magnitudes and roundings as in |v|), so that the last step is
// max(v, 0) + u / y'^16 as one fused multiply-add; the polynomial, the squarings and that step
// run as packed f32x2 operations.  Evaluated in fp32 over [-8, 8] its error stays below
// 1.25e-6 |v|, far below the bf16 rounding of the output (2^-9 relative).
__device__ __forceinline__ void gelu2(float& a, float& b) {
    const uint64_t u = f2pk(-fabsf(a), -fabsf(b));
    uint64_t y = f2fma(u, f2pk(5.6212996640e-06f, 5.6212996640e-06f), f2pk(-5.1055209009e-05f, -5.1055209009e-05f));
    y = f2fma(u, y, f2pk(3.9686137011e-05f, 3.9686137011e-05f));
    y = f2fma(u, y, f2pk(-3.4227392389e-03f, -3.4227392389e-03f));
    y = f2fma(u, y, f2pk(2.2076998457e-02f, 2.2076998457e-02f));
    y = f2fma(u, y, f2pk(-5.2075163037e-02f, -5.2075163037e-02f));
    y = f2fma(u, y, f2pk(1.0442737824e+00f, 1.0442737824e+00f));
    y = f2mul(y, y); y = f2mul(y, y); y = f2mul(y, y); y = f2mul(y, y);   // (.)^16
    float ya, yb;
    f2up(y, ya, yb);
    f2up(f2fma(u, f2pk(rcp_approx(ya), rcp_approx(yb)), f2pk(fmaxf(a, 0.0f), fmaxf(b, 0.0f))), a, b);
}

}  // namespace convfwd
