// GELU epilogue arithmetic shared by the library's kernels (device code only).
//
// GELU(v) = v * Phi(v) = v * (1 + erf(v / sqrt 2)) / 2, the erf form.  erf comes from
// Abramowitz & Stegun, Handbook of Mathematical Functions, eq. 7.1.28 (after Hastings):
// erf(z) = 1 - (1 + a1 z + ... + a6 z^6)^-16 for z >= 0, |error| <= 3e-7.  Then
// GELU(v) = v - h for v >= 0 and h for v < 0, with h = v (1 - erf(|v|/sqrt 2)) / 2, at one
// reciprocal and no exponential per value.  The absolute GELU error, <= 1.5e-7 |v|, is far
// below both output bounds (bf16 rounding; fp32: 1e-5 of the sum of |x w|).
#pragma once
#include <stdint.h>

namespace convfwd {

__device__ __forceinline__ float gelu(float v) {
    const float z = fabsf(v) * 0.70710678118654752f;
    float y = fmaf(z, 0.0000430638f, 0.0002765672f);
    y = fmaf(z, y, 0.0001520143f);
    y = fmaf(z, y, 0.0092705272f);
    y = fmaf(z, y, 0.0422820123f);
    y = fmaf(z, y, 0.0705230784f);
    y = fmaf(z, y, 1.0f);
    y = y * y; y = y * y; y = y * y; y = y * y;         // (.)^16
    const float h = __fdividef(0.5f * v, y);            // 0 once y overflows
    return v >= 0.0f ? v - h : h;
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

// gelu on two values at once: the polynomial and the squarings as packed f32x2 operations,
// so each value gets bit for bit the result of the scalar form.
__device__ __forceinline__ void gelu2(float& a, float& b) {
    const uint64_t z = f2pk(fabsf(a) * 0.70710678118654752f, fabsf(b) * 0.70710678118654752f);
    uint64_t y = f2fma(z, f2pk(0.0000430638f, 0.0000430638f), f2pk(0.0002765672f, 0.0002765672f));
    y = f2fma(z, y, f2pk(0.0001520143f, 0.0001520143f));
    y = f2fma(z, y, f2pk(0.0092705272f, 0.0092705272f));
    y = f2fma(z, y, f2pk(0.0422820123f, 0.0422820123f));
    y = f2fma(z, y, f2pk(0.0705230784f, 0.0705230784f));
    y = f2fma(z, y, f2pk(1.0f, 1.0f));
    y = f2mul(y, y); y = f2mul(y, y); y = f2mul(y, y); y = f2mul(y, y);   // (.)^16
    float ya, yb;
    f2up(y, ya, yb);
    const float ha = __fdividef(0.5f * a, ya), hb = __fdividef(0.5f * b, yb);
    a = a >= 0.0f ? a - ha : ha;
    b = b >= 0.0f ? b - hb : hb;
}

}  // namespace convfwd
