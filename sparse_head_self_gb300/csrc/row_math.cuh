// Mixed-precision and packed fp32 arithmetic on row data, inline PTX for
// sm_100+ / sm_103a: the building blocks of every banded kernel's dot
// products, row updates and exponentials.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace fibatt {

// c + lo(a)*lo(b) + hi(a)*hi(b) for packed bf16 pairs a, b.  Each product of
// two bf16 values is exact in fp32, so this equals converting both operands
// to fp32 and using fmaf, rounding for rounding.
__device__ __forceinline__ float dot2_bf16(uint32_t a, uint32_t b, float c) {
    unsigned short al, ah, bl, bh;
    asm("mov.b32 {%0, %1}, %2;" : "=h"(al), "=h"(ah) : "r"(a));
    asm("mov.b32 {%0, %1}, %2;" : "=h"(bl), "=h"(bh) : "r"(b));
    float d;
    asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(al), "h"(bl), "f"(c));
    asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(ah), "h"(bh), "f"(d));
    return d;
}

// (c.x + a.x*b.x, c.y + a.y*b.y), each an IEEE fma (packed f32x2, sm_100+).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// (c.x, c.y) + (lo(w), hi(w)) * (lo(p2), hi(p2)) for packed bf16 pairs w and
// p2, products exact and accumulated in fp32 (one mixed-precision FMA per
// element, no unpacking of w).
__device__ __forceinline__ float2 fma2_bf16(uint32_t p2, uint32_t w, float2 c) {
    asm("{\n\t.reg .b16 pl, ph, wl, wh;\n\t"
        "mov.b32 {pl, ph}, %2;\n\t"
        "mov.b32 {wl, wh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, pl, wl, %0;\n\t"
        "fma.rn.f32.bf16 %1, ph, wh, %1;\n\t}"
        : "+f"(c.x), "+f"(c.y)
        : "r"(p2), "r"(w));
    return c;
}

// p rounded to bf16 (nearest even) in both halves of a packed pair.
__device__ __forceinline__ uint32_t bf16x2_splat(float p) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(p));
    return r;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// 2^x on the SFU (ex2.approx.ftz, relative error about 2^-22; results below
// 2^-126 flush to zero, which only drops weights under 1e-38).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace fibatt
