// Row slices for the streaming kernels: G lanes share a 64-element row, lane
// `sub` owning one contiguous run of 64/G elements read and written with
// 256-bit accesses, and the mixed-precision arithmetic on such slices.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "row_math.cuh"

namespace fibatt {

// 256-bit read-only load and store of eight 32-bit words (32-byte aligned).
__device__ __forceinline__ void ld8(const uint8_t *p, uint32_t *w) {
    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                   "=r"(w[7])
                 : "l"(p));
}

__device__ __forceinline__ void st8(uint8_t *p, const uint32_t *w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// One lane's contiguous slice of a 64-dim row (64/G elements, as 32-bit
// words: packed bf16 pairs or fp32 values), and the matching fp32
// accumulator layout (float2 per element pair, in dim order).
template <typename T, int G>
struct Run {
    static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    static constexpr int kRowBytes = 64 * (int)sizeof(T);
    static constexpr int kBytes = kRowBytes / G;    // bytes of the slice: 32 or 64
    static constexpr int kWords = kBytes / 4;
    static constexpr int kPairs = 32 / G;           // float2 accumulators
    static_assert(kBytes % 32 == 0, "a slice is whole 256-bit loads");
    uint32_t w[kWords];

    __device__ __forceinline__ void load(const uint8_t *p) {
#pragma unroll
        for (int i = 0; i < kWords / 8; ++i) ld8(p + 32 * i, w + 8 * i);
    }
    // partial dot product over this lane's dims (four sums for ILP)
    __device__ __forceinline__ float dot(const Run &o) const {
        float a = 0.f, b = 0.f, c = 0.f, d = 0.f;
        if constexpr (kBf16) {
#pragma unroll
            for (int i = 0; i < kWords; i += 4) {
                a = dot2_bf16(w[i], o.w[i], a);
                b = dot2_bf16(w[i + 1], o.w[i + 1], b);
                c = dot2_bf16(w[i + 2], o.w[i + 2], c);
                d = dot2_bf16(w[i + 3], o.w[i + 3], d);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kWords; i += 4) {
                a = fmaf(__uint_as_float(w[i]), __uint_as_float(o.w[i]), a);
                b = fmaf(__uint_as_float(w[i + 1]), __uint_as_float(o.w[i + 1]), b);
                c = fmaf(__uint_as_float(w[i + 2]), __uint_as_float(o.w[i + 2]), c);
                d = fmaf(__uint_as_float(w[i + 3]), __uint_as_float(o.w[i + 3]), d);
            }
        }
        return (a + b) + (c + d);
    }
    // acc += p * this (fp32 weight)
    __device__ __forceinline__ void axpy(float p, float2 (&acc)[kPairs]) const {
        const float2 pp = make_float2(p, p);
        if constexpr (kBf16) {
#pragma unroll
            for (int i = 0; i < kWords; ++i) acc[i] = fma2(pp, make_float2(bf16_lo(w[i]), bf16_hi(w[i])), acc[i]);
        } else {
#pragma unroll
            for (int i = 0; i < kPairs; ++i)
                acc[i] = fma2(pp, make_float2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1])), acc[i]);
        }
    }
    // acc += p2 * this for a weight already rounded to bf16 (both halves of
    // p2); bf16 rows only: one mixed-precision FMA per element
    __device__ __forceinline__ void axpy_p2(uint32_t p2, float2 (&acc)[kPairs]) const {
#pragma unroll
        for (int i = 0; i < kWords; ++i) acc[i] = fma2_bf16(p2, w[i], acc[i]);
    }
    // acc * s to the I/O dtype (RNE for bf16), stored at p
    __device__ __forceinline__ static void store(uint8_t *p, const float2 (&acc)[kPairs], float s) {
        uint32_t o[kWords];
        if constexpr (kBf16) {
#pragma unroll
            for (int i = 0; i < kWords; ++i) o[i] = pack_bf16x2(acc[i].x * s, acc[i].y * s);
        } else {
#pragma unroll
            for (int i = 0; i < kPairs; ++i) {
                o[2 * i] = __float_as_uint(acc[i].x * s);
                o[2 * i + 1] = __float_as_uint(acc[i].y * s);
            }
        }
#pragma unroll
        for (int i = 0; i < kWords / 8; ++i) st8(p + 32 * i, o + 8 * i);
    }
};

template <int G>
__device__ __forceinline__ float lanes_sum(float x) {
#pragma unroll
    for (int m = 1; m < G; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

}  // namespace fibatt
