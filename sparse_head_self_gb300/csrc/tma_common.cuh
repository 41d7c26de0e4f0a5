// Bulk-copy (TMA) and mbarrier helpers, inline PTX for sm_100+ / sm_103a, and
// the row-slice arithmetic shared by the shared-memory-resident kernels.
//
// Every wait on an mbarrier is bounded by wall-clock time (%globaltimer):
// after kWaitLimitNs the waiting thread records kErrWaitTimeout in the
// device error word and raises the CTA's abort flag, after which no wait of
// the CTA blocks any more, so a bad byte count can never hang the GPU; a
// producer still waits (bounded) for the copies it issued before it leaves.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "row_math.cuh"

namespace fibatt {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// One-dimensional bulk copy global -> this CTA's shared memory, completion
// counted in bytes on `bar`.  dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Hint that [src, src + bytes) will be read soon: bulk prefetch into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Barrier among the first `threads` threads past warp 0 (named barrier 1).
__device__ __forceinline__ void consumer_sync(int threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// Barrier among `threads` threads on named barrier `id` (2..15; 1 is the
// consumers').
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Plain arrive (count 1) on `bar`.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Wait for phase `parity` of `bar` to complete; false on timeout (error
// recorded).  Each try_wait carries a suspend-time hint, so a waiting warp is
// parked by the hardware until the phase completes (or about 0.5 ms pass)
// instead of spinning and taking issue slots from the warps that compute.
//
// `abort` is a flag in the CTA's shared memory.  A wait that runs out of time
// sets it, and every wait of the CTA that starts (or is still spinning) once
// it is set gives up at once.  So when one wait fails, the whole CTA stops
// waiting: a caller that carries on after a false return (computing garbage
// that is never trusted, since the error word is set) still reaches every
// named barrier its peers reach, and no warp is left behind at one.
__device__ __forceinline__ bool mbar_try_wait(uint32_t b, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(b), "r"(parity), "r"(500000u)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const uint32_t b = smem_u32(bar);
    if (*abort) return false;
    if (mbar_try_wait(b, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(b, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_device_error, kErrWaitTimeout);
            *abort = 1;
            return false;
        }
    }
}

// Wait, bounded but regardless of `abort`, for phase `parity` of a stage's
// "full" barrier: the bulk copies a producer issued into the stage have
// landed.  A producer calls it for the last use of every stage before it
// leaves, so the CTA never exits with copies still writing into its shared
// memory (its consumers may have given up on them).
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    const uint32_t b = smem_u32(bar);
    if (mbar_try_wait(b, parity)) return;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(b, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_device_error, kErrDrainTimeout);
            return;
        }
    }
}

// ---- a slice of one 64-dim row ---------------------------------------------
//
// G lanes own one row, 64/G dims each (G = 2 or 4).  The lane at slot `sub`
// (0..G-1) of the row at position `pos` (0..8/G-1: the row's slot inside an
// eight-lane shared-memory phase) walks its 16-byte chunks in an order chosen
// so that the eight lanes of each phase touch eight different bank groups:
// rows are 128 B (bf16) or 256 B (fp32) and start on bank 0, so a chunk's
// bank group is its index modulo 8.  `acc` holds the lane's dims as float2
// pairs in the same chunk order.
template <typename T, int G>
struct Slice;

template <int G>
struct SliceBf16 {
    static constexpr int kChunks = 8 / G;    // 16-byte chunks per lane
    static constexpr int kRowBytes = 128;
    static constexpr int kPairs = 32 / G;    // float2 accumulators per lane
    __device__ static __forceinline__ int chunk(int sub, int pos, int i) {
        return kChunks * sub + ((i + pos) % kChunks);
    }
    uint4 w[kChunks];                        // packed bf16 pairs

    __device__ __forceinline__ void load(const uint8_t *row, const int (&c)[kChunks]) {
#pragma unroll
        for (int i = 0; i < kChunks; ++i) w[i] = *reinterpret_cast<const uint4 *>(row + c[i]);
    }
    __device__ __forceinline__ void load_global(const void *row, const int (&c)[kChunks]) {
#pragma unroll
        for (int i = 0; i < kChunks; ++i)
            w[i] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(row) + c[i]));
    }
    // partial <this, o> over the lane's dims (four interleaved sums for ILP)
    __device__ __forceinline__ float dot(const SliceBf16 &o) const {
        float a = 0.f, b = 0.f, c = 0.f, d = 0.f;
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            a = dot2_bf16(w[i].x, o.w[i].x, a);
            b = dot2_bf16(w[i].y, o.w[i].y, b);
            c = dot2_bf16(w[i].z, o.w[i].z, c);
            d = dot2_bf16(w[i].w, o.w[i].w, d);
        }
        return (a + b) + (c + d);
    }
    // acc[4i + e] += p * (element pair e of chunk i), fp32 weight
    __device__ __forceinline__ void axpy(float p, float2 (&acc)[kPairs]) const {
        const float2 pp = make_float2(p, p);
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            acc[4 * i + 0] = fma2(pp, make_float2(bf16_lo(w[i].x), bf16_hi(w[i].x)), acc[4 * i + 0]);
            acc[4 * i + 1] = fma2(pp, make_float2(bf16_lo(w[i].y), bf16_hi(w[i].y)), acc[4 * i + 1]);
            acc[4 * i + 2] = fma2(pp, make_float2(bf16_lo(w[i].z), bf16_hi(w[i].z)), acc[4 * i + 2]);
            acc[4 * i + 3] = fma2(pp, make_float2(bf16_lo(w[i].w), bf16_hi(w[i].w)), acc[4 * i + 3]);
        }
    }
    // The same update with a weight already rounded to bf16 (p2: both halves
    // of a packed pair, from bf16x2_splat): one mixed-precision FMA per
    // element (exact product, fp32 sum) instead of an unpack and half a
    // packed FMA.
    __device__ __forceinline__ void axpy_p2(uint32_t p2, float2 (&acc)[kPairs]) const {
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            acc[4 * i + 0] = fma2_bf16(p2, w[i].x, acc[4 * i + 0]);
            acc[4 * i + 1] = fma2_bf16(p2, w[i].y, acc[4 * i + 1]);
            acc[4 * i + 2] = fma2_bf16(p2, w[i].z, acc[4 * i + 2]);
            acc[4 * i + 3] = fma2_bf16(p2, w[i].w, acc[4 * i + 3]);
        }
    }
    // store acc (in this lane's chunk order) to a global row, RNE to bf16
    __device__ __forceinline__ static void store(void *row, const int (&c)[kChunks], const float2 (&acc)[kPairs]) {
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            uint4 t;
            t.x = pack_bf16x2(acc[4 * i + 0].x, acc[4 * i + 0].y);
            t.y = pack_bf16x2(acc[4 * i + 1].x, acc[4 * i + 1].y);
            t.z = pack_bf16x2(acc[4 * i + 2].x, acc[4 * i + 2].y);
            t.w = pack_bf16x2(acc[4 * i + 3].x, acc[4 * i + 3].y);
            *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(row) + c[i]) = t;
        }
    }
};

template <int G>
struct SliceF32 {
    static constexpr int kChunks = 16 / G;
    static constexpr int kRowBytes = 256;
    static constexpr int kPairs = 32 / G;
    // rows of 256 B: chunk c maps to bank group c mod 8
    __device__ static __forceinline__ int chunk(int sub, int pos, int i) {
        if (G == 2) return 8 * sub + ((i + 2 * pos + sub) & 7);
        return 4 * sub + ((i + 2 * (sub >> 1) + pos) & 3);
    }
    float4 w[kChunks];

    __device__ __forceinline__ void load(const uint8_t *row, const int (&c)[kChunks]) {
#pragma unroll
        for (int i = 0; i < kChunks; ++i) w[i] = *reinterpret_cast<const float4 *>(row + c[i]);
    }
    __device__ __forceinline__ void load_global(const void *row, const int (&c)[kChunks]) {
#pragma unroll
        for (int i = 0; i < kChunks; ++i)
            w[i] = __ldg(reinterpret_cast<const float4 *>(static_cast<const uint8_t *>(row) + c[i]));
    }
    __device__ __forceinline__ float dot(const SliceF32 &o) const {
        float a = 0.f, b = 0.f, c = 0.f, d = 0.f;
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            a = fmaf(w[i].x, o.w[i].x, a);
            b = fmaf(w[i].y, o.w[i].y, b);
            c = fmaf(w[i].z, o.w[i].z, c);
            d = fmaf(w[i].w, o.w[i].w, d);
        }
        return (a + b) + (c + d);
    }
    __device__ __forceinline__ void axpy(float p, float2 (&acc)[kPairs]) const {
        const float2 pp = make_float2(p, p);
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            acc[2 * i + 0] = fma2(pp, make_float2(w[i].x, w[i].y), acc[2 * i + 0]);
            acc[2 * i + 1] = fma2(pp, make_float2(w[i].z, w[i].w), acc[2 * i + 1]);
        }
    }
    __device__ __forceinline__ static void store(void *row, const int (&c)[kChunks], const float2 (&acc)[kPairs]) {
#pragma unroll
        for (int i = 0; i < kChunks; ++i)
            *reinterpret_cast<float4 *>(static_cast<uint8_t *>(row) + c[i]) =
                make_float4(acc[2 * i].x, acc[2 * i].y, acc[2 * i + 1].x, acc[2 * i + 1].y);
    }
};

template <int G>
struct Slice<__nv_bfloat16, G> : SliceBf16<G> {};
template <int G>
struct Slice<float, G> : SliceF32<G> {};

// Sum over the G lanes of a row (xor-shuffles).
template <int G>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int m = 1; m < G; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

}  // namespace fibatt
