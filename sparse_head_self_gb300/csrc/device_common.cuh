// Device helpers shared by the libfibatt kernels: row-slice loads/stores
// between global memory and fp32 registers for the two I/O dtypes.
#pragma once

#include <cstdint>
#include <cstdio>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fibatt {

// Device error word (bit flags), read and cleared by fibatt_device_error().
// The library is built without relocatable device code, so every .cu file
// has its own copy of the word; each defines a reader with
// FIBATT_DEFINE_ERROR_READER, and read_device_error() (resident.cu) combines
// them.
static __device__ unsigned int g_device_error = 0;
constexpr unsigned kErrWaitTimeout = 1u;    // a bounded mbarrier wait gave up
constexpr unsigned kErrDrainTimeout = 2u;   // a producer left before its last copies landed
constexpr unsigned kErrBounds = 4u;         // a bounds check of a FIBATT_CHECKS build failed

// Bounds checks of the debug build (-DFIBATT_CHECKS): FIBATT_CHECKED(cond)
// is `cond`, and a false one records kErrBounds and the first failing source
// line (this file's copy of g_check_line); the caller then skips the
// access.  In the regular build FIBATT_CHECKED(cond) is `true` and costs
// nothing.
#ifdef FIBATT_CHECKS
static __device__ unsigned int g_check_line = 0;
__device__ __forceinline__ bool check_ok(bool ok, unsigned line) {
    if (!ok) {
        atomicOr(&g_device_error, kErrBounds);
        atomicCAS(&g_check_line, 0u, line);
    }
    return ok;
}
#define FIBATT_CHECKED(cond) (::fibatt::check_ok((cond), __LINE__))
#define FIBATT_CHECK_READ_LINE(file)                                                                  \
    {                                                                                                  \
        unsigned line = 0;                                                                             \
        if (cudaMemcpyFromSymbol(&line, g_check_line, sizeof(unsigned)) == cudaSuccess && line) {      \
            fprintf(stderr, "libfibatt checks: a bounds check failed in %s, line %u\n", file, line); \
            if (clear) {                                                                               \
                const unsigned z = 0;                                                                  \
                cudaMemcpyToSymbol(g_check_line, &z, sizeof(unsigned));                                \
            }                                                                                          \
        }                                                                                              \
    }
#else
#define FIBATT_CHECKED(cond) true
#define FIBATT_CHECK_READ_LINE(file)
#endif

// Defines `cudaError_t fn(unsigned *code, bool clear)`, the reader of this
// file's error word (and, in a checks build, the line of its first failed
// check, printed to stderr).
#define FIBATT_DEFINE_ERROR_READER(fn, file)                                         \
    cudaError_t fn(unsigned *code, bool clear) {                                     \
        cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(unsigned)); \
        if (e != cudaSuccess) return e;                                              \
        FIBATT_CHECK_READ_LINE(file)                                                 \
        if (!clear || *code == 0) return cudaSuccess;                                \
        const unsigned zero = 0;                                                     \
        return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));          \
    }

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)
constexpr unsigned kFullMask = 0xffffffffu;

// Programmatic dependent launch (sm_90+).  launch_dependents lets the next
// kernel of the stream be scheduled while this one runs (its blocks take SMs
// as ours retire); wait blocks until every prerequisite grid has completed
// and its memory is visible.  Both are no-ops for an ordinary launch.  The
// kernels call wait first and launch_dependents after it, so a dependent
// grid is never scheduled before this grid's own prerequisites are done.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// bf16 -> fp32 is exact: the 16 bits are the high half of the fp32 pattern.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> packed bf16x2, round to nearest even (lo at the lower address).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Load 16 consecutive elements (16-byte aligned) as fp32.
__device__ __forceinline__ void load16(const float *p, float (&x)[16]) {
    const float4 *v = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 t = __ldg(v + i);
        x[4 * i + 0] = t.x;
        x[4 * i + 1] = t.y;
        x[4 * i + 2] = t.z;
        x[4 * i + 3] = t.w;
    }
}

__device__ __forceinline__ void load16(const __nv_bfloat16 *p, float (&x)[16]) {
    const uint4 *v = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint4 t = __ldg(v + i);
        x[8 * i + 0] = bf16_lo(t.x);
        x[8 * i + 1] = bf16_hi(t.x);
        x[8 * i + 2] = bf16_lo(t.y);
        x[8 * i + 3] = bf16_hi(t.y);
        x[8 * i + 4] = bf16_lo(t.z);
        x[8 * i + 5] = bf16_hi(t.z);
        x[8 * i + 6] = bf16_lo(t.w);
        x[8 * i + 7] = bf16_hi(t.w);
    }
}

__device__ __forceinline__ void store16(float *p, const float (&x)[16]) {
    float4 *v = reinterpret_cast<float4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
}

__device__ __forceinline__ void store16(__nv_bfloat16 *p, const float (&x)[16]) {
    uint4 *v = reinterpret_cast<uint4 *>(p);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint4 t;
        t.x = pack_bf16x2(x[8 * i + 0], x[8 * i + 1]);
        t.y = pack_bf16x2(x[8 * i + 2], x[8 * i + 3]);
        t.z = pack_bf16x2(x[8 * i + 4], x[8 * i + 5]);
        t.w = pack_bf16x2(x[8 * i + 6], x[8 * i + 7]);
        v[i] = t;
    }
}

}  // namespace fibatt
