// The global first token (Fibottention README, Algorithm 2: the mask keeps
// row 0 and column 0 all ones, so the class token attends every key and every
// query attends it).  The banded kernels add the pair (j, 0) to each query
// row j >= 1 whose band misses key 0, and the pair (0, k) to each key row
// k >= 1 whose band misses query 0; the kernels here handle what is dense:
//
//   fwd_global_row_kernel   O_0, LSE_0 over every key (overwrites the banded
//                           kernel's row 0)
//   bwd_global_row_kernel   P_0k, dS_0k for every key k (workspace, read by
//                           the banded backward for the pairs (0, k)) and
//                           dQ_0 over every key
//   bwd_global_col_kernel   dK_0, dV_0 over every query (the whole column of
//                           key 0, every query attends it)
//
// One block of kGtWarps warps per (b, h); a warp takes one key (or query) row
// at a time, two dims per lane, dot products reduced across the warp.
#include "device_common.cuh"
#include "fibatt_internal.h"

namespace fibatt {
namespace {

constexpr int kGtWarps = 8;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(kFullMask, x, m);
    return x;
}

// elements 2 * lane and 2 * lane + 1 of a 64-element row, as fp32
__device__ __forceinline__ float2 row_pair(const __nv_bfloat16 *row, int lane) {
    const uint32_t w = __ldg(reinterpret_cast<const unsigned int *>(row) + lane);
    return make_float2(bf16_lo(w), bf16_hi(w));
}
__device__ __forceinline__ float2 row_pair(const float *row, int lane) {
    return __ldg(reinterpret_cast<const float2 *>(row) + lane);
}
__device__ __forceinline__ void store_pair(__nv_bfloat16 *row, int lane, float2 v) {
    reinterpret_cast<unsigned int *>(row)[lane] = pack_bf16x2(v.x, v.y);
}
__device__ __forceinline__ void store_pair(float *row, int lane, float2 v) {
    reinterpret_cast<float2 *>(row)[lane] = v;
}

// Merge the warps' (m, l, acc) of a softmax taken in log2 units into the
// block's: returns (acc / l for this lane's two dims, m + log2 l) in warp 0.
__device__ __forceinline__ void merge_warps(float m, float l, float2 acc, float *s_m, float *s_l, float2 *s_acc,
                                            int warp, int lane, float2 *out, float *lse2) {
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    s_acc[warp * 32 + lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float M = -INFINITY;
        for (int w = 0; w < kGtWarps; ++w) M = fmaxf(M, s_m[w]);
        float L = 0.f;
        float2 A = make_float2(0.f, 0.f);
        for (int w = 0; w < kGtWarps; ++w) {
            const float f = s_l[w] > 0.f ? exp2f(s_m[w] - M) : 0.f;
            L += f * s_l[w];
            A.x += f * s_acc[w * 32 + lane].x;
            A.y += f * s_acc[w * 32 + lane].y;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        *out = make_float2(A.x * inv, A.y * inv);
        *lse2 = L > 0.f ? M + log2f(L) : -INFINITY;
    }
}

template <typename T>
__global__ void __launch_bounds__(kGtWarps * 32)
fwd_global_row_kernel(int N, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      float scale_log2, T *__restrict__ O, float *__restrict__ LSE) {
    __shared__ float s_m[kGtWarps], s_l[kGtWarps];
    __shared__ float2 s_acc[kGtWarps * 32];
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t base = (size_t)blockIdx.x * N * kHeadDim;
    const float2 q = row_pair(Q + base, lane);
    float m = -INFINITY, l = 0.f;
    float2 acc = make_float2(0.f, 0.f);
    for (int k = warp; k < N; k += kGtWarps) {
        const float2 kk = row_pair(K + base + (size_t)k * kHeadDim, lane);
        const float s = warp_sum(fmaf(q.x, kk.x, q.y * kk.y)) * scale_log2;
        if (s > m) {   // warp-uniform
            const float a = exp2f(m - s);
            l *= a;
            acc.x *= a;
            acc.y *= a;
            m = s;
        }
        const float p = exp2f(s - m);
        l += p;
        const float2 vv = row_pair(V + base + (size_t)k * kHeadDim, lane);
        acc.x = fmaf(p, vv.x, acc.x);
        acc.y = fmaf(p, vv.y, acc.y);
    }
    float2 o;
    float lse2;
    merge_warps(m, l, acc, s_m, s_l, s_acc, warp, lane, &o, &lse2);
    if (warp == 0) {
        store_pair(O + base, lane, o);
        if (lane == 0) LSE[(size_t)blockIdx.x * N] = lse2 * kLn2;
    }
}

// gw: [B*H][2][N] fp32: P_0k, then dS_0k.
template <typename T>
__global__ void __launch_bounds__(kGtWarps * 32)
bwd_global_row_kernel(int N, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      const T *__restrict__ O, const float *__restrict__ LSE, const T *__restrict__ dO,
                      float scale, float scale_log2, T *__restrict__ dQ, float *__restrict__ gw) {
    __shared__ float2 s_acc[kGtWarps * 32];
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t base = (size_t)blockIdx.x * N * kHeadDim;
    float *gP = gw + (size_t)blockIdx.x * 2 * N, *gS = gP + N;
    const float2 q = row_pair(Q + base, lane), g = row_pair(dO + base, lane), o = row_pair(O + base, lane);
    const float D0 = warp_sum(fmaf(g.x, o.x, g.y * o.y));
    const float lse2 = LSE[(size_t)blockIdx.x * N] * kLog2e;
    float2 dq = make_float2(0.f, 0.f);
    for (int k = warp; k < N; k += kGtWarps) {
        const float2 kk = row_pair(K + base + (size_t)k * kHeadDim, lane);
        const float2 vv = row_pair(V + base + (size_t)k * kHeadDim, lane);
        const float s = warp_sum(fmaf(q.x, kk.x, q.y * kk.y));
        const float dp = warp_sum(fmaf(g.x, vv.x, g.y * vv.y));
        const float P = exp2f(fmaf(s, scale_log2, -lse2));
        const float dS = P * (dp - D0);
        if (lane == 0) {
            gP[k] = P;
            gS[k] = dS;
        }
        dq.x = fmaf(dS, kk.x, dq.x);
        dq.y = fmaf(dS, kk.y, dq.y);
    }
    s_acc[warp * 32 + lane] = dq;
    __syncthreads();
    if (warp == 0) {
        float2 a = make_float2(0.f, 0.f);
        for (int w = 0; w < kGtWarps; ++w) {
            a.x += s_acc[w * 32 + lane].x;
            a.y += s_acc[w * 32 + lane].y;
        }
        store_pair(dQ + base, lane, make_float2(a.x * scale, a.y * scale));
    }
}

template <typename T>
__global__ void __launch_bounds__(kGtWarps * 32)
bwd_global_col_kernel(int N, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      const T *__restrict__ O, const float *__restrict__ LSE, const T *__restrict__ dO,
                      float scale, float scale_log2, T *__restrict__ dK, T *__restrict__ dV) {
    __shared__ float2 s_k[kGtWarps * 32], s_v[kGtWarps * 32];
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t base = (size_t)blockIdx.x * N * kHeadDim;
    const float2 k0 = row_pair(K + base, lane), v0 = row_pair(V + base, lane);
    float2 dk = make_float2(0.f, 0.f), dv = make_float2(0.f, 0.f);
    for (int j = warp; j < N; j += kGtWarps) {
        const size_t r = base + (size_t)j * kHeadDim;
        const float2 q = row_pair(Q + r, lane), g = row_pair(dO + r, lane), o = row_pair(O + r, lane);
        const float s = warp_sum(fmaf(q.x, k0.x, q.y * k0.y));
        const float dp = warp_sum(fmaf(g.x, v0.x, g.y * v0.y));
        const float Dj = warp_sum(fmaf(g.x, o.x, g.y * o.y));
        const float P = exp2f(fmaf(s, scale_log2, -LSE[(size_t)blockIdx.x * N + j] * kLog2e));
        const float dS = P * (dp - Dj);
        dk.x = fmaf(dS, q.x, dk.x);
        dk.y = fmaf(dS, q.y, dk.y);
        dv.x = fmaf(P, g.x, dv.x);
        dv.y = fmaf(P, g.y, dv.y);
    }
    s_k[warp * 32 + lane] = dk;
    s_v[warp * 32 + lane] = dv;
    __syncthreads();
    if (warp == 0) {
        float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
        for (int w = 0; w < kGtWarps; ++w) {
            a.x += s_k[w * 32 + lane].x;
            a.y += s_k[w * 32 + lane].y;
            b.x += s_v[w * 32 + lane].x;
            b.y += s_v[w * 32 + lane].y;
        }
        store_pair(dK + base, lane, make_float2(a.x * scale, a.y * scale));
        store_pair(dV + base, lane, b);
    }
}

template <typename T>
cudaError_t fwd_global(const FwdArgs &a) {
    const TableArg &tab = *a.tab;
    const cudaError_t e = launch_kernel(fwd_global_row_kernel<T>, dim3((unsigned)(a.B * tab.H)),
                                        dim3(kGtWarps * 32), 0, a.stream, pdl_enabled(), (int)tab.N,
                                        static_cast<const T *>(a.Q), static_cast<const T *>(a.K),
                                        static_cast<const T *>(a.V), a.scale * kLog2e, static_cast<T *>(a.O),
                                        a.LSE);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
cudaError_t bwd_global(const BwdArgs &a, bool row) {
    const TableArg &tab = *a.tab;
    const dim3 grid((unsigned)(a.B * tab.H)), block(kGtWarps * 32);
    cudaError_t e;
    if (row)
        e = launch_kernel(bwd_global_row_kernel<T>, grid, block, 0, a.stream, pdl_enabled(), (int)tab.N,
                          static_cast<const T *>(a.Q), static_cast<const T *>(a.K), static_cast<const T *>(a.V),
                          static_cast<const T *>(a.O), a.LSE, static_cast<const T *>(a.dO), a.scale,
                          a.scale * kLog2e, static_cast<T *>(a.dQ), a.gw);
    else
        e = launch_kernel(bwd_global_col_kernel<T>, grid, block, 0, a.stream, pdl_enabled(), (int)tab.N,
                          static_cast<const T *>(a.Q), static_cast<const T *>(a.K), static_cast<const T *>(a.V),
                          static_cast<const T *>(a.O), a.LSE, static_cast<const T *>(a.dO), a.scale,
                          a.scale * kLog2e, static_cast<T *>(a.dK), static_cast<T *>(a.dV));
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_global_row(const FwdArgs &a) {
    return a.dtype == FIBATT_F32 ? fwd_global<float>(a) : fwd_global<__nv_bfloat16>(a);
}

cudaError_t launch_bwd_global_row(const BwdArgs &a) {
    return a.dtype == FIBATT_F32 ? bwd_global<float>(a, true) : bwd_global<__nv_bfloat16>(a, true);
}

cudaError_t launch_bwd_global_col(const BwdArgs &a) {
    return a.dtype == FIBATT_F32 ? bwd_global<float>(a, false) : bwd_global<__nv_bfloat16>(a, false);
}

}  // namespace fibatt
