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
// One block of NW warps per (b, h) (8 for short sequences, 32 for long ones);
// a warp takes kGtRows key (or query) rows at a time (their loads issued
// together), two dims per lane, dot products reduced across the warp.
#include "device_common.cuh"
#include "fibatt_internal.h"

namespace fibatt {
namespace {

constexpr int kGtRows = 4;   // rows per warp step (backward kernels)
constexpr int kGtRowsFwd = 8;   // rows per warp step, forward row kernel (8 measured faster there, 4 in the backward)

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
template <int NW>
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
        for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w]);
        float L = 0.f;
        float2 A = make_float2(0.f, 0.f);
        for (int w = 0; w < NW; ++w) {
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

template <typename T, int NW>
__global__ void __launch_bounds__(NW * 32)
fwd_global_row_kernel(int N, long bh0, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      float scale_log2, T *__restrict__ O, float *__restrict__ LSE) {
    __shared__ float s_m[NW], s_l[NW];
    __shared__ float2 s_acc[NW * 32];
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = (size_t)bh0 + blockIdx.x;
    const size_t base = bh * N * kHeadDim;
    const float2 q = row_pair(Q + base, lane);
    float m = -INFINITY, l = 0.f;
    float2 acc = make_float2(0.f, 0.f);
    for (int k0 = warp * kGtRowsFwd; k0 < N; k0 += NW * kGtRowsFwd) {
        float2 kk[kGtRowsFwd], vv[kGtRowsFwd];
        float s[kGtRowsFwd];
#pragma unroll
        for (int i = 0; i < kGtRowsFwd; ++i) {
            const int k = min(k0 + i, N - 1);
            kk[i] = row_pair(K + base + (size_t)k * kHeadDim, lane);
            vv[i] = row_pair(V + base + (size_t)k * kHeadDim, lane);
        }
#pragma unroll
        for (int i = 0; i < kGtRowsFwd; ++i) {
            const float x = warp_sum(fmaf(q.x, kk[i].x, q.y * kk[i].y)) * scale_log2;
            s[i] = k0 + i < N ? x : -INFINITY;
        }
        float mb = s[0];
#pragma unroll
        for (int i = 1; i < kGtRowsFwd; ++i) mb = fmaxf(mb, s[i]);
        if (mb > m) {   // warp-uniform
            const float a = exp2f(m - mb);
            l *= a;
            acc.x *= a;
            acc.y *= a;
            m = mb;
        }
#pragma unroll
        for (int i = 0; i < kGtRowsFwd; ++i) {
            const float p = exp2f(s[i] - m);
            l += p;
            acc.x = fmaf(p, vv[i].x, acc.x);
            acc.y = fmaf(p, vv[i].y, acc.y);
        }
    }
    float2 o;
    float lse2;
    merge_warps<NW>(m, l, acc, s_m, s_l, s_acc, warp, lane, &o, &lse2);
    if (warp == 0) {
        store_pair(O + base, lane, o);
        if (lane == 0) LSE[bh * N] = lse2 * kLn2;
    }
}

// gw: [B*H][2][N] fp32: P_0k, then dS_0k.
template <typename T, int NW>
__global__ void __launch_bounds__(NW * 32)
bwd_global_row_kernel(int N, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      const T *__restrict__ O, const float *__restrict__ LSE, const T *__restrict__ dO,
                      float scale, float scale_log2, T *__restrict__ dQ, float *__restrict__ gw) {
    __shared__ float2 s_acc[NW * 32];
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t base = (size_t)blockIdx.x * N * kHeadDim;
    float *gP = gw + (size_t)blockIdx.x * 2 * N, *gS = gP + N;
    const float2 q = row_pair(Q + base, lane), g = row_pair(dO + base, lane), o = row_pair(O + base, lane);
    const float D0 = warp_sum(fmaf(g.x, o.x, g.y * o.y));
    const float lse2 = LSE[(size_t)blockIdx.x * N] * kLog2e;
    float2 dq = make_float2(0.f, 0.f);
    for (int k0 = warp * kGtRows; k0 < N; k0 += NW * kGtRows) {
        float2 kk[kGtRows], vv[kGtRows];
#pragma unroll
        for (int i = 0; i < kGtRows; ++i) {
            const int k = min(k0 + i, N - 1);
            kk[i] = row_pair(K + base + (size_t)k * kHeadDim, lane);
            vv[i] = row_pair(V + base + (size_t)k * kHeadDim, lane);
        }
#pragma unroll
        for (int i = 0; i < kGtRows; ++i) {
            const float s = warp_sum(fmaf(q.x, kk[i].x, q.y * kk[i].y));
            const float dp = warp_sum(fmaf(g.x, vv[i].x, g.y * vv[i].y));
            const bool in = k0 + i < N;
            const float P = in ? exp2f(fmaf(s, scale_log2, -lse2)) : 0.f;
            const float dS = P * (dp - D0);
            if (lane == 0 && in) {
                gP[k0 + i] = P;
                gS[k0 + i] = dS;
            }
            dq.x = fmaf(dS, kk[i].x, dq.x);
            dq.y = fmaf(dS, kk[i].y, dq.y);
        }
    }
    s_acc[warp * 32 + lane] = dq;
    __syncthreads();
    if (warp == 0) {
        float2 a = make_float2(0.f, 0.f);
        for (int w = 0; w < NW; ++w) {
            a.x += s_acc[w * 32 + lane].x;
            a.y += s_acc[w * 32 + lane].y;
        }
        store_pair(dQ + base, lane, make_float2(a.x * scale, a.y * scale));
    }
}

template <typename T, int NW>
__global__ void __launch_bounds__(NW * 32)
bwd_global_col_kernel(int N, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      const T *__restrict__ O, const float *__restrict__ LSE, const T *__restrict__ dO,
                      float scale, float scale_log2, T *__restrict__ dK, T *__restrict__ dV) {
    __shared__ float2 s_k[NW * 32], s_v[NW * 32];
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t base = (size_t)blockIdx.x * N * kHeadDim;
    const float2 k0 = row_pair(K + base, lane), v0 = row_pair(V + base, lane);
    float2 dk = make_float2(0.f, 0.f), dv = make_float2(0.f, 0.f);
    for (int j0 = warp * kGtRows; j0 < N; j0 += NW * kGtRows) {
        float2 q[kGtRows], g[kGtRows], o[kGtRows];
        float lse[kGtRows];
#pragma unroll
        for (int i = 0; i < kGtRows; ++i) {
            const int j = min(j0 + i, N - 1);
            const size_t r = base + (size_t)j * kHeadDim;
            q[i] = row_pair(Q + r, lane);
            g[i] = row_pair(dO + r, lane);
            o[i] = row_pair(O + r, lane);
            lse[i] = LSE[(size_t)blockIdx.x * N + j];
        }
#pragma unroll
        for (int i = 0; i < kGtRows; ++i) {
            const float s = warp_sum(fmaf(q[i].x, k0.x, q[i].y * k0.y));
            const float dp = warp_sum(fmaf(g[i].x, v0.x, g[i].y * v0.y));
            const float Dj = warp_sum(fmaf(g[i].x, o[i].x, g[i].y * o[i].y));
            const float P = j0 + i < N ? exp2f(fmaf(s, scale_log2, -lse[i] * kLog2e)) : 0.f;
            const float dS = P * (dp - Dj);
            dk.x = fmaf(dS, q[i].x, dk.x);
            dk.y = fmaf(dS, q[i].y, dk.y);
            dv.x = fmaf(P, g[i].x, dv.x);
            dv.y = fmaf(P, g[i].y, dv.y);
        }
    }
    s_k[warp * 32 + lane] = dk;
    s_v[warp * 32 + lane] = dv;
    __syncthreads();
    if (warp == 0) {
        float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
        for (int w = 0; w < NW; ++w) {
            a.x += s_k[w * 32 + lane].x;
            a.y += s_k[w * 32 + lane].y;
            b.x += s_v[w * 32 + lane].x;
            b.y += s_v[w * 32 + lane].y;
        }
        store_pair(dK + base, lane, make_float2(a.x * scale, a.y * scale));
        store_pair(dV + base, lane, b);
    }
}

template <typename T, int NW>
cudaError_t fwd_global(const FwdArgs &a, long bh0) {
    const TableArg &tab = *a.tab;
    const cudaError_t e = launch_kernel(fwd_global_row_kernel<T, NW>, dim3((unsigned)((long)a.B * tab.H - bh0)),
                                        dim3(NW * 32), 0, a.stream, pdl_enabled(), (int)tab.N, bh0,
                                        static_cast<const T *>(a.Q), static_cast<const T *>(a.K),
                                        static_cast<const T *>(a.V), a.scale * kLog2e, static_cast<T *>(a.O),
                                        a.LSE);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int NW>
cudaError_t bwd_global(const BwdArgs &a, bool row) {
    const TableArg &tab = *a.tab;
    const dim3 grid((unsigned)(a.B * tab.H)), block(NW * 32);
    cudaError_t e;
    if (row)
        e = launch_kernel(bwd_global_row_kernel<T, NW>, grid, block, 0, a.stream, pdl_enabled(), (int)tab.N,
                          static_cast<const T *>(a.Q), static_cast<const T *>(a.K), static_cast<const T *>(a.V),
                          static_cast<const T *>(a.O), a.LSE, static_cast<const T *>(a.dO), a.scale,
                          a.scale * kLog2e, static_cast<T *>(a.dQ), a.gw);
    else
        e = launch_kernel(bwd_global_col_kernel<T, NW>, grid, block, 0, a.stream, pdl_enabled(), (int)tab.N,
                          static_cast<const T *>(a.Q), static_cast<const T *>(a.K), static_cast<const T *>(a.V),
                          static_cast<const T *>(a.O), a.LSE, static_cast<const T *>(a.dO), a.scale,
                          a.scale * kLog2e, static_cast<T *>(a.dK), static_cast<T *>(a.dV));
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// 8 warps while a block's rows fit in a few steps, 32 beyond
constexpr int kGtShortN = 8 * kGtRows * 8;

cudaError_t launch_fwd_global_row(const FwdArgs &a, long bh0) {
    const bool wide = a.tab->N > kGtShortN;
    if (a.dtype == FIBATT_F32) return wide ? fwd_global<float, 32>(a, bh0) : fwd_global<float, 8>(a, bh0);
    return wide ? fwd_global<__nv_bfloat16, 32>(a, bh0) : fwd_global<__nv_bfloat16, 8>(a, bh0);
}

static cudaError_t bwd_global_any(const BwdArgs &a, bool row) {
    const bool wide = a.tab->N > kGtShortN;
    if (a.dtype == FIBATT_F32) return wide ? bwd_global<float, 32>(a, row) : bwd_global<float, 8>(a, row);
    return wide ? bwd_global<__nv_bfloat16, 32>(a, row) : bwd_global<__nv_bfloat16, 8>(a, row);
}

cudaError_t launch_bwd_global_row(const BwdArgs &a) { return bwd_global_any(a, true); }

cudaError_t launch_bwd_global_col(const BwdArgs &a) { return bwd_global_any(a, false); }

}  // namespace fibatt
