// Generic Fibottention kernels: any N, any table, both dtypes.
//
// Work split: four lanes own one query (or key) row, 16 of its 64 dims each;
// dot products are reduced with two xor-shuffles.  K/V (or Q/dO) rows are
// read straight from global memory through L1/L2.  These kernels are the
// always-available path; the shape-specialised kernels in other files take
// over where they apply.
//
// Per head h and query j the attended keys are k = j + off[t] for the head's
// ascending signed offsets off[t] with 0 <= k < N (Fibottention, Sec. 3,
// support set Omega_w^{Fib(a,b)}; scores outside Omega are excluded).
#include "device_common.cuh"
#include "fibatt_internal.h"

namespace fibatt {
namespace {

constexpr int kLanes = 4;             // lanes per row
constexpr int kThreads = 256;         // threads per block
constexpr int kRowsPerBlock = kThreads / kLanes;

__device__ __forceinline__ float group_sum(float x) {
    x += __shfl_xor_sync(kFullMask, x, 1);
    x += __shfl_xor_sync(kFullMask, x, 2);
    return x;
}

// Forward: online softmax over the head's offsets (Fibottention README,
// Algorithm 3: scores -> mask -> row softmax -> weighted sum of V), scores
// kept in log2 units; O = acc / l and LSE = ln(l) + max.
template <typename T>
__global__ void __launch_bounds__(kThreads)
fwd_generic_kernel(const __grid_constant__ TableArg tab, const T *__restrict__ Q,
                   const T *__restrict__ K, const T *__restrict__ V, float scale_log2,
                   T *__restrict__ O, float *__restrict__ LSE) {
    grid_dep_wait();
    grid_dep_launch();
    const int N = tab.N;
    const int bh = blockIdx.x;
    const int h = bh % tab.H;
    const int sub = threadIdx.x % kLanes;
    const int j = blockIdx.y * kRowsPerBlock + threadIdx.x / kLanes;
    const bool valid = j < N;
    const int jc = valid ? j : N - 1;
    const size_t base = (size_t)bh * N * kHeadDim + sub * 16;

    float q[16], acc[16];
    load16(Q + base + (size_t)jc * kHeadDim, q);
#pragma unroll
    for (int d = 0; d < 16; ++d) acc[d] = 0.f;
    float m = -INFINITY, l = 0.f;

    const int t0 = tab.start[h], t1 = tab.start[h + 1];
    for (int t = t0; t < t1; ++t) {
        const int k = j + tab.off[t];
        const bool in = valid && k >= 0 && k < N;
        const int kc = in ? k : jc;
        float kv[16];
        load16(K + base + (size_t)kc * kHeadDim, kv);
        float s = 0.f;
#pragma unroll
        for (int d = 0; d < 16; ++d) s = fmaf(q[d], kv[d], s);
        s = group_sum(s) * scale_log2;
        if (in) {
            const float mn = fmaxf(m, s);
            const float alpha = exp2f(m - mn);
            const float p = exp2f(s - mn);
            l = fmaf(l, alpha, p);
            float vv[16];
            load16(V + base + (size_t)k * kHeadDim, vv);
#pragma unroll
            for (int d = 0; d < 16; ++d) acc[d] = fmaf(p, vv[d], acc[d] * alpha);
            m = mn;
        }
    }
    if (valid) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int d = 0; d < 16; ++d) acc[d] *= inv;
        store16(O + base + (size_t)j * kHeadDim, acc);
        if (sub == 0) LSE[(size_t)bh * N + j] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
}

// D_j = <dO_j, O_j>, one fp32 per row.
template <typename T>
__global__ void __launch_bounds__(kThreads)
rowdot_kernel(int64_t rows, const T *__restrict__ O, const T *__restrict__ dO,
              float *__restrict__ Dout) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t r = (int64_t)blockIdx.x * kRowsPerBlock + threadIdx.x / kLanes;
    const int sub = threadIdx.x % kLanes;
    const int64_t rc = r < rows ? r : rows - 1;
    float o[16], g[16];
    load16(O + rc * kHeadDim + sub * 16, o);
    load16(dO + rc * kHeadDim + sub * 16, g);
    float s = 0.f;
#pragma unroll
    for (int d = 0; d < 16; ++d) s = fmaf(o[d], g[d], s);
    s = group_sum(s);
    if (r < rows && sub == 0) Dout[r] = s;
}

// dQ_j = scale * sum_t dS_{j, j+off[t]} K_{j+off[t]}, query-centric.
template <typename T>
__global__ void __launch_bounds__(kThreads)
dq_generic_kernel(const __grid_constant__ TableArg tab, const T *__restrict__ Q,
                  const T *__restrict__ K, const T *__restrict__ V, const T *__restrict__ dO,
                  const float *__restrict__ LSE, const float *__restrict__ Dws, float scale,
                  float scale_log2, T *__restrict__ dQ) {
    grid_dep_wait();
    grid_dep_launch();
    const int N = tab.N;
    const int bh = blockIdx.x;
    const int h = bh % tab.H;
    const int sub = threadIdx.x % kLanes;
    const int j = blockIdx.y * kRowsPerBlock + threadIdx.x / kLanes;
    const bool valid = j < N;
    const int jc = valid ? j : N - 1;
    const size_t base = (size_t)bh * N * kHeadDim + sub * 16;
    const size_t rowj = (size_t)bh * N + jc;

    float q[16], g[16], dq[16];
    load16(Q + base + (size_t)jc * kHeadDim, q);
    load16(dO + base + (size_t)jc * kHeadDim, g);
#pragma unroll
    for (int d = 0; d < 16; ++d) dq[d] = 0.f;
    const float lse2 = LSE[rowj] * kLog2e;
    const float Dj = Dws[rowj];

    const int t0 = tab.start[h], t1 = tab.start[h + 1];
    for (int t = t0; t < t1; ++t) {
        const int k = j + tab.off[t];
        const bool in = valid && k >= 0 && k < N;
        const int kc = in ? k : jc;
        float kv[16], vv[16];
        load16(K + base + (size_t)kc * kHeadDim, kv);
        load16(V + base + (size_t)kc * kHeadDim, vv);
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < 16; ++d) {
            s = fmaf(q[d], kv[d], s);
            dp = fmaf(g[d], vv[d], dp);
        }
        s = group_sum(s);
        dp = group_sum(dp);
        if (in) {
            const float p = exp2f(fmaf(s, scale_log2, -lse2));
            const float ds = p * (dp - Dj);
#pragma unroll
            for (int d = 0; d < 16; ++d) dq[d] = fmaf(ds, kv[d], dq[d]);
        }
    }
    if (valid) {
#pragma unroll
        for (int d = 0; d < 16; ++d) dq[d] *= scale;
        store16(dQ + base + (size_t)j * kHeadDim, dq);
    }
}

// dK_k = scale * sum_t dS_{k-off[t], k} Q_{k-off[t]} and
// dV_k = sum_t P_{k-off[t], k} dO_{k-off[t]}, key-centric: the queries that
// attend key k are j = k - off[t], so no two threads write the same row.
template <typename T>
__global__ void __launch_bounds__(kThreads)
dkv_generic_kernel(const __grid_constant__ TableArg tab, const T *__restrict__ Q,
                   const T *__restrict__ K, const T *__restrict__ V, const T *__restrict__ dO,
                   const float *__restrict__ LSE, const float *__restrict__ Dws, float scale,
                   float scale_log2, T *__restrict__ dK, T *__restrict__ dV) {
    grid_dep_wait();
    grid_dep_launch();
    const int N = tab.N;
    const int bh = blockIdx.x;
    const int h = bh % tab.H;
    const int sub = threadIdx.x % kLanes;
    const int k = blockIdx.y * kRowsPerBlock + threadIdx.x / kLanes;
    const bool valid = k < N;
    const int kc0 = valid ? k : N - 1;
    const size_t base = (size_t)bh * N * kHeadDim + sub * 16;
    const size_t rbase = (size_t)bh * N;

    float kk[16], vv[16], dk[16], dv[16];
    load16(K + base + (size_t)kc0 * kHeadDim, kk);
    load16(V + base + (size_t)kc0 * kHeadDim, vv);
#pragma unroll
    for (int d = 0; d < 16; ++d) dk[d] = dv[d] = 0.f;

    const int t0 = tab.start[h], t1 = tab.start[h + 1];
    for (int t = t0; t < t1; ++t) {
        const int j = k - tab.off[t];
        const bool in = valid && j >= 0 && j < N;
        const int jc = in ? j : kc0;
        float q[16], g[16];
        load16(Q + base + (size_t)jc * kHeadDim, q);
        load16(dO + base + (size_t)jc * kHeadDim, g);
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < 16; ++d) {
            s = fmaf(q[d], kk[d], s);
            dp = fmaf(g[d], vv[d], dp);
        }
        s = group_sum(s);
        dp = group_sum(dp);
        if (in) {
            const float lse2 = LSE[rbase + jc] * kLog2e;
            const float p = exp2f(fmaf(s, scale_log2, -lse2));
            const float ds = p * (dp - Dws[rbase + jc]);
#pragma unroll
            for (int d = 0; d < 16; ++d) {
                dv[d] = fmaf(p, g[d], dv[d]);
                dk[d] = fmaf(ds, q[d], dk[d]);
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int d = 0; d < 16; ++d) dk[d] *= scale;
        store16(dK + base + (size_t)k * kHeadDim, dk);
        store16(dV + base + (size_t)k * kHeadDim, dv);
    }
}

template <typename T>
cudaError_t fwd_generic(const FwdArgs &a) {
    const TableArg &tab = *a.tab;
    dim3 grid((unsigned)(a.B * tab.H), (unsigned)((tab.N + kRowsPerBlock - 1) / kRowsPerBlock));
    const cudaError_t e = launch_kernel(fwd_generic_kernel<T>, grid, dim3(kThreads), 0, a.stream, pdl_enabled(), tab,
                                        static_cast<const T *>(a.Q), static_cast<const T *>(a.K),
                                        static_cast<const T *>(a.V), a.scale * kLog2e, static_cast<T *>(a.O), a.LSE);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
cudaError_t bwd_generic(const BwdArgs &a) {
    const TableArg &tab = *a.tab;
    const int64_t rows = (int64_t)a.B * tab.H * tab.N;
    const bool pdl = pdl_enabled();
    cudaError_t e = launch_kernel(rowdot_kernel<T>, dim3((unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock)),
                                  dim3(kThreads), 0, a.stream, pdl, rows, static_cast<const T *>(a.O),
                                  static_cast<const T *>(a.dO), a.Dws);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(a.B * tab.H), (unsigned)((tab.N + kRowsPerBlock - 1) / kRowsPerBlock));
    const float sl2 = a.scale * kLog2e;
    e = launch_kernel(dq_generic_kernel<T>, grid, dim3(kThreads), 0, a.stream, pdl, tab, static_cast<const T *>(a.Q),
                      static_cast<const T *>(a.K), static_cast<const T *>(a.V), static_cast<const T *>(a.dO),
                      static_cast<const float *>(a.LSE), static_cast<const float *>(a.Dws), a.scale, sl2,
                      static_cast<T *>(a.dQ));
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_kernel(dkv_generic_kernel<T>, grid, dim3(kThreads), 0, a.stream, pdl, tab,
                      static_cast<const T *>(a.Q), static_cast<const T *>(a.K), static_cast<const T *>(a.V),
                      static_cast<const T *>(a.dO), static_cast<const float *>(a.LSE),
                      static_cast<const float *>(a.Dws), a.scale, sl2, static_cast<T *>(a.dK),
                      static_cast<T *>(a.dV));
    count_launches(3);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_generic(const FwdArgs &a) {
    return a.dtype == FIBATT_F32 ? fwd_generic<float>(a) : fwd_generic<__nv_bfloat16>(a);
}

cudaError_t launch_bwd_generic(const BwdArgs &a) {
    return a.dtype == FIBATT_F32 ? bwd_generic<float>(a) : bwd_generic<__nv_bfloat16>(a);
}

FIBATT_DEFINE_ERROR_READER(read_error_generic, "generic.cu")

}  // namespace fibatt
