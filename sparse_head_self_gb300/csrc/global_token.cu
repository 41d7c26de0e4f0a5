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
// Each (b, h) is one thread-block cluster of C CTAs (C = 1 when there are
// enough heads to fill the GPU, up to 8 otherwise) of 8 or 16 warps: CTA r
// of the cluster takes the r-th slice of the keys (or queries).  Four lanes
// share a row (16
// dims each, 32-byte pieces), so a warp takes eight rows per step, and each
// group of four lanes keeps its own partial result.  The partials are merged
// across the warp's groups with shuffles, across the warps in the CTA's
// shared memory, and across the CTAs in CTA 0 of the cluster, which reads the
// others' shared memory (distributed shared memory) between two cluster
// barriers: the merge order is fixed, so the results do not depend on
// scheduling.
#include <algorithm>
#include <cstdlib>
#include <initializer_list>

#include "device_common.cuh"
#include "fibatt_internal.h"
#include "row_math.cuh"
#include "row_run.cuh"
#include "cluster.cuh"
#include "dense_row.cuh"

namespace fibatt {
namespace {

template <typename T, int NW, bool A32>
__global__ void __launch_bounds__(NW * 32)
fwd_global_row_kernel(int N, long bh0, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      float scale_log2, T *__restrict__ O, float *__restrict__ LSE) {
    __shared__ DenseRowSmem<NW> sm;
    grid_dep_wait();
    grid_dep_launch();
    const size_t bh = (size_t)bh0 + blockIdx.x / cluster_size();
    const uint8_t *head = reinterpret_cast<const uint8_t *>(Q) + bh * N * Run<T, kGtG>::kRowBytes;
    int kb, ke;
    cluster_slice(N, kb, ke);
    dense_row0_fwd<T, NW, A32>(head, reinterpret_cast<const uint8_t *>(K) - reinterpret_cast<const uint8_t *>(Q),
                               reinterpret_cast<const uint8_t *>(V) - reinterpret_cast<const uint8_t *>(Q), kb, ke,
                               scale_log2, O + bh * N * kHeadDim, LSE + bh * N, sm);
}

// Sum over the warps of s_acc[w][lane] (warp 0), then over the cluster's
// CTAs (CTA 0): the result is valid in warp 0 of CTA 0.
template <int NW>
__device__ __forceinline__ float2 block_cluster_sum(float2 (*s_acc)[32], float2 *c_acc) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (warp == 0) {
        float2 a = make_float2(0.f, 0.f);
        for (int w = 0; w < NW; ++w) {
            a.x += s_acc[w][lane].x;
            a.y += s_acc[w][lane].y;
        }
        c_acc[lane] = a;
    }
    cluster_sync();
    float2 r = make_float2(0.f, 0.f);
    if (cluster_rank() == 0 && warp == 0) r = cluster_sum2(&c_acc[lane]);
    return r;
}

// gw: [B*H][2][N] fp32: P_0k, then dS_0k.
template <typename T, int NW, bool A32>
__global__ void __launch_bounds__(NW * 32)
bwd_global_row_kernel(int N, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      const T *__restrict__ O, const float *__restrict__ LSE, const T *__restrict__ dO,
                      float scale, float scale_log2, T *__restrict__ dQ, float *__restrict__ gw) {
    using S = Run<T, kGtG>;
    constexpr int RB = S::kRowBytes, P = S::kPairs;
    __shared__ float2 s_acc[NW][32];
    __shared__ float2 c_acc[32];   // this CTA's partial dQ_0, read by CTA 0 of the cluster
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane % kGtG, grp = lane / kGtG;
    const size_t bh = blockIdx.x / cluster_size();
    const size_t off0 = bh * N * RB + sub * S::kBytes;
    const uint8_t *q8 = reinterpret_cast<const uint8_t *>(Q), *k8 = reinterpret_cast<const uint8_t *>(K),
                  *v8 = reinterpret_cast<const uint8_t *>(V);
    float *gP = gw + bh * 2 * N, *gS = gP + N;
    int kb, ke;
    cluster_slice(N, kb, ke);
    S q, g, o;
    load_slice<A32>(q, q8 + off0);
    load_slice<A32>(g, reinterpret_cast<const uint8_t *>(dO) + off0);
    load_slice<A32>(o, reinterpret_cast<const uint8_t *>(O) + off0);
    const float D0 = lanes_sum<kGtG>(g.dot(o));
    const float lse2 = LSE[bh * N] * kLog2e;
    float2 dq[P];
#pragma unroll
    for (int i = 0; i < P; ++i) dq[i] = make_float2(0.f, 0.f);
    for (int k0 = kb + warp * kGtRows; k0 < ke; k0 += NW * kGtRows) {
        const int k = k0 + grp;
        const bool in = k < ke;
        const size_t r = off0 + (size_t)(in ? k : kb) * RB;
        S kr, vr;
        load_slice<A32>(kr, k8 + r);
        load_slice<A32>(vr, v8 + r);
        const float s = lanes_sum<kGtG>(q.dot(kr));
        const float dp = lanes_sum<kGtG>(g.dot(vr));
        const float Pk = in ? exp2f(fmaf(s, scale_log2, -lse2)) : 0.f;
        const float dS = Pk * (dp - D0);
        if (sub == 0 && in) {
            gP[k] = Pk;
            gS[k] = dS;
        }
        kr.axpy(dS, dq);
    }
    groups_sum(dq);
    group0_store(dq, s_acc[warp]);
    const float2 a = block_cluster_sum<NW>(s_acc, c_acc);
    if (cluster_rank() == 0 && warp == 0) store_pair(dQ + bh * N * kHeadDim, lane, make_float2(a.x * scale, a.y * scale));
    cluster_sync();   // no CTA leaves while CTA 0 reads its shared memory
}

template <typename T, int NW, bool A32>
__global__ void __launch_bounds__(NW * 32)
bwd_global_col_kernel(int N, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      const T *__restrict__ O, const float *__restrict__ LSE, const T *__restrict__ dO,
                      float scale, float scale_log2, T *__restrict__ dK, T *__restrict__ dV) {
    using S = Run<T, kGtG>;
    constexpr int RB = S::kRowBytes, P = S::kPairs;
    __shared__ float2 s_k[NW][32], s_v[NW][32];
    __shared__ float2 c_k[32], c_v[32];   // this CTA's partial dK_0, dV_0, read by CTA 0 of the cluster
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane % kGtG, grp = lane / kGtG;
    const size_t bh = blockIdx.x / cluster_size();
    const size_t off0 = bh * N * RB + sub * S::kBytes;
    const uint8_t *q8 = reinterpret_cast<const uint8_t *>(Q), *g8 = reinterpret_cast<const uint8_t *>(dO),
                  *o8 = reinterpret_cast<const uint8_t *>(O);
    int qb, qe;
    cluster_slice(N, qb, qe);
    S k0r, v0r;
    load_slice<A32>(k0r, reinterpret_cast<const uint8_t *>(K) + off0);
    load_slice<A32>(v0r, reinterpret_cast<const uint8_t *>(V) + off0);
    float2 dk[P], dv[P];
#pragma unroll
    for (int i = 0; i < P; ++i) dk[i] = dv[i] = make_float2(0.f, 0.f);
    for (int j0 = qb + warp * kGtRows; j0 < qe; j0 += NW * kGtRows) {
        const int j = j0 + grp;
        const bool in = j < qe;
        const int jc = in ? j : qb;
        const size_t r = off0 + (size_t)jc * RB;
        S qr, gr, orw;
        load_slice<A32>(qr, q8 + r);
        load_slice<A32>(gr, g8 + r);
        load_slice<A32>(orw, o8 + r);
        const float lse2 = LSE[bh * N + jc] * kLog2e;
        const float s = lanes_sum<kGtG>(qr.dot(k0r));
        const float dp = lanes_sum<kGtG>(gr.dot(v0r));
        const float Dj = lanes_sum<kGtG>(gr.dot(orw));
        const float Pj = in ? exp2f(fmaf(s, scale_log2, -lse2)) : 0.f;
        qr.axpy(Pj * (dp - Dj), dk);
        gr.axpy(Pj, dv);
    }
    groups_sum(dk);
    groups_sum(dv);
    group0_store(dk, s_k[warp]);
    group0_store(dv, s_v[warp]);
    const float2 a = block_cluster_sum<NW>(s_k, c_k);
    const float2 b = block_cluster_sum<NW>(s_v, c_v);
    if (cluster_rank() == 0 && warp == 0) {
        store_pair(dK + bh * N * kHeadDim, lane, make_float2(a.x * scale, a.y * scale));
        store_pair(dV + bh * N * kHeadDim, lane, b);
    }
    cluster_sync();   // no CTA leaves while CTA 0 reads its shared memory
}

// CTAs per (b, h): enough clusters for two CTAs per SM, at most 8 (the
// portable cluster size), 1 when the heads alone fill the GPU.  (Video
// shape, 96 heads, with the global token: 4 CTAs per head fwd 51.4 us, bwd
// 147.8 us; 7: 50.7 / 157.2 us; 1: 55.2 / 159.8 us.  128 x 128 image shape,
// 32 heads: 8 CTAs 197.8 / 599.8 us against 284.2 / 934.7 us for 1.)
int gt_cluster(long heads) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    long c = (2L * sms + heads - 1) / heads;
    if (const char *e = getenv("FIBATT_GT_CLUSTER")) c = atoi(e);
    return (int)std::max(1L, std::min(8L, c));
}

// Launch `kern` with clusters of c CTAs along x (and, as launch_kernel, as a
// programmatic dependent launch when pdl is set).
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kern)(KArgs...), unsigned heads, int c, unsigned threads, cudaStream_t stream,
                           Args &&...args) {
    const ProfileLaunch prof(stream, reinterpret_cast<const void *>(kern));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(heads * (unsigned)c);
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename T, int NW, bool A32>
cudaError_t fwd_global(const FwdArgs &a, long bh0) {
    const TableArg &tab = *a.tab;
    const long heads = (long)a.B * tab.H - bh0;
    const cudaError_t e =
        launch_cluster(fwd_global_row_kernel<T, NW, A32>, (unsigned)heads, gt_cluster(heads), NW * 32, a.stream,
                       (int)tab.N, bh0, static_cast<const T *>(a.Q), static_cast<const T *>(a.K),
                       static_cast<const T *>(a.V), a.scale * kLog2e, static_cast<T *>(a.O), a.LSE);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int NW, bool A32>
cudaError_t bwd_global(const BwdArgs &a, bool row) {
    const TableArg &tab = *a.tab;
    const long heads = (long)a.B * tab.H;
    const int c = gt_cluster(heads);
    cudaError_t e;
    if (row)
        e = launch_cluster(bwd_global_row_kernel<T, NW, A32>, (unsigned)heads, c, NW * 32, a.stream, (int)tab.N,
                           static_cast<const T *>(a.Q), static_cast<const T *>(a.K), static_cast<const T *>(a.V),
                           static_cast<const T *>(a.O), a.LSE, static_cast<const T *>(a.dO), a.scale,
                           a.scale * kLog2e, static_cast<T *>(a.dQ), a.gw);
    else
        e = launch_cluster(bwd_global_col_kernel<T, NW, A32>, (unsigned)heads, c, NW * 32, a.stream, (int)tab.N,
                           static_cast<const T *>(a.Q), static_cast<const T *>(a.K), static_cast<const T *>(a.V),
                           static_cast<const T *>(a.O), a.LSE, static_cast<const T *>(a.dO), a.scale,
                           a.scale * kLog2e, static_cast<T *>(a.dK), static_cast<T *>(a.dV));
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// 8 warps per CTA unless its slice of the rows takes them more than 32
// steps, 16 beyond (larger CTAs fit fewer per SM and, at 32 warps, spill)
constexpr int kGtShortN = 8 * kGtRows * 32;

static bool gt_wide(const TableArg &tab, long heads) {
    const int c = gt_cluster(heads);
    return (tab.N + c - 1) / c > kGtShortN;
}

static bool aligned32(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) % 32 != 0) return false;
    return true;
}

template <typename T>
static cudaError_t fwd_global_any(const FwdArgs &a, long bh0) {
    const bool wide = gt_wide(*a.tab, (long)a.B * a.tab->H - bh0), a32 = aligned32({a.Q, a.K, a.V});
    if (wide) return a32 ? fwd_global<T, 16, true>(a, bh0) : fwd_global<T, 16, false>(a, bh0);
    return a32 ? fwd_global<T, 8, true>(a, bh0) : fwd_global<T, 8, false>(a, bh0);
}

cudaError_t launch_fwd_global_row(const FwdArgs &a, long bh0) {
    return a.dtype == FIBATT_F32 ? fwd_global_any<float>(a, bh0) : fwd_global_any<__nv_bfloat16>(a, bh0);
}

template <typename T>
static cudaError_t bwd_global_any(const BwdArgs &a, bool row) {
    const bool wide = gt_wide(*a.tab, (long)a.B * a.tab->H), a32 = aligned32({a.Q, a.K, a.V, a.O, a.dO});
    if (wide) return a32 ? bwd_global<T, 16, true>(a, row) : bwd_global<T, 16, false>(a, row);
    return a32 ? bwd_global<T, 8, true>(a, row) : bwd_global<T, 8, false>(a, row);
}

cudaError_t launch_bwd_global_row(const BwdArgs &a) {
    return a.dtype == FIBATT_F32 ? bwd_global_any<float>(a, true) : bwd_global_any<__nv_bfloat16>(a, true);
}

cudaError_t launch_bwd_global_col(const BwdArgs &a) {
    return a.dtype == FIBATT_F32 ? bwd_global_any<float>(a, false) : bwd_global_any<__nv_bfloat16>(a, false);
}

FIBATT_DEFINE_ERROR_READER(read_error_global_token, "global_token.cu")

}  // namespace fibatt
