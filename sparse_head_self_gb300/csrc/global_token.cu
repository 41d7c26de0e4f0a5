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

namespace fibatt {
namespace {

constexpr int kGtG = 4;                  // lanes per row
constexpr int kGtRows = 32 / kGtG;       // rows per warp step

__device__ __forceinline__ void store_pair(__nv_bfloat16 *row, int i, float2 v) {
    reinterpret_cast<unsigned int *>(row)[i] = pack_bf16x2(v.x, v.y);
}
__device__ __forceinline__ void store_pair(float *row, int i, float2 v) { reinterpret_cast<float2 *>(row)[i] = v; }

// A lane's slice of a row: 256-bit loads when every row pointer is 32-byte
// aligned (A32), else two 128-bit loads (the boundary only asks for 16).
template <bool A32, typename S>
__device__ __forceinline__ void load_slice(S &r, const uint8_t *p) {
    if constexpr (A32) {
        r.load(p);
    } else {
#pragma unroll
        for (int i = 0; i < S::kWords / 4; ++i) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p) + i);
            r.w[4 * i] = v.x;
            r.w[4 * i + 1] = v.y;
            r.w[4 * i + 2] = v.z;
            r.w[4 * i + 3] = v.w;
        }
    }
}

// Sum of acc over the warp's eight row groups (lanes with the same slice);
// every lane ends with the sum for its slice.
template <int P>
__device__ __forceinline__ void groups_sum(float2 (&acc)[P]) {
#pragma unroll
    for (int d = kGtG; d < 32; d <<= 1)
#pragma unroll
        for (int i = 0; i < P; ++i) {
            acc[i].x += __shfl_xor_sync(kFullMask, acc[i].x, d);
            acc[i].y += __shfl_xor_sync(kFullMask, acc[i].y, d);
        }
}

// Lanes 0..3 (group 0) write the warp's 64-dim result, float2 index
// sub * P + i = dims (2 (sub P + i), +1), into dst[32].
template <int P>
__device__ __forceinline__ void group0_store(const float2 (&acc)[P], float2 *dst) {
    const int lane = threadIdx.x & 31;
    if (lane < kGtG)
#pragma unroll
        for (int i = 0; i < P; ++i) dst[lane * P + i] = acc[i];
}

// ---- thread-block clusters ----------------------------------------------

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_size() {
    unsigned n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}
// Every thread of every CTA of the cluster: writes to shared memory before
// it are visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of `p` (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, unsigned rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(a)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
    return a;
}
__device__ __forceinline__ float ld_cluster(uint32_t a) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ float2 ld_cluster2(uint32_t a) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
    return v;
}

// Rows [lo, hi) of this CTA's slice of n rows.
__device__ __forceinline__ void cluster_slice(int n, int &lo, int &hi) {
    const int c = (int)cluster_size(), r = (int)cluster_rank();
    const int per = (n + c - 1) / c;
    lo = min(n, r * per);
    hi = min(n, lo + per);
}

// Sum over the cluster's CTAs of the float2 at `mine` (each CTA's partial in
// its shared memory, lane `lane`'s element), read by CTA 0 in rank order.
__device__ __forceinline__ float2 cluster_sum2(const float2 *mine) {
    float2 a = make_float2(0.f, 0.f);
    for (unsigned r = 0; r < cluster_size(); ++r) {
        const float2 v = ld_cluster2(cluster_addr(mine, r));
        a.x += v.x;
        a.y += v.y;
    }
    return a;
}

template <typename T, int NW, bool A32>
__global__ void __launch_bounds__(NW * 32)
fwd_global_row_kernel(int N, long bh0, const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                      float scale_log2, T *__restrict__ O, float *__restrict__ LSE) {
    using S = Run<T, kGtG>;
    constexpr int RB = S::kRowBytes, P = S::kPairs;
    __shared__ float s_m[NW], s_l[NW];
    __shared__ float2 s_acc[NW][32];
    __shared__ float c_m, c_l;       // this CTA's state, read by CTA 0 of the cluster
    __shared__ float2 c_acc[32];
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane % kGtG, grp = lane / kGtG;
    const size_t bh = (size_t)bh0 + blockIdx.x / cluster_size();
    const uint8_t *head = reinterpret_cast<const uint8_t *>(Q) + bh * N * RB;
    const ptrdiff_t dk = reinterpret_cast<const uint8_t *>(K) - reinterpret_cast<const uint8_t *>(Q);
    const ptrdiff_t dv = reinterpret_cast<const uint8_t *>(V) - reinterpret_cast<const uint8_t *>(Q);
    int kb, ke;
    cluster_slice(N, kb, ke);
    S q;
    load_slice<A32>(q, head + sub * S::kBytes);
    // each row group's own online softmax (log2 units, running maximum raised
    // only when a score exceeds it by more than 8)
    float m = -1.0e30f, l = 0.f;
    float2 acc[P];
#pragma unroll
    for (int i = 0; i < P; ++i) acc[i] = make_float2(0.f, 0.f);
    for (int k0 = kb + warp * kGtRows; k0 < ke; k0 += NW * kGtRows) {
        const int k = k0 + grp;
        const bool in = k < ke;
        const uint8_t *row = head + (size_t)(in ? k : kb) * RB + sub * S::kBytes;
        S kr, vr;
        load_slice<A32>(kr, row + dk);
        load_slice<A32>(vr, row + dv);
        float s = lanes_sum<kGtG>(q.dot(kr)) * scale_log2;
        s = in ? s : -INFINITY;
        if (s > m + 8.f) {
            const float a = fast_exp2(m - s);
            l *= a;
#pragma unroll
            for (int i = 0; i < P; ++i) acc[i] = mul2(acc[i], make_float2(a, a));
            m = s;
        }
        const float p = fast_exp2(s - m);
        l += p;
        vr.axpy(p, acc);
    }
    // merge the warp's row groups (every lane takes part)
#pragma unroll
    for (int d = kGtG; d < 32; d <<= 1) {
        const float mo = __shfl_xor_sync(kFullMask, m, d), lo = __shfl_xor_sync(kFullMask, l, d);
        const float M = fmaxf(m, mo);
        const float fa = fast_exp2(m - M), fb = fast_exp2(mo - M);
        l = fa * l + fb * lo;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const float2 o = make_float2(__shfl_xor_sync(kFullMask, acc[i].x, d), __shfl_xor_sync(kFullMask, acc[i].y, d));
            acc[i] = make_float2(fa * acc[i].x + fb * o.x, fa * acc[i].y + fb * o.y);
        }
        m = M;
    }
    group0_store(acc, s_acc[warp]);
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    __syncthreads();
    if (warp == 0) {   // merge the warps in order, lane L taking dims 2L, 2L + 1
        float M = -INFINITY;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w]);
        float L = 0.f;
        float2 A = make_float2(0.f, 0.f);
        for (int w = 0; w < NW; ++w) {
            const float f = s_l[w] > 0.f ? exp2f(s_m[w] - M) : 0.f;
            L += f * s_l[w];
            A.x += f * s_acc[w][lane].x;
            A.y += f * s_acc[w][lane].y;
        }
        c_acc[lane] = A;
        if (lane == 0) {
            c_m = M;
            c_l = L;
        }
    }
    cluster_sync();
    if (cluster_rank() == 0 && warp == 0) {   // merge the CTAs' states in rank order
        float M = -INFINITY;
        for (unsigned r = 0; r < cluster_size(); ++r) M = fmaxf(M, ld_cluster(cluster_addr(&c_m, r)));
        float L = 0.f;
        float2 A = make_float2(0.f, 0.f);
        for (unsigned r = 0; r < cluster_size(); ++r) {
            const float lr = ld_cluster(cluster_addr(&c_l, r));
            const float f = lr > 0.f ? exp2f(ld_cluster(cluster_addr(&c_m, r)) - M) : 0.f;
            const float2 ar = ld_cluster2(cluster_addr(&c_acc[lane], r));
            L += f * lr;
            A.x += f * ar.x;
            A.y += f * ar.y;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        store_pair(O + bh * N * kHeadDim, lane, make_float2(A.x * inv, A.y * inv));
        if (lane == 0) LSE[bh * N] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    cluster_sync();   // no CTA leaves while CTA 0 reads its shared memory
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

}  // namespace fibatt
