// Dense rows of the global first token (Fibottention README, Algorithm 2:
// row 0 and column 0 of the mask all ones), computed by the CTAs of a
// thread-block cluster, each over its slice of the keys (or queries).  Four
// lanes share a row (16 dims each), so a warp takes eight rows per step and
// each group of four lanes keeps its own partial result, merged across the
// warp's groups with shuffles, across the warps in shared memory and across
// the CTAs in CTA 0 of the cluster through distributed shared memory, in a
// fixed order (the results do not depend on scheduling).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cluster.cuh"
#include "device_common.cuh"
#include "row_math.cuh"
#include "row_run.cuh"

namespace fibatt {

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

// Shared memory of dense_row0_fwd: the warps' states and the CTA's merged
// state (read by CTA 0 of the cluster).
template <int NW>
struct DenseRowSmem {
    float m[NW], l[NW];
    float2 acc[NW][32];
    float cm, cl;
    float2 cacc[32];
};

// O_0 and LSE_0 of one head: query row 0 (at q_head) against the keys
// [kb, ke) of this CTA (key and value rows at q_head + dk and + dv, rows of
// RB bytes), an online softmax in log2 units per row group (running maximum
// raised only when a score exceeds it by more than 8), merged over the
// cluster; CTA 0 writes O0 and *LSE0.  Every thread of every CTA of the
// cluster calls it with NW = blockDim.x / 32: it holds a CTA barrier and two
// cluster barriers.  CLUSTER = false: one CTA computes the whole row (no
// cluster, warp 0 writes the result after the CTA barrier).
template <typename T, int NW, bool A32, bool CLUSTER = true>
__device__ __forceinline__ void dense_row0_fwd(const uint8_t *head, ptrdiff_t dk, ptrdiff_t dv, int kb, int ke,
                                               float scale_log2, T *O0, float *LSE0, DenseRowSmem<NW> &sm) {
    using S = Run<T, kGtG>;
    constexpr int RB = S::kRowBytes, P = S::kPairs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane % kGtG, grp = lane / kGtG;
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
    group0_store(acc, sm.acc[warp]);
    if (lane == 0) {
        sm.m[warp] = m;
        sm.l[warp] = l;
    }
    __syncthreads();
    if (warp == 0) {   // merge the warps in order, lane L taking dims 2L, 2L + 1
        float M = -INFINITY;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm.m[w]);
        float L = 0.f;
        float2 A = make_float2(0.f, 0.f);
        for (int w = 0; w < NW; ++w) {
            const float f = sm.l[w] > 0.f ? exp2f(sm.m[w] - M) : 0.f;
            L += f * sm.l[w];
            A.x += f * sm.acc[w][lane].x;
            A.y += f * sm.acc[w][lane].y;
        }
        if constexpr (!CLUSTER) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
            store_pair(O0, lane, make_float2(A.x * inv, A.y * inv));
            if (lane == 0) *LSE0 = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
            return;
        }
        sm.cacc[lane] = A;
        if (lane == 0) {
            sm.cm = M;
            sm.cl = L;
        }
    }
    if constexpr (!CLUSTER) return;
    cluster_sync();
    if (cluster_rank() == 0 && warp == 0) {   // merge the CTAs' states in rank order
        float M = -INFINITY;
        for (unsigned r = 0; r < cluster_size(); ++r) M = fmaxf(M, ld_cluster(cluster_addr(&sm.cm, r)));
        float L = 0.f;
        float2 A = make_float2(0.f, 0.f);
        for (unsigned r = 0; r < cluster_size(); ++r) {
            const float lr = ld_cluster(cluster_addr(&sm.cl, r));
            const float f = lr > 0.f ? exp2f(ld_cluster(cluster_addr(&sm.cm, r)) - M) : 0.f;
            const float2 ar = ld_cluster2(cluster_addr(&sm.cacc[lane], r));
            L += f * lr;
            A.x += f * ar.x;
            A.y += f * ar.y;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        store_pair(O0, lane, make_float2(A.x * inv, A.y * inv));
        if (lane == 0) *LSE0 = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    cluster_sync();   // no CTA leaves while CTA 0 reads its shared memory
}


}  // namespace fibatt
