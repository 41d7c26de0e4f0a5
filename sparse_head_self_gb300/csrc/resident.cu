// Shared-memory-resident Fibottention kernels: persistent, warp-specialised,
// TMA-fed.
//
// Work unit: (batch b, head h, query chunk [q0, q1)).  Because every offset
// of a head is a fixed diagonal, the keys a chunk attends form the contiguous
// row window [q0 + min_off, q1 + max_off) clipped to [0, N) (Fibottention
// Sec. 3: |j - k| in Fib(a,b), |j - k| <= w), so one unit is three contiguous
// row ranges: the chunk's Q rows and the K and V windows.
//
// One CTA per SM.  Warp 0 is the producer: one lane issues the three bulk
// copies (TMA, cp.async.bulk) of each unit into a ring of shared-memory
// stages, each stage guarded by a "full" mbarrier (byte count) and an "empty"
// mbarrier (released by the consumer warps).  The other warps form consumer
// groups; group g computes units g, g + groups, ... of this CTA, so loads of
// later units overlap the arithmetic of earlier ones and HBM stays busy.
// Every mbarrier wait is bounded in time (tma_common.cuh).
//
// Arithmetic (two lanes per query row, 32 dims each):
//   s   = scale * <q_j, k_{j+d}>  -- bf16 x bf16 products with the
//         mixed-precision fma.rn.f32.bf16 (exact products, fp32 sums),
//         reduced over the lane pair with one xor-shuffle;
//   online softmax in log2 units whose running maximum is only raised when
//         a score exceeds it by more than 8 (then acc and l are rescaled),
//         so the rescale is rare and p = 2^(s - m) <= 2^8 never overflows;
//   acc += p * v_{j+d} with packed f32x2 fmas;
//   O = acc / l (RNE to the I/O dtype), LSE = ln 2 * (m + log2 l).
// Edges are branch-free: per round, two warp ballots drop the offsets that
// reach no key for any row of the round; the rest read a clamped row and
// mask the score of an out-of-range key to -inf.
//
// The flat kernels further down run the same round code on rows read from
// global memory, for heads whose key windows do not fit in shared memory.
#include <algorithm>
#include <cstdlib>
#include <initializer_list>
#include <type_traits>

#include "fibatt_internal.h"
#include "tma_common.cuh"

namespace fibatt {
namespace {

constexpr int kMaxStages = 4;

struct PipeParams {
    const void *Q, *K, *V;
    void *O;
    float *LSE;
    float scale_log2;
    int qsplit;        // query chunks per (b, h)
    int chunk;         // queries per chunk (multiple of 16)
    int kv_cap;        // rows reserved for each of the K and V windows
    int n_units;       // B * H * qsplit
    int stages;        // ring depth
    int groups;        // consumer groups
    int gwarps;        // warps per consumer group
    uint32_t stage_bytes;
    int prefetch;      // units beyond the ring warmed in L2
    // The last wave: units [n_keep, n_keep + (qsplit units left) * qsub) are
    // the regular units n_keep, n_keep + 1, ... cut into qsub sub-units of
    // sub_rows query rows, so the wave that does not fill every CTA is
    // spread thin instead of landing whole on a few CTAs.
    int n_keep;
    int qsub;
    int sub_rows;
    int early_prefetch;   // L2-prefetch the first units before the grid-dependency wait
    int snake;            // odd full waves take the CTAs in reverse order
    int fuse_row0;        // global first token: row 0 of each whole-head unit computed here
};

// Row 0 of a whole-head unit with the global first token: query 0 attends
// every key.  Consumer warp wg of the group takes batches of 16 keys
// (keys wg 16 + i 16 gwarps ...): two lanes per key score it (half the
// dims each, 16-byte chunks in an order rotated by key and half, so a
// quarter warp hits eight distinct bank groups), the batch enters the
// warp's running softmax state, and every lane then adds the batch's
// weighted value rows for its two dims.  The warp leaves its state in the
// stage's partial slot (pacc: gwarps x 32 float2, pm and pl: gwarps floats)
// and counts itself in; the warp that arrives last merges the states, writes
// O_0 and LSE_0 and resets the count.  No warp waits for another.  The slot
// is the stage's own: it is used again only by the stage's next unit, whose
// data arrives after every consumer warp, the merging one included, has
// released the stage.
template <typename T>
__device__ __forceinline__ void fused_row0(const uint8_t *sQ, const uint8_t *sK, ptrdiff_t vdelta, int N, int wg,
                                           int gwarps, float sl2, float2 *pacc, float *pm, float *pl, int *count,
                                           T *O0, float *LSE0) {
    constexpr bool F32 = std::is_same<T, float>::value;
    constexpr int RB = (int)sizeof(T) * kHeadDim;
    constexpr int HC = RB / 32;   // 16-byte chunks in half a row
    const int lane = threadIdx.x & 31, kl = lane >> 1, half = lane & 1;
    auto vpair = [&](int k) {
        const uint8_t *row = sK + vdelta + (size_t)k * RB;
        if constexpr (F32) {
            return reinterpret_cast<const float2 *>(row)[lane];
        } else {
            const uint32_t w = reinterpret_cast<const uint32_t *>(row)[lane];
            return make_float2(bf16_lo(w), bf16_hi(w));
        }
    };
    float m = -INFINITY, l = 0.f;
    float2 acc = make_float2(0.f, 0.f);
    for (int kb = wg * 16; kb < N; kb += 16 * gwarps) {
        const int k = kb + kl;
        float xa = 0.f, xb = 0.f;
        if (k < N) {
            const uint8_t *kr = sK + (size_t)k * RB;
#pragma unroll
            for (int c = 0; c < HC; ++c) {
                const int cc = half * HC + ((c + kl + 4 * half) & (HC - 1));
                const uint4 qv = *reinterpret_cast<const uint4 *>(sQ + cc * 16);
                const uint4 kv = *reinterpret_cast<const uint4 *>(kr + cc * 16);
                if constexpr (F32) {
                    xa = fmaf(__uint_as_float(qv.x), __uint_as_float(kv.x), xa);
                    xb = fmaf(__uint_as_float(qv.y), __uint_as_float(kv.y), xb);
                    xa = fmaf(__uint_as_float(qv.z), __uint_as_float(kv.z), xa);
                    xb = fmaf(__uint_as_float(qv.w), __uint_as_float(kv.w), xb);
                } else {   // mixed-precision FMAs on the packed pairs: no unpacking
                    xa = dot2_bf16(qv.x, kv.x, xa);
                    xb = dot2_bf16(qv.y, kv.y, xb);
                    xa = dot2_bf16(qv.z, kv.z, xa);
                    xb = dot2_bf16(qv.w, kv.w, xb);
                }
            }
        }
        float x = xa + xb;
        x += __shfl_xor_sync(kFullMask, x, 1);
        x = k < N ? x * sl2 : -INFINITY;
        float mb = x;
#pragma unroll
        for (int o = 2; o <= 16; o <<= 1) mb = fmaxf(mb, __shfl_xor_sync(kFullMask, mb, o));
        const float mn = fmaxf(m, mb);   // finite: key kb < N is in the batch
        const float f = fast_exp2(m - mn);
        const float pw = fast_exp2(x - mn);
        float ps = pw;
#pragma unroll
        for (int o = 2; o <= 16; o <<= 1) ps += __shfl_xor_sync(kFullMask, ps, o);
        l = fmaf(l, f, ps);
        acc.x *= f;
        acc.y *= f;
        m = mn;
        // keys past N have weight 0 and read row N - 1 (finite data)
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const float pt = __shfl_sync(kFullMask, pw, 2 * t);
            const float2 vv = vpair(min(kb + t, N - 1));
            acc.x = fmaf(pt, vv.x, acc.x);
            acc.y = fmaf(pt, vv.y, acc.y);
        }
    }
    if (lane == 0) {
        pm[wg] = m;
        pl[wg] = l;
    }
    pacc[wg * 32 + lane] = acc;
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(count, 1) == gwarps - 1;
    }
    if (!__shfl_sync(kFullMask, last, 0)) return;
    __threadfence_block();
    float M = -INFINITY;
#pragma unroll 4
    for (int w = 0; w < gwarps; ++w) M = fmaxf(M, pm[w]);
    float L = 0.f;
    float2 A = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int w = 0; w < gwarps; ++w) {
        const float fw = pl[w] > 0.f ? fast_exp2(pm[w] - M) : 0.f;
        L = fmaf(fw, pl[w], L);
        A.x = fmaf(fw, pacc[w * 32 + lane].x, A.x);
        A.y = fmaf(fw, pacc[w * 32 + lane].y, A.y);
    }
    const float inv = L > 0.f ? __frcp_rn(L) : 0.f;
    if constexpr (F32) {
        reinterpret_cast<float2 *>(O0)[lane] = make_float2(A.x * inv, A.y * inv);
    } else {
        reinterpret_cast<uint32_t *>(O0)[lane] = pack_bf16x2(A.x * inv, A.y * inv);
    }
    if (lane == 0) {
        *LSE0 = L > 0.f ? (M + fast_log2(L)) * kLn2 : -INFINITY;
        *count = 0;
    }
}

// Unit of this CTA's slot k (-1 past the end).  Slot k of CTA c is wave k,
// position c; with `snake`, odd full waves run the positions backwards, so a
// CTA alternates between the two ends of each wave (query chunks and heads
// otherwise repeat with the wave, since the grid and the units per batch
// element share factors).
__device__ __forceinline__ int fwd_slot_unit(const PipeParams &p, int k) {
    const int c = (int)blockIdx.x, g = (int)gridDim.x;
    const long L = (long)k * g + c;
    if (L >= p.n_units) return -1;
    if (p.snake && (k & 1) && (long)(k + 1) * g <= p.n_keep) return k * g + (g - 1 - c);
    return (int)L;
}

struct Unit {
    int bh, h, q0, q1, t0, t1, lo, nrows;
};

// Geometry of unit u; start and off are the table's head starts and offsets
// (the kernel parameter's, or a shared-memory copy of them).
__device__ __forceinline__ Unit unit_geometry(const TableArg &tab, const int *start, const int *off,
                                              const PipeParams &p, int u) {
    Unit g;
    if (u < p.n_keep) {
        g.bh = u / p.qsplit;
        g.q0 = (u % p.qsplit) * p.chunk;
        g.q1 = min(tab.N, g.q0 + p.chunk);
    } else {
        const int s = u - p.n_keep, ur = p.n_keep + s / p.qsub;
        g.bh = ur / p.qsplit;
        const int cb = (ur % p.qsplit) * p.chunk, ce = min(tab.N, cb + p.chunk);
        g.q0 = min(ce, cb + (s % p.qsub) * p.sub_rows);
        g.q1 = min(ce, g.q0 + p.sub_rows);
    }
    g.h = g.bh % tab.H;
    g.t0 = start[g.h];
    g.t1 = start[g.h + 1];
    g.lo = 0;
    g.nrows = 0;
    if (g.t1 > g.t0 && g.q1 > g.q0) {
        g.lo = max(0, g.q0 + off[g.t0]);
        g.nrows = max(0, min(tab.N, g.q1 + off[g.t1 - 1]) - g.lo);
    }
    // with the dense row 0 fused (whole-head units), the unit or last-wave
    // piece that holds query 0 stages every key row for it
    if (p.fuse_row0 && g.q0 == 0 && g.q1 > 0) {
        g.lo = 0;
        g.nrows = tab.N;
    }
    return g;
}

// Running state of one query row: acc = sum of weight x value row, m the
// running maximum (log2 units), l the sum of the weights (for the LSE) and
// lt the sum of the weights as they entered acc (rounded to bf16 when the
// P.V update takes bf16 weights), which normalises O.
template <int G>
struct SoftmaxState {
    float2 acc[32 / G];
    float m, l, lt;
};

template <int G>
__device__ __forceinline__ void softmax_raise(SoftmaxState<G> &st, float s) {
    if (s > st.m + 8.f) {
        const float a = fast_exp2(st.m - s);
        st.l *= a;
        st.lt *= a;
#pragma unroll
        for (int i = 0; i < 32 / G; ++i) st.acc[i] = mul2(st.acc[i], make_float2(a, a));
        st.m = s;
    }
}

// Per-lane geometry of a row slice: byte offsets of the lane's chunks.
template <typename T, int G>
struct LaneGeom {
    using S = Slice<T, G>;
    int c[S::kChunks];
    __device__ __forceinline__ LaneGeom() {
        const int lane = threadIdx.x & 31;
        const int sub = lane % G, pos = (lane / G) % (8 / G);
#pragma unroll
        for (int i = 0; i < S::kChunks; ++i) c[i] = 16 * S::chunk(sub, pos, i);
    }
};

// Running-max start: finite, so a prefix of masked scores (-inf) gives
// 2^(-inf - m) = 0 instead of a NaN, and any real score raises it.
constexpr float kMaxInit = -1.0e30f;

// Weight p of value row vr into the state.  W16 (bf16 rows): p is rounded
// to bf16 for the row update, as bf16 attention kernels round P before their
// P.V product, which makes the update one mixed-precision FMA per element;
// O is normalised by the sum of the rounded weights, so it stays a convex
// combination of the value rows and the largest weight's rounding cancels.
template <typename T, int G, bool W16>
__device__ __forceinline__ void softmax_accumulate(SoftmaxState<G> &st, const Slice<T, G> &vr, float p) {
    st.l += p;
    if constexpr (W16 && std::is_same<T, __nv_bfloat16>::value) {
        const uint32_t p2 = bf16x2_splat(p);
        st.lt += __uint_as_float(p2 << 16);
        vr.axpy_p2(p2, st.acc);
    } else {
        vr.axpy(p, st.acc);   // lt is l here (softmax_norm reads l)
    }
}

// The sum that normalises O (see softmax_accumulate).
template <typename T, int G, bool W16>
__device__ __forceinline__ float softmax_norm(const SoftmaxState<G> &st) {
    if constexpr (W16 && std::is_same<T, __nv_bfloat16>::value) return st.lt;
    else return st.l;
}

// One pass over offsets [tb, te) (read from the shared-memory copy `off`) for
// query row j, branch-free: the key row is clamped into the staged window
// [lo, lo + nrows) and a score whose key lies outside [0, N) (or whose row is
// padding) becomes -inf, so its weight is exactly 0 and the raise never
// triggers.  Two offsets per step so their shared-memory loads overlap.
// W16: bf16 weights in the P.V update (softmax_accumulate; the
// shared-memory kernels, where it saves issue slots), else fp32 weights.
template <typename T, int G, int UNROLL, bool W16>
__device__ __forceinline__ void fwd_offsets(const int *off, int N, int tb, int te, int j, bool valid, int lo,
                                            int nrows, const uint8_t *sK, ptrdiff_t vdelta, const Slice<T, G> &q,
                                            const LaneGeom<T, G> &lg, float sl2, SoftmaxState<G> &st) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    const int kmin = max(lo, 0), kmax = min(lo + nrows, N) - 1;   // keys present in the window
    int t = tb;
    if (UNROLL == 2) {
        for (; t + 1 < te; t += 2) {
            const int k0 = j + off[t], k1 = j + off[t + 1];
            const bool in0 = valid && k0 >= 0 && k0 < N, in1 = valid && k1 >= 0 && k1 < N;
            const uint8_t *a0 = sK + (ptrdiff_t)(min(max(k0, kmin), kmax) - lo) * RB;
            const uint8_t *a1 = sK + (ptrdiff_t)(min(max(k1, kmin), kmax) - lo) * RB;
            S k0r, k1r;
            k0r.load(a0, lg.c);
            k1r.load(a1, lg.c);
            float s0 = group_sum<G>(q.dot(k0r)) * sl2;
            float s1 = group_sum<G>(q.dot(k1r)) * sl2;
            s0 = in0 ? s0 : -INFINITY;
            s1 = in1 ? s1 : -INFINITY;
            softmax_raise(st, fmaxf(s0, s1));
            const float p0 = fast_exp2(s0 - st.m), p1 = fast_exp2(s1 - st.m);
            k0r.load(a0 + vdelta, lg.c);
            k1r.load(a1 + vdelta, lg.c);
            softmax_accumulate<T, G, W16>(st, k0r, p0);
            softmax_accumulate<T, G, W16>(st, k1r, p1);
        }
    }
    for (; t < te; ++t) {
        const int k = j + off[t];
        const bool in = valid && k >= 0 && k < N;
        const uint8_t *a = sK + (ptrdiff_t)(min(max(k, kmin), kmax) - lo) * RB;
        S kv;
        kv.load(a, lg.c);
        float s = group_sum<G>(q.dot(kv)) * sl2;
        s = in ? s : -INFINITY;
        softmax_raise(st, s);
        const float pr = fast_exp2(s - st.m);
        kv.load(a + vdelta, lg.c);
        softmax_accumulate<T, G, W16>(st, kv, pr);
    }
}

// Offsets of a head (ascending off[t0..t1)) that reach a key in [0, N) for
// at least one row of the round [jfirst, jlast]: [tb, te).  Warp-collective.
__device__ __forceinline__ void round_range(const int *off, int N, int t0, int t1, int jfirst, int jlast, int &tb,
                                            int &te) {
    const int lane = threadIdx.x & 31;
    int below = 0, above = 0;
    for (int base = t0; base < t1; base += 32) {
        const int t = base + lane;
        const bool e = t < t1;
        const int o = e ? off[t] : 0;
        below += __popc(__ballot_sync(kFullMask, e && jlast + o < 0));
        above += __popc(__ballot_sync(kFullMask, e && jfirst + o >= N));
    }
    tb = t0 + below;
    te = max(tb, t1 - above);
}

// Global first token: bit i set when the band of row first + i (i < nrows
// <= 32) reaches position 0, i.e. offset -(first + i) is in off[t0, t1) (the
// tables are symmetric, so the same bit says whether +(first + i) is).  The
// warp scans the head's table 32 entries at a time; call it warp-uniformly.
__device__ __forceinline__ unsigned band_reaches_zero(const int *off, int t0, int t1, int first, int nrows) {
    const int lane = threadIdx.x & 31;
    unsigned hit = 0;
    for (int t = t0; t < t1; t += 32) {
        const int i = t + lane < t1 ? -off[t + lane] - first : -1;
        hit |= __reduce_or_sync(kFullMask, i >= 0 && i < nrows ? 1u << i : 0u);
    }
    return hit;
}

// Round r of a unit: query rows [q0 + r R, q0 + r R + R) with R = 32 / G.
template <typename T, int G, int UNROLL, bool GT, bool W16>
__device__ __forceinline__ void fwd_round(const TableArg &tab, const int *off, const PipeParams &p, const Unit &g,
                                          const uint8_t *sQ, const uint8_t *sK, ptrdiff_t vdelta, int r,
                                          const LaneGeom<T, G> &lg, const uint8_t *sK0 = nullptr,
                                          const uint8_t *sV0 = nullptr) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    constexpr int R = 32 / G;
    const int N = tab.N;
    const int lane = threadIdx.x & 31;
    const int nq = g.q1 - g.q0;
    if (r * R >= nq) return;
    const size_t row0 = (size_t)g.bh * N;
    T *gO = static_cast<T *>(p.O) + row0 * kHeadDim;
    const int jl = r * R + lane / G;
    const bool valid = jl < nq;
    const int j = g.q0 + (valid ? jl : nq - 1);
    const int jfirst = g.q0 + r * R;
    const int jlast = g.q0 + min(nq, r * R + R) - 1;
    int tb = g.t0, te = g.t0;
    if (g.nrows) round_range(off, N, g.t0, g.t1, jfirst, jlast, tb, te);

    S q;
    q.load(sQ + (size_t)(j - g.q0) * RB, lg.c);
    SoftmaxState<G> st;
#pragma unroll
    for (int i = 0; i < 32 / G; ++i) st.acc[i] = make_float2(0.f, 0.f);
    st.m = kMaxInit;
    st.l = 0.f;
    st.lt = 0.f;
    fwd_offsets<T, G, UNROLL, W16>(off, N, tb, te, j, valid, g.lo, g.nrows, sK, vdelta, q, lg, p.scale_log2, st);
    if constexpr (GT) {
        // global first token: key 0 for every query row j >= 1 whose band
        // misses it
        const unsigned band0 = band_reaches_zero(off, g.t0, g.t1, jfirst, jlast - jfirst + 1);
        const bool need = valid && j >= 1 && !((band0 >> (j - jfirst)) & 1u);
        S kr;
        kr.load(sK0, lg.c);
        float s0 = group_sum<G>(q.dot(kr)) * p.scale_log2;
        s0 = need ? s0 : -INFINITY;
        softmax_raise(st, s0);
        const float pr = fast_exp2(s0 - st.m);
        kr.load(sV0, lg.c);
        softmax_accumulate<T, G, W16>(st, kr, pr);
    }
    if (valid && !(GT && p.fuse_row0 && j == 0)) {   // fused: row 0 is written by fused_row0
        const float ln = softmax_norm<T, G, W16>(st);
        const float inv = ln > 0.f ? __frcp_rn(ln) : 0.f;
#pragma unroll
        for (int i = 0; i < 32 / G; ++i) st.acc[i] = mul2(st.acc[i], make_float2(inv, inv));
        S::store(gO + (size_t)j * kHeadDim, lg.c, st.acc);
        if (lane % G == 0) p.LSE[row0 + j] = st.l > 0.f ? (st.m + fast_log2(st.l)) * kLn2 : -INFINITY;
    }
}

// L2 prefetch of unit u's three row ranges (a hint: nothing waits on it).
template <typename T>
__device__ __forceinline__ void prefetch_unit(const TableArg &tab, const PipeParams &p, int u) {
    constexpr int RB = sizeof(T) * kHeadDim;
    const Unit g = unit_geometry(tab, tab.start, tab.off, p, u);
    const size_t row0 = (size_t)g.bh * tab.N;
    if (g.q1 > g.q0)
        bulk_prefetch_l2(static_cast<const T *>(p.Q) + (row0 + g.q0) * kHeadDim, (uint32_t)(g.q1 - g.q0) * RB);
    if (g.nrows) {
        bulk_prefetch_l2(static_cast<const T *>(p.K) + (row0 + g.lo) * kHeadDim, (uint32_t)g.nrows * RB);
        bulk_prefetch_l2(static_cast<const T *>(p.V) + (row0 + g.lo) * kHeadDim, (uint32_t)g.nrows * RB);
    }
}

template <typename T, int G, int UNROLL, int MAXT, bool GT = false>
__global__ void __launch_bounds__(MAXT, 1)
fwd_pipe_kernel(const __grid_constant__ TableArg tab, const PipeParams p) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    constexpr int R = 32 / G;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
    __shared__ int s_off[kMaxEntries];
    __shared__ int s_row0_count[kMaxStages];   // fused row 0: warps done with the stage's unit
    __shared__ Unit s_unit[kMaxStages];        // geometry of the stage's unit, written by the producer
    __shared__ int s_start[kMaxHeads + 1];     // the heads' table starts
    __shared__ int s_abort;                    // a bounded wait of this CTA gave up (mbar_wait)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0 && (p.early_prefetch & 1)) {
        // Warm L2 with the first units' rows while the previous kernel drains.
        // A prefetch only moves lines into L2, the point of coherence: the
        // copies issued after the grid-dependency wait below still read what
        // the previous kernel wrote.
        for (int i = 0; i < ((p.early_prefetch & 2) ? 1 : p.stages); ++i) {
            const int u = fwd_slot_unit(p, i);
            if (u >= 0) prefetch_unit<T>(tab, p, u);
        }
    }
    for (int t = threadIdx.x; t < tab.start[tab.H]; t += blockDim.x) s_off[t] = tab.off[t];
    for (int t = threadIdx.x; t <= tab.H; t += blockDim.x) s_start[t] = tab.start[t];
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], p.gwarps);
            s_row0_count[s] = 0;
        }
        s_abort = 0;
    }
    __syncthreads();
    // touch no global memory before the previous kernel has completed; then
    // let the next kernel of the stream take SMs as this grid retires (only
    // after the wait, so a dependent never runs ahead of our prerequisites)
    grid_dep_wait();
    grid_dep_launch();

    const size_t q_off = 0, k_off = (size_t)p.chunk * RB, v_off = k_off + (size_t)p.kv_cap * RB;
    const size_t g0_off = v_off + (size_t)p.kv_cap * RB;   // K and V row 0 (global first token)
    if (warp == 0) {
        // producer: one lane streams every unit of this CTA into the ring and
        // keeps the next `prefetch` units warming in L2
        if (lane != 0) return;
        int issued = 0;   // units whose copies this lane issued (stage i % stages, use i / stages)
        for (int i = 0;; ++i) {
            const int u = fwd_slot_unit(p, i);
            if (u < 0) break;
            const int s = i % p.stages;
            if (i == 0)
                for (int d = p.stages; d < p.stages + p.prefetch; ++d) {
                    const int un = fwd_slot_unit(p, d);
                    if (un >= 0) prefetch_unit<T>(tab, p, un);
                }
            const Unit g = unit_geometry(tab, s_start, s_off, p, u);   // before the wait: off the critical path
            if (i >= p.stages && !mbar_wait(&empty_bar[s], ((i / p.stages) - 1) & 1, &s_abort)) break;
            // the second unit's copies wait for the first unit's rows to land, so
            // that every CTA's first unit has the DRAM to itself at the start
            if (i == 1 && (p.early_prefetch & 2) && !mbar_wait(&full_bar[0], 0, &s_abort)) break;
            uint8_t *st = smem + (size_t)s * p.stage_bytes;
            const size_t row0 = (size_t)g.bh * tab.N;
            uint32_t qb = (uint32_t)(g.q1 - g.q0) * RB, kvb = (uint32_t)g.nrows * RB;
            if (!FIBATT_CHECKED(g.q1 - g.q0 <= p.chunk && g.nrows <= p.kv_cap)) qb = kvb = 0;   // the stage's room
            // the consumers read the geometry after the full phase, which
            // this arrive (a release) belongs to
            s_unit[s] = g;
            mbar_expect_tx(&full_bar[s], qb + 2 * kvb + (GT ? 2u * RB : 0u));
            if (qb)   // a last-wave piece past the end of its chunk has no rows
                bulk_g2s(st + q_off, static_cast<const T *>(p.Q) + (row0 + g.q0) * kHeadDim, qb, &full_bar[s]);
            if (kvb) {
                bulk_g2s(st + k_off, static_cast<const T *>(p.K) + (row0 + g.lo) * kHeadDim, kvb, &full_bar[s]);
                bulk_g2s(st + v_off, static_cast<const T *>(p.V) + (row0 + g.lo) * kHeadDim, kvb, &full_bar[s]);
            }
            if (GT) {   // key and value row 0, for the global first token
                bulk_g2s(st + g0_off, static_cast<const T *>(p.K) + row0 * kHeadDim, RB, &full_bar[s]);
                bulk_g2s(st + g0_off + RB, static_cast<const T *>(p.V) + row0 * kHeadDim, RB, &full_bar[s]);
            }
            issued = i + 1;
            if (i >= 1 && p.prefetch > 0) {
                const int un = fwd_slot_unit(p, i + p.stages + p.prefetch - 1);
                if (un >= 0) prefetch_unit<T>(tab, p, un);
            }
        }
        // leave only once the last copies into every stage have landed
        for (int s = 0; s < p.stages && s < issued; ++s)
            mbar_drain(&full_bar[s], ((issued - 1 - s) / p.stages) & 1);
        return;
    }
    // Consumers.  Use k of stage s is the CTA's slot i = s + k * stages (its
    // unit from fwd_slot_unit), taken by group i % groups.  An mbarrier
    // parity wait cannot tell a phase that completed from one two phases
    // ahead, so before waiting for use k to be full the group waits for use
    // k - 1 to be released.  That release wait is itself unambiguous when use
    // k - 2 belonged to this group -- true when groups <= 2, or when stages is
    // a multiple of groups (each stage then always serves the same group) --
    // the plan allows nothing else.
    const int cw = warp - 1;
    const int grp = cw / p.gwarps, wg = cw % p.gwarps;
    if (grp >= p.groups) return;
    const LaneGeom<T, G> lg;
    const int rpu = p.chunk / R;
    const int rot_step = rpu % p.gwarps;
    int rot = 0;
    for (int i = grp;; i += p.groups) {
        const int u = fwd_slot_unit(p, i);
        if (u < 0) break;
        const int s = i % p.stages, k = i / p.stages;
        // the consumers meet at no named barrier, so a group that gave up may leave
        if (k >= 1 && !mbar_wait(&empty_bar[s], (k - 1) & 1, &s_abort)) return;
        if (!mbar_wait(&full_bar[s], k & 1, &s_abort)) return;
        const Unit g = s_unit[s];
        const uint8_t *st = smem + (size_t)s * p.stage_bytes;
        if constexpr (GT) {
            if (p.fuse_row0 && g.q0 == 0 && g.q1 > 0 && g.lo == 0 && g.nrows == tab.N) {
                // stage s's partial slot, after the stages: gwarps x 32
                // float2 partial accumulators, then gwarps maxima and sums
                const size_t row0 = (size_t)g.bh * tab.N;
                float2 *pacc = reinterpret_cast<float2 *>(smem + (size_t)p.stages * p.stage_bytes) +
                               (size_t)s * p.gwarps * 33;
                float *pm = reinterpret_cast<float *>(pacc + 32 * p.gwarps);
                fused_row0<T>(st + q_off, st + k_off, (ptrdiff_t)(v_off - k_off), tab.N, wg, p.gwarps,
                              p.scale_log2, pacc, pm, pm + p.gwarps, &s_row0_count[s],
                              static_cast<T *>(p.O) + row0 * kHeadDim, p.LSE + row0);
            }
        }
        // round r of the group's k-th unit goes to warp (r + k rpu) mod gwarps:
        // with fewer warps than rounds the extra rounds circulate over the
        // warps from unit to unit (rot = k rpu mod gwarps, kept incrementally)
        const int r0 = wg >= rot ? wg - rot : wg - rot + p.gwarps;
        rot += rot_step;
        if (rot >= p.gwarps) rot -= p.gwarps;
        for (int r = r0; r < rpu; r += p.gwarps)
            fwd_round<T, G, UNROLL, GT, true>(tab, s_off, p, g, st + q_off, st + k_off, (ptrdiff_t)(v_off - k_off), r, lg,
                                    st + g0_off, st + g0_off + RB);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
}

// ------------------------------------------------------------ flat forward
//
// The same rounds with nothing staged: the query, key and value rows are read
// from global memory (L1/L2) at the addresses the round would have used in
// shared memory.  For heads whose key windows do not fit in shared memory
// (long sequences with wide windows).  Block: kFlatWarps warps of one
// (b, h); warp w of block y takes round y * kFlatWarps + w.
constexpr int kFlatWarps = 4;   // 128-thread blocks measured fastest (4 to 32 warps tried)

template <typename T, int G, int UNROLL, int W = kFlatWarps, bool GT = false>
__global__ void __launch_bounds__(W * 32)
fwd_flat_kernel(const __grid_constant__ TableArg tab, const PipeParams p) {
    __shared__ int s_off[kMaxEntries];
    constexpr int RB = Slice<T, G>::kRowBytes;
    const int N = tab.N;
    const int bh = blockIdx.x, h = bh % tab.H;
    const int t0 = tab.start[h], t1 = tab.start[h + 1];
    for (int t = t0 + (int)threadIdx.x; t < t1; t += blockDim.x) s_off[t] = tab.off[t];
    __syncthreads();
    grid_dep_wait();
    grid_dep_launch();
    Unit g;
    g.bh = bh;
    g.h = h;
    g.q0 = 0;
    g.q1 = N;
    g.t0 = t0;
    g.t1 = t1;
    g.lo = 0;
    g.nrows = t1 > t0 ? N : 0;
    const size_t row0 = (size_t)bh * N * RB;
    const uint8_t *gQ = static_cast<const uint8_t *>(p.Q) + row0;
    const uint8_t *gK = static_cast<const uint8_t *>(p.K) + row0;
    const ptrdiff_t vdelta = static_cast<const uint8_t *>(p.V) - static_cast<const uint8_t *>(p.K);
    const LaneGeom<T, G> lg;
    const int r = blockIdx.y * W + (threadIdx.x >> 5);
    fwd_round<T, G, UNROLL, GT, false>(tab, s_off, p, g, gQ, gK, vdelta, r, lg, gK, gK + vdelta);
}

// ---------------------------------------------------------------- backward
//
// Work unit: one (batch b, head h), whole sequence resident.  A stage holds
// the head's Q, K, V and dO rows (four bulk copies); the producer also
// prefetches the next unit's O rows and LSE into L2.  All consumer warps share
// a unit in two phases separated by a named barrier:
//   A (query-centric, row j): s = <q_j, k>, dP = <dO_j, v> for k = j + off[t];
//     P = exp(s - LSE_j), dS = P (dP - D_j) with D_j = <dO_j, O_j>;
//     dQ_j = scale * sum dS k; P and dS go to a shared scratch [t][j].
//   B (key-centric, row k): the tables are symmetric (built from distances),
//     so the queries attending key k are j = k + off[t'] over the same table,
//     and the pair's forward offset index is the mirror t0 + t1 - 1 - t';
//     dK_k = scale * sum dS q_j, dV_k = sum P dO_j -- each key row owned by
//     one lane group, no atomics.

// <O_j, dO_j> over the full row: O from global memory, dO from shared
// memory; the lane walks the 16-byte chunks starting at its own index so a
// warp's lanes (one row each) touch different bank groups.
__device__ __forceinline__ float row_dot_global_shared(const __nv_bfloat16 *o, const uint8_t *g, int lane) {
    const uint4 *o4 = reinterpret_cast<const uint4 *>(o);
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int cc = (c + lane) & 7;
        const uint4 x = __ldg(o4 + cc);
        const uint4 y = *reinterpret_cast<const uint4 *>(g + 16 * cc);
        a = dot2_bf16(x.x, y.x, a);
        b = dot2_bf16(x.y, y.y, b);
        a = dot2_bf16(x.z, y.z, a);
        b = dot2_bf16(x.w, y.w, b);
    }
    return a + b;
}

__device__ __forceinline__ float row_dot_global_shared(const float *o, const uint8_t *g, int lane) {
    const float4 *o4 = reinterpret_cast<const float4 *>(o);
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const int cc = (c + lane) & 15;
        const float4 x = __ldg(o4 + cc);
        const float4 y = *reinterpret_cast<const float4 *>(g + 16 * cc);
        a = fmaf(x.x, y.x, a);
        b = fmaf(x.y, y.y, b);
        a = fmaf(x.z, y.z, a);
        b = fmaf(x.w, y.w, b);
    }
    return a + b;
}

struct BwdParams {
    const void *Q, *K, *V, *O, *dO;
    const float *LSE;
    void *dQ, *dK, *dV;
    float scale, scale_log2;
    int n_units;       // B * H
    int stages;        // ring depth (1 or 2)
    int cwarps;        // consumer warps
    uint32_t stage_bytes;
    uint32_t scratch_off;   // byte offset of the P/dS scratch in dynamic smem
    int max_count;          // max table entries of one head (scratch rows)
    const float *gw;        // global first token: P_0k, dS_0k ([B*H][2][N]), or NULL
    int early_prefetch;     // L2-prefetch the first units before the grid-dependency wait
    // Items: [0, n_keep) are whole units; then the units n_keep, n_keep + 1,
    // ... (the partial last wave) as `pieces` pieces each, piece q holding
    // rounds [q piece_rounds, (q + 1) piece_rounds) of both phases, with P and
    // dS recomputed in phase B so a piece needs no other piece's scratch.
    // n_units counts items.
    int n_keep;
    int pieces;
    int piece_rounds;
    uint32_t piece_off;   // per phase-B warp of a piece: [max_count][R] (P, dS) pairs
    int snake;            // odd full waves take the CTAs in reverse order (as the forward)
    int piece_par;        // one-round pieces spread over kPieceA + kPieceB warps (see the kernel)
    int fuse_gt;          // global first token: row 0 and column 0 inside each unit (gt_fused_*)
    uint32_t gt_off;      // fused global token: byte offset of w0r [2N], w0c [2N], partial sums [3 kGtParts][64]
};

constexpr int kGtParts = 4;   // fused global token: row ranges per dense sum

constexpr int kPieceA = 3;   // warps on a piece's query round, a third of its offsets each
constexpr int kPieceB = 6;   // warps on the first pass of its key round, a sixth each

// Unit of item u: item c + k * grid is wave k, position c; with `snake` odd
// full waves run the positions backwards (see fwd_slot_unit); the items past
// n_keep are pieces of the last units, in order.
__device__ __forceinline__ int bwd_item_unit(const BwdParams &p, int u) {
    if (u >= p.n_keep) return p.n_keep + (u - p.n_keep) / p.pieces;
    const int g = (int)gridDim.x, k = u / g;
    if (p.snake && (k & 1) && (k + 1) * g <= p.n_keep) return k * g + (g - 1 - u % g);
    return u;
}

// acc (this lane's slice of a row, in its chunk order) stored to a fp32 row of
// 64 dims in shared memory.
template <typename T, int G>
__device__ __forceinline__ void acc_store_shared(float *row, const int (&c)[Slice<T, G>::kChunks],
                                                 const float2 (&acc)[32 / G]) {
    constexpr int kPerChunk = 16 / (int)sizeof(T) / 2;   // element pairs per 16-byte chunk
#pragma unroll
    for (int i = 0; i < Slice<T, G>::kChunks; ++i) {
        const int base = c[i] / (int)sizeof(T);
#pragma unroll
        for (int e = 0; e < kPerChunk; e += 2)
            *reinterpret_cast<float4 *>(row + base + 2 * e) =
                make_float4(acc[kPerChunk * i + e].x, acc[kPerChunk * i + e].y, acc[kPerChunk * i + e + 1].x,
                            acc[kPerChunk * i + e + 1].y);
    }
}

// acc += the fp32 row of 64 dims at `row` in shared memory (this lane's slice,
// in its chunk order): the inverse of acc_store_shared.
template <typename T, int G>
__device__ __forceinline__ void acc_add_from_shared(const float *row, const int (&c)[Slice<T, G>::kChunks],
                                                    float2 (&acc)[32 / G]) {
    constexpr int kPerChunk = 16 / (int)sizeof(T) / 2;
#pragma unroll
    for (int i = 0; i < Slice<T, G>::kChunks; ++i) {
        const int base = c[i] / (int)sizeof(T);
#pragma unroll
        for (int e = 0; e < kPerChunk; e += 2) {
            const float4 v = *reinterpret_cast<const float4 *>(row + base + 2 * e);
            acc[kPerChunk * i + e] = add2(acc[kPerChunk * i + e], make_float2(v.x, v.y));
            acc[kPerChunk * i + e + 1] = add2(acc[kPerChunk * i + e + 1], make_float2(v.z, v.w));
        }
    }
}

// First pass of a piece's key round over offsets [ta, tz): (P, dS) of the
// pairs (k + off, k) from the staged rows into pw[(t - tb) R + row].
template <typename T, int G>
__device__ __forceinline__ void bwd_b_weights(const int *off, int N, int tb, int ta, int tz, int k, bool valid,
                                              const uint8_t *sQ, const uint8_t *sK, ptrdiff_t tens,
                                              const float *sD, const float *sL, float sl2,
                                              const LaneGeom<T, G> &lg, float2 *pw) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    constexpr int R = 32 / G;
    const int lane = threadIdx.x & 31, row = lane / G;
    const bool writer = (lane & (G - 1)) == 0;
    S kk, vv;
    kk.load(sK + (ptrdiff_t)k * RB, lg.c);
    vv.load(sK + tens + (ptrdiff_t)k * RB, lg.c);
    for (int t = ta; t < tz; ++t) {
        const int j = k + off[t];
        const bool in = valid && j >= 0 && j < N;
        const int jc = min(max(j, 0), N - 1);
        const uint8_t *a = sQ + (ptrdiff_t)jc * RB;
        S qq, gg;
        qq.load(a, lg.c);
        gg.load(a + 3 * tens, lg.c);
        const float sc = group_sum<G>(qq.dot(kk));
        const float dp = group_sum<G>(gg.dot(vv));
        const float P = in ? fast_exp2(fmaf(sc, sl2, -sL[jc])) : 0.f;
        if (writer) pw[(t - tb) * R + row] = make_float2(P, P * (dp - sD[jc]));
    }
}

// Phase B for one round of key rows with P and dS recomputed from the staged
// rows (pieces of a split unit), in two passes that keep the register count
// of the two-phase path: first s = <q_j, k>, dP = <dO_j, v>, P from the row's
// LSE and dS = P (dP - D_j) for every offset into this warp's area pw
// ([te - tb][R] pairs of P, dS), then the row updates as in bwd_b_offsets.
template <typename T, int G>
__device__ __forceinline__ void bwd_b_recompute_offsets(const int *off, int N, int tb, int te, int k, bool valid,
                                                        const uint8_t *sQ, const uint8_t *sK, ptrdiff_t tens,
                                                        const float *sD, const float *sL, float sl2,
                                                        const LaneGeom<T, G> &lg, float2 *pw,
                                                        float2 (&dk)[32 / G], float2 (&dv)[32 / G]) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    constexpr int R = 32 / G;
    const int lane = threadIdx.x & 31, row = lane / G;
    const bool writer = (lane & (G - 1)) == 0;
    {
        S kk, vv;
        kk.load(sK + (ptrdiff_t)k * RB, lg.c);
        vv.load(sK + tens + (ptrdiff_t)k * RB, lg.c);
        for (int t = tb; t < te; ++t) {
            const int j = k + off[t];
            const bool in = valid && j >= 0 && j < N;
            const int jc = min(max(j, 0), N - 1);
            const uint8_t *a = sQ + (ptrdiff_t)jc * RB;
            S qq, gg;
            qq.load(a, lg.c);
            gg.load(a + 3 * tens, lg.c);
            const float sc = group_sum<G>(qq.dot(kk));
            const float dp = group_sum<G>(gg.dot(vv));
            const float P = in ? fast_exp2(fmaf(sc, sl2, -sL[jc])) : 0.f;
            if (writer) pw[(t - tb) * R + row] = make_float2(P, P * (dp - sD[jc]));
        }
    }
    __syncwarp();
    for (int t = tb; t < te; ++t) {
        const int jc = min(max(k + off[t], 0), N - 1);
        const float2 w = pw[(t - tb) * R + row];
        const uint8_t *a = sQ + (ptrdiff_t)jc * RB;
        S qq, gg;
        qq.load(a, lg.c);
        gg.load(a + 3 * tens, lg.c);
        qq.axpy(w.y, dk);
        gg.axpy(w.x, dv);
    }
}

// Phase A for one round of query rows, branch-free: the key row is clamped
// into [0, N) and an out-of-range pair gets P = 0 (so dS = 0 too); only
// in-range pairs are written to the scratch.
template <typename T, int G, bool STORE = true>
__device__ __forceinline__ void bwd_a_offsets(const int *off, int N, int t0, int tb, int te, int j, bool valid,
                                              const uint8_t *sK, ptrdiff_t vdelta, const Slice<T, G> &q,
                                              const Slice<T, G> &g, float Dj, float lse2, float sl2,
                                              const LaneGeom<T, G> &lg, float2 *scr,
                                              float2 (&dq)[32 / G]) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    const bool writer = (threadIdx.x & (G - 1)) == 0;
    for (int t = tb; t < te; ++t) {
        const int k = j + off[t];
        const bool in = valid && k >= 0 && k < N;
        const uint8_t *a = sK + (ptrdiff_t)min(max(k, 0), N - 1) * RB;
        S kk, vv;
        kk.load(a, lg.c);
        vv.load(a + vdelta, lg.c);
        const float s = group_sum<G>(q.dot(kk));
        const float dp = group_sum<G>(g.dot(vv));
        const float P = in ? fast_exp2(fmaf(s, sl2, -lse2)) : 0.f;
        const float dS = P * (dp - Dj);
        if (STORE && writer && in) scr[(t - t0) * N + j] = make_float2(P, dS);
        kk.axpy(dS, dq);
    }
}

// Phase B for one round of key rows, branch-free: the query row is clamped
// into [0, N) and an out-of-range pair contributes P = dS = 0.
template <typename T, int G>
__device__ __forceinline__ void bwd_b_offsets(const int *off, int N, int t0, int t1, int tb, int te, int k,
                                              bool valid, const uint8_t *sQ, ptrdiff_t gdelta,
                                              const LaneGeom<T, G> &lg, const float2 *scr,
                                              float2 (&dk)[32 / G], float2 (&dv)[32 / G]) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    for (int t = tb; t < te; ++t) {
        const int j = k + off[t];
        const bool in = valid && j >= 0 && j < N;
        const int jc = min(max(j, 0), N - 1);
        const int m = t0 + t1 - 1 - t;            // forward offset index of the pair (j, k)
        const float2 w = scr[(m - t0) * N + jc];   // a stale pair when out of range: masked below
        const float P = in ? w.x : 0.f;
        const float dS = in ? w.y : 0.f;
        const uint8_t *a = sQ + (ptrdiff_t)jc * RB;
        S qq, gg;
        qq.load(a, lg.c);
        gg.load(a + gdelta, lg.c);
        qq.axpy(dS, dk);
        gg.axpy(P, dv);
    }
}

// Global first token, phase A: the pair (j, 0) for a query row j >= 1 whose
// band misses key 0 (sK0: key row 0; value row 0 at sK0 + vdelta).
template <typename T, int G>
__device__ __forceinline__ void bwd_a_global(const int *off, int t0, int t1, int j, bool valid, const uint8_t *sK0,
                                             ptrdiff_t vdelta, const Slice<T, G> &q, const Slice<T, G> &g, float Dj,
                                             float lse2, float sl2, const LaneGeom<T, G> &lg, float2 (&dq)[32 / G]) {
    // every lane takes part in the warp-wide scan, whatever its row
    const int first = __shfl_sync(kFullMask, j, 0);   // the warp's rows are first + lane / G
    const unsigned hit = band_reaches_zero(off, t0, t1, first, 32 / G);
    const bool need = valid && j >= 1 && !((hit >> (j - first)) & 1u);
    Slice<T, G> kk, vv;
    kk.load(sK0, lg.c);
    vv.load(sK0 + vdelta, lg.c);
    const float s = group_sum<G>(q.dot(kk));
    const float dp = group_sum<G>(g.dot(vv));
    const float P = need ? fast_exp2(fmaf(s, sl2, -lse2)) : 0.f;
    kk.axpy(P * (dp - Dj), dq);
}

// Global first token, phase B: the pair (0, k) for a key row k >= 1 whose
// band misses query 0, with P_0k and dS_0k from the dense-row kernel (gw of
// this (b, h)); sQ0: query row 0, its dO row at sQ0 + gdelta.
template <typename T, int G>
__device__ __forceinline__ void bwd_b_global(const int *off, int t0, int t1, int k, bool valid, const float *gw,
                                             int N, const uint8_t *sQ0, ptrdiff_t gdelta, const LaneGeom<T, G> &lg,
                                             float2 (&dk)[32 / G], float2 (&dv)[32 / G]) {
    // every lane takes part in the warp-wide scan, whatever its row
    const int first = __shfl_sync(kFullMask, k, 0);   // the warp's rows are first + lane / G
    const unsigned hit = band_reaches_zero(off, t0, t1, first, 32 / G);
    const bool need = valid && k >= 1 && !((hit >> (k - first)) & 1u);
    const float P = need ? gw[k] : 0.f;
    const float dS = need ? gw[N + k] : 0.f;
    Slice<T, G> qq, gg;
    qq.load(sQ0, lg.c);
    gg.load(sQ0 + gdelta, lg.c);
    qq.axpy(dS, dk);
    gg.axpy(P, dv);
}

// Global first token in a last-wave piece, phase B: the pair (0, k) for a
// key row k >= 1 whose band misses query 0, with P_0k and dS_0k computed
// here from the staged rows (query and dO row 0 at sQ and sQ + gdelta; key
// and value row k at sK + k RB and sK + vdelta + k RB; D_0, LSE_0 in log2
// units); acc += dS_0k q_0 (dk, which = 0) or P_0k dO_0 (dv, which = 1).
template <typename T, int G>
__device__ __forceinline__ void bwd_b_global_local(const int *off, int t0, int t1, int k, bool valid,
                                                   const uint8_t *sQ, ptrdiff_t gdelta, const uint8_t *sK,
                                                   ptrdiff_t vdelta, float D0, float L0, float sl2,
                                                   const LaneGeom<T, G> &lg, int which, float2 (&acc)[32 / G]) {
    constexpr int RB = Slice<T, G>::kRowBytes;
    // every lane takes part in the warp-wide scan, whatever its row
    const int first = __shfl_sync(kFullMask, k, 0);   // the warp's rows are first + lane / G
    const unsigned hit = band_reaches_zero(off, t0, t1, first, 32 / G);
    const bool need = valid && k >= 1 && !((hit >> (k - first)) & 1u);
    Slice<T, G> q0, g0, kk, vv;
    q0.load(sQ, lg.c);
    g0.load(sQ + gdelta, lg.c);
    kk.load(sK + (ptrdiff_t)k * RB, lg.c);
    vv.load(sK + vdelta + (ptrdiff_t)k * RB, lg.c);
    const float sc = group_sum<G>(q0.dot(kk));
    const float dp = group_sum<G>(g0.dot(vv));
    const float P = need ? fast_exp2(fmaf(sc, sl2, -L0)) : 0.f;
    if (which == 0)
        q0.axpy(P * (dp - D0), acc);
    else
        g0.axpy(P, acc);
}

// Half of the dot product of two 64-element rows in shared memory: the
// lane's half (lane & 1) of the dims, in 16-byte chunks whose order is
// rotated by rot and the half, so that the eight lanes of a quarter warp (four
// rows, both halves) read eight distinct bank groups.
template <typename T>
__device__ __forceinline__ float half_row_dot(const uint8_t *a, const uint8_t *b, int rot) {
    constexpr int HC = (int)sizeof(T) * kHeadDim / 32;   // 16-byte chunks in half a row
    const int half = threadIdx.x & 1;
    float xa = 0.f, xb = 0.f;
#pragma unroll
    for (int c = 0; c < HC; ++c) {
        const int cc = half * HC + ((c + rot + 4 * half) & (HC - 1));
        const uint4 x = *reinterpret_cast<const uint4 *>(a + cc * 16);
        const uint4 y = *reinterpret_cast<const uint4 *>(b + cc * 16);
        if constexpr (std::is_same<T, float>::value) {
            xa = fmaf(__uint_as_float(x.x), __uint_as_float(y.x), xa);
            xb = fmaf(__uint_as_float(x.y), __uint_as_float(y.y), xb);
            xa = fmaf(__uint_as_float(x.z), __uint_as_float(y.z), xa);
            xb = fmaf(__uint_as_float(x.w), __uint_as_float(y.w), xb);
        } else {
            xa = dot2_bf16(x.x, y.x, xa);
            xb = dot2_bf16(x.y, y.y, xb);
            xa = dot2_bf16(x.z, y.z, xa);
            xb = dot2_bf16(x.w, y.w, xb);
        }
    }
    return xa + xb;
}

// Global first token inside a whole-head unit of the backward, phase A: the
// weights of the dense row 0 (pairs (0, k), every key k) into w0r = [P_0k |
// dS_0k], and of the dense column 0 (pairs (j, 0), every query j) into w0c =
// [P_j0 | dS_j0], with P = exp(s - LSE) and dS = P (dP - D) of the row's own
// query.  Two lanes per row, 16 rows per warp batch.  The stage holds Q, K,
// V, dO at sQ + {0, 1, 2, 3} tens; sD and sL are D_j and LSE_j (log2 units).
template <typename T>
__device__ __forceinline__ void gt_fused_weights(const uint8_t *sQ, size_t tens, const float *sD, const float *sL,
                                                 int N, int cw, int cwarps, float sl2, float *w0r, float *w0c) {
    constexpr int RB = (int)sizeof(T) * kHeadDim;
    const int lane = threadIdx.x & 31, kl = lane >> 1;
    const uint8_t *sK = sQ + tens, *sV = sQ + 2 * tens, *sG = sQ + 3 * tens;
    for (int rb = cw * 16; rb < N; rb += 16 * cwarps) {
        const int r = min(rb + kl, N - 1);   // rows past N repeat row N - 1 and are not stored
        float s = half_row_dot<T>(sQ, sK + (size_t)r * RB, kl);
        float dp = half_row_dot<T>(sG, sV + (size_t)r * RB, kl);
        float sc = half_row_dot<T>(sQ + (size_t)r * RB, sK, kl);
        float dpc = half_row_dot<T>(sG + (size_t)r * RB, sV, kl);
        s += __shfl_xor_sync(kFullMask, s, 1);
        dp += __shfl_xor_sync(kFullMask, dp, 1);
        sc += __shfl_xor_sync(kFullMask, sc, 1);
        dpc += __shfl_xor_sync(kFullMask, dpc, 1);
        if ((lane & 1) == 0 && rb + kl < N) {
            const float P = fast_exp2(fmaf(s, sl2, -sL[0]));
            w0r[r] = P;
            w0r[N + r] = P * (dp - sD[0]);
            const float Pc = fast_exp2(fmaf(sc, sl2, -sL[r]));
            w0c[r] = Pc;
            w0c[N + r] = Pc * (dpc - sD[r]);
        }
    }
}

// Phase B: the three dense sums of the global first token, dQ_0 = scale
// sum_k dS_0k K_k, dK_0 = scale sum_j dS_j0 Q_j and dV_0 = sum_j P_j0 dO_j.
// Item = sum x row range (kGtParts ranges); the warp sums its item's rows,
// two dims per lane, into its partial slot and counts itself in; the warp
// whose item arrives last adds the partials in a fixed order (so the result
// does not depend on which warp that is), writes the three rows and resets
// the count.
template <typename T>
__device__ __forceinline__ void gt_fused_sums(const uint8_t *sQ, size_t tens, int N, int item, const float *w0r,
                                              const float *w0c, float2 *part, int *count, float scale, T *dQ0,
                                              T *dK0, T *dV0) {
    constexpr int RB = (int)sizeof(T) * kHeadDim;
    const int lane = threadIdx.x & 31;
    const int v = item / kGtParts, q = item % kGtParts;
    const float *w = v == 0 ? w0r + N : (v == 1 ? w0c + N : w0c);
    const uint8_t *X = v == 0 ? sQ + tens : (v == 1 ? sQ : sQ + 3 * tens);
    const int r0 = q * N / kGtParts, r1 = (q + 1) * N / kGtParts;
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int r = r0; r < r1; ++r) {
        const float wr = w[r];
        float2 x;
        if constexpr (std::is_same<T, float>::value) {
            x = reinterpret_cast<const float2 *>(X + (size_t)r * RB)[lane];
        } else {
            const uint32_t b = reinterpret_cast<const uint32_t *>(X + (size_t)r * RB)[lane];
            x = make_float2(bf16_lo(b), bf16_hi(b));
        }
        acc.x = fmaf(wr, x.x, acc.x);
        acc.y = fmaf(wr, x.y, acc.y);
    }
    part[item * 32 + lane] = acc;
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(count, 1) == 3 * kGtParts - 1;
    }
    if (!__shfl_sync(kFullMask, last, 0)) return;
    __threadfence_block();
#pragma unroll
    for (int vv = 0; vv < 3; ++vv) {
        float2 t = part[(vv * kGtParts) * 32 + lane];
#pragma unroll
        for (int qq = 1; qq < kGtParts; ++qq) {
            const float2 y = part[(vv * kGtParts + qq) * 32 + lane];
            t.x += y.x;
            t.y += y.y;
        }
        const float f = vv == 2 ? 1.f : scale;
        T *dst = vv == 0 ? dQ0 : (vv == 1 ? dK0 : dV0);
        if constexpr (std::is_same<T, float>::value) {
            reinterpret_cast<float2 *>(dst)[lane] = make_float2(t.x * f, t.y * f);
        } else {
            reinterpret_cast<uint32_t *>(dst)[lane] = pack_bf16x2(t.x * f, t.y * f);
        }
    }
    if (lane == 0) *count = 0;
}

// MAXT: threads per CTA the register budget is sized for (65536 / MAXT each).
template <typename T, int G, int MAXT, bool GT = false>
__global__ void __launch_bounds__(MAXT, 1)
bwd_pipe_kernel(const __grid_constant__ TableArg tab, const BwdParams p) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    constexpr int R = 32 / G;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full_bar[2], empty_bar[2], aux_bar[2];
    __shared__ int s_off[kMaxEntries];
    __shared__ int s_start[kMaxHeads + 1];   // the heads' table starts (per-unit reads from shared memory)
    __shared__ int s_gt_count;               // fused global token: dense-sum items done in this unit
    __shared__ int s_abort;                  // a bounded wait of this CTA gave up (mbar_wait)

    const int N = tab.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0 && (p.early_prefetch & 1)) {
        // as in the forward: warm L2 with the first units' rows early
        const uint32_t b = (uint32_t)((size_t)N * RB);
        for (int i = 0; i < ((p.early_prefetch & 2) ? 1 : p.stages); ++i) {
            const int it = (int)blockIdx.x + i * (int)gridDim.x;
            if (it >= p.n_units) break;
            const size_t row0 = (size_t)bwd_item_unit(p, it) * N * kHeadDim;
            bulk_prefetch_l2(static_cast<const T *>(p.Q) + row0, b);
            bulk_prefetch_l2(static_cast<const T *>(p.K) + row0, b);
            bulk_prefetch_l2(static_cast<const T *>(p.V) + row0, b);
            bulk_prefetch_l2(static_cast<const T *>(p.dO) + row0, b);
        }
    }
    for (int t = threadIdx.x; t < tab.start[tab.H]; t += blockDim.x) s_off[t] = tab.off[t];
    for (int t = threadIdx.x; t <= tab.H; t += blockDim.x) s_start[t] = tab.start[t];
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
            mbar_init(&aux_bar[s], 1);
        }
        s_gt_count = 0;
        s_abort = 0;
    }
    __syncthreads();
    grid_dep_wait();
    grid_dep_launch();
    const size_t tens = (size_t)N * RB;   // one tensor's rows in a stage: Q | K | V | dO | D | LSE2
    if (warp == 0) {
        // producer warp: lane 0 streams the unit's four tensors in; then the
        // whole warp fills the stage's per-row terms D_j = <dO_j, O_j> (O read
        // from global memory, prefetched into L2 a unit ahead) and LSE_j in
        // log2 units, so no consumer waits on a global load
        int i = 0;
        for (int it = blockIdx.x; it < p.n_units; it += gridDim.x, ++i) {
            const int s = i % p.stages;
            // the lanes agree, so the warp leaves the loop together
            if (i >= p.stages && !__all_sync(kFullMask, mbar_wait(&empty_bar[s], ((i / p.stages) - 1) & 1, &s_abort)))
                break;
            // as in the forward: the second unit's copies wait for the first
            // unit's rows to land
            if (i == 1 && (p.early_prefetch & 2) && !__all_sync(kFullMask, mbar_wait(&full_bar[0], 0, &s_abort)))
                break;
            uint8_t *st = smem + (size_t)s * p.stage_bytes;
            const bool fill_by_consumers = i == 0;
            const size_t row0 = (size_t)bwd_item_unit(p, it) * N;
            if (lane == 0) {
                // the stage holds Q, K, V, dO and the rows' D_j, LSE_j
                const uint32_t b = FIBATT_CHECKED(4 * tens + 8 * (size_t)N <= p.stage_bytes) ? (uint32_t)tens : 0u;
                mbar_expect_tx(&full_bar[s], 4 * b);
                if (b) {
                    bulk_g2s(st, static_cast<const T *>(p.Q) + row0 * kHeadDim, b, &full_bar[s]);
                    bulk_g2s(st + tens, static_cast<const T *>(p.K) + row0 * kHeadDim, b, &full_bar[s]);
                    bulk_g2s(st + 2 * tens, static_cast<const T *>(p.V) + row0 * kHeadDim, b, &full_bar[s]);
                    bulk_g2s(st + 3 * tens, static_cast<const T *>(p.dO) + row0 * kHeadDim, b, &full_bar[s]);
                }
                if (fill_by_consumers) {   // the consumers compute these D_j
                    bulk_prefetch_l2(static_cast<const T *>(p.O) + row0 * kHeadDim, b);
                    if ((N * 4) % 16 == 0 && (row0 * 4) % 16 == 0) bulk_prefetch_l2(p.LSE + row0, (uint32_t)N * 4);
                }
                const int itn = it + gridDim.x;
                if (itn < p.n_units) {
                    const int un = bwd_item_unit(p, itn);
                    bulk_prefetch_l2(static_cast<const T *>(p.O) + (size_t)un * N * kHeadDim, b);
                    if ((N * 4) % 16 == 0 && ((size_t)un * N * 4) % 16 == 0)
                        bulk_prefetch_l2(p.LSE + (size_t)un * N, (uint32_t)N * 4);
                }
            }
            __syncwarp();
            if (fill_by_consumers) {
                // a CTA's first unit: the consumers, idle until the rows land,
                // fill D_j and LSE_j in one pass of one row per thread instead
                // of waiting for this warp's round trips (later units, pieces
                // included, have a whole unit of lead for them here)
                if (lane == 0) mbar_arrive(&aux_bar[s]);
                continue;
            }
            if (!__all_sync(kFullMask, mbar_wait(&full_bar[s], (i / p.stages) & 1, &s_abort))) {
                ++i;   // this unit's copies were issued
                break;
            }
            float *sD = reinterpret_cast<float *>(st + 4 * tens), *sL = sD + N;
            // kDRows rows per lane and step, every dot product formed before
            // any store, so the rows' global loads are in flight together
            constexpr int kDRows = 4;
            for (int j = lane; j < N; j += 32 * kDRows) {
                float d[kDRows], l[kDRows];
#pragma unroll
                for (int x = 0; x < kDRows; ++x) {
                    const int jx = min(j + 32 * x, N - 1);
                    d[x] = row_dot_global_shared(static_cast<const T *>(p.O) + (row0 + jx) * kHeadDim,
                                                 st + 3 * tens + (size_t)jx * RB, lane);
                    l[x] = p.LSE[row0 + jx];
                }
#pragma unroll
                for (int x = 0; x < kDRows; ++x)
                    if (j + 32 * x < N) {
                        sD[j + 32 * x] = d[x];
                        sL[j + 32 * x] = l[x] * kLog2e;
                    }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&aux_bar[s]);
        }
        // i units issued: leave only once the last copies into every stage
        // have landed
        if (lane == 0)
            for (int s = 0; s < p.stages && s < i; ++s) mbar_drain(&full_bar[s], ((i - 1 - s) / p.stages) & 1);
        return;
    }
    const int cw = warp - 1;
    if (cw >= p.cwarps) return;
    const int cthreads = 32 * p.cwarps;
    const LaneGeom<T, G> lg;
    float2 *scr = reinterpret_cast<float2 *>(smem + p.scratch_off);   // (P, dS) [offset][row]
    const int nrounds = (N + R - 1) / R;
    int i = 0;
    for (int it = blockIdx.x; it < p.n_units; it += gridDim.x, ++i) {
        const int s = i % p.stages;
        // A failed wait does not end the warp: the consumers meet at named
        // barriers, so every warp carries on (every later wait of the CTA
        // then returns at once) and all of them leave together.  What they
        // compute after a failure is never trusted: the error word is set.
        mbar_wait(&full_bar[s], (i / p.stages) & 1, &s_abort);
        mbar_wait(&aux_bar[s], (i / p.stages) & 1, &s_abort);
        const uint8_t *st = smem + (size_t)s * p.stage_bytes;
        const uint8_t *sQ = st, *sK = st + tens;
        const float *sD = reinterpret_cast<const float *>(st + 4 * tens), *sL = sD + N;
        const int u = bwd_item_unit(p, it);
        // with the global token the plan cuts units into one-round pieces only
        // (the piece_par path below), with the dense parts fused
        const bool piece = it >= p.n_keep;
        const int h = u % tab.H;
        const int t0 = s_start[h];
        // the (P, dS) scratch and the pieces' areas hold max_count entries per row
        const int t1 = FIBATT_CHECKED(s_start[h + 1] - t0 <= p.max_count) ? s_start[h + 1] : t0;
        const size_t row0 = (size_t)u * N;
        if (i == 0) {
            // D_j = <dO_j, O_j> and LSE_j (log2 units), one row per consumer
            // thread: the producer warp would take all the rows' global-load
            // round trips in turn while every consumer waits
            float *wD = reinterpret_cast<float *>(smem + (size_t)s * p.stage_bytes + 4 * tens), *wL = wD + N;
            for (int j = cw * 32 + lane; j < N; j += cthreads) {
                wD[j] = row_dot_global_shared(static_cast<const T *>(p.O) + (row0 + j) * kHeadDim,
                                              st + 3 * tens + (size_t)j * RB, lane);
                wL[j] = p.LSE[row0 + j] * kLog2e;
            }
            consumer_sync(cthreads);
        }
        if (piece && p.piece_par) {
            // a one-round piece spread over the warps: kPieceA warps take a
            // share of the query round's offsets each (partial dQ rows in the
            // scratch area, which pieces do not use otherwise), kPieceB warps
            // compute the key round's (P, dS) for a share of the offsets each,
            // then one warp accumulates dK and one dV over all of them.  A
            // piece is always its CTA's last item (the plan keeps the pieces
            // within one wave).  With the global token, the pairs (j, 0) and
            // (0, k) of the round's rows are added by the warps that store
            // them, and the piece of round 0 has its spare warps compute the
            // dense row 0 and column 0 over the staged head.
            const int r = (it - p.n_keep) % p.pieces;
            const int lr = lane / G;
            int tb = t0, te = t0;
            if (t1 > t0) round_range(s_off, N, t0, t1, r * R, min(N, r * R + R) - 1, tb, te);
            const int m = te - tb;
            float *pa = reinterpret_cast<float *>(smem + p.scratch_off);   // [kPieceA - 1][R][64] partial dQ
            float2 *pw = reinterpret_cast<float2 *>(smem + p.piece_off);   // [m][R] (P, dS)
            if (cw < kPieceA) {
                const int jl = r * R + lr;
                const bool valid = jl < N;
                const int j = valid ? jl : N - 1;
                S qr, g;
                qr.load(sQ + (size_t)j * RB, lg.c);
                g.load(sQ + 3 * tens + (size_t)j * RB, lg.c);
                float2 dq[32 / G];
#pragma unroll
                for (int x = 0; x < 32 / G; ++x) dq[x] = make_float2(0.f, 0.f);
                bwd_a_offsets<T, G, false>(s_off, N, t0, tb + (m * cw) / kPieceA, tb + (m * (cw + 1)) / kPieceA, j,
                                           valid, sK, (ptrdiff_t)tens, qr, g, sD[j], sL[j], p.scale_log2, lg, scr,
                                           dq);
                // warps 1 .. kPieceA-1 hand their partial rows to warp 0,
                // which adds them (in order) and stores the dQ rows
                if (cw > 0) acc_store_shared<T, G>(pa + ((size_t)(cw - 1) * R + lr) * kHeadDim, lg.c, dq);
                named_sync(3, 32 * kPieceA);
                if (cw == 0) {
                    for (int a = 0; a < kPieceA - 1; ++a)
                        acc_add_from_shared<T, G>(pa + ((size_t)a * R + lr) * kHeadDim, lg.c, dq);
                    if constexpr (GT)
                        bwd_a_global<T, G>(s_off, t0, t1, j, valid, sK, (ptrdiff_t)tens, qr, g, sD[j], sL[j],
                                           p.scale_log2, lg, dq);
                    if (valid && !(GT && j == 0)) {   // dQ_0: the dense row (spare warps of round 0's piece)
#pragma unroll
                        for (int x = 0; x < 32 / G; ++x) dq[x] = mul2(dq[x], make_float2(p.scale, p.scale));
                        S::store(static_cast<T *>(p.dQ) + (row0 + j) * kHeadDim, lg.c, dq);
                    }
                }
            } else if (cw < kPieceA + kPieceB) {
                const int b = cw - kPieceA;
                const int kl = r * R + lr;
                const bool valid = kl < N;
                const int k = valid ? kl : N - 1;
                bwd_b_weights<T, G>(s_off, N, tb, tb + (m * b) / kPieceB, tb + (m * (b + 1)) / kPieceB, k, valid, sQ,
                                    sK, (ptrdiff_t)tens, sD, sL, p.scale_log2, lg, pw);
                named_sync(2, 32 * kPieceB);   // every (P, dS) of the round written
                if (b < 2) {   // b = 0: dK = scale sum dS q_j; b = 1: dV = sum P dO_j
                    float2 acc[32 / G];
#pragma unroll
                    for (int x = 0; x < 32 / G; ++x) acc[x] = make_float2(0.f, 0.f);
                    const uint8_t *src = b == 0 ? sQ : sQ + 3 * tens;
                    int t = tb;
                    for (; t + 1 < te; t += 2) {   // two offsets per step: their loads overlap
                        const int j0 = min(max(k + s_off[t], 0), N - 1), j1 = min(max(k + s_off[t + 1], 0), N - 1);
                        const float2 w0 = pw[(t - tb) * R + lr], w1 = pw[(t + 1 - tb) * R + lr];   // (0, 0) out of range
                        S r0, r1;
                        r0.load(src + (size_t)j0 * RB, lg.c);
                        r1.load(src + (size_t)j1 * RB, lg.c);
                        r0.axpy(b == 0 ? w0.y : w0.x, acc);
                        r1.axpy(b == 0 ? w1.y : w1.x, acc);
                    }
                    for (; t < te; ++t) {
                        const int jc = min(max(k + s_off[t], 0), N - 1);
                        const float2 w = pw[(t - tb) * R + lr];
                        S rr;
                        rr.load(src + (size_t)jc * RB, lg.c);
                        rr.axpy(b == 0 ? w.y : w.x, acc);
                    }
                    if constexpr (GT)
                        bwd_b_global_local<T, G>(s_off, t0, t1, k, valid, sQ, (ptrdiff_t)(3 * tens), sK,
                                                 (ptrdiff_t)tens, sD[0], sL[0], p.scale_log2, lg, b, acc);
                    if (valid && !(GT && k == 0)) {   // dK_0, dV_0: the dense column (round 0's piece)
                        if (b == 0) {
#pragma unroll
                            for (int x = 0; x < 32 / G; ++x) acc[x] = mul2(acc[x], make_float2(p.scale, p.scale));
                        }
                        S::store(static_cast<T *>(b == 0 ? p.dK : p.dV) + (row0 + k) * kHeadDim, lg.c, acc);
                    }
                }
            } else if (GT && r == 0) {
                // spare warps of round 0's piece: the weights of row 0 and
                // column 0 over the staged head, then the three dense sums
                // (gt_fused_weights / gt_fused_sums, as in a whole unit)
                const int sw = cw - (kPieceA + kPieceB), nsw = p.cwarps - (kPieceA + kPieceB);
                float *w0r = reinterpret_cast<float *>(smem + p.gt_off), *w0c = w0r + 2 * N;
                gt_fused_weights<T>(sQ, tens, sD, sL, N, sw, nsw, p.scale_log2, w0r, w0c);
                named_sync(4, 32 * nsw);
                float2 *part = reinterpret_cast<float2 *>(w0c + 2 * N);
                for (int item = sw; item < 3 * kGtParts; item += nsw)
                    gt_fused_sums<T>(sQ, tens, N, item, w0r, w0c, part, &s_gt_count, p.scale,
                                     static_cast<T *>(p.dQ) + row0 * kHeadDim, static_cast<T *>(p.dK) + row0 * kHeadDim,
                                     static_cast<T *>(p.dV) + row0 * kHeadDim);
            }
            consumer_sync(cthreads);   // stage free
            if (cw == 0 && lane == 0) mbar_arrive(&empty_bar[s]);
            continue;
        }
        if (piece) {
            // rounds [r0, r1) of this unit: warps 0 .. n-1 take the query
            // rounds (phase A), warps n .. 2n-1 the key rounds with P and dS
            // recomputed (phase B), concurrently
            const int q = (it - p.n_keep) % p.pieces;
            const int r0 = q * p.piece_rounds, r1 = min(nrounds, r0 + p.piece_rounds);
            const int n = r1 - r0;
            if (cw < n) {
                const int r = r0 + cw;
                const int jl = r * R + lane / G;
                const bool valid = jl < N;
                const int j = valid ? jl : N - 1;
                int tb = t0, te = t0;
                if (t1 > t0) round_range(s_off, N, t0, t1, r * R, min(N, r * R + R) - 1, tb, te);
                S qr, g;
                qr.load(sQ + (size_t)j * RB, lg.c);
                g.load(sQ + 3 * tens + (size_t)j * RB, lg.c);
                float2 dq[32 / G];
#pragma unroll
                for (int x = 0; x < 32 / G; ++x) dq[x] = make_float2(0.f, 0.f);
                bwd_a_offsets<T, G>(s_off, N, t0, tb, te, j, valid, sK, (ptrdiff_t)tens, qr, g, sD[j], sL[j],
                                    p.scale_log2, lg, scr, dq);
                if (valid) {
#pragma unroll
                    for (int x = 0; x < 32 / G; ++x) dq[x] = mul2(dq[x], make_float2(p.scale, p.scale));
                    S::store(static_cast<T *>(p.dQ) + (row0 + j) * kHeadDim, lg.c, dq);
                }
            } else if (cw < 2 * n) {
                const int r = r0 + cw - n;
                const int kl = r * R + lane / G;
                const bool valid = kl < N;
                const int k = valid ? kl : N - 1;
                int tb = t0, te = t0;
                if (t1 > t0) round_range(s_off, N, t0, t1, r * R, min(N, r * R + R) - 1, tb, te);
                float2 dk[32 / G], dv[32 / G];
#pragma unroll
                for (int x = 0; x < 32 / G; ++x) dk[x] = dv[x] = make_float2(0.f, 0.f);
                float2 *pw = reinterpret_cast<float2 *>(smem + p.piece_off) + (size_t)(cw - n) * R * p.max_count;
                bwd_b_recompute_offsets<T, G>(s_off, N, tb, te, k, valid, sQ, sK, (ptrdiff_t)tens, sD, sL,
                                              p.scale_log2, lg, pw, dk, dv);
                if (valid) {
#pragma unroll
                    for (int x = 0; x < 32 / G; ++x) dk[x] = mul2(dk[x], make_float2(p.scale, p.scale));
                    S::store(static_cast<T *>(p.dK) + (row0 + k) * kHeadDim, lg.c, dk);
                    S::store(static_cast<T *>(p.dV) + (row0 + k) * kHeadDim, lg.c, dv);
                }
            }
            consumer_sync(cthreads);   // stage free
            if (cw == 0 && lane == 0) mbar_arrive(&empty_bar[s]);
            continue;
        }
        // ---- phase A: query rows
        for (int r = cw; r < nrounds; r += p.cwarps) {
            const int jl = r * R + lane / G;
            const bool valid = jl < N;
            const int j = valid ? jl : N - 1;
            const int jfirst = r * R, jlast = min(N, r * R + R) - 1;
            int tb = t0, te = t0;
            if (t1 > t0) round_range(s_off, N, t0, t1, jfirst, jlast, tb, te);
            S q, g;
            q.load(sQ + (size_t)j * RB, lg.c);
            g.load(sQ + 3 * tens + (size_t)j * RB, lg.c);
            const float Dj = sD[j];
            const float lse2 = sL[j];
            float2 dq[32 / G];
#pragma unroll
            for (int x = 0; x < 32 / G; ++x) dq[x] = make_float2(0.f, 0.f);
            bwd_a_offsets<T, G>(s_off, N, t0, tb, te, j, valid, sK, (ptrdiff_t)tens, q, g, Dj, lse2, p.scale_log2, lg,
                                scr, dq);
            if constexpr (GT)
                bwd_a_global<T, G>(s_off, t0, t1, j, valid, sK, (ptrdiff_t)tens, q, g, Dj, lse2, p.scale_log2, lg, dq);
            if (valid && !(GT && j == 0)) {   // dQ_0: the dense row (fused below or the row kernel)
#pragma unroll
                for (int x = 0; x < 32 / G; ++x) dq[x] = mul2(dq[x], make_float2(p.scale, p.scale));
                S::store(static_cast<T *>(p.dQ) + (row0 + j) * kHeadDim, lg.c, dq);
            }
        }
        float *w0r = reinterpret_cast<float *>(smem + p.gt_off), *w0c = w0r + 2 * N;
        if constexpr (GT) {
            if (p.fuse_gt) gt_fused_weights<T>(sQ, tens, sD, sL, N, cw, p.cwarps, p.scale_log2, w0r, w0c);
        }
        consumer_sync(cthreads);
        // ---- phase B: key rows
        for (int r = cw; r < nrounds; r += p.cwarps) {
            const int kl = r * R + lane / G;
            const bool valid = kl < N;
            const int k = valid ? kl : N - 1;
            const int kfirst = r * R, klast = min(N, r * R + R) - 1;
            int tb = t0, te = t0;
            if (t1 > t0) round_range(s_off, N, t0, t1, kfirst, klast, tb, te);
            float2 dk[32 / G], dv[32 / G];
#pragma unroll
            for (int x = 0; x < 32 / G; ++x) dk[x] = dv[x] = make_float2(0.f, 0.f);
            bwd_b_offsets<T, G>(s_off, N, t0, t1, tb, te, k, valid, sQ, (ptrdiff_t)(3 * tens), lg, scr, dk,
                                dv);
            if constexpr (GT)
                bwd_b_global<T, G>(s_off, t0, t1, k, valid, p.fuse_gt ? w0r : p.gw + (size_t)u * 2 * N, N, sQ,
                                   (ptrdiff_t)(3 * tens), lg, dk, dv);
            if (valid && !(GT && k == 0)) {   // dK_0, dV_0: the dense column (fused below or the column kernel)
#pragma unroll
                for (int x = 0; x < 32 / G; ++x) dk[x] = mul2(dk[x], make_float2(p.scale, p.scale));
                S::store(static_cast<T *>(p.dK) + (row0 + k) * kHeadDim, lg.c, dk);
                S::store(static_cast<T *>(p.dV) + (row0 + k) * kHeadDim, lg.c, dv);
            }
        }
        if constexpr (GT) {
            if (p.fuse_gt) {
                float2 *part = reinterpret_cast<float2 *>(w0c + 2 * N);
                for (int item = cw; item < 3 * kGtParts; item += p.cwarps)
                    gt_fused_sums<T>(sQ, tens, N, item, w0r, w0c, part, &s_gt_count, p.scale,
                                     static_cast<T *>(p.dQ) + row0 * kHeadDim, static_cast<T *>(p.dK) + row0 * kHeadDim,
                                     static_cast<T *>(p.dV) + row0 * kHeadDim);
            }
        }
        consumer_sync(cthreads);   // scratch and stage free for the next unit
        if (cw == 0 && lane == 0) mbar_arrive(&empty_bar[s]);
    }
}

// ------------------------------------------------------------ flat backward
//
// The two phases as two kernels over rows read from global memory, with the
// pair weights P and dS in a global scratch [b, h][2][max_count][N] (phase A
// writes the pairs in range, phase B reads exactly those).  Phase A: dQ;
// phase B: dK, dV.  Block: kFlatWarps warps of one (b, h), one round each.
template <typename T, int G, bool GT>
__device__ __forceinline__ void bwd_flat_a_round(const TableArg &tab, const BwdParams &p, const int *s_off,
                                                 float *scr, int bh, int r) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    constexpr int R = 32 / G;
    const int N = tab.N;
    const int h = bh % tab.H;
    const int t0 = tab.start[h], t1 = tab.start[h + 1];
    const int lane = threadIdx.x & 31;
    const size_t row0 = (size_t)bh * N;
    const uint8_t *gK = static_cast<const uint8_t *>(p.K) + row0 * RB;
    const ptrdiff_t vdelta = static_cast<const uint8_t *>(p.V) - static_cast<const uint8_t *>(p.K);
    float2 *scr2 = reinterpret_cast<float2 *>(scr);   // this unit's (P, dS) [offset][row]
    const LaneGeom<T, G> lg;
    const int jl = r * R + lane / G;
    const bool valid = jl < N;
    const int j = valid ? jl : N - 1;
    const int jfirst = r * R, jlast = min(N, r * R + R) - 1;
    int tb = t0, te = t0;
    if (t1 > t0) round_range(s_off, N, t0, t1, jfirst, jlast, tb, te);
    S q, g, o;
    q.load_global(static_cast<const T *>(p.Q) + (row0 + j) * kHeadDim, lg.c);
    g.load_global(static_cast<const T *>(p.dO) + (row0 + j) * kHeadDim, lg.c);
    o.load_global(static_cast<const T *>(p.O) + (row0 + j) * kHeadDim, lg.c);
    const float Dj = group_sum<G>(g.dot(o));
    const float lse2 = p.LSE[row0 + j] * kLog2e;
    float2 dq[32 / G];
#pragma unroll
    for (int x = 0; x < 32 / G; ++x) dq[x] = make_float2(0.f, 0.f);
    bwd_a_offsets<T, G>(s_off, N, t0, tb, te, j, valid, gK, vdelta, q, g, Dj, lse2, p.scale_log2, lg, scr2,
                        dq);
    if constexpr (GT) bwd_a_global<T, G>(s_off, t0, t1, j, valid, gK, vdelta, q, g, Dj, lse2, p.scale_log2, lg, dq);
    if (valid && !(GT && j == 0)) {
#pragma unroll
        for (int x = 0; x < 32 / G; ++x) dq[x] = mul2(dq[x], make_float2(p.scale, p.scale));
        S::store(static_cast<T *>(p.dQ) + (row0 + j) * kHeadDim, lg.c, dq);
    }
}

template <typename T, int G, int W = kFlatWarps, bool GT = false>
__global__ void __launch_bounds__(W * 32)
bwd_flat_a_kernel(const __grid_constant__ TableArg tab, const BwdParams p, float *scr, int bh0) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    constexpr int R = 32 / G;
    __shared__ int s_off[kMaxEntries];
    const int N = tab.N;
    const int bh = bh0 + blockIdx.x, h = bh % tab.H;
    const int t0 = tab.start[h], t1 = tab.start[h + 1];
    for (int t = t0 + (int)threadIdx.x; t < t1; t += blockDim.x) s_off[t] = tab.off[t];
    __syncthreads();
    grid_dep_wait();
    grid_dep_launch();
    const int r = blockIdx.y * W + (threadIdx.x >> 5);
    if (r * R < N) bwd_flat_a_round<T, G, GT>(tab, p, s_off, scr + (size_t)blockIdx.x * 2 * p.max_count * N, bh, r);
}

template <typename T, int G, int W = kFlatWarps, bool GT = false>
__global__ void __launch_bounds__(W * 32)
bwd_flat_b_kernel(const __grid_constant__ TableArg tab, const BwdParams p, const float *scr, int bh0) {
    using S = Slice<T, G>;
    constexpr int RB = S::kRowBytes;
    constexpr int R = 32 / G;
    __shared__ int s_off[kMaxEntries];
    const int N = tab.N;
    const int bh = bh0 + blockIdx.x, h = bh % tab.H;
    const int t0 = tab.start[h], t1 = tab.start[h + 1];
    for (int t = t0 + (int)threadIdx.x; t < t1; t += blockDim.x) s_off[t] = tab.off[t];
    __syncthreads();
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.y * W + (threadIdx.x >> 5);
    if (r * R >= N) return;
    const size_t row0 = (size_t)bh * N;
    const uint8_t *gQ = static_cast<const uint8_t *>(p.Q) + row0 * RB;
    const ptrdiff_t gdelta = static_cast<const uint8_t *>(p.dO) - static_cast<const uint8_t *>(p.Q);
    const float2 *scr2 = reinterpret_cast<const float2 *>(scr + (size_t)blockIdx.x * 2 * p.max_count * N);
    const LaneGeom<T, G> lg;
    const int kl = r * R + lane / G;
    const bool valid = kl < N;
    const int k = valid ? kl : N - 1;
    const int kfirst = r * R, klast = min(N, r * R + R) - 1;
    int tb = t0, te = t0;
    if (t1 > t0) round_range(s_off, N, t0, t1, kfirst, klast, tb, te);
    float2 dk[32 / G], dv[32 / G];
#pragma unroll
    for (int x = 0; x < 32 / G; ++x) dk[x] = dv[x] = make_float2(0.f, 0.f);
    bwd_b_offsets<T, G>(s_off, N, t0, t1, tb, te, k, valid, gQ, gdelta, lg, scr2, dk, dv);
    if constexpr (GT) bwd_b_global<T, G>(s_off, t0, t1, k, valid, p.gw + (size_t)bh * 2 * N, N, gQ, gdelta, lg, dk, dv);
    if (valid && !(GT && k == 0)) {
#pragma unroll
        for (int x = 0; x < 32 / G; ++x) dk[x] = mul2(dk[x], make_float2(p.scale, p.scale));
        S::store(static_cast<T *>(p.dK) + (row0 + k) * kHeadDim, lg.c, dk);
        S::store(static_cast<T *>(p.dV) + (row0 + k) * kHeadDim, lg.c, dv);
    }
}

size_t row_bytes(fibatt_dtype dt) { return dt == FIBATT_F32 ? 256 : 128; }

// Early L2 prefetch of each CTA's first units (FIBATT_EARLY_PREFETCH=0 turns
// it off); it only pays with dependent launches.
// Bit 0: L2 prefetch of a CTA's first units before the grid-dependency wait
// (FIBATT_EARLY_PREFETCH=0: off).  Bit 1: the first unit alone at the start,
// its copies and prefetch issued before any other unit's (FIBATT_FIRST_ALONE:
// 1, the default, for the forward; 2 for both kernels; 0 off).  Measured on
// the ViT-B shape: forward 20.64 -> 20.57 us at B = 64, 19.28 -> 19.13 us
// without the diagonal, 13.72 -> 13.21 us at B = 38; the backward 1-3%
// slower (its producer's per-row pass for the second unit starts later).
int early_prefetch(bool backward) {
    static const int on = [] {
        const char *e = getenv("FIBATT_EARLY_PREFETCH");
        return (e && atoi(e) == 0) ? 0 : 1;
    }();
    const char *f = getenv("FIBATT_FIRST_ALONE");
    const int mode = f ? atoi(f) : 1;
    const bool alone = backward ? mode == 2 : mode >= 1;
    return (on && pdl_enabled() ? 1 : 0) | (alone ? 2 : 0);
}

// Snake order of the forward's waves (FIBATT_FWD_SNAKE=0 turns it off; read
// per call, so a test can compare both orders in one process).
static int fwd_snake() {
    const char *e = getenv("FIBATT_FWD_SNAKE");
    return (e && atoi(e) == 0) ? 0 : 1;
}

// The same for the resident backward (FIBATT_BWD_SNAKE=0 turns it off).
static int bwd_snake() {
    const char *e = getenv("FIBATT_BWD_SNAKE");
    return (e && atoi(e) == 0) ? 0 : 1;
}

int g_sm_count[64] = {0};
size_t g_fwd_smem_set[32][64] = {{0}};
size_t g_bwd_smem_set[16][64] = {{0}};

int sm_count(int dev) {
    if (dev < 0 || dev >= 64) return 148;
    if (!g_sm_count[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = n > 0 ? n : 148;
    }
    return g_sm_count[dev];
}

// Largest K/V window over every head and chunk.
int window_cap(const TableArg &tab, int qsplit, int chunk) {
    int cap = 1;
    for (int h = 0; h < tab.H; ++h) {
        const int t0 = tab.start[h], t1 = tab.start[h + 1];
        if (t1 == t0) continue;
        for (int c = 0; c < qsplit; ++c) {
            const int q0 = c * chunk, q1 = std::min(tab.N, q0 + chunk);
            if (q1 <= q0) continue;
            cap = std::max(cap, std::min(tab.N, q1 + tab.off[t1 - 1]) - std::max(0, q0 + tab.off[t0]));
        }
    }
    return cap;
}

}  // namespace

// Plan of the pipelined resident forward; false when not even one stage fits
// in shared memory (the generic kernel is used then).
bool plan_fwd_resident(const TableArg &tab, int B, fibatt_dtype dt, ResidentPlan *pl) {
    const int N = tab.N;
    const size_t RB = row_bytes(dt);
    const size_t budget = 210 * 1024;
    int dev = 0;
    cudaGetDevice(&dev);
    const int sms = sm_count(dev);
    // two lanes per row, one offset per step, measured fastest on the ViT-B
    // shapes with whole-head units (tuning overrides below)
    int G = 2, unroll = 1, maxt = 1024;
    if (const char *e = getenv("FIBATT_LANES")) G = atoi(e) == 2 ? 2 : 4;
    if (G == 2) maxt = 512;
    if (const char *e = getenv("FIBATT_UNROLL")) unroll = atoi(e) == 1 ? 1 : 2;
    if (const char *e = getenv("FIBATT_FWD_THREADS")) maxt = atoi(e) == 768 ? 768 : (atoi(e) == 512 ? 512 : 1024);
    if (G == 4) maxt = 1024;
    if (tab.global0) {   // the global-token kernels exist in the two-lane, 512-thread shape only
        G = 2;
        maxt = 512;
        if (!getenv("FIBATT_UNROLL")) unroll = 2;
    }
    const int R = 32 / G;                                  // rows per warp round
    const int maxw = maxt / 32;
    // Query chunks of a multiple of R rows.  Whole heads when there are at
    // least as many heads as SMs (each K/V window is then loaded once and a
    // unit's rounds fill the CTA's warps), else enough chunks to give every
    // SM a unit; and a ring of at least two stages.
    int qsplit = 1;
    const char *env = getenv("FIBATT_QSPLIT");
    if (env) {
        qsplit = std::max(1, atoi(env));
    } else {
        const long units = (long)B * tab.H;
        while (qsplit < 64 && units * qsplit < sms && (N + qsplit) / (qsplit + 1) >= 32) ++qsplit;
    }
    // Smallest possible stage (one round of rows): if even that does not fit,
    // the windows are too wide for this kernel.
    {
        const int qs_min = (N + R - 1) / R;
        const size_t smallest = (size_t)R * RB + 2 * (size_t)window_cap(tab, qs_min, R) * RB + 2 * RB;
        if (smallest > budget) return false;
    }
    int chunk = 0, kv_cap = 0;
    size_t stage = 0;
    // grow the split geometrically until two stages fit (or rows run out)
    for (;; qsplit = std::max(qsplit + 1, qsplit * 5 / 4)) {
        chunk = ((N + qsplit - 1) / qsplit + R - 1) / R * R;
        const int qs = (N + chunk - 1) / chunk;
        kv_cap = window_cap(tab, qs, chunk);
        stage = ((size_t)chunk * RB + 2 * (size_t)kv_cap * RB + (tab.global0 ? 2 * RB : 0) + 127) / 128 * 128;
        if (env || 2 * stage <= budget || chunk <= R) {
            qsplit = qs;
            break;
        }
    }
    int stages = (int)std::min<size_t>(kMaxStages, budget / stage);
    if (stages < 1) return false;
    if (const char *e = getenv("FIBATT_STAGES")) stages = std::max(1, std::min(stages, atoi(e)));
    // consumer groups: at most two (the kernel's release-then-full wait needs
    // groups <= 2, or stages a multiple of groups), and two only when a
    // unit's rounds leave warps for a second group; one group keeps a whole
    // stage of lead on every load
    const int rounds = chunk / R;
    int groups = stages >= 2 && 2 * rounds <= maxw - 1 ? 2 : 1;
    if (const char *e = getenv("FIBATT_GROUPS")) groups = std::max(1, std::min(2, atoi(e)));
    int gwarps = std::max(1, std::min(rounds, (maxw - 1) / groups));
    if (const char *e = getenv("FIBATT_FWD_GWARPS")) gwarps = std::max(1, std::min(gwarps, atoi(e)));
    int prefetch = 0;   // L2 warming of later units measured slower: off by default
    if (const char *e = getenv("FIBATT_PREFETCH")) prefetch = std::max(0, std::min(8, atoi(e)));
    pl->prefetch = prefetch;
    pl->lanes = G;
    pl->unroll = unroll;
    pl->maxt = maxt;
    pl->qsplit = qsplit;
    pl->chunk = chunk;
    pl->kv_cap = kv_cap;
    pl->stages = stages;
    pl->groups = groups;
    pl->gwarps = gwarps;
    pl->stage_bytes = stage;
    pl->threads = 32 * (1 + groups * gwarps);
    const long units = (long)B * tab.H * qsplit;
    pl->grid = (int)std::min<long>(units, sms);
    const long left = units > pl->grid ? units % pl->grid : 0;   // units of the last, partial wave
    // With the global first token and whole-head units, row 0 of every head
    // is computed inside its unit (fused_row0), or, for the last wave's
    // pieces, inside the piece that holds query 0 (which then stages every
    // key row of its head).  That needs every head's table non-empty (so that
    // a whole unit stages all N key rows) and room for a partial-state slot
    // per stage.
    bool staged_all = true;
    for (int h = 0; h < tab.H; ++h) staged_all = staged_all && tab.start[h + 1] > tab.start[h];
    pl->fuse_row0 = tab.global0 && qsplit == 1 && staged_all && kv_cap >= N;
    if (const char *e = getenv("FIBATT_GT_FUSE"))   // 0: never (the dense row kernel runs after)
        pl->fuse_row0 = pl->fuse_row0 && atoi(e) != 0;
    const size_t slot_bytes = (size_t)gwarps * 33 * sizeof(float2);   // one partial slot per stage
    if (pl->fuse_row0)
        while (stages > 2 && (stage + slot_bytes) * stages > budget) pl->stages = --stages;
    if (pl->fuse_row0 && (stage + slot_bytes) * stages > budget) pl->fuse_row0 = 0;
    pl->smem = (stage + (pl->fuse_row0 ? slot_bytes : 0)) * stages;
    // cut the units of the last, partial wave into single rounds (at most as
    // many pieces as there are CTAs)
    pl->n_keep = (int)units;
    pl->qsub = 1;
    pl->sub_rows = chunk;
    const char *st = getenv("FIBATT_SPLIT_TAIL");
    if (left > 0 && !(st && atoi(st) == 0)) {
        const int qsub = (int)std::max<long>(1, std::min<long>(chunk / R, pl->grid / left));
        if (qsub > 1) {
            pl->n_keep = (int)(units - left);
            pl->qsub = qsub;
            pl->sub_rows = ((chunk + qsub - 1) / qsub + R - 1) / R * R;
        }
    }
    return true;
}

template <typename T, int G, int UNROLL, int MAXT, bool GT = false>
static cudaError_t fwd_resident(const FwdArgs &a, const ResidentPlan &pl) {
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = fwd_pipe_kernel<T, G, UNROLL, MAXT, GT>;
    const int ti = (GT ? 16 : 0) + (std::is_same<T, float>::value ? 0 : 8) + (G == 2 ? 0 : 4) +
                   (UNROLL == 2 ? 0 : 2) + (MAXT == 1024 ? 0 : (MAXT == 768 ? 1 : 0));
    if (dev >= 0 && dev < 64 && g_fwd_smem_set[ti][dev] < pl.smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (e != cudaSuccess) return e;
        g_fwd_smem_set[ti][dev] = pl.smem;
    }
    const int n_reg = a.B * a.tab->H * pl.qsplit;
    PipeParams p{a.Q, a.K, a.V, a.O, a.LSE, a.scale * kLog2e, pl.qsplit, pl.chunk, pl.kv_cap,
                 pl.n_keep + (n_reg - pl.n_keep) * pl.qsub, pl.stages, pl.groups, pl.gwarps,
                 (uint32_t)pl.stage_bytes, pl.prefetch, pl.n_keep, pl.qsub, pl.sub_rows, early_prefetch(false),
                 fwd_snake(), pl.fuse_row0};
    const cudaError_t e =
        launch_kernel(kern, dim3(pl.grid), dim3(pl.threads), pl.smem, a.stream, pdl_enabled(), *a.tab, p);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
static cudaError_t fwd_resident_dispatch(const FwdArgs &a, const ResidentPlan &pl) {
    if (a.tab->global0)   // the plan keeps the default shapes for it
        return pl.lanes == 4 ? fwd_resident<T, 4, 2, 1024, true>(a, pl)
                             : (pl.unroll == 2 ? fwd_resident<T, 2, 2, 512, true>(a, pl)
                                               : fwd_resident<T, 2, 1, 512, true>(a, pl));
    if (pl.lanes == 4) return pl.unroll == 2 ? fwd_resident<T, 4, 2, 1024>(a, pl) : fwd_resident<T, 4, 1, 1024>(a, pl);
    if (pl.maxt == 768) return pl.unroll == 2 ? fwd_resident<T, 2, 2, 768>(a, pl) : fwd_resident<T, 2, 1, 768>(a, pl);
    return pl.unroll == 2 ? fwd_resident<T, 2, 2, 512>(a, pl) : fwd_resident<T, 2, 1, 512>(a, pl);
}

// Plan of the resident backward: the whole head's Q, K, V, dO in one stage,
// plus a P/dS scratch of max_count x N floats each.  False when one stage and
// the scratch do not fit.
bool plan_bwd_resident(const TableArg &tab, int B, fibatt_dtype dt, ResidentPlan *pl) {
    const int N = tab.N;
    const size_t RB = row_bytes(dt);
    const size_t budget = 218 * 1024;
    int dev = 0;
    cudaGetDevice(&dev);
    const int sms = sm_count(dev);
    // two lanes per row for bf16 (fewer shuffles and less per-pair scalar
    // work than four; measured faster), four for fp32 rows (two would spill)
    int G = dt == FIBATT_F32 ? 4 : 2;
    if (const char *e = getenv("FIBATT_BWD_LANES")) G = atoi(e) == 2 ? 2 : 4;
    if (dt == FIBATT_F32 || tab.global0) G = dt == FIBATT_F32 ? 4 : 2;   // global token: default shape only
    const int R = 32 / G;
    int maxt = 512;
    if (const char *e = getenv("FIBATT_BWD_THREADS")) maxt = atoi(e) == 1024 ? 1024 : 512;
    if (G == 2 || tab.global0) maxt = 512;
    const int maxw = maxt / 32;
    const size_t stage = (4 * (size_t)N * RB + 2 * (size_t)N * sizeof(float) + 127) / 128 * 128;
    const size_t scratch = (2 * (size_t)std::max(1, tab.max_count) * N * 4 + 127) / 128 * 128;
    int stages = stage * 2 + scratch <= budget ? 2 : (stage + scratch <= budget ? 1 : 0);
    if (const char *e = getenv("FIBATT_STAGES")) stages = std::min(stages, std::max(1, atoi(e)));
    if (stages < 1) return false;
    const int rounds = (N + R - 1) / R;
    pl->lanes = G;
    pl->unroll = 1;
    pl->maxt = maxt;
    pl->prefetch = 0;
    pl->qsplit = 1;
    pl->chunk = N;
    pl->kv_cap = N;
    pl->stages = stages;
    pl->groups = 1;
    pl->gwarps = std::max(1, std::min(rounds, maxw - 1));
    pl->grid = (int)std::min<long>((long)B * tab.H, sms);
    pl->stage_bytes = stage;
    pl->smem = stage * stages + scratch;
    // The partial last wave: its units cut into pieces of one or two rounds
    // (each run by 2 or 4 warps of a CTA, phase B recomputing P and dS) when
    // the pieces fit in one wave of CTAs; otherwise whole units.
    const int units = B * tab.H;
    const int left = units % pl->grid;
    pl->n_keep = units;
    pl->qsub = 1;       // pieces per unit
    pl->sub_rows = rounds;   // rounds per piece
    bool pieces = left > 0 && units > pl->grid;
    if (const char *e = getenv("FIBATT_BWD_PIECES")) pieces = pieces && atoi(e) != 0;
    pl->split_off = 0;
    pl->piece_par = 0;
    if (pieces) {
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        const size_t static_smem = 2048 + sizeof(int) * kMaxEntries;   // barriers + offsets, rounded up
        // one-round pieces: the partial dQ rows of warps 1 .. kPieceA-1, then (if there is room) the
        // round's (P, dS), in the unit scratch, which pieces use for nothing else
        const size_t pa_bytes = (size_t)(kPieceA - 1) * R * kHeadDim * sizeof(float);
        const size_t pw_bytes = (size_t)R * std::max(1, tab.max_count) * 8;   // one round's (P, dS)
        // the fewest rounds per piece whose pieces fit in one wave (up to
        // gwarps / 2: each round takes a phase-A and a phase-B warp); ViT-B
        // shape, B = 256 (32 units in the last wave, four-round pieces):
        // 182.2 -> 179.2 us against whole units
        int max_pr = pl->gwarps / 2;
        if (const char *e = getenv("FIBATT_BWD_PIECE_ROUNDS")) max_pr = std::max(1, std::min(max_pr, atoi(e)));
        for (int pr = 1; pr <= max_pr; ++pr) {
            const int np = (rounds + pr - 1) / pr;
            // one-round pieces over kPieceA + kPieceB warps
            bool par = pr == 1 && pl->gwarps >= kPieceA + kPieceB && scratch >= pa_bytes;
            if (const char *e = getenv("FIBATT_BWD_PIECE_PAR")) par = par && atoi(e) != 0;
            const bool pw_in_scratch = par && scratch >= pa_bytes + pw_bytes;
            // global token: one-round pieces only, with spare warps for the dense parts
            if (tab.global0 && !(par && pl->gwarps > kPieceA + kPieceB)) continue;
            // the (P, dS) area of each phase-B warp, unless it went to the scratch
            const size_t area = pw_in_scratch ? 0 : (size_t)pr * R * std::max(1, tab.max_count) * 8;
            if ((long)left * np <= pl->grid && 2 * pr <= pl->gwarps &&
                pl->smem + area + static_smem <= (size_t)optin) {
                pl->n_keep = units - left;
                pl->qsub = np;
                pl->sub_rows = pr;
                pl->split_off = pw_in_scratch ? stage * stages + pa_bytes : pl->smem;
                pl->smem += area;
                pl->piece_par = par;
                break;
            }
        }
    }
    // Global first token: the dense row 0 and column 0 inside each unit
    // (gt_fused_weights, gt_fused_sums) when their weights and partial sums
    // fit beside the stages; otherwise the row and column kernels.
    pl->fuse_row0 = 0;
    pl->gt_off = 0;
    if (tab.global0) {
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        const size_t static_smem = 2048 + sizeof(int) * kMaxEntries;   // barriers, starts + offsets, rounded up
        const size_t gt_bytes = ((4 * (size_t)N + 3 * kGtParts * kHeadDim) * sizeof(float) + 127) / 128 * 128;
        bool fuse = pl->smem + gt_bytes + static_smem <= (size_t)optin;
        if (const char *e = getenv("FIBATT_GT_FUSE")) fuse = fuse && atoi(e) != 0;
        if (fuse) {
            pl->fuse_row0 = 1;
            pl->gt_off = pl->smem;
            pl->smem += gt_bytes;
        } else if (pl->qsub > 1) {   // the pieces compute the dense parts only when fused: whole units
            pl->n_keep = units;
            pl->qsub = 1;
            pl->sub_rows = rounds;
            pl->split_off = 0;
            pl->piece_par = 0;
        }
    }
    pl->threads = 32 * (1 + pl->gwarps);
    return true;
}

template <typename T>
static cudaError_t bwd_resident(const BwdArgs &a, const ResidentPlan &pl, int units) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int ti = std::is_same<T, float>::value ? 0 : 1;
    const bool gt = a.tab->global0 != 0;
    decltype(&bwd_pipe_kernel<T, 4, 512>) kern;
    if constexpr (std::is_same<T, float>::value)   // fp32 rows: four lanes per row only
        kern = gt ? bwd_pipe_kernel<T, 4, 512, true>
                  : (pl.threads > 512 ? bwd_pipe_kernel<T, 4, 1024> : bwd_pipe_kernel<T, 4, 512>);
    else
        kern = gt ? (pl.lanes == 2 ? bwd_pipe_kernel<T, 2, 512, true> : bwd_pipe_kernel<T, 4, 512, true>)
                  : pl.lanes == 2 ? bwd_pipe_kernel<T, 2, 512>
                                  : (pl.threads > 512 ? bwd_pipe_kernel<T, 4, 1024> : bwd_pipe_kernel<T, 4, 512>);
    const int ki = ti * 8 + (gt ? 4 : 0) + (pl.lanes == 2 ? 2 : (pl.threads > 512 ? 1 : 0));
    if (dev >= 0 && dev < 64 && g_bwd_smem_set[ki][dev] < pl.smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (e != cudaSuccess) return e;
        g_bwd_smem_set[ki][dev] = pl.smem;
    }
    const int items = pl.n_keep + (units - pl.n_keep) * pl.qsub;
    BwdParams p{a.Q, a.K, a.V, a.O, a.dO, a.LSE, a.dQ, a.dK, a.dV, a.scale, a.scale * kLog2e,
                items, pl.stages, pl.gwarps, (uint32_t)pl.stage_bytes,
                (uint32_t)(pl.stage_bytes * pl.stages), std::max(1, (int)a.tab->max_count), a.gw, early_prefetch(true),
                pl.n_keep, pl.qsub, pl.sub_rows, (uint32_t)pl.split_off, bwd_snake(), pl.piece_par,
                pl.fuse_row0, (uint32_t)pl.gt_off};
    const cudaError_t e =
        launch_kernel(kern, dim3(pl.grid), dim3(pl.threads), pl.smem, a.stream, pdl_enabled(), *a.tab, p);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Units [bh0, bh0 + count); the scratch a.Dws holds `count` units' weights.
template <typename T, int G, int W = kFlatWarps, bool GT = false>
static cudaError_t bwd_flat(const BwdArgs &a, int bh0, int count) {
    constexpr int R = 32 / G;
    const TableArg &tab = *a.tab;
    BwdParams p{a.Q, a.K, a.V, a.O, a.dO, a.LSE, a.dQ, a.dK, a.dV, a.scale, a.scale * kLog2e,
                a.B * tab.H, 0, 0, 0, 0, std::max(1, (int)tab.max_count), a.gw, 0, a.B * tab.H, 1, 1, 0, 0, 0};
    const dim3 grid((unsigned)count, (unsigned)((tab.N + R * W - 1) / (R * W)));
    const bool pdl = pdl_enabled();
    float *scr = a.Dws;   // unit bh0 + x at x * 2 * max_count * N
    cudaError_t e =
        launch_kernel(bwd_flat_a_kernel<T, G, W, GT>, grid, dim3(W * 32), 0, a.stream, pdl, tab, p, scr, bh0);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_kernel(bwd_flat_b_kernel<T, G, W, GT>, grid, dim3(W * 32), 0, a.stream, pdl, tab, p,
                      static_cast<const float *>(scr), bh0);
    count_launches(2);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The streaming kernels (stream.cu) need 32-byte aligned rows (256-bit
// accesses); FIBATT_STREAM=0 selects the kernels below for every call.
static bool use_stream(const TableArg &tab, std::initializer_list<const void *> ptrs) {
    const char *e = getenv("FIBATT_STREAM");
    (void)tab;
    if (e && atoi(e) == 0) return false;
    for (const void *q : ptrs)
        if (reinterpret_cast<uintptr_t>(q) % 32 != 0) return false;
    return true;
}

bool flat_fwd_fuses_global(const FwdArgs &a) {
    return a.tab->global0 && stream_row0_in_grid(*a.tab) && use_stream(*a.tab, {a.Q, a.K, a.V, a.O});
}

bool flat_bwd_fuses_global(const BwdArgs &a) {
    return a.tab->global0 && use_stream(*a.tab, {a.Q, a.K, a.V, a.O, a.dO, a.dQ, a.dK, a.dV});
}

cudaError_t launch_bwd_flat(const BwdArgs &a) {
    if (use_stream(*a.tab, {a.Q, a.K, a.V, a.O, a.dO, a.dQ, a.dK, a.dV})) return launch_bwd_stream(a);
    int G = 4;
    if (const char *e = getenv("FIBATT_FLAT_LANES")) G = atoi(e) == 2 ? 2 : 4;
    const int units = a.B * a.tab->H;
    if (a.tab->global0)
        return a.dtype == FIBATT_F32 ? bwd_flat<float, 4, kFlatWarps, true>(a, 0, units)
                                     : bwd_flat<__nv_bfloat16, 4, kFlatWarps, true>(a, 0, units);
    if (a.dtype == FIBATT_F32) return bwd_flat<float, 4>(a, 0, units);
    return G == 2 ? bwd_flat<__nv_bfloat16, 2>(a, 0, units) : bwd_flat<__nv_bfloat16, 4>(a, 0, units);
}

size_t flat_bwd_scratch_bytes(const TableArg &tab, int B) {
    return std::max(stream_bwd_scratch_bytes(tab, B),
                    (size_t)B * tab.H * 2 * std::max(1, (int)tab.max_count) * tab.N * sizeof(float));
}

cudaError_t launch_bwd_resident(const BwdArgs &a, const ResidentPlan &pl) {
    const int units = a.B * a.tab->H;
    return a.dtype == FIBATT_F32 ? bwd_resident<float>(a, pl, units) : bwd_resident<__nv_bfloat16>(a, pl, units);
}

template <typename T, int G, int W = kFlatWarps, int U = 2, bool GT = false>
static cudaError_t fwd_flat(const FwdArgs &a) {
    constexpr int R = 32 / G;
    const TableArg &tab = *a.tab;
    PipeParams p{};
    p.Q = a.Q;
    p.K = a.K;
    p.V = a.V;
    p.O = a.O;
    p.LSE = a.LSE;
    p.scale_log2 = a.scale * kLog2e;
    const dim3 grid((unsigned)(a.B * tab.H), (unsigned)((tab.N + R * W - 1) / (R * W)));
    const cudaError_t e = launch_kernel(fwd_flat_kernel<T, G, U, W, GT>, grid, dim3(W * 32), 0, a.stream,
                                        pdl_enabled(), tab, p);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_fwd_flat(const FwdArgs &a) {
    if (use_stream(*a.tab, {a.Q, a.K, a.V, a.O})) return launch_fwd_stream(a);
    int G = 4;   // four lanes per row: more warps in flight to cover global-load latency (measured faster)
    if (const char *e = getenv("FIBATT_FLAT_LANES")) G = atoi(e) == 2 ? 2 : 4;
    if (a.tab->global0)
        return a.dtype == FIBATT_F32 ? fwd_flat<float, 4, kFlatWarps, 2, true>(a)
                                     : fwd_flat<__nv_bfloat16, 4, kFlatWarps, 2, true>(a);
    if (a.dtype == FIBATT_F32) return G == 4 ? fwd_flat<float, 4>(a) : fwd_flat<float, 2>(a);
    return G == 4 ? fwd_flat<__nv_bfloat16, 4>(a) : fwd_flat<__nv_bfloat16, 2>(a);
}

cudaError_t launch_fwd_resident(const FwdArgs &a, const ResidentPlan &pl) {
    return a.dtype == FIBATT_F32 ? fwd_resident_dispatch<float>(a, pl) : fwd_resident_dispatch<__nv_bfloat16>(a, pl);
}

// Read (and optionally clear) the device error word of the current device.
FIBATT_DEFINE_ERROR_READER(read_error_resident, "resident.cu")

// The device error words of every kernel file, OR-ed (and cleared).
cudaError_t read_device_error(unsigned *code, bool clear) {
    cudaError_t (*const readers[])(unsigned *, bool) = {read_error_resident, read_error_stream, read_error_generic,
                                                        read_error_global_token};
    *code = 0;
    for (auto r : readers) {
        unsigned c = 0;
        const cudaError_t e = r(&c, clear);
        if (e != cudaSuccess) return e;
        *code |= c;
    }
    return cudaSuccess;
}

}  // namespace fibatt
