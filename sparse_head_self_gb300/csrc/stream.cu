// Streaming Fibottention kernels: the banded forward and backward for heads
// whose key windows do not fit in shared memory (long sequences with wide
// windows, e.g. 8 video frames of 196 patches, or 128 x 128 patches).
//
// Every row comes straight from global memory through L1/L2.  A row is
// 64 elements; G lanes share it, lane `sub` owning one contiguous run of
// 64/G dims, read with 256-bit loads (ld.global.nc.v8.b32) so that the G
// lanes of a row cover the whole row in full 32-byte sectors.  (Slices whose
// 16-byte pieces alternate between lanes touch every sector twice per row.)
// Blocks are numbered head-major: all row blocks of one (b, h) run next to
// each other, so the K/V rows the resident blocks reach -- one head's, a few
// MB -- stay in L2 instead of the rows of every head at once.
//
// Forward (Fibottention Sec. 3; README Algorithm 3 restricted to the
// support): query row j, offsets off[t] of its head, key k = j + off[t]:
//   s = scale <q_j, k_k>, online softmax in log2 units, O_j = sum P v_k / l,
//   LSE_j = ln l + max.
// Backward, three launches, no atomics:
//   LSE_j log2(e) and D_j = <dO_j, O_j> for every row;
//   key-centric (key k stationary in registers; queries j = k + off[t], the
//   table being symmetric): P = exp(s - LSE_j), dS = P (<dO_j, v_k> - D_j),
//   dV_k = sum P dO_j, dK_k = scale sum dS q_j, and dS of each pair into a
//   scratch indexed by the query's own table entry;
//   query-centric: dQ_j = scale sum dS k_k over the same pairs.
// So the backward reads q, dO (key pass) and k (query pass) per pair: three
// rows instead of four, and one fp32 of scratch each way.
#include <algorithm>
#include <cstdlib>
#include <type_traits>

#include <cuda.h>

#include "fibatt_internal.h"
#include "row_math.cuh"
#include "row_run.cuh"
#include "dense_row.cuh"
#include "tma_common.cuh"

namespace fibatt {
namespace {

// Register budgets (bf16): the forward at 64 registers (32 warps per SM;
// video 36.7 -> 34.4 us, 128 x 128 image 156.4 -> 149.8 us against its own
// choice of 78; 48 registers spill: 43.4 / 184.3 us), the key pass at 80 (24
// warps; 100.2 -> 98.2 and 444.0 -> 429.8 us against 94; 64 spill: 136.0 /
// 626.2 us); with the global token the key pass takes 96 (20 warps; 80
// spill: 128 x 128 image 539 -> 582 us); the query pass 48 (40 warps; 97.4 ->
// 95.0 and 428.1 -> 413.2 us against 52; 40 spill: 96.9 / 421.5 us).
//
// Warps per block (consecutive row groups of one head).  Larger blocks
// raise the L1 hits between neighbouring offsets (the 128 x 128 image shape's
// forward: L2-to-SM bytes 2.80 -> 2.44 GB with 8 warps) but hold fewer warps
// per SM at these register counts, which costs more: 4 measured fastest.
constexpr int kStreamWarps = 4;

// Entries [tb, te) of the head's ascending offsets off[0, cnt) that reach a
// row in [0, N) from at least one of the rows [first, last]: the others are
// dropped for the whole warp.  Warp-collective.
__device__ __forceinline__ void trim(const int *off, int cnt, int N, int first, int last, int &tb, int &te) {
    const int lane = threadIdx.x & 31;
    int below = 0, above = 0;
    for (int base = 0; base < cnt; base += 32) {
        const int t = base + lane;
        const bool e = t < cnt;
        const int o = e ? off[t] : 0;
        below += __popc(__ballot_sync(kFullMask, e && last + o < 0));
        above += __popc(__ballot_sync(kFullMask, e && first + o >= N));
    }
    tb = below;
    te = max(tb, cnt - above);
}

// Global first token: bit i set when the band of row first + i (i < nrows
// <= 32) reaches position 0, i.e. offset -(first + i) is among off[0, cnt)
// (the tables are symmetric, so the same bit says whether +(first + i) is).
// Warp-collective: every lane takes part, whatever its row.
__device__ __forceinline__ unsigned band_to_zero(const int *off, int cnt, int first, int nrows) {
    const int lane = threadIdx.x & 31;
    unsigned hit = 0;
    for (int t = 0; t < cnt; t += 32) {
        const int i = t + lane < cnt ? -off[t + lane] - first : -1;
        hit |= __reduce_or_sync(kFullMask, i >= 0 && i < nrows ? 1u << i : 0u);
    }
    return hit;
}

// Copy of head h's offsets into shared memory; returns the count.
__device__ __forceinline__ int load_offsets(const TableArg &tab, int h, int *s_off) {
    const int t0 = tab.start[h], cnt = tab.start[h + 1] - t0;
    for (int t = threadIdx.x; t < cnt; t += blockDim.x) s_off[t] = tab.off[t0 + t];
    __syncthreads();
    return cnt;
}

// L2 prefetch (a hint: nothing waits on it) of the row windows the block's
// rows [first, first + rows) reach through each table entry, clipped to
// [0, N): rows first + off[t] ... of the head whose row 0 is at `base`, `rb`
// bytes per row; one entry per thread.  Every row a block reads is then on
// its way to L2 before the block's first use of it, instead of each warp
// meeting the compulsory misses of its own loads one step at a time.
__device__ __forceinline__ void prefetch_windows(const uint8_t *base, int rb, const int *off, int cnt, int N,
                                                 int first, int rows) {
    for (int t = threadIdx.x; t < cnt; t += blockDim.x) {
        const int lo = max(0, first + off[t]), hi = min(N, first + rows + off[t]);
        if (hi > lo)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + (size_t)lo * rb),
                         "r"((uint32_t)(hi - lo) * (uint32_t)rb)
                         : "memory");
    }
}

struct StreamParams {
    const void *Q, *K, *V, *O, *dO;
    const float *LSE;
    void *Out, *dK, *dV;   // forward: O; backward: dQ (query pass) or nothing
    float *LSEout;         // forward: LSE
    float2 *LD;            // backward: (LSE_j log2(e), D_j) per row
    float *scr;            // backward: dS per (b, h, table entry, query row), rows of `ns` floats
    int ns;                // scratch row stride (N rounded up to 32: 128-byte rows)
    int prefetch;          // L2 prefetch of the block's row windows: 1 forward, 2 key pass, 4 query pass
    float *gw;             // global first token, backward: dS_j0 of column 0, a row of `ns` floats per (b, h)
    int row0_heads;        // global token: B * H when the dense blocks (forward: rows 0; key pass: dQ_0 and
                           // column 0) run in the kernel's own grid ahead of the banded blocks, else 0
    float scale, scale_log2;
    int nblk;              // row blocks per (b, h)
    int max_count;         // scratch entries per (b, h)
};

// Running maximum start: finite, so a masked score (-inf) gives weight 0.
constexpr float kMInit = -1.0e30f;

// ------------------------------------------------------------------ forward

// Rows [first, first + 32/G) of head bh (one warp; first < N).
template <typename T, int G, bool W16, bool GT>
__device__ __forceinline__ void fwd_stream_rows(const TableArg &tab, const StreamParams &p, const int *s_off, int cnt,
                                                int bh, int first) {
    using S = Run<T, G>;
    constexpr int R = 32 / G;
    constexpr int RB = S::kRowBytes;
    const int N = tab.N;
    const int lane = threadIdx.x & 31, sub = lane % G;
    const int last = min(N, first + R) - 1;
    const bool valid = first + lane / G < N;
    const int j = valid ? first + lane / G : last;
    int tb, te;
    trim(s_off, cnt, N, first, last, tb, te);

    const size_t row0 = (size_t)bh * N;
    const uint8_t *gK = static_cast<const uint8_t *>(p.K) + row0 * RB + sub * S::kBytes;
    const uint8_t *gV = static_cast<const uint8_t *>(p.V) + row0 * RB + sub * S::kBytes;
    S q;
    q.load(static_cast<const uint8_t *>(p.Q) + (row0 + j) * RB + sub * S::kBytes);
    float2 acc[S::kPairs];
#pragma unroll
    for (int i = 0; i < S::kPairs; ++i) acc[i] = make_float2(0.f, 0.f);
    float m = kMInit, l = 0.f, lt = 0.f;   // lt: the weights as they entered acc (bf16-rounded with W16)
    const float sl2 = p.scale_log2;
    auto raise = [&](float s) {
        if (s > m + 8.f) {   // rare: p = 2^(s - m) <= 2^8 between raises
            const float a = fast_exp2(m - s);
            l *= a;
            lt *= a;
#pragma unroll
            for (int i = 0; i < S::kPairs; ++i) acc[i] = mul2(acc[i], make_float2(a, a));
            m = s;
        }
    };
    auto add = [&](const S &v, float pr) {
        l += pr;
        if constexpr (W16 && S::kBf16) {
            const uint32_t p2 = bf16x2_splat(pr);
            lt += __uint_as_float(p2 << 16);
            v.axpy_p2(p2, acc);
        } else {
            v.axpy(pr, acc);
        }
    };
    int t = tb;
    for (; t + 1 < te; t += 2) {   // two offsets per step: four row loads in flight
        const int k0 = j + s_off[t], k1 = j + s_off[t + 1];
        const bool in0 = valid && k0 >= 0 && k0 < N, in1 = valid && k1 >= 0 && k1 < N;
        const size_t c0 = (size_t)min(max(k0, 0), N - 1) * RB, c1 = (size_t)min(max(k1, 0), N - 1) * RB;
        S ka, kb, va, vb;
        ka.load(gK + c0);
        kb.load(gK + c1);
        va.load(gV + c0);
        vb.load(gV + c1);
        float s0 = lanes_sum<G>(q.dot(ka)) * sl2, s1 = lanes_sum<G>(q.dot(kb)) * sl2;
        s0 = in0 ? s0 : -INFINITY;
        s1 = in1 ? s1 : -INFINITY;
        raise(fmaxf(s0, s1));
        add(va, fast_exp2(s0 - m));
        add(vb, fast_exp2(s1 - m));
    }
    if (t < te) {
        const int k0 = j + s_off[t];
        const bool in0 = valid && k0 >= 0 && k0 < N;
        const size_t c0 = (size_t)min(max(k0, 0), N - 1) * RB;
        S ka, va;
        ka.load(gK + c0);
        va.load(gV + c0);
        float s0 = lanes_sum<G>(q.dot(ka)) * sl2;
        s0 = in0 ? s0 : -INFINITY;
        raise(s0);
        add(va, fast_exp2(s0 - m));
    }
    if constexpr (GT) {
        // global first token: key 0 for every row j >= 1 whose band misses
        // it (row 0 itself is dense: fwd_row0_block)
        const unsigned band0 = band_to_zero(s_off, cnt, first, last - first + 1);
        const bool need = valid && j >= 1 && !((band0 >> (j - first)) & 1u);
        S k0r, v0r;
        k0r.load(gK);
        v0r.load(gV);
        float s0 = lanes_sum<G>(q.dot(k0r)) * sl2;
        s0 = need ? s0 : -INFINITY;
        raise(s0);
        add(v0r, fast_exp2(s0 - m));
    }
    if (!valid || (GT && j == 0)) return;
    const float ln = (W16 && S::kBf16) ? lt : l;
    S::store(static_cast<uint8_t *>(p.Out) + (row0 + j) * RB + sub * S::kBytes, acc, ln > 0.f ? __frcp_rn(ln) : 0.f);
    if (sub == 0) p.LSEout[row0 + j] = l > 0.f ? (m + fast_log2(l)) * kLn2 : -INFINITY;
}

// Global first token: the dense row 0 of head blockIdx.x, one block per
// head over every key.  Launched ahead of the banded blocks in the same
// grid (fwd_stream_kernel takes blocks past the heads), so these longer
// blocks start first and run beside the banded ones.
template <typename T, int W>
__device__ __forceinline__ void fwd_row0_block(const TableArg &tab, const StreamParams &p, int bh) {
    constexpr int RB = Run<T, 4>::kRowBytes;
    __shared__ DenseRowSmem<W> sm;
    const int N = tab.N;
    const uint8_t *head = static_cast<const uint8_t *>(p.Q) + (size_t)bh * N * RB;
    dense_row0_fwd<T, W, true, false>(head, static_cast<const uint8_t *>(p.K) - static_cast<const uint8_t *>(p.Q),
                                      static_cast<const uint8_t *>(p.V) - static_cast<const uint8_t *>(p.Q), 0, N,
                                      p.scale_log2, static_cast<T *>(p.Out) + (size_t)bh * N * kHeadDim,
                                      p.LSEout + (size_t)bh * N, sm);
}

template <typename T, int G, int W, bool W16, bool GT>
__global__ void __launch_bounds__(W * 32, (G == 4 && sizeof(T) == 2) ? (32 / W > 0 ? 32 / W : 1) : (16 / W > 0 ? 16 / W : 1))
fwd_stream_kernel(const __grid_constant__ TableArg tab, const StreamParams p) {
    constexpr int R = 32 / G;
    constexpr int RB = Run<T, G>::kRowBytes;
    extern __shared__ int s_off[];
    const int N = tab.N;
    int b = (int)blockIdx.x;
    if constexpr (GT) {   // the first B*H blocks: the dense rows 0 (fwd_row0_block), when in this grid
        if (b < p.row0_heads) {
            grid_dep_wait();
            grid_dep_launch();
            fwd_row0_block<T, W>(tab, p, b);
            return;
        }
        b -= p.row0_heads;
    }
    const int bh = b / p.nblk, yb = b % p.nblk;
    const int cnt = load_offsets(tab, bh % tab.H, s_off);
    if (p.prefetch & 1) {   // Q, K and V are inputs: their rows may be prefetched into L2 while
        // the previous kernel drains (L2 is the point of coherence, so the
        // loads after the wait still see what that kernel wrote)
        const size_t head = (size_t)bh * N * RB;
        const int bfirst = yb * W * R;
        prefetch_windows(static_cast<const uint8_t *>(p.K) + head, RB, s_off, cnt, N, bfirst, W * R);
        prefetch_windows(static_cast<const uint8_t *>(p.V) + head, RB, s_off, cnt, N, bfirst, W * R);
    }
    grid_dep_wait();
    grid_dep_launch();
    const int first = (yb * W + (int)(threadIdx.x >> 5)) * R;
    if (first < N) fwd_stream_rows<T, G, W16, GT>(tab, p, s_off, cnt, bh, first);   // whole warps
}

// ----------------------------------------------- forward, near window staged
//
// The table entries with |off| <= dmax reach, from a block of Tq = 8W query
// rows j0 .. j0 + Tq - 1, the key rows j0 + off[nb] .. j0 + Tq - 1 +
// off[ne - 1]: at most Tq + 2 dmax rows, shared by every near entry (the
// small Fibonacci distances lie within a few dozen rows of each other).  The
// block stages that window of K and V once in shared memory with bulk tensor
// copies (boxes of kWinBox rows, 128-byte swizzle), computes its far entries
// from global memory as fwd_stream_rows does while the copies land, then the
// near ones from the window.  The far entries read every key row once per
// pair either way; the near ones read a staged row once per block instead of
// once per pair.

constexpr int kWinRows = 256;                        // staged key (and value) rows per block
constexpr int kWinBox = 32;                          // rows per tensor copy
constexpr int kWinBytes = 2 * kWinRows * 128;        // K window, then V window

struct WinMaps {
    CUtensorMap k, v;   // K and V as [rows][64] bf16, boxes of kWinBox rows, 128-byte swizzle
};

// Rows [row, row + kWinBox) of the tensor `map` describes into shared memory
// at dst (1024-byte aligned), completion counted in bytes on `bar`; rows
// past the tensor's end arrive as zeros.
__device__ __forceinline__ void tma_rows(void *dst, const CUtensorMap *map, int row, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(smem_u32(bar))
        : "memory");
}

// The lane's 32-byte run (16-byte chunks 2 sub and 2 sub + 1) of local row
// kl of a window written with the 128-byte swizzle, under which chunk c of
// row r sits at byte 16 (c ^ (r & 7)) of the row.  In words, the same order
// as a 256-bit global load of the run.  The eight lanes of a shared-memory
// phase (two consecutive rows, four lanes each) meet eight bank groups.
__device__ __forceinline__ void win_run(const uint8_t *win, int kl, int sub, uint32_t *w) {
    if (!FIBATT_CHECKED((unsigned)kl < (unsigned)kWinRows)) kl = 0;
    const int a0 = kl * 128 + ((((2 * sub) ^ kl) & 7) << 4);
    const uint4 x = *reinterpret_cast<const uint4 *>(win + a0);
    const uint4 y = *reinterpret_cast<const uint4 *>(win + (a0 ^ 16));
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    w[4] = y.x; w[5] = y.y; w[6] = y.z; w[7] = y.w;
}

// Entries [nb, ne) of the ascending table with |off| <= dmax.  Warp-collective.
__device__ __forceinline__ void near_range(const int *off, int cnt, int dmax, int &nb, int &ne) {
    const int lane = threadIdx.x & 31;
    int below = 0, upto = 0;
    for (int base = 0; base < cnt; base += 32) {
        const int t = base + lane;
        const bool e = t < cnt;
        const int o = e ? off[t] : 0;
        below += __popc(__ballot_sync(kFullMask, e && o < -dmax));
        upto += __popc(__ballot_sync(kFullMask, e && o <= dmax));
    }
    nb = below;
    ne = max(nb, upto);
}

// Rows [first, first + 8) of head bh (one warp; first < N); the block's
// window holds key rows [wb, we) of the head for the entries [nb, ne).
template <bool W16>
__device__ __forceinline__ void fwd_window_rows(const TableArg &tab, const StreamParams &p, const int *s_off, int cnt,
                                                int bh, int first, const uint8_t *win, int wb, int we, int nb, int ne,
                                                uint64_t *bar, volatile int *abort) {
    using S = Run<__nv_bfloat16, 4>;
    constexpr int G = 4, R = 8, RB = 128;
    const int N = tab.N;
    const int lane = threadIdx.x & 31, sub = lane % G;
    const int last = min(N, first + R) - 1;
    const bool valid = first + lane / G < N;
    const int j = valid ? first + lane / G : last;
    int tb, te;
    trim(s_off, cnt, N, first, last, tb, te);

    const size_t row0 = (size_t)bh * N;
    const uint8_t *gK = static_cast<const uint8_t *>(p.K) + row0 * RB + sub * S::kBytes;
    const uint8_t *gV = static_cast<const uint8_t *>(p.V) + row0 * RB + sub * S::kBytes;
    S q;
    q.load(static_cast<const uint8_t *>(p.Q) + (row0 + j) * RB + sub * S::kBytes);
    float2 acc[S::kPairs];
#pragma unroll
    for (int i = 0; i < S::kPairs; ++i) acc[i] = make_float2(0.f, 0.f);
    float m = kMInit, l = 0.f, lt = 0.f;
    const float sl2 = p.scale_log2;
    auto raise = [&](float s) {
        if (s > m + 8.f) {
            const float a = fast_exp2(m - s);
            l *= a;
            lt *= a;
#pragma unroll
            for (int i = 0; i < S::kPairs; ++i) acc[i] = mul2(acc[i], make_float2(a, a));
            m = s;
        }
    };
    auto add = [&](const S &v, float pr) {
        l += pr;
        if constexpr (W16) {
            const uint32_t p2 = bf16x2_splat(pr);
            lt += __uint_as_float(p2 << 16);
            v.axpy_p2(p2, acc);
        } else {
            v.axpy(pr, acc);
        }
    };
    // far entries [ta, tz) from global memory, two per step
    auto far = [&](int ta, int tz) {
        int t = ta;
        for (; t + 1 < tz; t += 2) {
            const int k0 = j + s_off[t], k1 = j + s_off[t + 1];
            const bool in0 = valid && k0 >= 0 && k0 < N, in1 = valid && k1 >= 0 && k1 < N;
            const size_t c0 = (size_t)min(max(k0, 0), N - 1) * RB, c1 = (size_t)min(max(k1, 0), N - 1) * RB;
            S ka, kb, va, vb;
            ka.load(gK + c0);
            kb.load(gK + c1);
            va.load(gV + c0);
            vb.load(gV + c1);
            float s0 = lanes_sum<G>(q.dot(ka)) * sl2, s1 = lanes_sum<G>(q.dot(kb)) * sl2;
            s0 = in0 ? s0 : -INFINITY;
            s1 = in1 ? s1 : -INFINITY;
            raise(fmaxf(s0, s1));
            add(va, fast_exp2(s0 - m));
            add(vb, fast_exp2(s1 - m));
        }
        if (t < tz) {
            const int k0 = j + s_off[t];
            const bool in0 = valid && k0 >= 0 && k0 < N;
            const size_t c0 = (size_t)min(max(k0, 0), N - 1) * RB;
            S ka, va;
            ka.load(gK + c0);
            va.load(gV + c0);
            float s0 = lanes_sum<G>(q.dot(ka)) * sl2;
            s0 = in0 ? s0 : -INFINITY;
            raise(s0);
            add(va, fast_exp2(s0 - m));
        }
    };
    far(tb, min(te, nb));
    far(max(tb, ne), te);
    const int na = max(tb, nb), nz = min(te, ne);
    if (na < nz) {
        // near entries from the window (its copies were issued before the far loop)
        mbar_wait(bar, 0, abort);
        const int jw = j - wb, wl = we - wb - 1;   // key j + off at local row jw + off, clamped into [0, wl]
        const uint8_t *wV = win + kWinRows * RB;
        int t = na;
        for (; t + 1 < nz; t += 2) {
            const int k0 = j + s_off[t], k1 = j + s_off[t + 1];
            const bool in0 = valid && k0 >= 0 && k0 < N, in1 = valid && k1 >= 0 && k1 < N;
            const int l0 = min(max(jw + s_off[t], 0), wl), l1 = min(max(jw + s_off[t + 1], 0), wl);
            S ka, kb, va, vb;
            win_run(win, l0, sub, ka.w);
            win_run(win, l1, sub, kb.w);
            win_run(wV, l0, sub, va.w);
            win_run(wV, l1, sub, vb.w);
            float s0 = lanes_sum<G>(q.dot(ka)) * sl2, s1 = lanes_sum<G>(q.dot(kb)) * sl2;
            s0 = in0 ? s0 : -INFINITY;
            s1 = in1 ? s1 : -INFINITY;
            raise(fmaxf(s0, s1));
            add(va, fast_exp2(s0 - m));
            add(vb, fast_exp2(s1 - m));
        }
        if (t < nz) {
            const int k0 = j + s_off[t];
            const bool in0 = valid && k0 >= 0 && k0 < N;
            const int l0 = min(max(jw + s_off[t], 0), wl);
            S ka, va;
            win_run(win, l0, sub, ka.w);
            win_run(wV, l0, sub, va.w);
            float s0 = lanes_sum<G>(q.dot(ka)) * sl2;
            s0 = in0 ? s0 : -INFINITY;
            raise(s0);
            add(va, fast_exp2(s0 - m));
        }
    }
    if (!valid) return;
    const float ln = W16 ? lt : l;
    S::store(static_cast<uint8_t *>(p.Out) + (row0 + j) * RB + sub * S::kBytes, acc, ln > 0.f ? __frcp_rn(ln) : 0.f);
    if (sub == 0) p.LSEout[row0 + j] = l > 0.f ? (m + fast_log2(l)) * kLn2 : -INFINITY;
}

// Dynamic shared memory: up to 1 KB of alignment, the K and V windows, the
// head's offsets.
size_t window_smem_bytes(int max_count) { return 1024 + kWinBytes + sizeof(int) * (size_t)std::max(1, max_count); }

// W warps (8W query rows) per block, MINB blocks per SM.
template <int W, int MINB, bool W16>
__global__ void __launch_bounds__(W * 32, MINB)
fwd_window_kernel(const __grid_constant__ TableArg tab, const StreamParams p, const __grid_constant__ WinMaps wm) {
    constexpr int R = 8;
    extern __shared__ uint8_t w_smem[];
    __shared__ uint64_t bar;
    __shared__ int s_abort;
    uint8_t *win = w_smem + ((1024u - (smem_u32(w_smem) & 1023u)) & 1023u);
    int *s_off = reinterpret_cast<int *>(win + kWinBytes);
    const int N = tab.N;
    const int bh = (int)blockIdx.x / p.nblk, yb = (int)blockIdx.x % p.nblk;
    const int h = bh % tab.H, t0 = tab.start[h], cnt = tab.start[h + 1] - t0;
    for (int t = threadIdx.x; t < cnt; t += blockDim.x) s_off[t] = tab.off[t0 + t];
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        s_abort = 0;
    }
    __syncthreads();
    const int j0 = yb * W * R, jlast = min(N, j0 + W * R) - 1;
    int nb, ne;
    near_range(s_off, cnt, (kWinRows - W * R) / 2, nb, ne);
    int wb = 0, we = 0;
    if (nb < ne) {
        wb = max(0, j0 + s_off[nb]);
        we = min(N, jlast + s_off[ne - 1] + 1);
        if (we <= wb) nb = ne;
    }
    int nbox = nb < ne ? (we - wb + kWinBox - 1) / kWinBox : 0;   // nbox * kWinBox <= kWinRows
    if (!FIBATT_CHECKED(nbox * kWinBox <= kWinRows)) nbox = 0, nb = ne;
    grid_dep_wait();
    grid_dep_launch();
    if (threadIdx.x == 0 && nbox > 0) {
        mbar_expect_tx(&bar, (uint32_t)nbox * kWinBox * 128 * 2);
        const int y = bh * N + wb;
        for (int i = 0; i < nbox; ++i) {
            tma_rows(win + i * kWinBox * 128, &wm.k, y + i * kWinBox, &bar);
            tma_rows(win + kWinRows * 128 + i * kWinBox * 128, &wm.v, y + i * kWinBox, &bar);
        }
    }
    const int first = j0 + (int)(threadIdx.x >> 5) * R;
    if (first < N)
        fwd_window_rows<W16>(tab, p, s_off, cnt, bh, first, win, wb, we, nb, ne, &bar, &s_abort);   // whole warps
    // the copies land before the block leaves, whatever its warps did
    if (threadIdx.x == 0 && nbox > 0) mbar_drain(&bar, 0);
}

// ----------------------------------------------------------------- backward

// Per row: LSE_j log2(e) and D_j = <dO_j, O_j>, rows [0, rows).
template <typename T, int G, int W>
__global__ void __launch_bounds__(W * 32) rowdot_stream_kernel(const StreamParams p, long rows) {
    using S = Run<T, G>;
    constexpr int RB = S::kRowBytes;
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31, sub = lane % G;
    const long r = ((long)blockIdx.x * W + (threadIdx.x >> 5)) * (32 / G) + lane / G;
    const long rc = r < rows ? r : rows - 1;
    S o, g;
    o.load(static_cast<const uint8_t *>(p.O) + rc * RB + sub * S::kBytes);
    g.load(static_cast<const uint8_t *>(p.dO) + rc * RB + sub * S::kBytes);
    const float l = p.LSE[rc];
    const float d = lanes_sum<G>(o.dot(g));
    if (r < rows && sub == 0) p.LD[r] = make_float2(l * kLog2e, d);
}

// Global first token, key pass: the dense parts of row 0 and column 0, one
// block per head each, placed ahead of the banded blocks in the key pass's
// grid so that they start first and run beside them.  Four lanes per row,
// eight rows per warp step; the warps' sums merged in shared memory in warp
// order.
//   dense_dq0_block: dQ_0 = scale sum over every key k of dS_0k k_k.
//   dense_col_block: for every query j, dS_j0 (into gw, for the query pass),
//                    dK_0 = scale sum dS_j0 q_j and dV_0 = sum P_j0 dO_j.
template <typename T, int W>
__device__ __forceinline__ void dense_dq0_block(const TableArg &tab, const StreamParams &p, int bh) {
    using S = Run<T, 4>;
    constexpr int RB = S::kRowBytes, P = S::kPairs;
    __shared__ float2 s_sum[W][32];
    const int N = tab.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane % 4, grp = lane / 4;
    const size_t row0 = (size_t)bh * N, lo = sub * S::kBytes;
    const uint8_t *gK = static_cast<const uint8_t *>(p.K) + row0 * RB + lo;
    const uint8_t *gV = static_cast<const uint8_t *>(p.V) + row0 * RB + lo;
    S q0, g0;
    q0.load(static_cast<const uint8_t *>(p.Q) + row0 * RB + lo);
    g0.load(static_cast<const uint8_t *>(p.dO) + row0 * RB + lo);
    const float2 l0 = p.LD[row0];
    float2 dq[P];
#pragma unroll
    for (int i = 0; i < P; ++i) dq[i] = make_float2(0.f, 0.f);
    for (int k0 = warp * 8; k0 < N; k0 += W * 8) {
        const int k = k0 + grp;
        const bool in = k < N;
        const size_t r = (size_t)(in ? k : 0) * RB;
        S kr, vr;
        kr.load(gK + r);
        vr.load(gV + r);
        const float sc = lanes_sum<4>(q0.dot(kr)), dp = lanes_sum<4>(g0.dot(vr));
        const float P0 = in ? fast_exp2(fmaf(sc, p.scale_log2, -l0.x)) : 0.f;
        kr.axpy(P0 * (dp - l0.y), dq);
    }
    groups_sum(dq);
    group0_store(dq, s_sum[warp]);
    __syncthreads();
    if (warp == 0) {
        float2 a = make_float2(0.f, 0.f);
        for (int w = 0; w < W; ++w) a = add2(a, s_sum[w][lane]);
        store_pair(static_cast<T *>(p.Out) + row0 * kHeadDim, lane, make_float2(a.x * p.scale, a.y * p.scale));
    }
}

template <typename T, int W>
__device__ __forceinline__ void dense_col_block(const TableArg &tab, const StreamParams &p, int bh) {
    using S = Run<T, 4>;
    constexpr int RB = S::kRowBytes, P = S::kPairs;
    __shared__ float2 s_sum[2][W][32];
    const int N = tab.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane % 4, grp = lane / 4;
    const size_t row0 = (size_t)bh * N, lo = sub * S::kBytes;
    const uint8_t *gQ = static_cast<const uint8_t *>(p.Q) + row0 * RB + lo;
    const uint8_t *gG = static_cast<const uint8_t *>(p.dO) + row0 * RB + lo;
    float *gw = p.gw + (size_t)bh * p.ns;
    S k0r, v0r;
    k0r.load(static_cast<const uint8_t *>(p.K) + row0 * RB + lo);
    v0r.load(static_cast<const uint8_t *>(p.V) + row0 * RB + lo);
    float2 dk[P], dv[P];
#pragma unroll
    for (int i = 0; i < P; ++i) dk[i] = dv[i] = make_float2(0.f, 0.f);
    for (int j0 = warp * 8; j0 < N; j0 += W * 8) {
        const int j = j0 + grp;
        const bool in = j < N;
        const int jc = in ? j : 0;
        S qj, gj;
        qj.load(gQ + (size_t)jc * RB);
        gj.load(gG + (size_t)jc * RB);
        const float2 lj = p.LD[row0 + jc];
        const float sc = lanes_sum<4>(qj.dot(k0r)), dp = lanes_sum<4>(gj.dot(v0r));
        const float Pj = in ? fast_exp2(fmaf(sc, p.scale_log2, -lj.x)) : 0.f, dS = Pj * (dp - lj.y);
        if (in && sub == 0) gw[j] = dS;
        qj.axpy(dS, dk);
        gj.axpy(Pj, dv);
    }
    groups_sum(dk);
    groups_sum(dv);
    group0_store(dk, s_sum[0][warp]);
    group0_store(dv, s_sum[1][warp]);
    __syncthreads();
    if (warp < 2) {
        float2 a = make_float2(0.f, 0.f);
        for (int w = 0; w < W; ++w) a = add2(a, s_sum[warp][w][lane]);
        const float sc = warp == 0 ? p.scale : 1.f;
        store_pair(static_cast<T *>(warp == 0 ? p.dK : p.dV) + row0 * kHeadDim, lane, make_float2(a.x * sc, a.y * sc));
    }
}

// The key rows [first, first + 32/G) of head bh (one warp; first < N).
template <typename T, int G, bool GT, int KU = 1>
__device__ __forceinline__ void key_rows(const TableArg &tab, const StreamParams &p, const int *s_off, int cnt, int bh,
                                         int first) {
    using S = Run<T, G>;
    constexpr int R = 32 / G;
    constexpr int RB = S::kRowBytes;
    const int N = tab.N;
    const int lane = threadIdx.x & 31, sub = lane % G;
    const int last = min(N, first + R) - 1;
    const bool valid = first + lane / G < N;
    const int k = valid ? first + lane / G : last;
    int tb, te;
    trim(s_off, cnt, N, first, last, tb, te);

    const size_t row0 = (size_t)bh * N;
    const size_t lo = sub * S::kBytes;
    const uint8_t *gQ = static_cast<const uint8_t *>(p.Q) + row0 * RB + lo;
    const uint8_t *gG = static_cast<const uint8_t *>(p.dO) + row0 * RB + lo;
    const float2 *ld = p.LD + row0;
    float *scr = p.scr + ((size_t)bh * p.max_count + cnt - 1) * p.ns;   // entry cnt-1-t at -t ns
    float2 dk[S::kPairs], dv[S::kPairs];
#pragma unroll
    for (int i = 0; i < S::kPairs; ++i) dk[i] = dv[i] = make_float2(0.f, 0.f);
    const float sl2 = p.scale_log2;
    S kk, vv;
    kk.load(static_cast<const uint8_t *>(p.K) + (row0 + k) * RB + lo);
    vv.load(static_cast<const uint8_t *>(p.V) + (row0 + k) * RB + lo);
    int t = tb;
    if constexpr (KU == 2) {   // two entries per step: both pairs' row loads in flight together
        for (; t + 1 < te; t += 2) {
            const int j0 = k + s_off[t], j1 = k + s_off[t + 1];
            const bool in0 = valid && (unsigned)j0 < (unsigned)N, in1 = valid && (unsigned)j1 < (unsigned)N;
            const int c0 = in0 ? j0 : k, c1 = in1 ? j1 : k;
            S q0, g0, q1, g1;
            q0.load(gQ + (size_t)c0 * RB);
            g0.load(gG + (size_t)c0 * RB);
            q1.load(gQ + (size_t)c1 * RB);
            g1.load(gG + (size_t)c1 * RB);
            const float2 l0 = ld[c0], l1 = ld[c1];
            const float s0 = lanes_sum<G>(q0.dot(kk)), dp0 = lanes_sum<G>(g0.dot(vv));
            const float s1 = lanes_sum<G>(q1.dot(kk)), dp1 = lanes_sum<G>(g1.dot(vv));
            const float P0 = in0 ? fast_exp2(fmaf(s0, sl2, -l0.x)) : 0.f;
            const float P1 = in1 ? fast_exp2(fmaf(s1, sl2, -l1.x)) : 0.f;
            const float dS0 = P0 * (dp0 - l0.y), dS1 = P1 * (dp1 - l1.y);
            g0.axpy(P0, dv);
            q0.axpy(dS0, dk);
            g1.axpy(P1, dv);
            q1.axpy(dS1, dk);
            if (in0 && sub == 0 && FIBATT_CHECKED(t < cnt && cnt <= p.max_count && j0 < p.ns))
                scr[(ptrdiff_t)j0 - (ptrdiff_t)t * p.ns] = dS0;
            if (in1 && sub == 0 && FIBATT_CHECKED(t + 1 < cnt && cnt <= p.max_count && j1 < p.ns))
                scr[(ptrdiff_t)j1 - (ptrdiff_t)(t + 1) * p.ns] = dS1;
        }
    }
    for (; t < te; ++t) {
        const int j = k + s_off[t];
        const bool in = valid && (unsigned)j < (unsigned)N;
        const int jc = in ? j : k;   // any row in range: its pair is masked
        S qq, gg;
        qq.load(gQ + (size_t)jc * RB);
        gg.load(gG + (size_t)jc * RB);
        const float2 lj = ld[jc];
        const float s = lanes_sum<G>(qq.dot(kk));
        const float dp = lanes_sum<G>(gg.dot(vv));
        const float P = in ? fast_exp2(fmaf(s, sl2, -lj.x)) : 0.f;
        const float dS = P * (dp - lj.y);
        // fp32 weights: bf16-rounded P and dS (one mixed-precision FMA per
        // element instead of an unpack and half a packed FMA) put the dK and
        // dQ errors within a few thousandths of the bf16 bound
        gg.axpy(P, dv);
        qq.axpy(dS, dk);
        if (in && sub == 0 && FIBATT_CHECKED(t < cnt && cnt <= p.max_count && j < p.ns))
            scr[(ptrdiff_t)j - (ptrdiff_t)t * p.ns] = dS;
    }
    if constexpr (GT) {
        // global first token: the pair (0, k) for every key k >= 1 whose band
        // misses query 0, computed here from the key and value rows already
        // in registers; key 0's whole column is the dense column block's
        const unsigned band0 = band_to_zero(s_off, cnt, first, last - first + 1);
        const bool need = valid && k >= 1 && !((band0 >> (k - first)) & 1u);
        S q0, g0;
        q0.load(gQ);
        g0.load(gG);
        const float2 l0 = ld[0];
        const float s0 = lanes_sum<G>(q0.dot(kk)), dp0 = lanes_sum<G>(g0.dot(vv));
        const float P0 = need ? fast_exp2(fmaf(s0, sl2, -l0.x)) : 0.f;
        g0.axpy(P0, dv);
        q0.axpy(P0 * (dp0 - l0.y), dk);
    }
    if (!valid || (GT && k == 0)) return;
    S::store(static_cast<uint8_t *>(p.dK) + (row0 + k) * RB + lo, dk, p.scale);
    S::store(static_cast<uint8_t *>(p.dV) + (row0 + k) * RB + lo, dv, 1.f);
}

// Key-centric pass: key row k stationary; the queries attending it are
// j = k + off[t] (symmetric table), whose pair is query j's entry cnt-1-t.
template <typename T, int G, int W, bool GT, int KU = 1>
__global__ void __launch_bounds__(W * 32, (G == 4 && sizeof(T) == 2) ? ((GT || KU == 2 ? 20 : 24) / W > 0 ? (GT || KU == 2 ? 20 : 24) / W : 1) : 1)
bwd_key_stream_kernel(const __grid_constant__ TableArg tab, const StreamParams p) {
    using S = Run<T, G>;
    constexpr int R = 32 / G;
    constexpr int RB = S::kRowBytes;
    extern __shared__ int s_off[];
    const int N = tab.N;
    int b = (int)blockIdx.x;
    if constexpr (GT) {   // the first 2 B H blocks: row 0's dQ_0, then column 0 (dense_*_block)
        if (b < 2 * p.row0_heads) {
            grid_dep_wait();
            grid_dep_launch();
            if (b < p.row0_heads)
                dense_dq0_block<T, W>(tab, p, b);
            else
                dense_col_block<T, W>(tab, p, b - p.row0_heads);
            return;
        }
        b -= 2 * p.row0_heads;
    }
    const int bh = b / p.nblk, yb = b % p.nblk;
    const int cnt = load_offsets(tab, bh % tab.H, s_off);
    if (p.prefetch & 2) {   // the query and dO rows are inputs (see the forward)
        const size_t head = (size_t)bh * N * RB;
        const int bfirst = yb * W * R;
        prefetch_windows(static_cast<const uint8_t *>(p.Q) + head, RB, s_off, cnt, N, bfirst, W * R);
        prefetch_windows(static_cast<const uint8_t *>(p.dO) + head, RB, s_off, cnt, N, bfirst, W * R);
    }
    grid_dep_wait();
    grid_dep_launch();
    const int first = (yb * W + (int)(threadIdx.x >> 5)) * R;
    if (first < N) key_rows<T, G, GT, KU>(tab, p, s_off, cnt, bh, first);   // whole warps
}

// Query-centric pass: dQ_j = scale sum over in-range entries t of
// dS(j, t) k_{j + off[t]}, dS from the key pass's scratch.
template <typename T, int G, int W, bool GT>
__global__ void __launch_bounds__(W * 32, (G == 4 && sizeof(T) == 2) ? (40 / W > 0 ? 40 / W : 1) : 1)
bwd_query_stream_kernel(const __grid_constant__ TableArg tab, const StreamParams p) {
    using S = Run<T, G>;
    constexpr int R = 32 / G;
    constexpr int RB = S::kRowBytes;
    extern __shared__ int s_off[];
    const int N = tab.N;
    const int bh = blockIdx.x / p.nblk, yb = blockIdx.x % p.nblk;
    const int cnt = load_offsets(tab, bh % tab.H, s_off);
    const int bfirst = yb * W * R;
    // the key rows are an input (see the forward); the dS rows are the key
    // pass's output, so they wait for it
    if (p.prefetch & 4)
        prefetch_windows(static_cast<const uint8_t *>(p.K) + (size_t)bh * N * RB, RB, s_off, cnt, N, bfirst, W * R);
    grid_dep_wait();
    grid_dep_launch();
    for (int t = threadIdx.x; (p.prefetch & 4) && t < cnt; t += blockDim.x) {
        const int n = (min(N, bfirst + W * R) - bfirst + 3) / 4 * 4;   // whole 16-byte pieces, inside the row stride
        if (n > 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                             p.scr + ((size_t)bh * p.max_count + t) * p.ns + bfirst),
                         "r"((uint32_t)n * 4u)
                         : "memory");
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane % G;
    const int first = (yb * W + warp) * R;
    if (first >= N) return;
    const int last = min(N, first + R) - 1;
    const bool valid = first + lane / G < N;
    const int j = valid ? first + lane / G : last;
    int tb, te;
    trim(s_off, cnt, N, first, last, tb, te);

    const size_t row0 = (size_t)bh * N;
    const size_t lo = sub * S::kBytes;
    const uint8_t *gK = static_cast<const uint8_t *>(p.K) + row0 * RB + lo;
    const float *scr = p.scr + (size_t)bh * p.max_count * p.ns + j;
    if (!FIBATT_CHECKED(te <= cnt && cnt <= p.max_count && j < p.ns)) te = tb;   // the scratch's rows
    float2 dq[S::kPairs];
#pragma unroll
    for (int i = 0; i < S::kPairs; ++i) dq[i] = make_float2(0.f, 0.f);
    // four offsets per step: their key-row and weight loads all in flight
    // before the first update
    constexpr int U = 4;
    int t = tb;
    for (; t + U <= te; t += U) {
        S kr[U];
        float wt[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int kk = j + s_off[t + u];
            const bool in = valid && (unsigned)kk < (unsigned)N;
            kr[u].load(gK + (size_t)(in ? kk : j) * RB);
            // out-of-range entries were never written: select, never multiply
            wt[u] = in ? scr[(size_t)(t + u) * p.ns] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) kr[u].axpy(wt[u], dq);
    }
    for (; t < te; ++t) {
        const int kk = j + s_off[t];
        const bool in = valid && (unsigned)kk < (unsigned)N;
        S kr;
        kr.load(gK + (size_t)(in ? kk : j) * RB);
        const float w0 = in ? scr[(size_t)t * p.ns] : 0.f;
        kr.axpy(w0, dq);
    }
    if constexpr (GT) {
        // global first token: the pair (j, 0) for every row j >= 1 whose band
        // misses key 0, its dS from the key pass's dense column block; row 0
        // is dense: its dQ_0 is the dense dQ_0 block's
        const unsigned band0 = band_to_zero(s_off, cnt, first, last - first + 1);
        const bool need = valid && j >= 1 && !((band0 >> (j - first)) & 1u);
        const float dS = need ? p.gw[(size_t)bh * p.ns + j] : 0.f;
        S k0r;
        k0r.load(gK);
        k0r.axpy(dS, dq);
    }
    if (!valid || (GT && j == 0)) return;
    S::store(static_cast<uint8_t *>(p.Out) + (row0 + j) * RB + lo, dq, p.scale);
}

}  // namespace

// Global first token: the streaming forward computes the dense rows 0 in
// blocks of its own grid (one block of kStreamWarps warps per head, over
// every key) while they take little longer than the banded blocks; for long
// sequences one block per head would outlast the whole banded grid (128 x
// 128 image shape, 16385 keys: forward 336 us against 193 us with the
// cluster kernel of global_token.cu), so there the dense row kernel runs.
// Video shape (1569 keys): forward 49.3 -> 39.9 us.
bool stream_row0_in_grid(const TableArg &tab) { return tab.N <= 4096; }

namespace {

int stream_lanes() {
    const char *e = getenv("FIBATT_FLAT_LANES");
    return (e && atoi(e) == 2) ? 2 : 4;
}

// bf16 weights in the forward's P.V update (FIBATT_FLAT_W16=0: fp32
// weights); measured faster on the 128 x 128 image shape
// FIBATT_STREAM_PREFETCH: bit mask of the kernels that L2-prefetch their
// row windows (1 forward, 2 key pass, 4 query pass).  Only the query pass
// gains (long backward 467.9 -> 455.9 us): its key and dS rows are read once
// each from DRAM, and the prefetch takes those misses off the warps' path;
// the forward (156.8 -> 205.7 us) and the key pass (467.9 -> 493.0 us) lose,
// their extra bulk traffic competing with the loads of a kernel that is
// already at two thirds of the issue rate.
int stream_prefetch() {
    const char *e = getenv("FIBATT_STREAM_PREFETCH");
    return e ? atoi(e) & 7 : 4;
}

// Table entries per step of the key pass (FIBATT_KEY_UNROLL: 2, the
// default for bf16 rows, four lanes, four warps, no global token; 1).  Two entries keep both
// pairs' query and dO rows in flight together, at 96 registers (20 warps per
// SM against 24): video backward 95.0 -> 93.2 us, 128 x 128 image 413.4 ->
// 406.0 us.
int key_unroll() {
    const char *e = getenv("FIBATT_KEY_UNROLL");
    return e && atoi(e) == 1 ? 1 : 2;
}

bool stream_w16() {
    const char *e = getenv("FIBATT_FLAT_W16");
    return !(e && atoi(e) == 0);
}

template <typename T, int G, bool W16, int W = kStreamWarps, bool GT = false>
cudaError_t fwd_stream(const FwdArgs &a) {
    constexpr int R = 32 / G;
    const TableArg &tab = *a.tab;
    StreamParams p{};
    p.Q = a.Q;
    p.K = a.K;
    p.V = a.V;
    p.Out = a.O;
    p.LSEout = a.LSE;
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.nblk = (tab.N + R * W - 1) / (R * W);
    p.prefetch = stream_prefetch();
    p.row0_heads = GT && stream_row0_in_grid(tab) ? a.B * tab.H : 0;
    const size_t smem = sizeof(int) * std::max(1, (int)tab.max_count);
    const long blocks = (long)a.B * tab.H * p.nblk + p.row0_heads;   // the dense row-0 blocks first
    const cudaError_t e = launch_kernel(fwd_stream_kernel<T, G, W, W16, GT>, dim3((unsigned)blocks), dim3(W * 32), smem,
                                        a.stream, pdl_enabled(), tab, p);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// cuTensorMapEncodeTiled from the driver (through the runtime's entry-point
// query, so the library needs no link against libcuda); null if unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// A bf16 tensor of `rows` rows of 64 elements (128-byte rows) at `base`,
// read in boxes of kWinBox rows with the 128-byte swizzle.
bool window_map(CUtensorMap *m, const void *base, long rows) {
    const EncodeTiledFn f = encode_tiled();
    if (!f) return false;
    const cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {64, kWinBox};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The near-window forward, on request (FIBATT_STREAM_WINDOW=1): bf16 rows,
// no global token, row coordinates within int32.  Measured slower than the
// plain streaming forward (video 43.2 against 34.3 us, 128 x 128 image 189.9
// against 149.8 us): 18% more instructions (a 32-byte run takes two 128-bit
// shared-memory loads where one 256-bit global load did, plus the swizzled
// addressing), 21 instead of 29 warps per SM (64 KB of shared memory and 80
// registers per block), for 17% less L2-to-SM traffic.
bool window_enabled(const FwdArgs &a) {
    const char *e = getenv("FIBATT_STREAM_WINDOW");
    if (!(e && atoi(e) == 1)) return false;
    return a.dtype == FIBATT_BF16 && !a.tab->global0 &&
           (long)a.B * a.tab->H * a.tab->N + kWinRows < 0x7fffffffL;
}

// Returns cudaErrorNotSupported (nothing launched) when the tensor maps
// cannot be made; the caller then takes the plain streaming forward.
template <int W, int MINB, bool W16>
cudaError_t fwd_window(const FwdArgs &a) {
    constexpr int R = 8;
    const TableArg &tab = *a.tab;
    const long rows = (long)a.B * tab.H * tab.N;
    WinMaps wm;
    if (!window_map(&wm.k, a.K, rows) || !window_map(&wm.v, a.V, rows)) return cudaErrorNotSupported;
    StreamParams p{};
    p.Q = a.Q;
    p.K = a.K;
    p.V = a.V;
    p.Out = a.O;
    p.LSEout = a.LSE;
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.nblk = (tab.N + R * W - 1) / (R * W);
    const size_t smem = window_smem_bytes(tab.max_count);
    static size_t smem_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = fwd_window_kernel<W, MINB, W16>;
    if (dev < 0 || dev >= 64 || smem_set[dev] < smem) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) smem_set[dev] = smem;
    }
    const long blocks = (long)a.B * tab.H * p.nblk;
    const cudaError_t e =
        launch_kernel(kern, dim3((unsigned)blocks), dim3(W * 32), smem, a.stream, pdl_enabled(), tab, p, wm);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int G, int W = kStreamWarps, bool GT = false>
cudaError_t bwd_stream(const BwdArgs &a) {
    constexpr int R = 32 / G;
    const TableArg &tab = *a.tab;
    const long rows = (long)a.B * tab.H * tab.N;
    StreamParams p{};
    p.Q = a.Q;
    p.K = a.K;
    p.V = a.V;
    p.O = a.O;
    p.dO = a.dO;
    p.LSE = a.LSE;
    p.dK = a.dK;
    p.dV = a.dV;
    p.LD = reinterpret_cast<float2 *>(a.Dws);
    p.scr = a.Dws + (2 * rows + 63) / 64 * 64;   // 256-byte aligned, after LD
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.nblk = (tab.N + R * W - 1) / (R * W);
    p.max_count = std::max(1, (int)tab.max_count);
    p.ns = (tab.N + 31) / 32 * 32;
    p.prefetch = stream_prefetch();
    const size_t heads = (size_t)a.B * tab.H;
    p.gw = p.scr + heads * p.max_count * p.ns;   // global token: after the scratch
    p.row0_heads = GT ? (int)heads : 0;
    const bool pdl = pdl_enabled();
    const size_t smem = sizeof(int) * p.max_count;
    const dim3 block(W * 32);
    const unsigned row_blocks = (unsigned)((rows + R * W - 1) / (R * W));
    const unsigned blocks = (unsigned)((long)a.B * tab.H * p.nblk);
    cudaError_t e = launch_kernel(rowdot_stream_kernel<T, G, W>, dim3(row_blocks), block, 0, a.stream, pdl, p, rows);
    if (e == cudaSuccess) e = cudaGetLastError();
    p.Out = a.dQ;   // the key pass's dense dQ_0 blocks write row 0 of dQ
    if (e == cudaSuccess)
        e = [&] {
            // the default shape without the global token (with it, whose key pass already runs at 96
            // registers, two entries per step measured slower: 128 x 128 image 524.0 -> 541.3 us)
            if constexpr (sizeof(T) == 2 && G == 4 && W == kStreamWarps && !GT) {
                if (key_unroll() == 2)
                    return launch_kernel(bwd_key_stream_kernel<T, G, W, GT, 2>,
                                         dim3(blocks + 2 * (unsigned)p.row0_heads), block, smem, a.stream, pdl, tab, p);
            }
            return launch_kernel(bwd_key_stream_kernel<T, G, W, GT>, dim3(blocks + 2 * (unsigned)p.row0_heads), block,
                                 smem, a.stream, pdl, tab, p);
        }();
    if (e == cudaSuccess) e = cudaGetLastError();
    p.Out = a.dQ;
    if (e == cudaSuccess)
        e = launch_kernel(bwd_query_stream_kernel<T, G, W, GT>, dim3(blocks), block, smem, a.stream, pdl, tab, p);
    count_launches(3);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// Warps per block (FIBATT_STREAM_WARPS: 4 or 8).
int stream_warps() {
    const char *e = getenv("FIBATT_STREAM_WARPS");
    return e && atoi(e) == 8 ? 8 : kStreamWarps;
}

cudaError_t launch_fwd_stream(const FwdArgs &a) {
    const bool w16 = stream_w16();
    if (a.tab->global0)   // the global first token: the default shape only
        return a.dtype == FIBATT_F32 ? fwd_stream<float, 4, false, kStreamWarps, true>(a)
                                     : fwd_stream<__nv_bfloat16, 4, true, kStreamWarps, true>(a);
    if (a.dtype == FIBATT_F32) return fwd_stream<float, 4, false>(a);
    if (window_enabled(a) && stream_lanes() == 4) {
        // FIBATT_WINDOW_SHAPE: 0 (8 warps, 3 blocks per SM, 80 registers) or 1 (10 warps, 2 blocks, 84
        // registers)
        const char *e = getenv("FIBATT_WINDOW_SHAPE");
        const int shape = e ? atoi(e) : 0;
        cudaError_t r;
        if (!w16)
            r = fwd_window<8, 3, false>(a);
        else if (shape == 1)
            r = fwd_window<10, 2, true>(a);
        else
            r = fwd_window<8, 3, true>(a);
        if (r != cudaErrorNotSupported) return r;
    }
    if (stream_lanes() == 2)
        return w16 ? fwd_stream<__nv_bfloat16, 2, true>(a) : fwd_stream<__nv_bfloat16, 2, false>(a);
    if (!w16) return fwd_stream<__nv_bfloat16, 4, false>(a);
    return stream_warps() == 8 ? fwd_stream<__nv_bfloat16, 4, true, 8>(a) : fwd_stream<__nv_bfloat16, 4, true, 4>(a);
}

cudaError_t launch_bwd_stream(const BwdArgs &a) {
    if (a.tab->global0)
        return a.dtype == FIBATT_F32 ? bwd_stream<float, 4, kStreamWarps, true>(a)
                                     : bwd_stream<__nv_bfloat16, 4, kStreamWarps, true>(a);
    if (a.dtype == FIBATT_F32) return bwd_stream<float, 4>(a);
    if (stream_lanes() == 2) return bwd_stream<__nv_bfloat16, 2>(a);
    return stream_warps() == 8 ? bwd_stream<__nv_bfloat16, 4, 8>(a) : bwd_stream<__nv_bfloat16, 4, 4>(a);
}

FIBATT_DEFINE_ERROR_READER(read_error_stream, "stream.cu")

size_t stream_bwd_scratch_bytes(const TableArg &tab, int B) {
    const size_t rows = (size_t)B * tab.H * tab.N, heads = (size_t)B * tab.H;
    const size_t ns = (tab.N + 31) / 32 * 32;
    size_t floats = (2 * rows + 63) / 64 * 64 + heads * std::max(1, (int)tab.max_count) * ns;
    if (tab.global0) floats += heads * ns;   // the global token's column weights dS_j0
    return floats * sizeof(float);
}

}  // namespace fibatt
