// libfibatt C ABI: argument checks, support construction and dispatch.
// The operation and every argument rule are documented in include/fibatt.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <set>
#include <tuple>
#include <string>
#include <vector>

#include "fibatt_internal.h"

struct fibatt_support {
    fibatt::SupportImpl impl;
};

namespace fibatt {
namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

std::string fmt(const char *f, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, f);
    vsnprintf(buf, sizeof buf, f, ap);
    va_end(ap);
    return buf;
}

// Host-side fault injection for the error paths: FIBATT_FAULT=launch makes
// fwd/bwd report a CUDA launch failure without launching anything,
// FIBATT_FAULT=arg makes them report an invalid argument.
bool fault(const char *kind) {
    const char *e = std::getenv("FIBATT_FAULT");
    return e && std::strcmp(e, kind) == 0;
}

// floor(sqrt(n)) for 0 <= n <= 2^62: start from the long double root and
// correct by whole steps.
int64_t int_sqrt(int64_t n) {
    int64_t r = (int64_t)std::sqrt((long double)n);
    while (r > 0 && (__int128)r * r > n) --r;
    while ((__int128)(r + 1) * (r + 1) <= n) ++r;
    return r;
}

// floor(n * phi) = floor((n + sqrt(5 n^2)) / 2); sqrt(5 n^2) is irrational
// for n >= 1, so its floor can replace it.
int64_t floor_phi(int64_t n) { return n <= 0 ? 0 : (n + int_sqrt(5 * n * n)) / 2; }

// Kernel family override for tests and tuning: FIBATT_PATH=generic forces the
// generic kernels, FIBATT_PATH=resident forbids falling back to them.
enum class PathSel { Auto, Generic, Resident, Flat };
PathSel path_sel() {
    const char *e = std::getenv("FIBATT_PATH");
    if (!e) return PathSel::Auto;
    if (std::strcmp(e, "generic") == 0) return PathSel::Generic;
    if (std::strcmp(e, "resident") == 0) return PathSel::Resident;
    if (std::strcmp(e, "flat") == 0) return PathSel::Flat;
    return PathSel::Auto;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Build one support from per-head distance sets (already cut to <= N-1).
fibatt_status finish_support(int H, int N, const std::vector<std::set<int64_t>> &dist,
                             int include_diag, fibatt_support_t *out) {
    fibatt_support *s = new (std::nothrow) fibatt_support;
    if (!s) return set_error(FIBATT_ERR_OOM, "support: host allocation failed");
    TableArg &tab = s->impl.tab;
    std::memset(&tab, 0, sizeof tab);
    tab.H = H;
    tab.N = N;
    s->impl.pairs.assign(H, 0);
    s->impl.global_pairs.assign(H, 0);
    int n = 0;
    for (int h = 0; h < H; ++h) {
        tab.start[h] = n;
        const std::set<int64_t> &d = dist[h];
        const bool zero = include_diag || d.count(0);
        std::vector<int32_t> row;
        for (auto it = d.rbegin(); it != d.rend(); ++it)
            if (*it > 0) row.push_back((int32_t)-*it);
        if (zero) row.push_back(0);
        for (int64_t f : d)
            if (f > 0) row.push_back((int32_t)f);
        if (n + (int)row.size() > kMaxEntries) {
            delete s;
            return set_error(FIBATT_ERR_UNSUPPORTED,
                             fmt("support: more than %d signed offsets in total", kMaxEntries));
        }
        int64_t pairs = zero ? N : 0;
        for (int64_t f : d)
            if (f > 0) pairs += 2 * (int64_t)(N - f);
        s->impl.pairs[h] = pairs;
        // row 0 and column 0 hold 2N - 1 pairs; the banded ones among them
        // are (0, f) and (f, 0) for every distance f, and (0, 0) once
        int64_t npos = 0;
        for (int64_t f : d) npos += f > 0;
        s->impl.global_pairs[h] = 2 * (int64_t)N - 1 - 2 * npos - (zero ? 1 : 0);
        for (int32_t o : row) {
            tab.off[n++] = o;
            tab.max_abs = std::max(tab.max_abs, o < 0 ? -o : o);
        }
        tab.max_count = std::max(tab.max_count, (int32_t)row.size());
    }
    tab.start[H] = n;
    *out = s;
    return FIBATT_OK;
}

fibatt_status check_tensor(const void *p, const char *name) {
    if (!p) return set_error(FIBATT_ERR_INVALID_ARG, fmt("%s is NULL", name));
    if (!aligned(p, 16)) return set_error(FIBATT_ERR_INVALID_ARG, fmt("%s is not 16-byte aligned", name));
    return FIBATT_OK;
}

fibatt_status check_common(fibatt_support_t s, int B, int D, fibatt_dtype dtype, float scale) {
    if (!s) return set_error(FIBATT_ERR_INVALID_ARG, "support handle is NULL");
    if (B < 1) return set_error(FIBATT_ERR_INVALID_ARG, fmt("B must be >= 1 (got %d)", B));
    if (D != kHeadDim)
        return set_error(FIBATT_ERR_UNSUPPORTED, fmt("head dim %d unsupported (only %d)", D, kHeadDim));
    if (dtype != FIBATT_F32 && dtype != FIBATT_BF16)
        return set_error(FIBATT_ERR_UNSUPPORTED, fmt("unknown dtype %d", (int)dtype));
    if (!std::isfinite(scale)) return set_error(FIBATT_ERR_INVALID_ARG, "scale is not finite");
    const TableArg &tab = s->impl.tab;
    if ((int64_t)B * tab.H > 0x7fffffffLL)
        return set_error(FIBATT_ERR_INVALID_ARG, "B*H exceeds 2^31-1");
    if ((int64_t)tab.N > 65535LL * 64)
        return set_error(FIBATT_ERR_UNSUPPORTED, "N above 4194240 is not supported");
    if (fault("arg")) return set_error(FIBATT_ERR_INVALID_ARG, "injected argument fault (FIBATT_FAULT=arg)");
    return FIBATT_OK;
}

}  // namespace

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

fibatt_status set_error(fibatt_status st, const std::string &msg) {
    g_last_error = msg;
    return st;
}

namespace {
struct PlanKey {
    const void *support;
    bool backward;
    int B, dt, dev;
    std::string env;
    bool operator<(const PlanKey &o) const {
        return std::tie(support, backward, B, dt, dev, env) < std::tie(o.support, o.backward, o.B, o.dt, o.dev, o.env);
    }
};
struct PlanEntry {
    bool ok;
    ResidentPlan plan;
};
std::mutex g_plan_mu;
std::map<PlanKey, PlanEntry> g_plans;

std::string tuning_env() {
    std::string r;
    for (const char *n : {"FIBATT_QSPLIT", "FIBATT_LANES", "FIBATT_GROUPS", "FIBATT_STAGES", "FIBATT_BWD_THREADS",
                          "FIBATT_UNROLL", "FIBATT_FWD_THREADS", "FIBATT_PREFETCH", "FIBATT_BWD_LANES", "FIBATT_SPLIT_TAIL",
                          "FIBATT_BWD_PIECES", "FIBATT_BWD_PIECE_PAR", "FIBATT_GT_FUSE", "FIBATT_FWD_GWARPS", "FIBATT_BWD_PIECE_ROUNDS"}) {
        const char *e = std::getenv(n);
        r += e ? e : "-";
        r += ',';
    }
    return r;
}
}  // namespace

bool cached_plan(const void *support, bool backward, const TableArg &tab, int B, fibatt_dtype dt,
                 ResidentPlan *pl) {
    int dev = 0;
    cudaGetDevice(&dev);
    PlanKey key{support, backward, B, (int)dt, dev, tuning_env()};
    {
        std::lock_guard<std::mutex> lock(g_plan_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            *pl = it->second.plan;
            return it->second.ok;
        }
    }
    PlanEntry e;
    e.ok = backward ? plan_bwd_resident(tab, B, dt, &e.plan) : plan_fwd_resident(tab, B, dt, &e.plan);
    std::lock_guard<std::mutex> lock(g_plan_mu);
    if (g_plans.size() > 4096) g_plans.clear();
    g_plans[key] = e;
    *pl = e.plan;
    return e.ok;
}

void forget_plans(const void *support) {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    for (auto it = g_plans.begin(); it != g_plans.end();) {
        if (it->first.support == support) it = g_plans.erase(it);
        else ++it;
    }
}

fibatt_status check_bwd_args(fibatt_support_t s, int B, int D, fibatt_dtype dtype, const void *Q, const void *K,
                             const void *V, const void *O, const float *LSE, const void *dO, float scale,
                             const void *dQ, const void *dK, const void *dV) {
    fibatt_status st = check_common(s, B, D, dtype, scale);
    if (st != FIBATT_OK) return st;
    if ((st = check_tensor(Q, "Q")) || (st = check_tensor(K, "K")) || (st = check_tensor(V, "V")) ||
        (st = check_tensor(O, "O")) || (st = check_tensor(dO, "dO")) || (st = check_tensor(dQ, "dQ")) ||
        (st = check_tensor(dK, "dK")) || (st = check_tensor(dV, "dV")))
        return st;
    if (!LSE || !aligned(LSE, 4)) return set_error(FIBATT_ERR_INVALID_ARG, "LSE is NULL or misaligned");
    return FIBATT_OK;
}

const TableArg &support_table(fibatt_support_t s) { return s->impl.tab; }

fibatt_status cuda_error(cudaError_t e, const char *what) {
    cudaGetLastError();  // clear a sticky-free launch error so the next call starts clean
    return set_error(FIBATT_ERR_CUDA, fmt("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e)));
}

bool pdl_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("FIBATT_PDL");
        return !(e && std::atoi(e) == 0);
    }();
    return on;
}

}  // namespace fibatt

using namespace fibatt;

extern "C" {

fibatt_status fibatt_wythoff_row(int64_t i, int64_t *a, int64_t *b) {
    if (i < 1 || i > 100000000 || !a || !b)
        return set_error(FIBATT_ERR_INVALID_ARG, "wythoff row index must be in [1, 1e8]");
    const int64_t r = floor_phi(i);
    *a = floor_phi(r);
    *b = *a + r;  // floor(r*phi^2) = floor(r*phi) + r since phi^2 = phi + 1
    return FIBATT_OK;
}

fibatt_status fibatt_wythoff_row_modified(int64_t i, int64_t *a, int64_t *b) {
    int64_t x, y;
    fibatt_status st = fibatt_wythoff_row(i, &x, &y);
    if (st != FIBATT_OK) return st;
    *b = y - x;
    *a = x - *b;
    return FIBATT_OK;
}

fibatt_status fibatt_window_schedule(int h, int64_t w_min, int64_t w_max, int64_t *w) {
    if (h < 1 || !w || w_min < 1 || w_max < w_min)
        return set_error(FIBATT_ERR_INVALID_ARG, "window schedule needs h >= 1 and 1 <= w_min <= w_max");
    for (int i = 1; i <= h; ++i)
        w[i - 1] = h == 1 ? w_min : w_min + ((w_max - w_min) * (int64_t)(i - 1)) / (h - 1);
    return FIBATT_OK;
}

fibatt_status fibatt_support_build(int H, int N, const int64_t *a, const int64_t *b, const int64_t *w,
                                   int include_diag, fibatt_support_t *out) {
    if (!out) return set_error(FIBATT_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (H < 1 || N < 1) return set_error(FIBATT_ERR_INVALID_ARG, fmt("H=%d and N=%d must be >= 1", H, N));
    if (H > kMaxHeads) return set_error(FIBATT_ERR_UNSUPPORTED, fmt("H=%d above %d", H, kMaxHeads));
    if (!a || !b || !w) return set_error(FIBATT_ERR_INVALID_ARG, "a, b or w is NULL");
    std::vector<std::set<int64_t>> dist(H);
    for (int h = 0; h < H; ++h) {
        if (a[h] < 0 || b[h] < 0 || (a[h] == 0 && b[h] == 0))
            return set_error(FIBATT_ERR_INVALID_ARG,
                             fmt("head %d: need a, b >= 0 and not both 0 (a=%lld b=%lld)", h,
                                 (long long)a[h], (long long)b[h]));
        if (w[h] < 1 || w[h] > N)
            return set_error(FIBATT_ERR_INVALID_ARG,
                             fmt("head %d: window %lld outside [1, N=%d]", h, (long long)w[h], N));
        // Generalised Fibonacci list, extended while its last term is below
        // w (README Algorithm 1); keep the terms inside the window and the
        // sequence (Sec. 3: |j-k| in Fib(a,b) and |j-k| <= w).
        const int64_t lim = std::min<int64_t>(w[h], N - 1);
        int64_t x = a[h], y = b[h];
        if (x <= lim) dist[h].insert(x);
        if (y <= lim) dist[h].insert(y);
        while (y < w[h]) {
            const int64_t z = x + y;
            x = y;
            y = z;
            if (y <= lim) dist[h].insert(y);
        }
    }
    return finish_support(H, N, dist, include_diag, out);
}

fibatt_status fibatt_support_build_distances(int H, int N, const int32_t *counts, const int32_t *distances,
                                             int include_diag, fibatt_support_t *out) {
    if (!out) return set_error(FIBATT_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (H < 1 || N < 1) return set_error(FIBATT_ERR_INVALID_ARG, fmt("H=%d and N=%d must be >= 1", H, N));
    if (H > kMaxHeads) return set_error(FIBATT_ERR_UNSUPPORTED, fmt("H=%d above %d", H, kMaxHeads));
    if (!counts) return set_error(FIBATT_ERR_INVALID_ARG, "counts is NULL");
    std::vector<std::set<int64_t>> dist(H);
    int64_t pos = 0;
    for (int h = 0; h < H; ++h) {
        if (counts[h] < 0) return set_error(FIBATT_ERR_INVALID_ARG, fmt("counts[%d] < 0", h));
        if (counts[h] > 0 && !distances) return set_error(FIBATT_ERR_INVALID_ARG, "distances is NULL");
        for (int32_t c = 0; c < counts[h]; ++c, ++pos) {
            const int32_t f = distances[pos];
            if (f < 0) return set_error(FIBATT_ERR_INVALID_ARG, fmt("negative distance %d", f));
            if (f <= N - 1) dist[h].insert(f);
        }
    }
    return finish_support(H, N, dist, include_diag, out);
}

fibatt_status fibatt_support_info(fibatt_support_t s, int *H, int *N, int *total_entries) {
    if (!s) return set_error(FIBATT_ERR_INVALID_ARG, "support handle is NULL");
    const TableArg &tab = s->impl.tab;
    if (H) *H = tab.H;
    if (N) *N = tab.N;
    if (total_entries) *total_entries = tab.start[tab.H];
    return FIBATT_OK;
}

fibatt_status fibatt_support_get(fibatt_support_t s, int32_t *counts, int32_t *signed_offsets, int64_t *pairs) {
    if (!s) return set_error(FIBATT_ERR_INVALID_ARG, "support handle is NULL");
    const TableArg &tab = s->impl.tab;
    for (int h = 0; h < tab.H; ++h) {
        if (counts) counts[h] = tab.start[h + 1] - tab.start[h];
        if (pairs) pairs[h] = s->impl.pairs[h] + (tab.global0 ? s->impl.global_pairs[h] : 0);
    }
    if (signed_offsets) std::memcpy(signed_offsets, tab.off, sizeof(int32_t) * tab.start[tab.H]);
    return FIBATT_OK;
}

fibatt_status fibatt_support_set_global_token(fibatt_support_t s, int enabled) {
    if (!s) return set_error(FIBATT_ERR_INVALID_ARG, "support handle is NULL");
    forget_plans(s);   // stage sizes depend on it
    s->impl.tab.global0 = enabled ? 1 : 0;
    return FIBATT_OK;
}

void fibatt_support_destroy(fibatt_support_t s) {
    if (s) forget_plans(s);
    delete s;
}

fibatt_status fibatt_fwd(fibatt_support_t s, int B, int D, fibatt_dtype dtype, const void *Q, const void *K,
                         const void *V, float scale, void *O, float *LSE, cudaStream_t stream) {
    const ProfileReport report("fibatt_fwd");
    fibatt_status st = check_common(s, B, D, dtype, scale);
    if (st != FIBATT_OK) return st;
    if ((st = check_tensor(Q, "Q")) || (st = check_tensor(K, "K")) || (st = check_tensor(V, "V")) ||
        (st = check_tensor(O, "O")))
        return st;
    if (!LSE || !aligned(LSE, 4)) return set_error(FIBATT_ERR_INVALID_ARG, "LSE is NULL or misaligned");
    if (fault("launch")) return set_error(FIBATT_ERR_CUDA, "injected launch failure (FIBATT_FAULT=launch)");
    FwdArgs a{&s->impl.tab, B, dtype, Q, K, V, O, LSE, scale, stream};
    const PathSel sel = path_sel();
    ResidentPlan pl;
    cudaError_t e;
    long row0_from = 0;   // global first token: heads from here on get row 0 from the row kernel
    if (s->impl.tab.global0 && sel == PathSel::Generic)
        return set_error(FIBATT_ERR_UNSUPPORTED, "FIBATT_PATH=generic has no global first token");
    if (sel == PathSel::Generic) {
        e = launch_fwd_generic(a);
    } else if (sel != PathSel::Flat && cached_plan(s, false, s->impl.tab, B, dtype, &pl)) {
        e = launch_fwd_resident(a, pl);
        // fused: every head's row 0 was written by its whole-head unit or by
        // the last-wave piece that holds query 0
        if (s->impl.tab.global0 && pl.fuse_row0) row0_from = (long)B * s->impl.tab.H;
    } else {
        if (sel == PathSel::Resident)
            return set_error(FIBATT_ERR_UNSUPPORTED, "FIBATT_PATH=resident: windows do not fit in shared memory");
        e = launch_fwd_flat(a);
        if (flat_fwd_fuses_global(a)) row0_from = (long)B * s->impl.tab.H;   // the streaming kernel wrote rows 0
    }
    if (e == cudaSuccess && s->impl.tab.global0 && row0_from < (long)B * s->impl.tab.H)
        e = launch_fwd_global_row(a, row0_from);
    if (e != cudaSuccess) return cuda_error(e, "fibatt_fwd launch");
    return FIBATT_OK;
}

static size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// P_0k and dS_0k of every key of every (b, h) when token 0 is global.
static size_t global_ws_bytes(const TableArg &tab, int B) {
    return tab.global0 ? (size_t)B * tab.H * 2 * tab.N * sizeof(float) : 0;
}

size_t fibatt_bwd_workspace_bytes(fibatt_support_t s, int B) {
    if (!s || B < 1) return 0;
    const size_t rows = (size_t)B * s->impl.tab.H * s->impl.tab.N;
    const size_t bytes = std::max(rows * sizeof(float), flat_bwd_scratch_bytes(s->impl.tab, B));
    return round256(bytes) + round256(global_ws_bytes(s->impl.tab, B));
}

enum class BwdPath { Resident, Flat, Generic };

// The backward path and the workspace it actually touches (0 for the
// resident kernel, which keeps its scratch in shared memory).
static size_t bwd_workspace_needed(fibatt_support_t s, int B, fibatt_dtype dt, BwdPath *path, ResidentPlan *pl) {
    const PathSel sel = path_sel();
    const TableArg &tab = s->impl.tab;
    const size_t gws = round256(global_ws_bytes(tab, B));   // placed after the path's own scratch
    if (sel == PathSel::Generic) {
        *path = BwdPath::Generic;
        return (size_t)B * tab.H * tab.N * sizeof(float);
    }
    if (sel != PathSel::Flat && cached_plan(s, true, tab, B, dt, pl)) {
        *path = BwdPath::Resident;
        return gws;
    }
    *path = BwdPath::Flat;
    return gws ? round256(flat_bwd_scratch_bytes(tab, B)) + gws : flat_bwd_scratch_bytes(tab, B);
}

fibatt_status fibatt_bwd(fibatt_support_t s, int B, int D, fibatt_dtype dtype, const void *Q, const void *K,
                         const void *V, const void *O, const float *LSE, const void *dO, float scale, void *dQ,
                         void *dK, void *dV, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    const ProfileReport report("fibatt_bwd");
    fibatt_status st = check_common(s, B, D, dtype, scale);
    if (st != FIBATT_OK) return st;
    if ((st = check_tensor(Q, "Q")) || (st = check_tensor(K, "K")) || (st = check_tensor(V, "V")) ||
        (st = check_tensor(O, "O")) || (st = check_tensor(dO, "dO")) || (st = check_tensor(dQ, "dQ")) ||
        (st = check_tensor(dK, "dK")) || (st = check_tensor(dV, "dV")))
        return st;
    if (!LSE || !aligned(LSE, 4)) return set_error(FIBATT_ERR_INVALID_ARG, "LSE is NULL or misaligned");
    BwdPath path = BwdPath::Generic;
    ResidentPlan pl;
    const size_t need = bwd_workspace_needed(s, B, dtype, &path, &pl);
    if (path != BwdPath::Resident && path_sel() == PathSel::Resident)
        return set_error(FIBATT_ERR_UNSUPPORTED, "FIBATT_PATH=resident: the backward does not fit in shared memory");
    if (need > 0) {
        if ((st = check_tensor(workspace, "workspace"))) return st;
        if (ws_bytes < need)
            return set_error(FIBATT_ERR_INVALID_ARG,
                             fmt("workspace holds %zu bytes, %zu needed", ws_bytes, need));
    }
    if (fault("launch")) return set_error(FIBATT_ERR_CUDA, "injected launch failure (FIBATT_FAULT=launch)");
    if (s->impl.tab.global0 && path == BwdPath::Generic)
        return set_error(FIBATT_ERR_UNSUPPORTED, "FIBATT_PATH=generic has no global first token");
    BwdArgs a{&s->impl.tab, B, dtype, Q, K, V, O, dO, LSE, dQ, dK, dV, static_cast<float *>(workspace),
              scale, stream};
    if (s->impl.tab.global0) {
        const size_t own = path == BwdPath::Flat ? round256(flat_bwd_scratch_bytes(s->impl.tab, B)) : 0;
        a.gw = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + own);
    }

    cudaError_t e = cudaSuccess;
    // the resident kernel computes the dense row and column itself when the plan fuses them
    const bool dense_kernels = a.gw && !(path == BwdPath::Resident && pl.fuse_row0) &&
                               !(path == BwdPath::Flat && flat_bwd_fuses_global(a));
    if (dense_kernels) e = launch_bwd_global_row(a);   // dQ_0 and the weights of the pairs (0, k)
    if (e == cudaSuccess)
        e = path == BwdPath::Resident ? launch_bwd_resident(a, pl)
            : path == BwdPath::Flat   ? launch_bwd_flat(a)
                                      : launch_bwd_generic(a);
    if (e == cudaSuccess && dense_kernels) e = launch_bwd_global_col(a);   // dK_0, dV_0
    if (e != cudaSuccess) return cuda_error(e, "fibatt_bwd launch");
    return FIBATT_OK;
}

const char *fibatt_last_error(void) { return g_last_error.c_str(); }

const char *fibatt_version(void) { return "libfibatt 0.1 (sm_103a)"; }

uint64_t fibatt_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

fibatt_status fibatt_device_error(int clear, unsigned *code) {
    if (!code) return set_error(FIBATT_ERR_INVALID_ARG, "code is NULL");
    *code = 0;
    cudaError_t e = read_device_error(code, clear != 0);
    if (e != cudaSuccess) return cuda_error(e, "fibatt_device_error");
    return FIBATT_OK;
}

}  // extern "C"
