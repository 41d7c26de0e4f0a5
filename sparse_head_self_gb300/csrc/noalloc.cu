// fibatt_bwd_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// fibatt_bwd needs a caller-provided workspace for its generic kernels (one
// fp32 per query row, D_j = <dO_j, O_j>).  Some callers have no way to get
// one: code running where the allocator is off limits (inside a captured or
// replayed region that must not touch the allocator, a plugin handed fixed
// buffers by its host framework, a real-time loop that forbids allocation
// after start-up).  For them this entry point keeps that scratch in a
// fixed-size array that is part of the library image on every GPU that loads
// it, so the call itself never allocates.
//
// The array is a file-scope __device__ variable.  Host code cannot use its
// name as a device address, so on the first call on each device (with that
// device current) the library asks the runtime for the array's address with
// cudaGetSymbolAddress and remembers it; do that first call before any stream
// capture.  Every call on a device shares the one array: calls that overlap on
// the GPU (on different streams, unordered) race on it.  Each call overwrites
// every entry it reads before reading it, so nothing needs clearing between
// calls.
#include <cstdio>
#include <mutex>

#include "fibatt_internal.h"

namespace fibatt {
namespace {

// Room for B * H * N query rows of scratch (4 MiB per device).
constexpr size_t kNoAllocRows = FIBATT_NOALLOC_MAX_ROWS;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocRows];

std::mutex g_noalloc_mu;
float *g_noalloc_ptr[64] = {nullptr};

// Device address of this device's scratch array (looked up once per device).
fibatt_status noalloc_scratch(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "fibatt_bwd_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= 64) return set_error(FIBATT_ERR_UNSUPPORTED, "fibatt_bwd_noalloc: device index above 63");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_error(e, "fibatt_bwd_noalloc: cudaGetSymbolAddress");
        g_noalloc_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return FIBATT_OK;
}

}  // namespace
}  // namespace fibatt

using namespace fibatt;

extern "C" fibatt_status fibatt_bwd_noalloc(fibatt_support_t s, int B, int D, fibatt_dtype dtype, const void *Q,
                                            const void *K, const void *V, const void *O, const float *LSE,
                                            const void *dO, float scale, void *dQ, void *dK, void *dV,
                                            cudaStream_t stream) {
    const ProfileReport report("fibatt_bwd_noalloc");
    fibatt_status st = check_bwd_args(s, B, D, dtype, Q, K, V, O, LSE, dO, scale, dQ, dK, dV);
    if (st != FIBATT_OK) return st;
    const TableArg &tab = support_table(s);
    if (tab.global0)
        return set_error(FIBATT_ERR_UNSUPPORTED, "fibatt_bwd_noalloc has no global first token; use fibatt_bwd");
    const size_t rows = (size_t)B * tab.H * tab.N;
    if (rows > kNoAllocRows) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "fibatt_bwd_noalloc: B*H*N = %zu query rows exceed the fixed scratch of %zu rows; "
                 "use fibatt_bwd with a workspace",
                 rows, kNoAllocRows);
        return set_error(FIBATT_ERR_INVALID_ARG, msg);
    }
    float *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != FIBATT_OK) return st;
    BwdArgs a{&tab, B, dtype, Q, K, V, O, dO, LSE, dQ, dK, dV, scratch, scale, stream};
    cudaError_t e = launch_bwd_generic(a);
    if (e != cudaSuccess) return cuda_error(e, "fibatt_bwd_noalloc launch");
    return FIBATT_OK;
}
