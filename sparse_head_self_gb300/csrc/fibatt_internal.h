// Internal declarations shared by the host API and the kernel launchers of
// libfibatt.  Not part of the public ABI (see include/fibatt.h).
#pragma once

#include <cstdint>
#include <string>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "fibatt.h"

namespace fibatt {

constexpr int kHeadDim = FIBATT_HEAD_DIM;
constexpr int kMaxHeads = FIBATT_MAX_HEADS;
constexpr int kMaxEntries = FIBATT_MAX_ENTRIES;

// Signed-offset tables of every head, passed to kernels by value as a
// __grid_constant__ argument (a few KB; no device allocation, valid on any
// device and inside CUDA graphs).  Head h owns entries [start[h], start[h+1])
// of `off`, ascending.  Query j of head h attends key j + off[t] whenever
// 0 <= j + off[t] < N.
struct TableArg {
    int32_t H;
    int32_t N;
    int32_t max_count;                 // max entries of one head
    int32_t max_abs;                   // max |offset| over all heads
    int32_t global0;                   // token 0 global (row 0 and column 0 attended)
    int32_t start[kMaxHeads + 1];
    int32_t off[kMaxEntries];
};

struct ResidentPlan;

struct SupportImpl {
    TableArg tab;
    std::vector<int64_t> pairs;        // |Omega_h| per head, banded part
    std::vector<int64_t> global_pairs; // pairs the global token adds per head
};

// ---- launch accounting (fibatt_launch_count) -------------------------------
void count_launches(int n);

// ---- error reporting (thread-local message) --------------------------------
fibatt_status set_error(fibatt_status st, const std::string &msg);
fibatt_status cuda_error(cudaError_t e, const char *what);

// Argument checks of fibatt_bwd minus the workspace, and a support's tables.
fibatt_status check_bwd_args(fibatt_support_t s, int B, int D, fibatt_dtype dtype, const void *Q, const void *K,
                             const void *V, const void *O, const float *LSE, const void *dO, float scale,
                             const void *dQ, const void *dK, const void *dV);
const TableArg &support_table(fibatt_support_t s);

// ---- launchers (return the CUDA launch status) -----------------------------
struct FwdArgs {
    const TableArg *tab;
    int B;
    fibatt_dtype dtype;
    const void *Q, *K, *V;
    void *O;
    float *LSE;
    float scale;
    cudaStream_t stream;
};

struct BwdArgs {
    const TableArg *tab;
    int B;
    fibatt_dtype dtype;
    const void *Q, *K, *V, *O, *dO;
    const float *LSE;
    void *dQ, *dK, *dV;
    float *Dws;                        // fp32 scratch: [B*H*N] (generic) or pair weights (flat)
    float scale;
    cudaStream_t stream;
    float *gw = nullptr;               // global token: P_0k, dS_0k per (b, h) ([B*H][2][N] fp32)
};

// Shared-memory-resident kernels: one CTA per (b, h, query chunk); the
// chunk's K/V row window is staged in shared memory (resident.cu).
struct ResidentPlan {
    int lanes;           // lanes per query row (2 or 4)
    int unroll;          // offsets per step in the interior loop (1 or 2)
    int maxt;            // threads the kernel's register budget is sized for
    int qsplit;          // query chunks per (b, h)
    int chunk;           // queries per chunk
    int kv_cap;          // rows reserved per staged window
    int stages;          // shared-memory ring depth
    int groups;          // consumer warp groups
    int gwarps;          // warps per consumer group
    int prefetch;        // units beyond the ring warmed in L2 (forward)
    int n_keep;          // whole units before the last partial wave
    int qsub;            // pieces each last-wave unit is cut into
    int sub_rows;        // forward: query rows per piece; backward: rounds per piece
    size_t split_off;    // backward: byte offset of the pieces' (P, dS) areas
    int piece_par;       // backward: one-round pieces spread over more warps
    int fuse_row0;       // global first token: row 0 (forward), row and column 0 (backward) computed inside each
                         // whole-head unit
    size_t gt_off;       // backward, fused global token: byte offset of its weights and partial sums
    size_t stage_bytes;  // bytes per ring stage
    size_t smem;         // dynamic shared memory bytes
    int threads;         // threads per CTA (producer warp + consumers)
    int grid;            // CTAs (persistent, one per SM at most)
};
bool plan_fwd_resident(const TableArg &tab, int B, fibatt_dtype dt, ResidentPlan *pl);
bool plan_bwd_resident(const TableArg &tab, int B, fibatt_dtype dt, ResidentPlan *pl);

// Plans memoised per (support, B, dtype, device, tuning overrides): planning
// is host work that would otherwise run on every call.
struct PlanCache;
bool cached_plan(const void *support, bool backward, const TableArg &tab, int B, fibatt_dtype dt,
                 ResidentPlan *pl);
void forget_plans(const void *support);

// ---- per-kernel timing (FIBATT_PROFILE=1; profile.cpp) ----------------------
// A ProfileLaunch around each launch records CUDA events on its stream while
// profiling is on; the ProfileReport of the public call prints the kernels'
// times to stderr when the call returns.
class ProfileLaunch {
  public:
    ProfileLaunch(cudaStream_t stream, const void *func);
    ~ProfileLaunch();

  private:
    cudaStream_t stream_;
    int slot_ = -1;
};

class ProfileReport {
  public:
    explicit ProfileReport(const char *call) : call_(call) {}
    ~ProfileReport();

  private:
    const char *call_;
};

// Launch `kern` on `stream`; with pdl set, as a programmatic dependent launch
// (the kernel calls grid_dep_wait before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                          Args &&...args) {
    const ProfileLaunch prof(stream, reinterpret_cast<const void *>(kern));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Programmatic dependent launches on (FIBATT_PDL unset or non-zero) or off.
bool pdl_enabled();

cudaError_t launch_fwd_generic(const FwdArgs &a);
cudaError_t launch_bwd_generic(const BwdArgs &a);
cudaError_t launch_fwd_resident(const FwdArgs &a, const ResidentPlan &pl);
cudaError_t launch_fwd_flat(const FwdArgs &a);
cudaError_t launch_bwd_flat(const BwdArgs &a);       // a.Dws: pair-weight scratch
size_t flat_bwd_scratch_bytes(const TableArg &tab, int B);
// Streaming kernels for wide windows (stream.cu): rows 32-byte aligned.  The
// backward's workspace: (LSE_j log2 e, D_j) per row, then dS per (b, h, table
// entry, query row); with the global first token, the dense pairs of row 0
// and column 0 and per-block sums, all computed inside the streaming kernels
// (no dense kernel launches).
cudaError_t launch_fwd_stream(const FwdArgs &a);
bool flat_fwd_fuses_global(const FwdArgs &a);   // the flat forward computes the dense row 0 itself
bool flat_bwd_fuses_global(const BwdArgs &a);   // the flat backward computes the dense row and column itself
cudaError_t launch_bwd_stream(const BwdArgs &a);
size_t stream_bwd_scratch_bytes(const TableArg &tab, int B);
bool stream_row0_in_grid(const TableArg &tab);   // global token: the streaming forward computes the rows 0
cudaError_t launch_bwd_resident(const BwdArgs &a, const ResidentPlan &pl);
cudaError_t read_device_error(unsigned *code, bool clear);
// Each kernel file's own copy of the device error word (device_common.cuh).
cudaError_t read_error_resident(unsigned *code, bool clear);
cudaError_t read_error_stream(unsigned *code, bool clear);
cudaError_t read_error_generic(unsigned *code, bool clear);
cudaError_t read_error_global_token(unsigned *code, bool clear);

// Global first token (global_token.cu): the dense row of token 0 (forward,
// after the banded kernel), its dense row before the banded backward, and
// the column of key 0 after it.
// Rows 0 of heads bh0 .. B H - 1 (every head when bh0 = 0).
cudaError_t launch_fwd_global_row(const FwdArgs &a, long bh0 = 0);
cudaError_t launch_bwd_global_row(const BwdArgs &a);
cudaError_t launch_bwd_global_col(const BwdArgs &a);

}  // namespace fibatt
