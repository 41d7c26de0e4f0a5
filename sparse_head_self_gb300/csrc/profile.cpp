// Per-kernel timing of the library's calls (FIBATT_PROFILE=1).
//
// While FIBATT_PROFILE is set to a non-zero value, every kernel launch goes
// between two CUDA events recorded on its stream (ProfileLaunch, used by
// the launch helpers), and each public call, before it returns, waits for
// its last event and prints one line per kernel to stderr:
//   libfibatt profile: fibatt_bwd bwd_key_stream_kernel<__nv_bfloat16, 4, 4, false> 283.10 us
// The events stop consecutive kernels from overlapping (programmatic
// dependent launches), so the times are each kernel's own, not the
// pipelined call's.  Nothing is recorded while the stream is being captured
// into a CUDA graph.
#include <cxxabi.h>

#include <cstdio>
#include <cstdlib>
#include <string>
#include <vector>

#include "fibatt_internal.h"

namespace fibatt {
namespace {

struct Rec {
    const void *func;
    cudaEvent_t start, stop;
};

thread_local std::vector<Rec> t_recs;

bool profiling() {
    const char *e = getenv("FIBATT_PROFILE");
    return e && atoi(e) != 0;
}

// "fwd_stream_kernel<__nv_bfloat16, 4, 4, true, false>": demangled, without
// the namespaces and the parameter list.
std::string kernel_name(const void *func) {
    const char *mangled = nullptr;
    if (cudaFuncGetName(&mangled, func) != cudaSuccess || !mangled) return "(unknown kernel)";
    int status = 0;
    char *d = abi::__cxa_demangle(mangled, nullptr, nullptr, &status);
    std::string n = status == 0 && d ? d : mangled;
    free(d);
    for (const char *ns : {"fibatt::(anonymous namespace)::", "(anonymous namespace)::", "fibatt::"})
        for (size_t at; (at = n.find(ns)) != std::string::npos;) n.erase(at, std::string(ns).size());
    if (n.compare(0, 5, "void ") == 0) n.erase(0, 5);
    const size_t paren = n.find('(');
    if (paren != std::string::npos) n.erase(paren);
    return n;
}

}  // namespace

ProfileLaunch::ProfileLaunch(cudaStream_t stream, const void *func) : stream_(stream) {
    if (!profiling()) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
    Rec r{func, nullptr, nullptr};
    if (cudaEventCreate(&r.start) != cudaSuccess) return;
    if (cudaEventCreate(&r.stop) != cudaSuccess) {
        cudaEventDestroy(r.start);
        return;
    }
    cudaEventRecord(r.start, stream);
    slot_ = (int)t_recs.size();
    t_recs.push_back(r);
}

ProfileLaunch::~ProfileLaunch() {
    if (slot_ >= 0) cudaEventRecord(t_recs[slot_].stop, stream_);
}

ProfileReport::~ProfileReport() {
    if (t_recs.empty()) return;
    cudaEventSynchronize(t_recs.back().stop);
    for (const Rec &r : t_recs) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess)
            fprintf(stderr, "libfibatt profile: %s %s %.2f us\n", call_, kernel_name(r.func).c_str(), ms * 1e3f);
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    t_recs.clear();
}

}  // namespace fibatt
