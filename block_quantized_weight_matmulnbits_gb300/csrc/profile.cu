// MNB_PROFILE=1: per-call profiling of the C entry points.  The CPU operator's
// env-gated phase timers (onnx-runtime-ep-cpu 0.1.0-dev.5, src/kernels/
// matmul_nbits.rs, mm_profile: widen / GEMV / narrow accumulated per call and
// printed every 512 calls) and its tracing spans around the decode and prefill
// work become, here:
//   - an NVTX range around each profiled call (visible to ncu's --nvtx filters);
//   - per kernel family: the host time inside the call (validation, selection,
//     launch) and the device time between two CUDA events recorded on the
//     call's stream around its launches (skipped while the stream is being
//     captured into a graph);
//   - a line on stderr every MNB_PROFILE_EVERY calls of a family (default 512).
// The events sit between the call's kernels and its neighbours on the stream,
// so a profiled run loses the programmatic-launch overlap: the device time is
// the call's own, not its share of a chained sequence.
#include <nvtx3/nvToolsExt.h>

#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "mnb_internal.h"

namespace mnb {
namespace {

struct Family {
    int64_t calls = 0, timed = 0;
    double host_us = 0, device_us = 0;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;  // recorded since the last report
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pool;     // free pairs (the spare family's only)
};

std::mutex g_prof_mu;
std::map<std::string, Family>& families() {
    static std::map<std::string, Family> f;
    return f;
}

int64_t report_every() {
    const char* v = std::getenv("MNB_PROFILE_EVERY");
    const long long n = v ? std::strtoll(v, nullptr, 10) : 0;
    return n > 0 ? (int64_t)n : 512;
}

// Sums the pending pairs of a family and returns them to the spare pool (the caller holds the lock).
void drain(Family& f, Family& spare) {
    for (auto& pr : f.pending) {
        float ms = 0;
        if (cudaEventSynchronize(pr.second) == cudaSuccess && cudaEventElapsedTime(&ms, pr.first, pr.second) ==
                                                                  cudaSuccess) {
            f.device_us += ms * 1e3;
            ++f.timed;
        }
        spare.pool.push_back(pr);
    }
    f.pending.clear();
}

}  // namespace

bool profile_enabled() {
    const char* v = std::getenv("MNB_PROFILE");
    return v && v[0] == '1';
}

ProfileScope::ProfileScope(const char* range, cudaStream_t s) : on_(profile_enabled()), stream_(s) {
    if (!on_) return;
    nvtxRangePushA(range);
    t0_ = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now().time_since_epoch()).count();
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    Family& spare = families()[""];  // event pairs not yet bound to a family
    if (spare.pool.empty()) {
        cudaEvent_t a = nullptr, b = nullptr;
        if (cudaEventCreate(&a) != cudaSuccess) return;
        if (cudaEventCreate(&b) != cudaSuccess) {
            cudaEventDestroy(a);
            return;
        }
        spare.pool.push_back({a, b});
    }
    ev_ = spare.pool.back();
    spare.pool.pop_back();
    if (cudaEventRecord(ev_.first, s) != cudaSuccess) {
        spare.pool.push_back(ev_);
        ev_ = {nullptr, nullptr};
    }
}

void ProfileScope::done(const char* kernel) {
    if (!on_ || done_) return;
    done_ = true;
    const double t1 =
        std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now().time_since_epoch()).count();
    const bool timed = ev_.first && cudaEventRecord(ev_.second, stream_) == cudaSuccess;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    Family& f = families()[kernel];
    ++f.calls;
    f.host_us += t1 - t0_;
    if (ev_.first) {
        if (timed) f.pending.push_back(ev_);
        else families()[""].pool.push_back(ev_);
        ev_ = {nullptr, nullptr};
    }
    if (f.calls % report_every() == 0) {
        drain(f, families()[""]);
        std::fprintf(stderr,
                     "[mnb profile] kernel=%s calls=%lld host_us_per_call=%.2f device_us_per_call=%.2f "
                     "timed_calls=%lld\n",
                     kernel, (long long)f.calls, f.host_us / (double)f.calls,
                     f.timed ? f.device_us / (double)f.timed : 0.0, (long long)f.timed);
        std::fflush(stderr);
    }
}

ProfileScope::~ProfileScope() {
    if (!on_) return;
    if (!done_ && ev_.first) {  // the call failed before its launch: return the events unused
        std::lock_guard<std::mutex> lk(g_prof_mu);
        families()[""].pool.push_back(ev_);
    }
    nvtxRangePop();
}

}  // namespace mnb
