// kda_profile.cu -- device-time profile of the library's own kernel launches
// (kda_profile_start / kda_profile_stop in include/kda.h).
//
// While a profile runs, every launch site brackets its kernel with two CUDA
// events recorded on the stream the kernel is launched on, so the summed
// event intervals are the kernels' device durations as they ran in the
// caller's schedule (overlapping side streams included).  Launches inside a
// stream capture are not timed.  No device memory is allocated: events only.
#include "kda_internal.h"

#include <atomic>
#include <mutex>
#include <vector>

namespace kda {
namespace {

struct Profile {
    std::mutex mu;
    std::atomic<bool> on{false};
    std::vector<cudaEvent_t> ev;  // two per timed launch: start, end
    std::vector<int> kind;        // kda_kernel_kind of each timed launch
    int used = 0;                 // timed launches so far
    int64_t dropped = 0;          // launches past the event budget
};

Profile &prof() {
    static Profile p;
    return p;
}

void destroy_events(Profile &g) {
    for (cudaEvent_t e : g.ev)
        if (e) cudaEventDestroy(e);
    g.ev.clear();
    g.kind.clear();
    g.used = 0;
    g.dropped = 0;
}

}  // namespace

ProfScope::ProfScope(int kind, cudaStream_t s) : s_(s) {
    Profile &g = prof();
    if (!g.on.load(std::memory_order_acquire)) return;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    if (cap != cudaStreamCaptureStatusNone) return;
    std::lock_guard<std::mutex> lock(g.mu);
    if (!g.on.load(std::memory_order_relaxed)) return;
    if (2 * (g.used + 1) > int(g.ev.size())) {
        ++g.dropped;
        return;
    }
    const int slot = g.used++;
    g.kind[size_t(slot)] = kind;
    if (cudaEventRecord(g.ev[2 * size_t(slot)], s) != cudaSuccess) {
        cudaGetLastError();
        g.kind[size_t(slot)] = -1;
        return;
    }
    slot_ = slot;
}

ProfScope::~ProfScope() {
    if (slot_ < 0) return;
    Profile &g = prof();
    std::lock_guard<std::mutex> lock(g.mu);
    if (size_t(2 * slot_ + 1) < g.ev.size() && cudaEventRecord(g.ev[2 * size_t(slot_) + 1], s_) != cudaSuccess) {
        cudaGetLastError();
        g.kind[size_t(slot_)] = -1;
    }
}

}  // namespace kda

extern "C" {

kda_status kda_profile_start(int32_t max_launches) {
    kda::Profile &g = kda::prof();
    if (max_launches <= 0 || max_launches > (1 << 20)) return KDA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g.mu);
    if (g.on.load()) return KDA_ERR_INVALID_ARG;
    kda::destroy_events(g);
    g.ev.assign(2 * size_t(max_launches), nullptr);
    g.kind.assign(size_t(max_launches), -1);
    for (cudaEvent_t &e : g.ev) {
        if (cudaEventCreate(&e) != cudaSuccess) {
            cudaGetLastError();
            e = nullptr;
            kda::destroy_events(g);
            return KDA_ERR_CUDA;
        }
    }
    g.on.store(true, std::memory_order_release);
    return KDA_OK;
}

kda_status kda_profile_stop(kda_profile *out) {
    kda::Profile &g = kda::prof();
    std::lock_guard<std::mutex> lock(g.mu);
    if (!g.on.load()) return KDA_ERR_INVALID_ARG;
    g.on.store(false, std::memory_order_release);
    kda_profile r = {};
    r.dropped = g.dropped;
    kda_status st = KDA_OK;
    for (int i = 0; i < g.used; ++i) {
        const int k = g.kind[size_t(i)];
        if (k < 0 || k >= KDA_KERNEL_COUNT) continue;
        float ms = 0.f;
        if (cudaEventSynchronize(g.ev[2 * size_t(i) + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, g.ev[2 * size_t(i)], g.ev[2 * size_t(i) + 1]) != cudaSuccess) {
            cudaGetLastError();
            st = KDA_ERR_CUDA;
            continue;
        }
        r.launches[k] += 1;
        r.ms[k] += double(ms);
    }
    kda::destroy_events(g);
    if (out) *out = r;
    return st;
}

}  // extern "C"
