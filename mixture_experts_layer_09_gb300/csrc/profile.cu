// profile.cu -- launch counter and optional per-kernel CUDA-event timing.
//
// Every kernel launch of the library passes through a KernelScope, which counts it.  When
// timing is switched on (moe_profile_enable), the scope also records a CUDA event pair on the
// launching stream around the kernel; moe_profile_read waits for the recorded events and
// returns the summed device time per kernel name.  Events come from a pool created on first
// use; this is host-side bookkeeping only and allocates no device memory.
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {
struct Pending {
    const char* name;
    cudaEvent_t b, e;
};
struct Acc {
    double ms = 0.0;
    long launches = 0;
};
std::mutex g_mu;
std::atomic<bool> g_enabled{false};
std::atomic<long long> g_launches{0};
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_pool;
std::map<std::string, Acc> g_acc;

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void settle_locked() {
    for (const Pending& p : g_pending) {
        float ms = 0.f;
        if (p.b && p.e && cudaEventSynchronize(p.e) == cudaSuccess && cudaEventElapsedTime(&ms, p.b, p.e) == cudaSuccess) {
            Acc& a = g_acc[p.name];
            a.ms += ms;
            a.launches += 1;
        }
        if (p.b) g_pool.push_back(p.b);
        if (p.e) g_pool.push_back(p.e);
    }
    g_pending.clear();
}
}  // namespace

KernelScope::KernelScope(const char* name, cudaStream_t st) : st_(st), idx_(-1) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_enabled.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    Pending p{name, take_event(), take_event()};
    if (p.b) cudaEventRecord(p.b, st);
    g_pending.push_back(p);
    idx_ = static_cast<int>(g_pending.size()) - 1;
}

KernelScope::~KernelScope() {
    if (idx_ < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (idx_ < static_cast<int>(g_pending.size()) && g_pending[idx_].e) cudaEventRecord(g_pending[idx_].e, st_);
}

}  // namespace moe

extern "C" {

MOE_API int moe_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(moe::g_mu);
    moe::settle_locked();
    moe::g_acc.clear();
    moe::g_enabled.store(on != 0);
    return MOE_OK;
}

MOE_API long long moe_launch_count(void) { return moe::g_launches.load(); }

MOE_API int moe_profile_read(int max_n, char* names, int name_len, double* ms, long* launches, int* n) {
    if (!n || max_n < 0 || (max_n > 0 && (!names || !ms || !launches || name_len < 2))) return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(moe::g_mu);
    moe::settle_locked();
    int i = 0;
    for (const auto& kv : moe::g_acc) {
        if (i >= max_n) break;
        std::string s = kv.first.substr(0, name_len - 1);
        std::copy(s.begin(), s.end(), names + static_cast<size_t>(i) * name_len);
        names[static_cast<size_t>(i) * name_len + s.size()] = 0;
        ms[i] = kv.second.ms;
        launches[i] = kv.second.launches;
        ++i;
    }
    *n = static_cast<int>(moe::g_acc.size());
    return MOE_OK;
}

}  // extern "C"
