// profile.cu -- optional per-kernel timing.  When enabled, every launch the
// library enqueues is bracketed by two CUDA events recorded on the launch
// stream; sparse_profile_read() waits for the recorded events and reports, per
// kernel name, the number of launches and the summed GPU time.  Off by default:
// then a launch site costs one relaxed atomic load.
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "profile.cuh"

namespace so {
namespace prof {

namespace {
struct Pending {
    const char* name;
    cudaEvent_t start, stop;
};
struct Total {
    const char* name;
    int64_t launches;
    double ms;
};
std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Pending> g_pending;
std::vector<Total> g_totals;
std::vector<cudaEvent_t> g_free;

cudaEvent_t take_event()
{
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

void drain_locked()
{
    for (const Pending& p : g_pending) {
        float ms = 0.0f;
        if (p.start && p.stop && cudaEventSynchronize(p.stop) == cudaSuccess &&
            cudaEventElapsedTime(&ms, p.start, p.stop) == cudaSuccess) {
            bool found = false;
            for (Total& t : g_totals)
                if (std::strcmp(t.name, p.name) == 0) {
                    t.launches += 1;
                    t.ms += ms;
                    found = true;
                    break;
                }
            if (!found) g_totals.push_back(Total{p.name, 1, static_cast<double>(ms)});
        }
        if (p.start) g_free.push_back(p.start);
        if (p.stop) g_free.push_back(p.stop);
    }
    g_pending.clear();
}

bool enabled() { return g_enabled.load(std::memory_order_relaxed) != 0; }

Scope::Scope(const char* name, cudaStream_t s) : name_(name), stream_(s), start_(nullptr)
{
    if (!enabled()) return;
    std::lock_guard<std::mutex> lk(g_mu);
    start_ = take_event();
    if (start_) cudaEventRecord(start_, stream_);
}

Scope::~Scope()
{
    if (!start_) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t stop = take_event();
    if (stop) cudaEventRecord(stop, stream_);
    g_pending.push_back(Pending{name_, start_, stop});
}

}  // namespace prof
}  // namespace so

extern "C" {

void sparse_profile_enable(int enable)
{
    so::prof::g_enabled.store(enable ? 1 : 0, std::memory_order_relaxed);
}

void sparse_profile_reset(void)
{
    std::lock_guard<std::mutex> lk(so::prof::g_mu);
    so::prof::drain_locked();
    so::prof::g_totals.clear();
}

int sparse_profile_read(int max_entries, const char** names, int64_t* launches, double* total_ms)
{
    std::lock_guard<std::mutex> lk(so::prof::g_mu);
    so::prof::drain_locked();
    const int n = static_cast<int>(so::prof::g_totals.size());
    for (int i = 0; i < n && i < max_entries; ++i) {
        if (names) names[i] = so::prof::g_totals[i].name;
        if (launches) launches[i] = so::prof::g_totals[i].launches;
        if (total_ms) total_ms[i] = so::prof::g_totals[i].ms;
    }
    return n;
}

}  // extern "C"
