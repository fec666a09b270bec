// Optional per-kernel timing: when enabled, every kernel launch of the
// library is bracketed by two CUDA events recorded on the launching stream;
// mhc_profiler_collect() waits for them and sums the elapsed time per
// kernel name.  Off by default; costs nothing when off.
#include <atomic>
#include <mutex>
#include <string.h>
#include <vector>

#include "../../include/mhc.h"
#include "launch.h"

namespace mhc {
namespace {

struct Rec {
    const char *name;
    cudaEvent_t a, b;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;
thread_local long g_open = -1;

cudaEvent_t take_event()
{
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

void prof_begin(const char *name, cudaStream_t s)
{
    if (!g_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    Rec r{name, take_event(), take_event()};
    if (!r.a || !r.b) return;
    cudaEventRecord(r.a, s);
    g_recs.push_back(r);
    g_open = long(g_recs.size()) - 1;
}

void prof_end(cudaStream_t s)
{
    if (!g_on.load(std::memory_order_relaxed) || g_open < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_open < long(g_recs.size())) cudaEventRecord(g_recs[g_open].b, s);
    g_open = -1;
}

}  // namespace mhc

extern "C" {

void mhc_profiler_enable(int on) { mhc::g_on.store(on != 0); }

int mhc_profiler_collect(mhc_kernel_time *out, int max)
{
    using namespace mhc;
    std::lock_guard<std::mutex> lk(g_mu);
    std::vector<mhc_kernel_time> agg;
    for (const Rec &r : g_recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
            cudaGetLastError();
            ms = 0.f;
        }
        size_t i = 0;
        for (; i < agg.size(); ++i)
            if (strncmp(agg[i].name, r.name, sizeof agg[i].name) == 0) break;
        if (i == agg.size()) {
            mhc_kernel_time k;
            memset(&k, 0, sizeof k);
            strncpy(k.name, r.name, sizeof k.name - 1);
            agg.push_back(k);
        }
        agg[i].launches += 1;
        agg[i].total_ms += ms;
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_recs.clear();
    int n = int(agg.size());
    for (int i = 0; i < n && i < max && out; ++i) out[i] = agg[i];
    return n;
}

}  // extern "C"
