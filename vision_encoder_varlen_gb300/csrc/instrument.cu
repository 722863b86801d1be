// Launch counting and optional per-launch CUDA-event timing of the library's kernels.
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

namespace vit {
namespace {

std::atomic<int64_t> g_launches{0};
std::atomic<int> g_timing{0};

struct Record {
    const char *name;
    cudaEvent_t start, stop;
};

std::mutex g_mutex;
std::vector<Record> g_records;           // launches timed since the last read
std::vector<cudaEvent_t> g_free_events;  // recycled events

cudaEvent_t take_event()
{
    if (!g_free_events.empty()) {
        cudaEvent_t e = g_free_events.back();
        g_free_events.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

LaunchScope::LaunchScope(const char *name, cudaStream_t stream) : name_(name), stream_(stream), slot_(nullptr)
{
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_timing.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_mutex);
    Record *r = new Record{name, take_event(), take_event()};
    if (r->start) cudaEventRecord(r->start, stream);
    slot_ = r;
}

LaunchScope::~LaunchScope()
{
    if (!slot_) return;
    Record *r = static_cast<Record *>(slot_);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (r->stop) cudaEventRecord(r->stop, stream_);
    g_records.push_back(*r);
    delete r;
}

}  // namespace vit

using namespace vit;

extern "C" {

int64_t vit_launch_count(void) { return g_launches.load(); }

int vit_kernel_timing(int enable) { return g_timing.exchange(enable ? 1 : 0); }

int vit_kernel_timing_read(vit_kernel_time_t *out, int max_entries)
{
    std::vector<Record> recs;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        recs.swap(g_records);
    }
    int n = 0;
    int rc = 0;
    for (const Record &r : recs) {
        float ms = 0.f;
        if (!r.start || !r.stop || cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
            rc = -1;
            continue;
        }
        int idx = -1;
        for (int i = 0; i < n; ++i)
            if (strcmp(out[i].name, r.name) == 0) idx = i;
        if (idx < 0) {
            if (n >= max_entries) continue;
            idx = n++;
            out[idx].name = r.name;
            out[idx].launches = 0;
            out[idx].total_ms = 0.0;
        }
        out[idx].launches += 1;
        out[idx].total_ms += ms;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    for (const Record &r : recs) {
        if (r.start) g_free_events.push_back(r.start);
        if (r.stop) g_free_events.push_back(r.stop);
    }
    return rc < 0 ? rc : n;
}

}  // extern "C"
