// Per-kernel CUDA-event timing behind fa_profile_start / fa_profile_stop.
// While a session is active every launch site brackets its kernel with two
// events recorded on the launch stream; stopping synchronises them and sums
// the durations per kernel kind.  On a stream that is being captured into a
// CUDA graph the two events become event-record nodes of the graph, so the
// durations are those of the graph's launch.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

struct Record {
    int kind;
    cudaEvent_t begin, end;
};

std::mutex g_mu;
bool g_active = false;
bool g_pending = false;
bool g_overflow = false;
int g_pending_kind = 0;
std::vector<cudaEvent_t> g_pool;
std::vector<Record> g_records;
long long g_launches[FA_KERNEL_COUNT];

// Records e on s; while s is being captured, as an external event-record node
// (a plain record there would only order the capture).
cudaError_t record(cudaEvent_t e, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    return cudaEventRecord(e, s);
}

bool ensure_pool(size_t n) {
    while (g_pool.size() < n) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return false;
        g_pool.push_back(e);
    }
    return true;
}

}  // namespace

namespace fa {

void prof_begin(int kind, cudaStream_t stream) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_active || kind < 0 || kind >= FA_KERNEL_COUNT) return;
    ++g_launches[kind];
    g_pending = false;
    const size_t i = g_records.size();
    if (i >= static_cast<size_t>(FA_PROFILE_MAX_LAUNCHES) || !ensure_pool(2 * i + 2)) {
        g_overflow = true;
        return;
    }
    if (record(g_pool[2 * i], stream) != cudaSuccess) {
        g_overflow = true;
        return;
    }
    g_pending = true;
    g_pending_kind = kind;
}

void prof_end(int kind, cudaStream_t stream) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_active || !g_pending || kind != g_pending_kind) return;
    const size_t i = g_records.size();
    if (record(g_pool[2 * i + 1], stream) != cudaSuccess) {
        g_overflow = true;
        g_pending = false;
        return;
    }
    g_records.push_back({kind, g_pool[2 * i], g_pool[2 * i + 1]});
    g_pending = false;
}

}  // namespace fa

extern "C" {

int fa_profile_start(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!ensure_pool(8192)) return FA_ERR_CUDA;
    g_records.clear();
    for (long long& c : g_launches) c = 0;
    g_overflow = false;
    g_pending = false;
    g_active = true;
    return FA_OK;
}

int fa_profile_stop(int n, int64_t* launches, double* total_ms) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_active = false;
    double ms[FA_KERNEL_COUNT] = {0};
    int rc = FA_OK;
    for (const Record& r : g_records) {
        if (cudaEventSynchronize(r.end) != cudaSuccess) {
            rc = FA_ERR_CUDA;
            continue;
        }
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.begin, r.end) != cudaSuccess) {
            rc = FA_ERR_CUDA;
            continue;
        }
        ms[r.kind] += t;
    }
    for (int k = 0; k < n && k < FA_KERNEL_COUNT; ++k) {
        if (launches) launches[k] = g_launches[k];
        if (total_ms) total_ms[k] = ms[k];
    }
    g_records.clear();
    if (rc == FA_OK && g_overflow) rc = FA_ERR_ALLOC;
    return rc;
}

}  // extern "C"
