// Optional per-kernel timing. When enabled (pkv_profile_enable), every
// kernel launch site brackets its launch with a pair of CUDA events recorded
// on the launching stream; pkv_profile_collect waits for them and returns the
// launch count and summed device time per kernel name. Off by default: a
// disabled ProfScope costs one relaxed atomic load.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace pkv {
namespace {

struct Record {
    const char* name;
    cudaEvent_t a, b;
};

std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Record> g_records;

void clear_records() {
    for (auto& r : g_records) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_records.clear();
}

}  // namespace

ProfScope::ProfScope(const char* n, cudaStream_t st) : name(n), s(st) {
    if (!g_enabled.load(std::memory_order_relaxed)) return;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    if (cudaEventCreate(&b) != cudaSuccess) {
        cudaEventDestroy(a);
        return;
    }
    cudaEventRecord(a, s);
    active = true;
}

ProfScope::~ProfScope() {
    if (!active) return;
    cudaEventRecord(b, s);
    std::lock_guard<std::mutex> lock(g_mu);
    g_records.push_back({name, a, b});
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_profile_enable(int32_t on) {
    std::lock_guard<std::mutex> lock(g_mu);
    clear_records();
    g_enabled.store(on ? 1 : 0);
    return PKV_OK;
}

extern "C" pkv_status pkv_profile_collect(int32_t max_kernels, char* names, double* total_ms,
                                          int64_t* launches, int32_t* n_kernels) {
    if (max_kernels < 0 || !n_kernels || (max_kernels > 0 && (!names || !total_ms || !launches)))
        return fail(PKV_ERR_INVALID, "pkv_profile_collect: bad argument");
    std::lock_guard<std::mutex> lock(g_mu);
    std::vector<std::string> order;
    std::vector<double> ms;
    std::vector<int64_t> cnt;
    for (auto& r : g_records) {
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e != cudaSuccess) return cuda_fail(e, "pkv_profile_collect: event");
        float t = 0.f;
        e = cudaEventElapsedTime(&t, r.a, r.b);
        if (e != cudaSuccess) return cuda_fail(e, "pkv_profile_collect: elapsed");
        size_t k = 0;
        while (k < order.size() && order[k] != r.name) ++k;
        if (k == order.size()) {
            order.push_back(r.name);
            ms.push_back(0.0);
            cnt.push_back(0);
        }
        ms[k] += t;
        cnt[k] += 1;
    }
    clear_records();
    *n_kernels = (int32_t)order.size();
    for (size_t k = 0; k < order.size() && (int32_t)k < max_kernels; ++k) {
        std::strncpy(names + 64 * k, order[k].c_str(), 63);
        names[64 * k + 63] = 0;
        total_ms[k] = ms[k];
        launches[k] = cnt[k];
    }
    return PKV_OK;
}
