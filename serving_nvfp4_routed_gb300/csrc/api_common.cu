// api_common.cu -- status strings, launch accounting and optional per-kernel
// event timing for libnvfp4moe.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace nvfp4 {

namespace {

std::mutex g_mu;
unsigned long long g_launches = 0;
std::atomic<int> g_kernel_choice{0};
bool g_profile = false;

struct Pending {
    std::string name;
    cudaEvent_t start, stop;
};
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_pool;
cudaEvent_t g_open = nullptr;

struct Total {
    int launches = 0;
    double ms = 0.0;
};
std::map<std::string, Total> g_totals;

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e;
    cudaEventCreate(&e);
    return e;
}

}  // namespace

void launch_begin(const char* name, cudaStream_t s) {
    (void)name;
    std::lock_guard<std::mutex> lk(g_mu);
    ++g_launches;
    if (g_profile) {
        g_open = take_event();
        cudaEventRecord(g_open, s);
    }
}

void launch_end(const char* name, cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_profile && g_open) {
        cudaEvent_t stop = take_event();
        cudaEventRecord(stop, s);
        g_pending.push_back({name, g_open, stop});
        g_open = nullptr;
    }
}

bool pdl_enabled() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("NVFP4_NO_PDL");
        v = (e && e[0] && e[0] != '0') ? 0 : 1;
    }
    return v == 1;
}

int kernel_choice() { return g_kernel_choice.load(std::memory_order_relaxed); }

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

int device_cc_major() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev);
    return v;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" const char* nvfp4_status_string(nvfp4_status s) {
    switch (s) {
        case NVFP4_OK: return "NVFP4_OK";
        case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
        case NVFP4_ERR_SHAPE: return "NVFP4_ERR_SHAPE";
        case NVFP4_ERR_ALIGN: return "NVFP4_ERR_ALIGN";
        case NVFP4_ERR_WORKSPACE: return "NVFP4_ERR_WORKSPACE";
        case NVFP4_ERR_UNSUPPORTED: return "NVFP4_ERR_UNSUPPORTED";
        case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
        case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
        case NVFP4_ERR_DEVICE_INPUT: return "NVFP4_ERR_DEVICE_INPUT";
    }
    return "NVFP4_ERR_UNKNOWN";
}

extern "C" nvfp4_status nvfp4_set_kernel_choice(int choice) {
    if (choice < 0 || choice > 4) return NVFP4_ERR_INVALID_ARG;
    g_kernel_choice.store(choice, std::memory_order_relaxed);
    return NVFP4_OK;
}

extern "C" uint64_t nvfp4_launch_count(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_launches;
}

extern "C" void nvfp4_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_profile = on != 0;
}

extern "C" int nvfp4_profile_collect(int max, char* names, int* launches, double* ms) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& p : g_pending) {
        float t = 0.0f;
        cudaEventSynchronize(p.stop);
        cudaEventElapsedTime(&t, p.start, p.stop);
        Total& tot = g_totals[p.name];
        tot.launches += 1;
        tot.ms += t;
        g_pool.push_back(p.start);
        g_pool.push_back(p.stop);
    }
    g_pending.clear();
    int n = 0;
    for (auto& kv : g_totals) {
        if (n >= max) break;
        if (names) {
            std::strncpy(names + 64 * n, kv.first.c_str(), 63);
            names[64 * n + 63] = 0;
        }
        if (launches) launches[n] = kv.second.launches;
        if (ms) ms[n] = kv.second.ms;
        ++n;
    }
    g_totals.clear();
    return n;
}
