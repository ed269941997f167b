// Host-side plumbing of libmlasparse: the device error word, SM-count cache,
// mla_get_error and mla_strerror.
#include <mutex>
#include <utility>
#include <vector>

#include "mla_device.cuh"

namespace {

// One error word per device; every kernel of the library receives its address.
__device__ int g_mla_error_word = 0;

constexpr int kMaxDevices = 64;
int* g_err_addr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::vector<std::pair<int, const void*>> g_smem_set;   // (device, kernel) pairs already raised
std::mutex g_mu;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

}  // namespace

namespace mla_host {

int* device_error_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_err_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mla_error_word) != cudaSuccess) return nullptr;
        g_err_addr[dev] = static_cast<int*>(p);
    }
    return g_err_addr[dev];
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

bool max_dynamic_smem(const void* kernel, int bytes) {
    const int dev = current_device();
    if (dev < 0) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    for (const auto& p : g_smem_set)
        if (p.first == dev && p.second == kernel) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    g_smem_set.emplace_back(dev, kernel);
    return true;
}

}  // namespace mla_host

extern "C" int mla_get_error(int32_t* host_code) {
    if (host_code == nullptr) return MLA_EINVAL;
    int* addr = mla_host::device_error_word();
    if (addr == nullptr) return MLA_ECUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ECUDA;
    int v = 0;
    if (cudaMemcpy(&v, addr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ECUDA;
    const int zero = 0;
    if (cudaMemcpy(addr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return MLA_ECUDA;
    *host_code = v;
    return MLA_OK;
}

extern "C" const char* mla_strerror(int code) {
    switch (code) {
        case MLA_OK: return "MLA_OK";
        case MLA_EINVAL: return "MLA_EINVAL: invalid argument";
        case MLA_EUNSUPPORTED: return "MLA_EUNSUPPORTED: unsupported shape";
        case MLA_ENOWORKSPACE: return "MLA_ENOWORKSPACE: workspace missing or too small";
        case MLA_ECUDA: return "MLA_ECUDA: CUDA runtime error";
        default: return "unknown libmlasparse error code";
    }
}
