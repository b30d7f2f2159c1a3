// Host runtime pieces of the library: device checks, status names, version.
#include <atomic>

#include "wgs_common.cuh"

namespace wgs {

namespace {

constexpr int kMaxDevices = 64;
// Per device: 0 = not probed yet, -1 = wrong architecture, > 0 = SM count.
std::atomic<int> g_device_sms[kMaxDevices];

}  // namespace

wgs_status current_device(DeviceInfo *info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WGS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return WGS_ERR_CUDA;
    int sms = g_device_sms[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        int major = 0, minor = 0, count = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return WGS_ERR_CUDA;
        sms = (major == 10 && minor == 3 && count > 0) ? count : -1;
        g_device_sms[dev].store(sms, std::memory_order_relaxed);
    }
    if (sms < 0) return WGS_ERR_ARCH;
    info->device = dev;
    info->sm_count = sms;
    return WGS_OK;
}

}  // namespace wgs

extern "C" const char *wgs_status_string(wgs_status s) {
    switch (s) {
        case WGS_OK: return "ok";
        case WGS_ERR_NULL: return "a required pointer is NULL";
        case WGS_ERR_SHAPE: return "invalid or inconsistent sizes";
        case WGS_ERR_WIDTH: return "width not supported by this entry point";
        case WGS_ERR_ALIGN: return "pointer not aligned as required";
        case WGS_ERR_DTYPE: return "unknown dtype";
        case WGS_ERR_ARCH: return "current CUDA device is not compute capability 10.3 (sm_103a)";
        case WGS_ERR_LAUNCH: return "kernel launch failed";
        case WGS_ERR_INDEX: return "a gather index was outside [-1, n_src)";
        case WGS_ERR_ALIAS: return "buffers overlap in a way the operation does not allow";
        case WGS_ERR_CUDA: return "a CUDA runtime call failed";
        case WGS_ERR_TOO_LARGE: return "problem larger than the library's fixed scratch array";
    }
    return "unknown status";
}

extern "C" int32_t wgs_abi_version(void) { return WGS_ABI_VERSION; }
