// abi.cu -- status strings, device queries and option handling for libwsw.so.
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace wsw {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices];
std::mutex g_mu;
}  // namespace

bool device_info(DeviceInfo *out, int *status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = WSW_ERR_CUDA;
        return false;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_have[dev]) {
            *out = g_info[dev];
            return true;
        }
    }
    int major = 0, minor = 0, sms = 0, smem = 0, l2 = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
        *status = WSW_ERR_CUDA;
        return false;
    }
    if (major != 10 || minor != 3) {
        *status = WSW_ERR_UNSUPPORTED;
        return false;
    }
    DeviceInfo d{dev, sms, smem, l2};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_info[dev] = d;
        g_have[dev] = true;
    }
    *out = d;
    return true;
}

int resolve_opts(const wsw_launch_opts *o, Opts *out) {
    Opts r{2, 32, false, 0, WSW_CHAIN_L2_PREFETCH_STEPS};
    if (o) {
        if (o->rows_per_warp != 0) {
            if (o->rows_per_warp != 1 && o->rows_per_warp != 2 && o->rows_per_warp != 4)
                return WSW_ERR_INVALID_ARG;
            r.rows_per_warp = o->rows_per_warp;
        }
        if (o->load_bytes != 0) {
            if (o->load_bytes != 32 && o->load_bytes != 16 && o->load_bytes != 8 &&
                o->load_bytes != 4 && o->load_bytes != 2)
                return WSW_ERR_INVALID_ARG;
            r.load_bytes = o->load_bytes;
        }
        if (o->pdl != 0 && o->pdl != 1) return WSW_ERR_INVALID_ARG;
        r.pdl = o->pdl == 1;
        if (o->ctas_per_sm < 0 || o->ctas_per_sm > 32) return WSW_ERR_INVALID_ARG;
        r.ctas_per_sm = o->ctas_per_sm;
        if (o->l2_prefetch_steps < -1 || o->l2_prefetch_steps > 64) return WSW_ERR_INVALID_ARG;
        if (o->l2_prefetch_steps != 0) r.l2_prefetch_steps = o->l2_prefetch_steps < 0 ? 0 : o->l2_prefetch_steps;
    }
    *out = r;
    return WSW_OK;
}

cudaError_t ensure_smem(const void *kernel, int bytes) {
    static std::map<std::pair<const void *, int>, int> granted;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = granted.find({kernel, dev});
        if (it != granted.end() && it->second >= bytes) return cudaSuccess;
    }
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lk(g_mu);
        int &g = granted[{kernel, dev}];
        if (g < bytes) g = bytes;
    }
    return e;
}

int load_width(const void *base, int64_t pitch_bytes, int cap) {
    uint64_t a = reinterpret_cast<uint64_t>(base) | static_cast<uint64_t>(pitch_bytes);
    int w = 32;
    while (w > 2 && (a % static_cast<uint64_t>(w)) != 0) w >>= 1;
    return w < cap ? w : cap;
}

}  // namespace wsw

extern "C" const char *wsw_status_string(int status) {
    switch (status) {
        case WSW_OK: return "WSW_OK";
        case WSW_ERR_INVALID_ARG: return "WSW_ERR_INVALID_ARG";
        case WSW_ERR_MISALIGNED: return "WSW_ERR_MISALIGNED";
        case WSW_ERR_UNSUPPORTED: return "WSW_ERR_UNSUPPORTED";
        case WSW_ERR_WORKSPACE: return "WSW_ERR_WORKSPACE";
        case WSW_ERR_CUDA: return "WSW_ERR_CUDA";
        case WSW_ERR_TIMEOUT: return "WSW_ERR_TIMEOUT";
        default: return "WSW_ERR_UNKNOWN";
    }
}

extern "C" int wsw_abi_version(void) { return WSW_ABI_VERSION; }
