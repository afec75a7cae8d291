// moe_noalloc.cu -- wsw_moe_gemv_q8_0_noalloc: the grouped q8_0 MoE mat-vec for callers
// that cannot allocate device memory.
//
// Some callers of this library have no way to allocate: a plugin or custom-operator
// interface of a serving engine that hands over only the input and output buffers, a
// runtime that reserves all device memory in its own pool at start-up and refuses later
// allocations, or a latency-critical path that cannot afford cudaMalloc's implicit
// device synchronisation.  Such callers cannot provide the workspace that the
// tensor-core form of wsw_moe_gemv_q8_0 needs.  This entry point uses a fixed scratch
// array that is part of the library image instead.
//
// The array is a file-scope __device__ variable of kScratchBytes (8 MiB).  Every GPU
// that loads the library holds it until the process exits.  In host code its name is
// only a stand-in for the device variable, so its device address is looked up once per
// device (cudaGetSymbolAddress, with that device current) and passed to the kernels.
#include <map>
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_moe_scratch[kScratchBytes];

std::mutex g_scratch_mu;
std::map<int, void *> g_scratch_ptr;  // device ordinal -> device address of g_moe_scratch

// The scratch array's device address on the current device (looked up on the first call
// there), or nullptr with *status set when the lookup fails.
void *scratch_on_current_device(int *status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        *status = WSW_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    auto it = g_scratch_ptr.find(dev);
    if (it != g_scratch_ptr.end()) return it->second;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_moe_scratch) != cudaSuccess || ptr == nullptr) {
        *status = WSW_ERR_CUDA;
        return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
    return ptr;
}

}  // namespace

extern "C" size_t wsw_moe_workspace_bytes(int64_t E, int64_t K, int64_t R);
extern "C" int wsw_moe_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K,
                                 const int8_t *xq, const uint16_t *xd, const int32_t *ids, int64_t R,
                                 float *y, int32_t *err_flag, void *ws, size_t ws_bytes, void *stream,
                                 const wsw_launch_opts *opts);

// Same contract and results as wsw_moe_gemv_q8_0 with a workspace, but the workspace is
// the library's own scratch array.  Sizes whose workspace would exceed it are refused
// with WSW_ERR_UNSUPPORTED before anything is launched.  Nothing in this call
// allocates: no cudaMalloc, cudaFree or allocating library routine.
extern "C" int wsw_moe_gemv_q8_0_noalloc(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K,
                                         const int8_t *xq, const uint16_t *xd, const int32_t *ids, int64_t R,
                                         float *y, int32_t *err_flag, void *stream, const wsw_launch_opts *opts) {
    const size_t need = wsw_moe_workspace_bytes(E, K, R);
    if (need > kScratchBytes) return WSW_ERR_UNSUPPORTED;
    if (need == 0)  // these sizes run without scratch
        return wsw_moe_gemv_q8_0(Wq, Wd, E, Mo, K, xq, xd, ids, R, y, err_flag, nullptr, 0, stream, opts);
    int st = WSW_OK;
    void *scratch = scratch_on_current_device(&st);
    if (scratch == nullptr) return st;
    return wsw_moe_gemv_q8_0(Wq, Wd, E, Mo, K, xq, xd, ids, R, y, err_flag, scratch, kScratchBytes, stream, opts);
}
