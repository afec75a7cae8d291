// wait_check.cu -- runs the bounded mbarrier wait of the tensor-core kernels on its own,
// so that its give-up path can be checked on a GPU without breaking a pipeline.
//
// One thread initialises a shared-memory mbarrier for one arrival, arrives on it or not,
// and waits for phase 0 with tc::mbar_wait.  With the arrival the phase completes and the
// wait returns at once; without it nothing can complete the phase, the wait gives up after
// its time limit (about a second) and the kernel writes WSW_ERR_TIMEOUT for the host to
// read.  The kernel then returns normally, so the context stays usable.
#include "tc_util.cuh"

namespace wsw {
namespace {

__global__ void bounded_wait_check_kernel(int arrive, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (arrive) tc::mbar_arrive(&bar);
    *status = tc::mbar_wait(&bar, 0) ? WSW_OK : WSW_ERR_TIMEOUT;
}

}  // namespace
}  // namespace wsw

extern "C" int wsw_bounded_wait_check(int32_t arrive, int32_t *status, void *stream) {
    using namespace wsw;
    if ((arrive != 0 && arrive != 1) || !status) return WSW_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(status) & 3) return WSW_ERR_MISALIGNED;
    DeviceInfo di;
    int st = WSW_OK;
    if (!device_info(&di, &st)) return st;
    const cudaError_t e = launch(bounded_wait_check_kernel, dim3(1), dim3(32), 0,
                                 static_cast<cudaStream_t>(stream), false, arrive, status);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
