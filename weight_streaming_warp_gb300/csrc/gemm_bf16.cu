// gemm_bf16.cu -- small-batch prefill product Y[n][r] = sum_k W[r][k] * X[n][k].
//
// Source: "ggml-cuda: pad matmul weight rows to avoid cache-set aliasing" (AMD-Ecosystem
// llama.cpp PR), Overview and Results: in small-batch prefill a short run of output
// rows streams the whole weight matrix, the weight's row stride may carry one extra
// 128-byte line, and the matmul takes its leading dimension from the row stride.
//
// Warp-level bf16 tensor-core tiles (m16n8k16, fp32 accumulation): a warp owns 16
// weight rows and 32 batch columns and walks K in steps of 16; fragments are read
// straight from global memory (each weight element is fetched by one warp per 32
// batch columns).
#include "common.cuh"

namespace wsw {
namespace {

constexpr int kWarps = 4;
constexpr int kNB = 4;  // 8-column MMA tiles per warp

__device__ __forceinline__ uint32_t ld_pair(const uint16_t *base, int64_t row, int64_t nrows,
                                            int64_t ld, int64_t k, int64_t K) {
    if (row >= nrows) return 0u;
    const uint16_t *p = base + row * ld + k;
    if (k + 1 < K) return *reinterpret_cast<const uint32_t *>(p);
    if (k < K) return static_cast<uint32_t>(p[0]);
    return 0u;
}

__global__ void __launch_bounds__(kWarps * 32) gemm_bf16_mma_kernel(
    const uint16_t *__restrict__ W, int64_t M, int64_t K, int64_t ld, const uint16_t *__restrict__ X,
    int64_t N, int64_t ldx, float *__restrict__ Y) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tg = lane & 3;
    const int64_t r0 = (static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * 16;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * 8 * kNB;
    if (r0 >= M) return;
    float c[kNB][4];
#pragma unroll
    for (int j = 0; j < kNB; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.0f;
    for (int64_t k0 = 0; k0 < K; k0 += 16) {
        const uint32_t a0 = ld_pair(W, r0 + g, M, ld, k0 + 2 * tg, K);
        const uint32_t a1 = ld_pair(W, r0 + g + 8, M, ld, k0 + 2 * tg, K);
        const uint32_t a2 = ld_pair(W, r0 + g, M, ld, k0 + 2 * tg + 8, K);
        const uint32_t a3 = ld_pair(W, r0 + g + 8, M, ld, k0 + 2 * tg + 8, K);
#pragma unroll
        for (int j = 0; j < kNB; ++j) {
            const int64_t n = n0 + 8 * j + g;
            const uint32_t b0 = ld_pair(X, n, N, ldx, k0 + 2 * tg, K);
            const uint32_t b1 = ld_pair(X, n, N, ldx, k0 + 2 * tg + 8, K);
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
#pragma unroll
    for (int j = 0; j < kNB; ++j) {
        const int64_t n = n0 + 8 * j + 2 * tg;
        const int64_t r = r0 + g;
        if (n < N && r < M) Y[n * M + r] = c[j][0];
        if (n + 1 < N && r < M) Y[(n + 1) * M + r] = c[j][1];
        if (n < N && r + 8 < M) Y[n * M + r + 8] = c[j][2];
        if (n + 1 < N && r + 8 < M) Y[(n + 1) * M + r + 8] = c[j][3];
    }
}

}  // namespace
}  // namespace wsw

extern "C" int wsw_gemm_bf16(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const uint16_t *X,
                             int64_t N, int64_t ldx, float *Y, void *stream, const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (M < 0 || N < 0 || K < 0 || ld < K || ldx < K) return WSW_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return WSW_OK;
    if (!W || !X || !Y) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15) || (reinterpret_cast<uintptr_t>(X) & 15) ||
        (reinterpret_cast<uintptr_t>(Y) & 3) || (K % 8) || (ld % 8) || (ldx % 8))
        return WSW_ERR_MISALIGNED;
    if (M > (int64_t(1) << 31) || N > 65535 * 8 * kNB) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return cudaMemsetAsync(Y, 0, static_cast<size_t>(M) * N * 4, s) == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
    const dim3 grid(static_cast<unsigned>((M + 16 * kWarps - 1) / (16 * kWarps)),
                    static_cast<unsigned>((N + 8 * kNB - 1) / (8 * kNB)));
    cudaError_t e = launch(gemm_bf16_mma_kernel, grid, dim3(kWarps * 32), 0, s, o.pdl, W, M, K, ld, X, N, ldx, Y);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
