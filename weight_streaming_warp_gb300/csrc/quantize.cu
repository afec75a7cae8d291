// quantize.cu -- block quantizer of the activation, q8_0 (32-element blocks, fp16
// scale) and the 256-element superblock (fp32 scale).
//
// Source: "QuantizeQ8KK is thread-per-superblock: 95.5us/call against llama.cpp's
// 1.6us ..." (vllm.cpp issue), sections Cause and The donor.  The page measures a
// thread-per-superblock decomposition (16 threads at a 4096-wide hidden state, two
// loads per element in the amax scan) against a per-element decomposition with a
// warp reduction for the scale.  Here every thread owns 8 consecutive values (two
// 16-byte loads, each value loaded once), a block is 4 (q8_0) or 32 (superblock)
// adjacent lanes, and amax is reduced with warp shuffles inside that lane group.
//
// The per-block arithmetic (q8_math.cuh): amax = max |x|; d = amax / 127 (IEEE fp32
// division); q = round-half-away(x / d) (IEEE fp32 division by the fp32 d, then
// roundf), clamped to [-127, 127]; an all-zero block stores d = +0 and q = 0.
#include <cuda_fp16.h>

#include "common.cuh"
#include "q8_math.cuh"

namespace wsw {
namespace {

constexpr int kQThreads = 256;

template <int BLOCK, bool VEC>
__global__ void __launch_bounds__(kQThreads)
    quantize_q8_kernel(const float *__restrict__ x, int64_t lanes_per_row, int64_t total,
                       int64_t n, int64_t ldx, int8_t *__restrict__ q, void *__restrict__ scales) {
    constexpr int LPB = BLOCK / 8;  // lanes per block
    // The consumer of q (a quantized mat-vec) may start streaming its weights now.
    pdl_launch_dependents();
    pdl_wait();  // x is written by the previous kernel in the stream

    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < total; base += stride) {
        const int64_t g = base + threadIdx.x;
        const bool active = g < total;  // lane groups are all active or all idle
        const int64_t row = active ? g / lanes_per_row : 0;
        const int64_t j = active ? g - row * lanes_per_row : 0;
        float v[8];
        if (active) {
            const float *src = x + row * ldx + 8 * j;
            if constexpr (VEC) {
                const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
                const float4 b = __ldg(reinterpret_cast<const float4 *>(src) + 1);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = __ldg(src + i);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        const float amax = q8m::block_amax<BLOCK>(v);
        if (!active) continue;

        const float d = q8m::scale(amax);
        uint32_t packed[2];
        q8m::codes(v, amax, d, packed);
        int8_t *dst = q + row * n + 8 * j;
        if (VEC) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = static_cast<int8_t>((packed[i >> 2] >> (8 * (i & 3))) & 0xffu);
        }
        if ((j % LPB) == 0) {
            const int64_t b = row * (n / BLOCK) + (8 * j) / BLOCK;
            if constexpr (BLOCK == 32)
                static_cast<__half *>(scales)[b] = __float2half_rn(d);
            else
                static_cast<float *>(scales)[b] = d;
        }
    }
}

template <int BLOCK>
cudaError_t launch_quantize(bool vec, dim3 grid, cudaStream_t s, bool pdl, const float *x,
                            int64_t lpr, int64_t total, int64_t n, int64_t ldx, int8_t *q,
                            void *scales) {
    if (vec)
        return launch(quantize_q8_kernel<BLOCK, true>, grid, dim3(kQThreads), 0, s, pdl, x, lpr,
                      total, n, ldx, q, scales);
    return launch(quantize_q8_kernel<BLOCK, false>, grid, dim3(kQThreads), 0, s, pdl, x, lpr, total,
                  n, ldx, q, scales);
}

}  // namespace
}  // namespace wsw

extern "C" int wsw_quantize_q8(const float *x, int64_t rows, int64_t n, int64_t ldx, int32_t block,
                               int8_t *q, void *scales, void *stream, const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (block != 32 && block != 256) return WSW_ERR_INVALID_ARG;
    if (rows < 0 || n < 0 || n % block != 0 || ldx < n) return WSW_ERR_INVALID_ARG;
    if (rows == 0 || n == 0) return WSW_OK;
    if (!x || !q || !scales) return WSW_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(x) % 4 != 0) return WSW_ERR_MISALIGNED;
    if (block == 32 && reinterpret_cast<uintptr_t>(scales) % 2 != 0) return WSW_ERR_MISALIGNED;
    if (block == 256 && reinterpret_cast<uintptr_t>(scales) % 4 != 0) return WSW_ERR_MISALIGNED;
    if (rows > (int64_t(1) << 40) / (n > 0 ? n : 1)) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;

    const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ldx % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(q) % 8 == 0);
    const int64_t lpr = n / 8;
    const int64_t total = rows * lpr;
    int64_t blocks = (total + kQThreads - 1) / kQThreads;
    const int64_t cap = static_cast<int64_t>(di.sm_count) * 8;
    if (blocks > cap) blocks = cap;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = block == 32
                        ? launch_quantize<32>(vec, dim3(static_cast<unsigned>(blocks)), s, o.pdl, x,
                                              lpr, total, n, ldx, q, scales)
                        : launch_quantize<256>(vec, dim3(static_cast<unsigned>(blocks)), s, o.pdl, x,
                                               lpr, total, n, ldx, q, scales);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
