// dequant_kv.cu -- one-pass dequantization of a q8_0 K or V cache into a
// per-head-contiguous binary16 buffer.
//
// Source: "vulkan : dequant q8_0 KV once in coopmat1" (llama.cpp PR), Overview and the
// stride discussion.  The cache is position-major with the heads interleaved
// (ne = [head_dim, KV, n_head_kv], nb[1] = head_dim * n_head_kv * elem), so one head's
// rows are head_dim * heads elements apart.  Dequantizing once and writing the result
// per head ([head][pos][dim]) lets the attention consumer read each head sequentially;
// the page measures the strided walk costing up to 3.2x on a low-bandwidth part.
//
//   out[h][p][i] = f16_rn(fp32(d[p][h][i/32]) * q[p][h][i])
// The fp32 product is exact (11 x 8 significant bits); __float2half_rn rounds once.
//
// Each thread converts 16 values (one 16-byte load, two 16-byte stores); a CTA covers
// 4 x 256 consecutive 16-value pieces of the input, requested into L2 before the
// dependency wait and loaded before the first conversion.  Reads are sequential in input order; each group of head_dim/16 threads
// writes one contiguous output row.
#include <cuda_fp16.h>

#include "common.cuh"

namespace wsw {
namespace {

constexpr int kThreads = 256;
constexpr int kPieces = 4;  // 16-value pieces per thread

template <bool VEC>
__global__ void __launch_bounds__(kThreads) dequant_q8_0_kv_kernel(
    const int8_t *__restrict__ q, const uint16_t *__restrict__ d, int64_t depth, int64_t heads,
    int64_t head_dim, uint16_t *__restrict__ out, int64_t npieces) {
    pdl_launch_dependents();
    // This CTA's input lines are requested into L2 before the dependency wait: L2 is the
    // point of coherence, so lines an earlier kernel is still writing (the newly appended
    // positions) are read correctly after the wait, and the rest arrive early.
    {
        const int64_t p0 = static_cast<int64_t>(blockIdx.x) * kPieces * kThreads;
        const int64_t p1 = p0 + kPieces * kThreads < npieces ? p0 + kPieces * kThreads : npieces;
        prefetch_range_l2(q + 16 * p0, 16 * (p1 - p0));
        prefetch_range_l2(d + p0 / 2, (p1 - p0));  // one binary16 scale per two pieces
    }
    pdl_wait();  // the cache is written by earlier kernels
    const int64_t per_pos = heads * head_dim / 16;  // pieces per position
    const int64_t per_head = head_dim / 16;         // pieces per head row
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kPieces * kThreads + threadIdx.x;
    uint4 v[kPieces];
    uint32_t db[kPieces];
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
        const int64_t t = base + static_cast<int64_t>(u) * kThreads;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        db[u] = 0u;
        if (t < npieces) {
            if (VEC) {
                v[u] = __ldg(reinterpret_cast<const uint4 *>(q) + t);
            } else {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
                for (int i = 0; i < 16; ++i)
                    w[i >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(q[16 * t + i])) << (8 * (i & 3));
                v[u] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            db[u] = __ldg(d + (t >> 1));  // 32 values per scale = two pieces
        }
    }
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
        const int64_t t = base + static_cast<int64_t>(u) * kThreads;
        if (t >= npieces) continue;
        const int64_t p = t / per_pos;
        const int64_t rem = t - p * per_pos;
        const int64_t h = rem / per_head;
        const int64_t i0 = (rem - h * per_head) * 16;
        const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(db[u])));
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int b0 = static_cast<int8_t>((w[i >> 1] >> (16 * (i & 1))) & 0xffu);
            const int b1 = static_cast<int8_t>((w[i >> 1] >> (16 * (i & 1) + 8)) & 0xffu);
            const uint32_t h0 = __half_as_ushort(__float2half_rn(s * static_cast<float>(b0)));
            const uint32_t h1 = __half_as_ushort(__float2half_rn(s * static_cast<float>(b1)));
            o[i] = h0 | (h1 << 16);
        }
        uint16_t *dst = out + (h * depth + p) * head_dim + i0;
        if (VEC) {
            reinterpret_cast<uint4 *>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
            for (int i = 0; i < 8; ++i) {
                dst[2 * i] = static_cast<uint16_t>(o[i] & 0xffffu);
                dst[2 * i + 1] = static_cast<uint16_t>(o[i] >> 16);
            }
        }
    }
}

}  // namespace
}  // namespace wsw

extern "C" int wsw_dequant_q8_0_kv(const int8_t *q, const uint16_t *d, int64_t depth, int64_t heads,
                                   int64_t head_dim, uint16_t *out, void *stream,
                                   const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (depth < 0 || heads < 0 || head_dim < 0 || head_dim % 32 != 0) return WSW_ERR_INVALID_ARG;
    if (depth == 0 || heads == 0 || head_dim == 0) return WSW_OK;
    if (!q || !d || !out) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d) & 1) || (reinterpret_cast<uintptr_t>(out) & 1))
        return WSW_ERR_MISALIGNED;
    if (depth > (int64_t(1) << 32) || heads > 65536 || head_dim > 65536) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    const int64_t npieces = depth * heads * head_dim / 16;
    const bool vec = (reinterpret_cast<uintptr_t>(q) % 16 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    const int64_t ctas = (npieces + kPieces * kThreads - 1) / (kPieces * kThreads);
    if (ctas > 0x7fffffffLL) return WSW_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = vec ? launch(dequant_q8_0_kv_kernel<true>, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), 0, s,
                                 o.pdl, q, d, depth, heads, head_dim, out, npieces)
                        : launch(dequant_q8_0_kv_kernel<false>, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), 0, s,
                                 o.pdl, q, d, depth, heads, head_dim, out, npieces);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
