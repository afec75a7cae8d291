// gemv_bf16.cu -- decode mat-vec y = alpha * W.x with bf16 weights, fp32 x and y.
//
// Source: "perf(vulkan): decode GEMV reads four elements per load, and the row lever
// is dead" (vllm.cpp PR).  Opening paragraph: the decode GEMV moves ~52 GB of bf16
// weights per token and is bound by DRAM bandwidth on weights streamed once.  "What
// shipped": wider loads cut load instructions (here 16-byte loads, degrading to 8, 4
// and 2 bytes when the base or row pitch is misaligned).  "What did NOT work": more
// output rows per workgroup halves the number of independent sequential read streams;
// results must be bit-identical for any rows-per-workgroup value.  Chaining: "cuda:
// prefetch the next PTQ1_0 mat-vec's weights into L2 from the last CTAs", Overview and
// Additional information (programmatic dependent launch on sm_90+).
//
// Design (GB300):
//  * One warp streams a contiguous run of output rows (one long sequential stream per
//    warp); the grid is one wave of 8-warp CTAs, sized so that every warp gets the
//    same number of row groups.
//  * Each lane owns "chunks" of 8 consecutive weights (16 bytes): in step s of a row
//    the lane reads chunk 32*s + lane.  The arithmetic is fixed by that mapping alone:
//    the lane accumulates its chunks in order with fp32 FMAs (element 0..7 of each
//    chunk), then a xor-butterfly over the 32 lanes.  Load width and rows per warp
//    only change how bytes are fetched, so the output is bit-identical across them.
//  * x is staged once per CTA into shared memory as two planes of float4 (elements
//    8c..8c+3 and 8c+4..8c+7 of chunk c) so that the per-lane reads are conflict-free.
//  * Weights use L1::no_allocate + L2 evict_first loads, double-buffered in registers.
//  * With PDL, a CTA issues its first weight loads and an L2 prefetch of the start of
//    its stream before griddepcontrol.wait, i.e. while the previous mat-vec drains.
#include "common.cuh"

namespace wsw {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSmemSteps = 100;  // x staged in shared memory up to K = 25600

struct GemvArgs {
    const uint16_t *W;
    int64_t M, K, ld;
    const float *x;
    float alpha;
    float *y;
    int64_t groups;      // ceil(M / R)
    int64_t per_warp;    // row groups per warp
    int64_t nsteps;      // ceil(K / 256)
};

// Load the 8 weights of chunk c of a row: full chunks in one 16-byte piece (split
// into LB-byte loads), a ragged final chunk element by element, absent chunks as 0.
template <int LB>
__device__ __forceinline__ void load_chunk(const uint16_t *row, int64_t c, int64_t K,
                                           uint32_t (&v)[4], uint64_t pol) {
    const int64_t e0 = 8 * c;
    if (e0 + 8 <= K) {
        load16<LB>(row + e0, v, pol);
    } else {
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t t = 0;
            if (e0 + i < K) StreamLoad<2>::run(row + e0 + i, &t, pol);
            h[i] = t;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = h[2 * i] | (h[2 * i + 1] << 16);
    }
}

__device__ __forceinline__ void x_chunk_global(const float *x, int64_t c, int64_t K, float (&xv)[8]) {
    const int64_t e0 = 8 * c;
    if (e0 + 8 <= K && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(x + e0));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(x + e0) + 1);
        xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
        xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xv[i] = (e0 + i < K) ? __ldg(x + e0 + i) : 0.0f;
    }
}

template <int R, int LB, bool XS>
__global__ void __launch_bounds__(kThreads, 2) gemv_bf16_kernel(const GemvArgs a) {
    constexpr int U = 4 / R;  // steps per register batch; two batches in flight
    extern __shared__ float4 xs[];  // [2][nsteps * 32]

    const int lane = threadIdx.x & 31;
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int64_t g0 = warp * a.per_warp;
    int64_t g1 = g0 + a.per_warp;
    if (g1 > a.groups) g1 = a.groups;
    const int64_t T = g1 > g0 ? (g1 - g0) * a.nsteps : 0;  // row-group steps of this warp
    const uint64_t pol = policy_evict_first();

    uint32_t bufA[U][R][4], bufB[U][R][4];
    // issue position (warp-uniform)
    int64_t it = 0, ig = g0, is = 0;

    auto issue = [&](uint32_t(&buf)[U][R][4]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (it < T) {
                const int64_t c = is * 32 + lane;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int64_t row = ig * R + r;
                    if (row < a.M)
                        load_chunk<LB>(a.W + row * a.ld, c, a.K, buf[u][r], pol);
                    else
                        buf[u][r][0] = buf[u][r][1] = buf[u][r][2] = buf[u][r][3] = 0u;
                }
                ++it;
                if (++is == a.nsteps) { is = 0; ++ig; }
            }
        }
    };

    // Before the dependency wait: first batch into registers, and the start of this
    // warp's stream into L2.
    issue(bufA);
    if (T > 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = g0 * R + r;
            if (row < a.M) {
                const char *p = reinterpret_cast<const char *>(a.W + row * a.ld);
                int64_t nbytes = 2 * a.K;
                if (nbytes > 16384 / R) nbytes = 16384 / R;
                for (int64_t off = 4096 / R + lane * 128; off < nbytes; off += 32 * 128) prefetch_l2(p + off);
            }
        }
    }

    pdl_wait();
    if constexpr (XS) {
        const int64_t nchunks = a.nsteps * 32;
        const bool xvec = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
        for (int64_t c = threadIdx.x; c < nchunks; c += kThreads) {
            const int64_t e0 = 8 * c;
            float v[8];
            if (xvec && e0 + 8 <= a.K) {
                const float4 p = __ldg(reinterpret_cast<const float4 *>(a.x + e0));
                const float4 q = __ldg(reinterpret_cast<const float4 *>(a.x + e0) + 1);
                v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w;
                v[4] = q.x; v[5] = q.y; v[6] = q.z; v[7] = q.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = (e0 + i < a.K) ? __ldg(a.x + e0 + i) : 0.0f;
            }
            xs[c] = make_float4(v[0], v[1], v[2], v[3]);
            xs[nchunks + c] = make_float4(v[4], v[5], v[6], v[7]);
        }
        __syncthreads();
    }
    pdl_launch_dependents();

    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.0f;
    int64_t ct = 0, cg = g0, cs = 0;  // compute position

    auto compute = [&](const uint32_t(&buf)[U][R][4]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (ct < T) {
                const int64_t c = cs * 32 + lane;
                float xv[8];
                if constexpr (XS) {
                    const float4 p = xs[c];
                    const float4 q = xs[a.nsteps * 32 + c];
                    xv[0] = p.x; xv[1] = p.y; xv[2] = p.z; xv[3] = p.w;
                    xv[4] = q.x; xv[5] = q.y; xv[6] = q.z; xv[7] = q.w;
                } else {
                    x_chunk_global(a.x, c, a.K, xv);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float s = acc[r];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        s = fmaf(bf16lo(buf[u][r][i]), xv[2 * i], s);
                        s = fmaf(bf16hi(buf[u][r][i]), xv[2 * i + 1], s);
                    }
                    acc[r] = s;
                }
                ++ct;
                if (++cs == a.nsteps) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float s = acc[r];
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(WSW_FULL_MASK, s, off);
                        const int64_t row = cg * R + r;
                        if (lane == r && row < a.M) a.y[row] = a.alpha * s;
                        acc[r] = 0.0f;
                    }
                    cs = 0;
                    ++cg;
                }
            }
        }
    };

    while (ct < T) {
        issue(bufB);
        compute(bufA);
        if (ct >= T) break;
        issue(bufA);
        compute(bufB);
    }
}

template <int R, int LB, bool XS>
cudaError_t launch_one(const GemvArgs &a, unsigned ctas, size_t smem, cudaStream_t s, bool pdl) {
    auto k = gemv_bf16_kernel<R, LB, XS>;
    if (XS) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k), kMaxSmemSteps * 1024);
        if (e != cudaSuccess) return e;
    }
    return launch(k, dim3(ctas), dim3(kThreads), smem, s, pdl, a);
}

template <int R>
cudaError_t launch_lb(int lb, bool xs, const GemvArgs &a, unsigned ctas, size_t smem,
                      cudaStream_t s, bool pdl) {
    switch (lb) {
        case 16: return xs ? launch_one<R, 16, true>(a, ctas, smem, s, pdl) : launch_one<R, 16, false>(a, ctas, smem, s, pdl);
        case 8: return xs ? launch_one<R, 8, true>(a, ctas, smem, s, pdl) : launch_one<R, 8, false>(a, ctas, smem, s, pdl);
        case 4: return xs ? launch_one<R, 4, true>(a, ctas, smem, s, pdl) : launch_one<R, 4, false>(a, ctas, smem, s, pdl);
        default: return xs ? launch_one<R, 2, true>(a, ctas, smem, s, pdl) : launch_one<R, 2, false>(a, ctas, smem, s, pdl);
    }
}

int validate(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const float *x, const float *y) {
    if (M < 0 || K < 0 || ld < K || ld < 0) return WSW_ERR_INVALID_ARG;
    if (M == 0) return WSW_OK;
    if (!y) return WSW_ERR_INVALID_ARG;
    if (K > 0 && (!W || !x)) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 1) || (reinterpret_cast<uintptr_t>(x) & 3) ||
        (reinterpret_cast<uintptr_t>(y) & 3))
        return WSW_ERR_MISALIGNED;
    if (M > (int64_t(1) << 40) || K > (int64_t(1) << 31)) return WSW_ERR_INVALID_ARG;
    return WSW_OK;
}

int gemv_launch(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const float *x, float alpha,
                float *y, cudaStream_t s, const Opts &o, const DeviceInfo &di, bool pdl) {
    if (M == 0) return WSW_OK;
    if (K == 0)
        return cudaMemsetAsync(y, 0, static_cast<size_t>(M) * 4, s) == cudaSuccess ? WSW_OK
                                                                                  : WSW_ERR_CUDA;
    GemvArgs a;
    a.W = W; a.M = M; a.K = K; a.ld = ld; a.x = x; a.alpha = alpha; a.y = y;
    const int R = o.rows_per_warp;
    a.groups = (M + R - 1) / R;
    a.nsteps = (K + 255) / 256;
    const int cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : 2;
    const int64_t target = static_cast<int64_t>(di.sm_count) * cps * kWarps;
    a.per_warp = (a.groups + target - 1) / target;
    const int64_t warps = (a.groups + a.per_warp - 1) / a.per_warp;
    const unsigned ctas = static_cast<unsigned>((warps + kWarps - 1) / kWarps);
    const bool xs = a.nsteps <= kMaxSmemSteps;
    const size_t smem = xs ? static_cast<size_t>(a.nsteps) * 1024 : 0;
    const int lb = load_width(W, ld * 2, o.load_bytes);
    cudaError_t e;
    switch (R) {
        case 1: e = launch_lb<1>(lb, xs, a, ctas, smem, s, pdl); break;
        case 2: e = launch_lb<2>(lb, xs, a, ctas, smem, s, pdl); break;
        default: e = launch_lb<4>(lb, xs, a, ctas, smem, s, pdl); break;
    }
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}

}  // namespace
}  // namespace wsw

extern "C" int wsw_gemv_bf16(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const float *x,
                             float alpha, float *y, void *stream, const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    st = validate(W, M, K, ld, x, y);
    if (st != WSW_OK || M == 0) return st;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    return gemv_launch(W, M, K, ld, x, alpha, y, static_cast<cudaStream_t>(stream), o, di, o.pdl);
}

extern "C" int wsw_gemv_bf16_chain(int64_t n_links, const wsw_gemv_link *links, void *stream,
                                   const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (n_links < 0 || (n_links > 0 && !links)) return WSW_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n_links; ++i) {
        const wsw_gemv_link &l = links[i];
        st = validate(l.W, l.M, l.K, l.ld, l.x, l.y);
        if (st != WSW_OK) return st;
    }
    if (n_links == 0) return WSW_OK;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    // Default for a chain is PDL on; an explicit opts->pdl = 0 turns it off.
    const bool pdl = opts ? o.pdl : true;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int64_t i = 0; i < n_links; ++i) {
        const wsw_gemv_link &l = links[i];
        st = gemv_launch(l.W, l.M, l.K, l.ld, l.x, l.alpha, l.y, s, o, di, pdl);
        if (st != WSW_OK) return st;
    }
    return WSW_OK;
}
