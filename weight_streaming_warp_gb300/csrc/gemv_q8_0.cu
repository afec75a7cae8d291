// gemv_q8_0.cu -- decode mat-vec over q8_0 weights and a q8_0 activation, dense and
// grouped over MoE experts.
//
// Source: "QuantizeQ8KK is thread-per-superblock: 95.5us/call ..." (vllm.cpp issue),
// sections Cause and Scope: the dense path quantizes x (m = 1) and runs the quantized
// GEMV; the MoE path quantizes m = T x top_k rows and runs a grouped GEMM over the
// experts.  Layout: q8_0 blocks of 32 int8 values with one binary16 scale, stored as
// an int8 matrix plus a separate scale matrix.
//
//   y[r] = sum_b fp32(Wd[r][b]) * fp32(xd[b]) * isum_b,
//   isum_b = sum_{i<32} Wq[r][32b+i] * xq[32b+i]   (exact int32).
//
// Canonical arithmetic (shared by the dense and the grouped kernels, which therefore
// agree bit for bit): a lane owns 16-byte chunks, chunk 32*s + lane in step s of a
// row; the two lanes of a block add their half sums with one shuffle; the even lane
// multiplies the exact fp32 product Wd*xd by the block sum and accumulates it with an
// fp32 FMA, blocks in increasing order; a xor-butterfly over the warp ends the row.
#include <cuda_fp16.h>

#include "common.cuh"

namespace wsw {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kU = 4;  // row steps per register batch; two batches in flight

__device__ __forceinline__ int dot16(const uint32_t (&w)[4], const uint4 &xv) {
    int s = 0;
    s = __dp4a(static_cast<int>(w[0]), static_cast<int>(xv.x), s);
    s = __dp4a(static_cast<int>(w[1]), static_cast<int>(xv.y), s);
    s = __dp4a(static_cast<int>(w[2]), static_cast<int>(xv.z), s);
    s = __dp4a(static_cast<int>(w[3]), static_cast<int>(xv.w), s);
    return s;
}

// One block's contribution: the pair's half sums are combined and the even lane
// accumulates; odd lanes keep their accumulator unchanged (it stays 0).
__device__ __forceinline__ float q8_accumulate(float acc, int half_sum, uint32_t wd_bits,
                                               uint32_t xd_bits, int lane) {
    const int isum = half_sum + __shfl_xor_sync(WSW_FULL_MASK, half_sum, 1);
    if ((lane & 1) == 0) {
        const float t = __half2float(__ushort_as_half(static_cast<unsigned short>(wd_bits))) *
                        __half2float(__ushort_as_half(static_cast<unsigned short>(xd_bits)));
        acc = fmaf(t, static_cast<float>(isum), acc);
    }
    return acc;
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(WSW_FULL_MASK, s, off);
    return s;
}

// ---------------------------------------------------------------- dense ----

struct Q8Args {
    const int8_t *Wq;
    const uint16_t *Wd;
    int64_t M, K, ldq;
    const int8_t *xq;
    const uint16_t *xd;
    float *y;
    int64_t groups, per_warp, nsteps;  // nsteps = ceil(K / 512)
};

template <int R, int LB>
__global__ void __launch_bounds__(kThreads, 2) gemv_q8_0_kernel(const Q8Args a) {
    constexpr int U = kU / R;
    extern __shared__ uint4 xs_q[];  // [nsteps * 32] chunks of xq, then xd as u16 [nsteps * 16]

    const int lane = threadIdx.x & 31;
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int64_t g0 = warp * a.per_warp;
    int64_t g1 = g0 + a.per_warp;
    if (g1 > a.groups) g1 = a.groups;
    const int64_t T = g1 > g0 ? (g1 - g0) * a.nsteps : 0;
    const int64_t nblk = a.K / 32;
    const uint64_t pol = policy_evict_first();

    uint32_t wA[U][R][4], wB[U][R][4];
    uint32_t dA[U][R], dB[U][R];
    int64_t it = 0, ig = g0, is = 0;

    auto issue = [&](uint32_t(&w)[U][R][4], uint32_t(&d)[U][R]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (it < T) {
                const int64_t c = is * 32 + lane;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int64_t row = ig * R + r;
                    d[u][r] = 0u;
                    if (row < a.M && 16 * c < a.K) {
                        load16<LB>(a.Wq + row * a.ldq + 16 * c, w[u][r], pol);
                        if ((lane & 1) == 0) StreamLoad<2>::run(a.Wd + row * nblk + (c >> 1), &d[u][r], pol);
                    } else {
                        w[u][r][0] = w[u][r][1] = w[u][r][2] = w[u][r][3] = 0u;
                    }
                }
                ++it;
                if (++is == a.nsteps) { is = 0; ++ig; }
            }
        }
    };

    issue(wA, dA);
    if (T > 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = g0 * R + r;
            if (row < a.M) {
                const char *p = reinterpret_cast<const char *>(a.Wq + row * a.ldq);
                int64_t nbytes = a.K;
                if (nbytes > 16384 / R) nbytes = 16384 / R;
                for (int64_t off = 4096 / R + lane * 128; off < nbytes; off += 32 * 128) prefetch_l2(p + off);
            }
        }
    }

    pdl_wait();
    {
        const int64_t nchunks = a.nsteps * 32;
        uint16_t *xs_d = reinterpret_cast<uint16_t *>(xs_q + nchunks);
        const bool xvec = (reinterpret_cast<uintptr_t>(a.xq) & 15) == 0;
        for (int64_t c = threadIdx.x; c < nchunks; c += kThreads) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (16 * c < a.K) {
                if (xvec) {
                    v = __ldg(reinterpret_cast<const uint4 *>(a.xq) + c);
                } else {
                    uint32_t t[4] = {0u, 0u, 0u, 0u};
                    for (int i = 0; i < 16; ++i)
                        t[i >> 2] |= (static_cast<uint32_t>(static_cast<uint8_t>(a.xq[16 * c + i])) << (8 * (i & 3)));
                    v = make_uint4(t[0], t[1], t[2], t[3]);
                }
            }
            xs_q[c] = v;
        }
        for (int64_t b = threadIdx.x; b < a.nsteps * 16; b += kThreads) xs_d[b] = b < nblk ? a.xd[b] : 0;
        __syncthreads();
    }
    pdl_launch_dependents();
    const uint16_t *xs_d = reinterpret_cast<const uint16_t *>(xs_q + a.nsteps * 32);

    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.0f;
    int64_t ct = 0, cg = g0, cs = 0;

    auto compute = [&](const uint32_t(&w)[U][R][4], const uint32_t(&d)[U][R]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (ct < T) {
                const int64_t c = cs * 32 + lane;
                const uint4 xv = xs_q[c];
                const uint32_t xdb = xs_d[c >> 1];
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] = q8_accumulate(acc[r], dot16(w[u][r], xv), d[u][r], xdb, lane);
                ++ct;
                if (++cs == a.nsteps) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float s = warp_sum(acc[r]);
                        const int64_t row = cg * R + r;
                        if (lane == r && row < a.M) a.y[row] = s;
                        acc[r] = 0.0f;
                    }
                    cs = 0;
                    ++cg;
                }
            }
        }
    };

    while (ct < T) {
        issue(wB, dB);
        compute(wA, dA);
        if (ct >= T) break;
        issue(wA, dA);
        compute(wB, dB);
    }
}

template <int R, int LB>
cudaError_t launch_q8(const Q8Args &a, unsigned ctas, size_t smem, cudaStream_t s, bool pdl) {
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(gemv_q8_0_kernel<R, LB>), static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch(gemv_q8_0_kernel<R, LB>, dim3(ctas), dim3(kThreads), smem, s, pdl, a);
}

template <int R>
cudaError_t launch_q8_lb(int lb, const Q8Args &a, unsigned ctas, size_t smem, cudaStream_t s, bool pdl) {
    switch (lb) {
        case 16: return launch_q8<R, 16>(a, ctas, smem, s, pdl);
        case 8: return launch_q8<R, 8>(a, ctas, smem, s, pdl);
        case 4: return launch_q8<R, 4>(a, ctas, smem, s, pdl);
        default: return launch_q8<R, 2>(a, ctas, smem, s, pdl);
    }
}

// ---------------------------------------------------------------- grouped ---

constexpr int kMoeNT = 4;         // tokens of one expert per pass over a weight row
constexpr int kMoeMaxE = 1024;
constexpr int kMoeMaxR = 16384;

struct MoeArgs {
    const int8_t *Wq;
    const uint16_t *Wd;
    int64_t E, Mo, K;
    const int8_t *xq;
    const uint16_t *xd;
    const int32_t *ids;
    int64_t R;
    float *y;
    int32_t *err;
    int64_t nsteps;
};

// Shared memory: cnt[E], off[E], cur[E], used[E], list[R], nused.
template <int LB>
__global__ void __launch_bounds__(kThreads, 2) moe_gemv_q8_0_kernel(const MoeArgs a) {
    extern __shared__ int moe_smem[];
    int *cnt = moe_smem;
    int *off = cnt + a.E;
    int *cur = off + a.E;
    int *used = cur + a.E;
    int *list = used + a.E;
    __shared__ int s_nused;
    __shared__ int s_warp_tot[kWarps];

    pdl_wait();  // ids and the activation come from earlier kernels
    pdl_launch_dependents();

    // Bucket the rows by expert (every CTA does this for itself; no global scratch).
    for (int64_t e = threadIdx.x; e < a.E; e += kThreads) { cnt[e] = 0; cur[e] = 0; }
    __syncthreads();
    bool bad = false;
    for (int64_t m = threadIdx.x; m < a.R; m += kThreads) {
        const int e = a.ids[m];
        if (e >= 0 && e < a.E) atomicAdd(&cnt[e], 1);
        else bad = true;
    }
    if (bad && blockIdx.x == 0 && a.err) atomicOr(a.err, 1);
    __syncthreads();
    if (threadIdx.x < 32) {
        // Exclusive scan of cnt and compaction of the used experts, in expert order.
        int run = 0, urun = 0;
        for (int64_t base = 0; base < a.E; base += 32) {
            const int64_t e = base + threadIdx.x;
            const int c = e < a.E ? cnt[e] : 0;
            int incl = c, uincl = c > 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(WSW_FULL_MASK, incl, o);
                const int ut = __shfl_up_sync(WSW_FULL_MASK, uincl, o);
                if (threadIdx.x >= o) { incl += t; uincl += ut; }
            }
            if (e < a.E) {
                off[e] = run + incl - c;
                if (c > 0) used[urun + uincl - 1] = static_cast<int>(e);
            }
            run += __shfl_sync(WSW_FULL_MASK, incl, 31);
            urun += __shfl_sync(WSW_FULL_MASK, uincl, 31);
        }
        if (threadIdx.x == 0) s_nused = urun;
    }
    __syncthreads();
    for (int64_t m = threadIdx.x; m < a.R; m += kThreads) {
        const int e = a.ids[m];
        if (e >= 0 && e < a.E) list[off[e] + atomicAdd(&cur[e], 1)] = static_cast<int>(m);
    }
    (void)s_warp_tot;
    __syncthreads();

    // Flattened (used expert, output row) work, split evenly over the grid's warps.
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int64_t total = static_cast<int64_t>(s_nused) * a.Mo;
    const int64_t per = (total + nwarps - 1) / nwarps;
    int64_t w0 = warp * per, w1 = w0 + per;
    if (w1 > total) w1 = total;
    const int64_t nblk = a.K / 32;
    const uint64_t pol = policy_evict_first();

    for (int64_t item = w0; item < w1; ++item) {
        const int64_t u = item / a.Mo;
        const int64_t o = item - u * a.Mo;
        const int e = used[u];
        const int ntok = cnt[e];
        const int *toks = list + off[e];
        const int8_t *wrow = a.Wq + (static_cast<int64_t>(e) * a.Mo + o) * a.K;
        const uint16_t *drow = a.Wd + (static_cast<int64_t>(e) * a.Mo + o) * nblk;
        for (int t0 = 0; t0 < ntok; t0 += kMoeNT) {
            int m[kMoeNT];
            float acc[kMoeNT];
#pragma unroll
            for (int j = 0; j < kMoeNT; ++j) {
                m[j] = (t0 + j < ntok) ? toks[t0 + j] : -1;
                acc[j] = 0.0f;
            }
            for (int64_t s = 0; s < a.nsteps; ++s) {
                const int64_t c = s * 32 + lane;
                uint32_t w[4] = {0u, 0u, 0u, 0u};
                uint32_t db = 0u;
                const bool valid = 16 * c < a.K;
                if (valid) {
                    load16<LB>(wrow + 16 * c, w, pol);
                    if ((lane & 1) == 0) StreamLoad<2>::run(drow + (c >> 1), &db, pol);
                }
#pragma unroll
                for (int j = 0; j < kMoeNT; ++j) {
                    if (m[j] < 0) continue;  // warp-uniform
                    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                    uint32_t xdb = 0u;
                    if (valid) {
                        const int8_t *xr = a.xq + static_cast<int64_t>(m[j]) * a.K + 16 * c;
                        if ((reinterpret_cast<uintptr_t>(xr) & 15) == 0) {
                            xv = __ldg(reinterpret_cast<const uint4 *>(xr));
                        } else {
                            uint32_t t[4] = {0u, 0u, 0u, 0u};
                            for (int i = 0; i < 16; ++i)
                                t[i >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(xr[i])) << (8 * (i & 3));
                            xv = make_uint4(t[0], t[1], t[2], t[3]);
                        }
                        xdb = __ldg(a.xd + static_cast<int64_t>(m[j]) * nblk + (c >> 1));
                    }
                    acc[j] = q8_accumulate(acc[j], dot16(w, xv), db, xdb, lane);
                }
            }
#pragma unroll
            for (int j = 0; j < kMoeNT; ++j) {
                if (m[j] < 0) continue;
                const float sum = warp_sum(acc[j]);
                if (lane == 0) a.y[static_cast<int64_t>(m[j]) * a.Mo + o] = sum;
            }
        }
    }
}

}  // namespace
}  // namespace wsw

extern "C" int wsw_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t M, int64_t K, int64_t ldq,
                             const int8_t *xq, const uint16_t *xd, float *y, void *stream,
                             const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (M < 0 || K < 0 || K % 32 != 0 || ldq % 32 != 0 || ldq < K) return WSW_ERR_INVALID_ARG;
    if (M == 0) return WSW_OK;
    if (!y) return WSW_ERR_INVALID_ARG;
    if (K > 0 && (!Wq || !Wd || !xq || !xd)) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Wd) & 1) || (reinterpret_cast<uintptr_t>(xd) & 1) ||
        (reinterpret_cast<uintptr_t>(y) & 3))
        return WSW_ERR_MISALIGNED;
    if (M > (int64_t(1) << 40) || K > (int64_t(1) << 24)) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return cudaMemsetAsync(y, 0, static_cast<size_t>(M) * 4, s) == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;

    Q8Args a;
    a.Wq = Wq; a.Wd = Wd; a.M = M; a.K = K; a.ldq = ldq; a.xq = xq; a.xd = xd; a.y = y;
    const int R = o.rows_per_warp;
    a.groups = (M + R - 1) / R;
    a.nsteps = (K + 511) / 512;
    const int cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : 2;
    const int64_t target = static_cast<int64_t>(di.sm_count) * cps * kWarps;
    a.per_warp = (a.groups + target - 1) / target;
    const int64_t warps = (a.groups + a.per_warp - 1) / a.per_warp;
    const unsigned ctas = static_cast<unsigned>((warps + kWarps - 1) / kWarps);
    const size_t smem = static_cast<size_t>(a.nsteps) * (512 + 32);
    if (smem > 48 * 1024) {
        // Large K: allow more dynamic shared memory (up to the device's opt-in limit).
        if (smem > static_cast<size_t>(di.max_smem_optin)) return WSW_ERR_UNSUPPORTED;
    }
    const int lb = load_width(Wq, ldq, o.load_bytes);
    cudaError_t e = cudaSuccess;
    switch (R) {
        case 1: e = launch_q8_lb<1>(lb, a, ctas, smem, s, o.pdl); break;
        case 2: e = launch_q8_lb<2>(lb, a, ctas, smem, s, o.pdl); break;
        default: e = launch_q8_lb<4>(lb, a, ctas, smem, s, o.pdl); break;
    }
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}

extern "C" int wsw_moe_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K,
                                 const int8_t *xq, const uint16_t *xd, const int32_t *ids, int64_t R,
                                 float *y, int32_t *err_flag, void *stream, const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (E < 0 || Mo < 0 || K < 0 || R < 0 || K % 32 != 0) return WSW_ERR_INVALID_ARG;
    if (E > kMoeMaxE || R > kMoeMaxR) return WSW_ERR_UNSUPPORTED;
    if (R == 0 || Mo == 0) return WSW_OK;
    if (!ids || !y || E == 0) return WSW_ERR_INVALID_ARG;
    if (K > 0 && (!Wq || !Wd || !xq || !xd)) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Wd) & 1) || (reinterpret_cast<uintptr_t>(xd) & 1) ||
        (reinterpret_cast<uintptr_t>(y) & 3) || (reinterpret_cast<uintptr_t>(ids) & 3) ||
        (reinterpret_cast<uintptr_t>(err_flag) & 3))
        return WSW_ERR_MISALIGNED;
    if (K > (int64_t(1) << 24) || Mo > (int64_t(1) << 24)) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MoeArgs a;
    a.Wq = Wq; a.Wd = Wd; a.E = E; a.Mo = Mo; a.K = K; a.xq = xq; a.xd = xd; a.ids = ids; a.R = R;
    a.y = y; a.err = err_flag;
    a.nsteps = (K + 511) / 512;
    const size_t smem = static_cast<size_t>(4 * E + R) * sizeof(int);
    const int cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : 2;
    const unsigned ctas = static_cast<unsigned>(di.sm_count * cps);
    // Weight rows are 16-byte aligned when Wq is and K is a multiple of 16 (it is).
    const int lb = load_width(Wq, K, o.load_bytes);
    auto run = [&](auto kernel) -> cudaError_t {
        if (smem > 48 * 1024) {
            cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kernel), static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        return launch(kernel, dim3(ctas), dim3(kThreads), smem, s, o.pdl, a);
    };
    cudaError_t e;
    switch (lb) {
        case 16: e = run(moe_gemv_q8_0_kernel<16>); break;
        case 8: e = run(moe_gemv_q8_0_kernel<8>); break;
        case 4: e = run(moe_gemv_q8_0_kernel<4>); break;
        default: e = run(moe_gemv_q8_0_kernel<2>); break;
    }
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
