// gemv_q8_0.cu -- decode mat-vec over q8_0 weights and a q8_0 activation (the grouped
// MoE form is in moe_cc.cu and moe_tc.cu).
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
// Canonical arithmetic (q8_dot.cuh; the grouped CUDA-core kernel follows it too, so the
// two agree bit for bit): a lane owns whole blocks, block 32*s + lane in step s of a row
// (one 256-bit load of 32 int8 values); the exact block sum comes from eight dp4a; the
// lane multiplies the exact fp32 product Wd*xd by it and accumulates with an fp32 FMA,
// its blocks in increasing order; at the end of each K-segment a xor-butterfly reduces
// the lanes, and the segment sums are added first to last (the segments and the work
// decomposition are in stream_gemv.cuh).
#include <cuda_fp16.h>

#include "q8_dot.cuh"
#include "q8_math.cuh"
#include "stream_gemv.cuh"

namespace wsw {
namespace {

using q8d::dot32;
using q8d::warp_sum;

__device__ __forceinline__ float q8_accumulate(float acc, int isum, uint32_t wd_bits, uint32_t xd_bits) {
    return q8d::accumulate(acc, isum, wd_bits, xd_bits);
}

// ---------------------------------------------------------------- dense ----

struct Q8 {
    static constexpr int kWarps = 8;  // warps per CTA
    static constexpr int kStepElems = 1024;
    static constexpr bool kGlobalX = false;  // x is always staged in shared memory
    static constexpr bool kWaitFirst = false;
    struct Args {
        sg::Common c;
        const int8_t *Wq;
        const uint16_t *Wd;
        int64_t K, ldq;
        const int8_t *xq;
        const uint16_t *xd;
        float *y;
    };
    __device__ __forceinline__ static const char *row_ptr(const Args &a, int64_t row) {
        return reinterpret_cast<const char *>(a.Wq + row * a.ldq);
    }
    __device__ __forceinline__ static int64_t row_bytes(const Args &a) { return a.K; }
    struct Buf { uint32_t w[8]; uint32_t d; };
    struct Acc { float a; };
    struct XVal { uint4 x0, x1; uint32_t d; };

    template <int LB>
    __device__ __forceinline__ static void load(const Args &a, int64_t row, int step, int lane, Buf &b,
                                                uint64_t pol) {
        const int64_t blk = static_cast<int64_t>(step) * 32 + lane;
        b.d = 0u;
        if (32 * blk < a.K) {
            load32<LB>(a.Wq + row * a.ldq + 32 * blk, b.w, pol);
            StreamLoad<2>::run(a.Wd + row * (a.K / 32) + blk, &b.d, pol);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) b.w[i] = 0u;
        }
    }
    __device__ __forceinline__ static void zero(Buf &b) {
#pragma unroll
        for (int i = 0; i < 8; ++i) b.w[i] = 0u;
        b.d = 0u;
    }
    __device__ __forceinline__ static void prefetch_x(const Args &a) {
        prefetch_range_l2(a.xq, a.K);
        prefetch_range_l2(a.xd, a.K / 16);
    }
    // Shared memory: xq as two planes of 16-byte halves [2][nsteps * 32], then xd.
    template <bool XS>
    __device__ __forceinline__ static void stage_x(const Args &a, unsigned char *xsm, int nsteps) {
        // 32-bit indices: K <= 2^24 (checked on the host)
        uint4 *xs = reinterpret_cast<uint4 *>(xsm);
        const int nslots = nsteps * 32;
        uint16_t *xs_d = reinterpret_cast<uint16_t *>(xs + 2 * nslots);
        const int K = static_cast<int>(a.K);
        const int nblk = K / 32;
        const int bd = static_cast<int>(blockDim.x);
        const bool xvec = (reinterpret_cast<uintptr_t>(a.xq) & 15) == 0;
        for (int h = static_cast<int>(threadIdx.x); h < 2 * nslots; h += bd) {
            // half h = bytes 16h .. 16h+15 = plane (h & 1) of block h >> 1
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (16 * h < K) {
                if (xvec) {
                    v = __ldg(reinterpret_cast<const uint4 *>(a.xq) + h);
                } else {
                    uint32_t t[4] = {0u, 0u, 0u, 0u};
                    for (int i = 0; i < 16; ++i)
                        t[i >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(a.xq[16 * h + i])) << (8 * (i & 3));
                    v = make_uint4(t[0], t[1], t[2], t[3]);
                }
            }
            xs[(h & 1) * nslots + (h >> 1)] = v;
        }
        for (int b = static_cast<int>(threadIdx.x); b < nslots; b += bd) xs_d[b] = b < nblk ? a.xd[b] : 0;
    }
    template <bool XS>
    __device__ __forceinline__ static XVal load_x(const Args &, const unsigned char *xsm, int step, int lane,
                                                  int nsteps, int64_t = 0) {
        const uint4 *xs = reinterpret_cast<const uint4 *>(xsm);
        const int64_t nslots = static_cast<int64_t>(nsteps) * 32;
        const uint16_t *xs_d = reinterpret_cast<const uint16_t *>(xs + 2 * nslots);
        const int64_t b = static_cast<int64_t>(step) * 32 + lane;
        XVal v;
        v.x0 = xs[b];
        v.x1 = xs[nslots + b];
        v.d = xs_d[b];
        return v;
    }
    __device__ __forceinline__ static void clear(Acc &c) { c.a = 0.0f; }
    __device__ __forceinline__ static void accumulate(Acc &c, const Buf &b, const XVal &x) {
        c.a = q8_accumulate(c.a, dot32(b.w, x.x0, x.x1), b.d, x.d);
    }
    __device__ __forceinline__ static float lane_total(const Acc &c) { return c.a; }
    __device__ __forceinline__ static void store(const Args &a, int64_t row, float s) { a.y[row] = s; }
};

// The dense mat-vec whose CTAs quantize the fp32 activation themselves, with the
// quantizer's block arithmetic (q8_math.cuh): y equals wsw_quantize_q8 (block 32)
// followed by wsw_gemv_q8_0, bit for bit, and the quantizer is off the critical path
// of a decode chain.  CTA 0 can also write the quantized activation out.
struct Q8X : Q8 {
    static constexpr int kWarps = 16;  // one CTA per SM: x is quantized once per SM
    struct Args : Q8::Args {
        const float *x;
        int8_t *xq_out;    // optional (with xd_out): q of x, K bytes
        uint16_t *xd_out;  // optional: binary16 scales, K / 32
    };
    __device__ __forceinline__ static void prefetch_x(const Args &a) { prefetch_range_l2(a.x, 4 * a.K); }
    template <bool XS>
    __device__ __forceinline__ static void stage_x(const Args &a, unsigned char *xsm, int nsteps) {
        constexpr int kB = 2;  // passes whose x loads are in flight together
        // 32-bit indices: K <= 2^24 (checked on the host), so every offset fits.
        const int K = static_cast<int>(a.K);
        const int nslots = nsteps * 32;
        uint16_t *xs_d = reinterpret_cast<uint16_t *>(xsm + 32 * nslots);
        const bool xvec = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
        const bool out = blockIdx.x == 0 && a.xq_out != nullptr;
        const bool ovec = (reinterpret_cast<uintptr_t>(a.xq_out) & 7) == 0;
        const int nt = 4 * nslots;  // a multiple of 128: whole warps iterate together
        const int bd = static_cast<int>(blockDim.x);
        // Thread t quantizes values 8t .. 8t+7, quarter (t & 3) of block t >> 2 (block
        // amax uses shuffles, so every lane of a warp takes part in a unit or none does:
        // nt is a multiple of 128 and a warp's 32 units are consecutive).  Blocks past K
        // are zero: d = +0 and q = 0, as the padding of Q8.
        for (int t0 = static_cast<int>(threadIdx.x); t0 < nt; t0 += kB * bd) {
            float v[kB][8];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int e0 = 8 * (t0 + u * bd);
                if (e0 < K) {  // K % 32 == 0: a block is entirely inside or outside
                    if (xvec) {
                        const float4 p = __ldg(reinterpret_cast<const float4 *>(a.x + e0));
                        const float4 q = __ldg(reinterpret_cast<const float4 *>(a.x + e0) + 1);
                        v[u][0] = p.x; v[u][1] = p.y; v[u][2] = p.z; v[u][3] = p.w;
                        v[u][4] = q.x; v[u][5] = q.y; v[u][6] = q.z; v[u][7] = q.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) v[u][i] = __ldg(a.x + e0 + i);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[u][i] = 0.0f;
                }
            }
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int t = t0 + u * bd;
                if (t >= nt) break;  // warp-uniform, and so are the later units
                const float amax = q8m::block_amax<32>(v[u]);
                const float d = q8m::scale(amax);
                uint32_t p[2];
                q8m::codes(v[u], amax, d, p);
                const int b = t >> 2;
                const int qt = t & 3;
                // bytes 8 qt .. 8 qt + 7 of block b: plane qt >> 1, offset 8 (qt & 1)
                *reinterpret_cast<uint2 *>(xsm + ((qt >> 1) * nslots + b) * 16 + 8 * (qt & 1)) = make_uint2(p[0], p[1]);
                const uint16_t dbits = __half_as_ushort(__float2half_rn(d));
                if (qt == 0) xs_d[b] = dbits;
                const int e0 = 8 * t;
                if (out && e0 < K) {
                    if (ovec) {
                        *reinterpret_cast<uint2 *>(a.xq_out + e0) = make_uint2(p[0], p[1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            a.xq_out[e0 + i] = static_cast<int8_t>((p[i >> 2] >> (8 * (i & 3))) & 0xffu);
                    }
                    if (qt == 0) a.xd_out[b] = dbits;
                }
            }
        }
    }
};

// The grouped MoE mat-vec for a few routed rows (wsw_moe_gemv_q8_0 with R <= 16): a
// dense mat-vec over R * Mo virtual rows, virtual row v = m * Mo + o multiplying row o of
// expert ids[m] with activation row m, so that y[m][o] = y[v] in the caller's [R][Mo]
// layout.  Nothing is bucketed: every routed row streams its expert's rows (a repeated
// expert among so few rows is read again).  The weight addresses come from the ids, which
// an earlier kernel writes, so the dependency wait comes first (kWaitFirst).  The rows per
// warp divide Mo and the K-segments are the dense model's for one Mo x K matrix, so every
// row equals wsw_gemv_q8_0 on its expert, bit for bit.
constexpr int kGatherMaxRows = 16;

struct Q8G : Q8 {
    static constexpr bool kWaitFirst = true;
    struct Args : Q8::Args {
        int64_t E, Mo;
        const int32_t *ids;
        int64_t R;
        int32_t *err;
    };
    // the routing ids of this launch (-1 for an id outside [0, E)), staged per CTA
    __device__ __forceinline__ static int *ids_smem() {
        __shared__ int ids_s[kGatherMaxRows];
        return ids_s;
    }
    // per-token bytes of the staged activation: Q8's two 16-byte planes and the scales
    __device__ __forceinline__ static int64_t token_bytes(int nsteps) { return static_cast<int64_t>(nsteps) * 1088; }
    // routed row of virtual row v: 32-bit division (v < R * Mo <= 16 * 2^24)
    __device__ __forceinline__ static uint32_t routed_row(const Args &a, int64_t v) {
        return static_cast<uint32_t>(v) / static_cast<uint32_t>(a.Mo);
    }
    __device__ __forceinline__ static int64_t expert_row(const Args &a, int64_t v, bool &valid) {
        const uint32_t m = routed_row(a, v);
        const int e = ids_smem()[m];
        valid = e >= 0;
        const uint32_t o = static_cast<uint32_t>(v) - m * static_cast<uint32_t>(a.Mo);
        return static_cast<int64_t>(valid ? e : 0) * a.Mo + o;
    }
    __device__ __forceinline__ static const char *row_ptr(const Args &a, int64_t v) {
        bool valid;
        return reinterpret_cast<const char *>(a.Wq + expert_row(a, v, valid) * a.ldq);
    }
    template <int LB>
    __device__ __forceinline__ static void load(const Args &a, int64_t v, int step, int lane, Buf &b, uint64_t pol) {
        bool valid;
        const int64_t row = expert_row(a, v, valid);
        if (valid) Q8::load<LB>(a, row, step, lane, b, pol);
        else Q8::zero(b);
    }
    __device__ __forceinline__ static void prefetch_x(const Args &) {}
    // The routing ids, before the first weight load.
    __device__ __forceinline__ static void stage_route(const Args &a) {
        if (threadIdx.x < a.R) {
            const int e = a.ids[threadIdx.x];
            const bool ok = e >= 0 && e < a.E;
            ids_smem()[threadIdx.x] = ok ? e : -1;
            if (!ok && blockIdx.x == 0 && a.err) atomicOr(a.err, 1);
        }
    }
    // All R activations in one pass over (routed row, 16-byte piece) pairs, four loads in
    // flight per thread before their stores, in Q8's layout per routed row.
    template <bool XS>
    __device__ __forceinline__ static void stage_x(const Args &a, unsigned char *xsm, int nsteps) {
        // 32-bit indices: R <= 16 and K <= 2^24
        const int nslots = nsteps * 32;
        const int tb = nsteps * 1088;
        const int K = static_cast<int>(a.K);
        const int nblk = K / 32;
        const int bd = static_cast<int>(blockDim.x);
        const bool xvec = (reinterpret_cast<uintptr_t>(a.xq) & 15) == 0;
        const int nh = 2 * nslots;  // 16-byte halves of one routed row (padded past K)
        const int total = static_cast<int>(a.R) * nh;
        for (int i0 = static_cast<int>(threadIdx.x); i0 < total; i0 += 4 * bd) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * bd;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (i < total) {
                    const int m = i / nh, h = i - m * nh;
                    const int8_t *row = a.xq + static_cast<int64_t>(m) * K;
                    if (16 * h < K) {
                        if (xvec) {
                            v[u] = __ldg(reinterpret_cast<const uint4 *>(row) + h);
                        } else {
                            uint32_t t[4] = {0u, 0u, 0u, 0u};
                            for (int j = 0; j < 16; ++j)
                                t[j >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(row[16 * h + j])) << (8 * (j & 3));
                            v[u] = make_uint4(t[0], t[1], t[2], t[3]);
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * bd;
                if (i < total) {
                    const int m = i / nh, h = i - m * nh;
                    // half h = bytes 16h .. 16h+15 = plane (h & 1) of block h >> 1
                    reinterpret_cast<uint4 *>(xsm + m * tb)[(h & 1) * nslots + (h >> 1)] = v[u];
                }
            }
        }
        const int dtotal = static_cast<int>(a.R) * nslots;
        for (int i0 = static_cast<int>(threadIdx.x); i0 < dtotal; i0 += 4 * bd) {
            uint16_t dv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * bd;
                dv[u] = 0;
                if (i < dtotal) {
                    const int m = i / nslots, b = i - m * nslots;
                    if (b < nblk) dv[u] = a.xd[m * nblk + b];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * bd;
                if (i < dtotal) {
                    const int m = i / nslots, b = i - m * nslots;
                    reinterpret_cast<uint16_t *>(xsm + m * tb + 32 * nslots)[b] = dv[u];
                }
            }
        }
    }
    template <bool XS>
    __device__ __forceinline__ static XVal load_x(const Args &a, const unsigned char *xsm, int step, int lane,
                                                  int nsteps, int64_t row) {
        return Q8::load_x<XS>(a, xsm + routed_row(a, row) * token_bytes(nsteps), step, lane, nsteps);
    }
    __device__ __forceinline__ static void store(const Args &a, int64_t v, float s) {
        if (ids_smem()[routed_row(a, v)] >= 0) a.y[v] = s;
    }
};

// Dense launch shared by the two entry points (arguments already validated).
template <class F>
int q8_dense_launch(typename F::Args &a, int64_t M, int64_t K, const Opts &o, const DeviceInfo &di,
                    cudaStream_t s) {
    const int R = o.rows_per_warp;
    const int64_t nsteps = (K + Q8::kStepElems - 1) / Q8::kStepElems;
    if (nsteps > 0x7fffffffLL) return WSW_ERR_UNSUPPORTED;
    a.c = sg::make_common(M, static_cast<int>(nsteps), R, di.sm_count, F::kWarps, Q8::kWarps);
    const int cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : 16 / F::kWarps;
    const unsigned ctas = sg::grid_ctas(a.c, static_cast<int64_t>(di.sm_count) * cps);
    const size_t x_smem = static_cast<size_t>(nsteps) * (1024 + 64);
    if (sg::kMaxPartials * 4 + x_smem > static_cast<size_t>(di.max_smem_optin)) return WSW_ERR_UNSUPPORTED;
    const int lb = load_width(a.Wq, a.ldq, o.load_bytes);
    const cudaError_t e = sg::launch_stream_gemv<F>(R, lb, true, a, ctas, x_smem, s, o.pdl);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}

}  // namespace

bool moe_q8_gather_takes(int64_t R) { return R > 0 && R <= kGatherMaxRows; }

int moe_q8_gather_launch(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K, const int8_t *xq,
                         const uint16_t *xd, const int32_t *ids, int64_t R, float *y, int32_t *err, const Opts &o,
                         const DeviceInfo &di, cudaStream_t s) {
    Q8G::Args a;
    a.Wq = Wq; a.Wd = Wd; a.K = K; a.ldq = K; a.xq = xq; a.xd = xd; a.y = y;
    a.E = E; a.Mo = Mo; a.ids = ids; a.R = R; a.err = err;
    const int64_t nsteps = (K + Q8::kStepElems - 1) / Q8::kStepElems;
    // rows of a warp never straddle two routed rows; the K-segments are those of one
    // expert's dense Mo x K mat-vec (neither choice changes a bit of a row)
    const int rw = Mo % o.rows_per_warp == 0 ? o.rows_per_warp : 1;
    const int ls = sg::choose_log2_seg(Mo, static_cast<int>(nsteps), di.sm_count, Q8::kWarps);
    a.c = sg::make_common_seg(R * Mo, static_cast<int>(nsteps), rw, Q8G::kWarps, ls);
    const int cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : 16 / Q8G::kWarps;
    const unsigned ctas = sg::grid_ctas(a.c, static_cast<int64_t>(di.sm_count) * cps);
    const size_t x_smem = static_cast<size_t>(R) * static_cast<size_t>(nsteps) * 1088;
    if (sg::kMaxPartials * 4 + x_smem > static_cast<size_t>(di.max_smem_optin)) return WSW_ERR_UNSUPPORTED;
    int lb = load_width(Wq, K, o.load_bytes);
    const cudaError_t e = sg::launch_stream_gemv<Q8G>(rw, lb, true, a, ctas, x_smem, s, o.pdl);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}

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

    Q8::Args a;
    a.Wq = Wq; a.Wd = Wd; a.K = K; a.ldq = ldq; a.xq = xq; a.xd = xd; a.y = y;
    return q8_dense_launch<Q8>(a, M, K, o, di, s);
}

extern "C" int wsw_quantize_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t M, int64_t K, int64_t ldq,
                                      const float *x, int8_t *xq_out, uint16_t *xd_out, float *y, void *stream,
                                      const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (M < 0 || K < 0 || K % 32 != 0 || ldq % 32 != 0 || ldq < K) return WSW_ERR_INVALID_ARG;
    if ((xq_out == nullptr) != (xd_out == nullptr)) return WSW_ERR_INVALID_ARG;
    if (M == 0 && xq_out == nullptr) return WSW_OK;
    if (M > 0 && !y) return WSW_ERR_INVALID_ARG;
    if (K > 0 && (!x || (M > 0 && (!Wq || !Wd)))) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Wd) & 1) || (reinterpret_cast<uintptr_t>(x) & 3) ||
        (reinterpret_cast<uintptr_t>(xd_out) & 1) || (reinterpret_cast<uintptr_t>(y) & 3))
        return WSW_ERR_MISALIGNED;
    if (M > (int64_t(1) << 40) || K > (int64_t(1) << 24)) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 0 || K == 0) {
        // Nothing to multiply: the quantizer alone (an empty x needs nothing at all).
        if (K > 0) {
            wsw_launch_opts qo = {0, 0, o.pdl, 0};
            const int qs = wsw_quantize_q8(x, 1, K, K, 32, xq_out, xd_out, stream, &qo);
            if (qs != WSW_OK) return qs;
        }
        if (M == 0) return WSW_OK;
        return cudaMemsetAsync(y, 0, static_cast<size_t>(M) * 4, s) == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
    }
    Q8X::Args a;
    a.Wq = Wq; a.Wd = Wd; a.K = K; a.ldq = ldq; a.xq = nullptr; a.xd = nullptr; a.y = y;
    a.x = x; a.xq_out = xq_out; a.xd_out = xd_out;
    return q8_dense_launch<Q8X>(a, M, K, o, di, s);
}
