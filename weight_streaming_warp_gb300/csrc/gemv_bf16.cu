// gemv_bf16.cu -- decode mat-vec y = alpha * W.x with bf16 weights, fp32 x and y.
//
// Source: "perf(vulkan): decode GEMV reads four elements per load, and the row lever
// is dead" (vllm.cpp PR).  Opening paragraph: the decode GEMV moves ~52 GB of bf16
// weights per token and is bound by DRAM bandwidth on weights streamed once.  "What
// shipped": wider loads cut load instructions (here 32-byte loads, degrading to 16, 8,
// 4 and 2 bytes when the base or row pitch is misaligned).  "What did NOT work": more
// output rows per workgroup halves the number of independent sequential read streams;
// results must be bit-identical for any rows-per-workgroup value.  Chaining: "cuda:
// prefetch the next PTQ1_0 mat-vec's weights into L2 from the last CTAs", Overview and
// Additional information (programmatic dependent launch on sm_90+).
//
// Design (GB300), see stream_gemv.cuh for the work decomposition:
//  * Each lane owns "chunks" of 16 consecutive weights (32 bytes): in step s of a row
//    the lane reads chunk 32*s + lane with one 256-bit load, so a warp step covers
//    1 KB of the row.  The lane keeps two fp32 FMA chains (even and odd elements of
//    its chunks, in order) and adds them at the end of each K-segment.
//  * x is staged once per CTA into shared memory as four planes of float4 (elements
//    16c + 4q .. 16c + 4q + 3 of chunk c in plane q), so per-lane reads are
//    conflict-free; for K > 25600 x is read through L1 instead.
//  * Weights use L1::no_allocate + L2 evict_first loads, double-buffered in registers.
//  * With PDL, each warp issues both register batches of weight loads before
//    griddepcontrol.wait, i.e. while the previous mat-vec drains.
#include "stream_gemv.cuh"

namespace wsw {
namespace {

constexpr int kMaxSmemSteps = 50;  // x staged in shared memory up to K = 25600

struct Bf16 {
    static constexpr int kWarps = 16;  // warps per CTA
    static constexpr int kStepElems = 512;
    static constexpr bool kGlobalX = true;  // x may be read through L1 instead of staged
    static constexpr bool kWaitFirst = false;
    struct Args {
        sg::Common c;
        const uint16_t *W;
        int64_t K, ld;
        const float *x;
        float alpha;
        float *y;
        sg::NextLink nx;  // the next link of a chain (nx.W == NULL: none)
    };
    __device__ __forceinline__ static const char *row_ptr(const Args &a, int64_t row) {
        return reinterpret_cast<const char *>(a.W + row * a.ld);
    }
    __device__ __forceinline__ static int64_t row_bytes(const Args &a) { return a.K * 2; }
    __device__ __forceinline__ static void prefetch_x(const Args &a) { prefetch_range_l2(a.x, 4 * a.K); }
    struct Buf { uint32_t w[8]; };
    struct Acc { float a0, a1; };
    struct XVal { float4 q[4]; };

    // The 16 weights of chunk c of a row (32 bytes): full chunks as LB-byte pieces, a
    // ragged final chunk element by element, absent chunks as zeros.
    template <int LB>
    __device__ __forceinline__ static void load(const Args &a, int64_t row, int step, int lane, Buf &b,
                                                uint64_t pol) {
        const uint16_t *rp = a.W + row * a.ld;
        const int64_t e0 = 16 * (static_cast<int64_t>(step) * 32 + lane);
        if (e0 + 16 <= a.K) {
            load32<LB>(rp + e0, b.w, pol);
        } else {
            uint32_t h[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                uint32_t t = 0;
                if (e0 + i < a.K) StreamLoad<2>::run(rp + e0 + i, &t, pol);
                h[i] = t;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) b.w[i] = h[2 * i] | (h[2 * i + 1] << 16);
        }
    }
    __device__ __forceinline__ static void zero(Buf &b) {
#pragma unroll
        for (int i = 0; i < 8; ++i) b.w[i] = 0u;
    }
    template <bool XS>
    __device__ __forceinline__ static void stage_x(const Args &a, unsigned char *xsm, int nsteps) {
        if constexpr (XS) {
            // 32-bit indices: x is staged only for K <= 25600 (kMaxSmemSteps)
            float4 *xs = reinterpret_cast<float4 *>(xsm);
            const int K = static_cast<int>(a.K);
            const int nchunks = nsteps * 32;
            const bool xvec = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
            for (int q = static_cast<int>(threadIdx.x); q < 4 * nchunks; q += static_cast<int>(blockDim.x)) {
                // quad q = elements 4q .. 4q+3 = plane (q & 3) of chunk q >> 2
                const int e0 = 4 * q;
                float4 v;
                if (xvec && e0 + 4 <= K) {
                    v = __ldg(reinterpret_cast<const float4 *>(a.x) + q);
                } else {
                    float t[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) t[i] = (e0 + i < K) ? __ldg(a.x + e0 + i) : 0.0f;
                    v = make_float4(t[0], t[1], t[2], t[3]);
                }
                xs[(q & 3) * nchunks + (q >> 2)] = v;
            }
        }
    }
    template <bool XS>
    __device__ __forceinline__ static XVal load_x(const Args &a, const unsigned char *xsm, int step, int lane,
                                                  int nsteps, int64_t) {
        XVal v;
        const int64_t c = static_cast<int64_t>(step) * 32 + lane;
        if constexpr (XS) {
            const float4 *xs = reinterpret_cast<const float4 *>(xsm);
            const int64_t nchunks = static_cast<int64_t>(nsteps) * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) v.q[q] = xs[q * nchunks + c];
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t e0 = 16 * c + 4 * q;
                if (e0 + 4 <= a.K && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0) {
                    v.q[q] = __ldg(reinterpret_cast<const float4 *>(a.x + e0));
                } else {
                    float t[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) t[i] = (e0 + i < a.K) ? __ldg(a.x + e0 + i) : 0.0f;
                    v.q[q] = make_float4(t[0], t[1], t[2], t[3]);
                }
            }
        }
        return v;
    }
    __device__ __forceinline__ static void clear(Acc &c) { c.a0 = c.a1 = 0.0f; }
    __device__ __forceinline__ static void accumulate(Acc &c, const Buf &b, const XVal &x) {
        float s0 = c.a0, s1 = c.a1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s0 = fmaf(bf16lo(b.w[2 * q]), x.q[q].x, s0);
            s1 = fmaf(bf16hi(b.w[2 * q]), x.q[q].y, s1);
            s0 = fmaf(bf16lo(b.w[2 * q + 1]), x.q[q].z, s0);
            s1 = fmaf(bf16hi(b.w[2 * q + 1]), x.q[q].w, s1);
        }
        c.a0 = s0;
        c.a1 = s1;
    }
    __device__ __forceinline__ static float lane_total(const Acc &c) { return c.a0 + c.a1; }
    __device__ __forceinline__ static void store(const Args &a, int64_t row, float s) { a.y[row] = a.alpha * s; }
};

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

// Rows per warp when the caller leaves the choice to the library: four for tall matrices
// (measured on GB300: 34816 x 5120 runs 2.6% faster than with two), two otherwise.  The
// choice never changes a result bit.
int auto_rows_per_warp(int64_t M) { return M >= 16384 ? 4 : 2; }
bool rows_left_to_library(const wsw_launch_opts *opts) { return opts == nullptr || opts->rows_per_warp == 0; }

// PDL: a single call follows opts->pdl (default off); a chain link is dependent unless
// the caller passes options with pdl = 0.
bool use_pdl(const wsw_launch_opts *opts, const Opts &o, bool chain) { return (chain && !opts) || o.pdl; }

// Every choice of a launch, made on the host from the shape, the weight pointer's
// alignment, the SM count and the options.  gemv_launch and wsw_gemv_bf16_plan both
// take their choices from make_plan.
struct Plan {
    sg::Common c;
    int rows_per_warp, load_bytes;
    unsigned ctas;  // 0: no kernel
    bool x_in_smem, pdl;
    size_t x_smem;
};

int make_plan(const uint16_t *W, int64_t M, int64_t K, int64_t ld, int sm_count, const Opts &o, bool pdl,
              bool auto_rows, Plan *p) {
    *p = Plan{};
    p->rows_per_warp = auto_rows ? auto_rows_per_warp(M) : o.rows_per_warp;
    p->load_bytes = load_width(W, ld * 2, o.load_bytes);
    p->pdl = pdl;
    if (M == 0 || K == 0) return WSW_OK;
    const int64_t nsteps = (K + Bf16::kStepElems - 1) / Bf16::kStepElems;
    if (nsteps > 0x7fffffffLL) return WSW_ERR_UNSUPPORTED;
    p->c = sg::make_common(M, static_cast<int>(nsteps), p->rows_per_warp, sm_count, Bf16::kWarps, Bf16::kWarps);
    const int cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : 16 / Bf16::kWarps;
    p->ctas = sg::grid_ctas(p->c, static_cast<int64_t>(sm_count) * cps);
    p->x_in_smem = nsteps <= kMaxSmemSteps;
    p->x_smem = p->x_in_smem ? static_cast<size_t>(nsteps) * 2048 : 0;
    return WSW_OK;
}

// What a chain link needs to know of the next link to prefetch its first loads: the
// next link's own plan, under the same options.
sg::NextLink next_link(const wsw_gemv_link &l, int sm_count, const Opts &o, bool pdl, bool auto_rows) {
    sg::NextLink nx{};
    Plan p;
    if (o.l2_prefetch_steps <= 0 ||
        make_plan(l.W, l.M, l.K, l.ld, sm_count, o, pdl, auto_rows, &p) != WSW_OK || p.ctas == 0)
        return nx;
    nx.W = reinterpret_cast<const char *>(l.W);
    nx.pitch = l.ld * 2;
    nx.row_bytes = l.K * 2;
    nx.c = p.c;
    nx.ctas = static_cast<int>(p.ctas);
    nx.R = p.rows_per_warp;
    nx.steps = o.l2_prefetch_steps;
    return nx;
}

int gemv_launch(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const float *x, float alpha,
                float *y, cudaStream_t s, const Opts &o, const DeviceInfo &di, bool pdl, bool auto_rows,
                const sg::NextLink &nx) {
    if (M == 0) return WSW_OK;
    if (K == 0)
        return cudaMemsetAsync(y, 0, static_cast<size_t>(M) * 4, s) == cudaSuccess ? WSW_OK
                                                                                  : WSW_ERR_CUDA;
    Plan p;
    const int st = make_plan(W, M, K, ld, di.sm_count, o, pdl, auto_rows, &p);
    if (st != WSW_OK) return st;
    Bf16::Args a;
    a.c = p.c;
    a.W = W; a.K = K; a.ld = ld; a.x = x; a.alpha = alpha; a.y = y;
    a.nx = nx;
    const cudaError_t e =
        sg::launch_stream_gemv<Bf16>(p.rows_per_warp, p.load_bytes, p.x_in_smem, a, p.ctas, p.x_smem, s, p.pdl);
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
    return gemv_launch(W, M, K, ld, x, alpha, y, static_cast<cudaStream_t>(stream), o, di,
                       use_pdl(opts, o, false), rows_left_to_library(opts), sg::NextLink{});
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
    const bool pdl = use_pdl(opts, o, true), auto_rows = rows_left_to_library(opts);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int64_t i = 0; i < n_links; ++i) {
        const wsw_gemv_link &l = links[i];
        const sg::NextLink nx =
            i + 1 < n_links ? next_link(links[i + 1], di.sm_count, o, pdl, auto_rows) : sg::NextLink{};
        st = gemv_launch(l.W, l.M, l.K, l.ld, l.x, l.alpha, l.y, s, o, di, pdl, auto_rows, nx);
        if (st != WSW_OK) return st;
    }
    return WSW_OK;
}

extern "C" int wsw_gemv_bf16_plan(const uint16_t *W, int64_t M, int64_t K, int64_t ld, int32_t sm_count,
                                  int32_t chain, const wsw_launch_opts *opts, wsw_gemv_plan *out) {
    using namespace wsw;
    if (!out || sm_count <= 0 || (chain != 0 && chain != 1)) return WSW_ERR_INVALID_ARG;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    // x and y are not part of the plan: stand-ins that pass their checks
    static const float stand_in[1] = {0.f};
    st = validate(W, M, K, ld, stand_in, stand_in);
    if (st != WSW_OK) return st;
    Plan p;
    st = make_plan(W, M, K, ld, sm_count, o, use_pdl(opts, o, chain == 1), rows_left_to_library(opts), &p);
    if (st != WSW_OK) return st;
    out->load_bytes = p.load_bytes;
    out->rows_per_warp = p.rows_per_warp;
    out->pdl = p.pdl ? 1 : 0;
    out->ctas = static_cast<int32_t>(p.ctas);
    out->threads = p.ctas ? Bf16::kWarps * 32 : 0;
    out->log2_segments = p.ctas ? p.c.log2_seg : 0;
    out->x_in_smem = p.x_in_smem ? 1 : 0;
    out->l2_prefetch_steps = chain ? o.l2_prefetch_steps : 0;
    return WSW_OK;
}
