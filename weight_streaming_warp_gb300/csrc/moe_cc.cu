// moe_cc.cu -- grouped q8_0 MoE mat-vec on the CUDA cores (few activation rows per
// expert), and the entry point that picks it or the tensor-core form (moe_tc.cu).
//
// Source: "QuantizeQ8KK is thread-per-superblock: 95.5us/call ..." (vllm.cpp issue),
// sections Cause and Scope: the MoE path quantizes m = T x top_k rows and runs a
// grouped GEMM over the experts.
//
// Every CTA buckets the routed rows by expert in shared memory (no global scratch):
// the ids are read once, each warp counts the experts of its own chunk of rows with
// shared-memory atomics, per-expert bases follow from the per-warp counts, and a second
// pass writes every expert's rows in row order (ranks within 32 rows by shuffles), so
// all CTAs build the same lists.
//
// Work units are (used expert e, a run of P row pairs of e's weights, batch j of up to
// 4 of e's rows), ordered by expert, then by run, then by batch, so the batches of one
// run follow each other and re-read those weight rows from L2.  P (1 .. 8) is chosen on
// the host from the number of routed rows so that the grid's warps all get work.
// Blocks of 8 units go to CTAs in grid-stride order and warp w of a CTA takes unit w of
// each block, so the grid streams one contiguous window of the experts' weights at a
// time.  A warp keeps two register batches of weight loads in flight like the dense
// kernel and reads the activation chunks from L1 when it computes (every weight row of
// the expert re-reads them).
//
// Per (weight row, activation row) the arithmetic is the dense kernel's (q8_dot.cuh):
// lane blocks in step order, K-segments of the dense model for an Mo x K matrix,
// butterfly, segments added in order -- so each y row equals wsw_gemv_q8_0 on its
// expert, bit for bit.
#include <cuda_fp16.h>

#include "moe_tc.cuh"
#include "q8_dot.cuh"
#include "stream_gemv.cuh"

namespace wsw {
namespace {

constexpr int kW = 8;  // warps per CTA
constexpr int kT = kW * 32;
constexpr int kNT = 4;    // activation rows per unit
constexpr int kRows = 2;  // weight rows per unit
constexpr int kU = 2;     // steps per register batch
constexpr int kMaxE = 1024;
constexpr int kMaxR = 16384;
constexpr int64_t kTcMinRows = 256;  // more routed rows than this: tensor-core form

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
    int nsteps;    // ceil(K / 1024)
    int log2_seg;  // K-segments (log2) of the dense model for one expert's Mo x K matrix
    int pairs;     // P: row pairs per unit
};

// 32 bytes of an activation row as LB-byte pieces, cached in L1; the words come out the
// same whatever LB is.
template <int LB>
__device__ __forceinline__ void load32_l1(const int8_t *p, uint32_t (&v)[8]) {
    if constexpr (LB == 32) {
        asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                     : "l"(p));
    } else if constexpr (LB == 16) {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint4 b = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if constexpr (LB == 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint2 a = __ldg(reinterpret_cast<const uint2 *>(p) + i);
            v[2 * i] = a.x;
            v[2 * i + 1] = a.y;
        }
    } else if constexpr (LB == 4) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __ldg(reinterpret_cast<const uint32_t *>(p) + i);
    } else {
        static_assert(LB == 2, "load width");
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = __ldg(reinterpret_cast<const unsigned short *>(p) + 2 * i);
            const uint32_t hi = __ldg(reinterpret_cast<const unsigned short *>(p) + 2 * i + 1);
            v[i] = lo | (hi << 16);
        }
    }
}

// Shared memory (ints unless noted): ids[R], cnt[E], off[E], used[E], wbase[kW][E],
// list[R], then ubase[E + 1] (int64, 8-byte aligned).
template <int LB, bool SPLIT>
__global__ void __launch_bounds__(kT, 2) moe_cc_kernel(const MoeArgs a) {
    extern __shared__ __align__(16) int moe_smem[];
    const int E = static_cast<int>(a.E);
    const int R = static_cast<int>(a.R);
    int *ids_s = moe_smem;
    int *cnt = ids_s + R;
    int *off = cnt + E;
    int *used = off + E;
    int *wbase = used + E;
    int *list = wbase + kW * E;
    int64_t *ubase = reinterpret_cast<int64_t *>(moe_smem + ((2 * R + (3 + kW) * E + 1) & ~1));
    __shared__ int s_nused;

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;

    pdl_wait();  // ids and activations come from earlier kernels
    pdl_launch_dependents();

    // ------------------------------------------------------------ bucketing
    bool bad = false;
    for (int m = threadIdx.x; m < R; m += kT) {
        const int e = a.ids[m];
        const bool ok = e >= 0 && e < E;
        ids_s[m] = ok ? e : -1;
        bad |= !ok;
    }
    if (bad && blockIdx.x == 0 && a.err) atomicOr(a.err, 1);
    for (int i = threadIdx.x; i < kW * E; i += kT) wbase[i] = 0;
    __syncthreads();
    const int r0 = static_cast<int>(static_cast<int64_t>(wid) * R / kW);
    const int r1 = static_cast<int>(static_cast<int64_t>(wid + 1) * R / kW);
    // per-warp counts of each expert (shared-memory atomics: a count does not depend on
    // the order; __match_any_sync costs a pass per distinct expert of the 32 ids)
    for (int base = r0; base < r1; base += 32) {
        const int m = base + lane;
        const int e = m < r1 ? ids_s[m] : -1;
        if (e >= 0) atomicAdd(&wbase[wid * E + e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kT) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            const int c = wbase[w * E + e];
            wbase[w * E + e] = run;
            run += c;
        }
        cnt[e] = run;
    }
    __syncthreads();
    const int64_t gpe = ((a.Mo + kRows - 1) / kRows + a.pairs - 1) / a.pairs;  // runs per expert
    if (wid == 0) {
        // exclusive scans over the experts (rows, units) and the used-expert list
        int run = 0, urun = 0;
        int64_t unit_run = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = e < E ? cnt[e] : 0;
            const int64_t units = gpe * ((c + kNT - 1) / kNT);
            int incl = c, uincl = c > 0;
            int64_t uninc = units;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(WSW_FULL_MASK, incl, o);
                const int ut = __shfl_up_sync(WSW_FULL_MASK, uincl, o);
                const int64_t nt = __shfl_up_sync(WSW_FULL_MASK, uninc, o);
                if (lane >= o) { incl += t; uincl += ut; uninc += nt; }
            }
            if (e < E) {
                off[e] = run + incl - c;
                if (c > 0) {
                    used[urun + uincl - 1] = e;
                    ubase[urun + uincl - 1] = unit_run + uninc - units;
                }
            }
            run += __shfl_sync(WSW_FULL_MASK, incl, 31);
            urun += __shfl_sync(WSW_FULL_MASK, uincl, 31);
            unit_run += __shfl_sync(WSW_FULL_MASK, uninc, 31);
        }
        if (lane == 0) {
            s_nused = urun;
            ubase[urun] = unit_run;
        }
    }
    __syncthreads();
    // stable lists: row m goes after the earlier rows of its expert in earlier warps,
    // earlier chunks of this warp and lower lanes of its chunk (counted by shuffles)
    for (int base = r0; base < r1; base += 32) {
        const int m = base + lane;
        const int e = m < r1 ? ids_s[m] : -1;
        int below = 0;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            const int ej = __shfl_sync(WSW_FULL_MASK, e, j);
            below += (j < lane) & (ej == e);
        }
        const int run = e >= 0 ? wbase[wid * E + e] : 0;
        __syncwarp();
        if (e >= 0) {
            list[off[e] + run + below] = m;
            atomicAdd(&wbase[wid * E + e], 1);
        }
        __syncwarp();
    }
    __syncthreads();

    // ------------------------------------------------------------ streaming
    const int nused = s_nused;
    const int64_t U = ubase[nused];
    const int64_t C = gridDim.x;
    // units of this warp: u = (blockIdx + q C) * kW + wid, q = 0, 1, ...
    const int64_t u_first = static_cast<int64_t>(blockIdx.x) * kW + wid;
    const int64_t u_step = C * kW;
    const int nq = u_first < U ? static_cast<int>((U - 1 - u_first) / u_step + 1) : 0;
    if (nq == 0) return;
    const int nsteps = a.nsteps;
    const int64_t nblk = a.K / 32;
    const uint64_t pol = policy_evict_first();

    struct Unit {
        int ui;       // used-expert index
        int e;        // expert
        int n;        // activation rows in the unit (1 .. kNT)
        int tok0;     // first of them in the expert-ordered row list
        int np;       // row pairs left in the unit, this one included
        int64_t o;    // first output row of the current row pair
    };
    // unit number q of this warp (q increases monotonically; ui is scanned forward)
    auto locate = [&](int q, Unit &t) {
        const int64_t u = u_first + q * u_step;
        while (ubase[t.ui + 1] <= u) ++t.ui;
        t.e = used[t.ui];
        const int c = cnt[t.e];
        const int nb = (c + kNT - 1) / kNT;
        const int64_t r = u - ubase[t.ui];
        const int64_t run = nb == 1 ? r : r / nb;
        const int j = static_cast<int>(r - run * nb);
        t.tok0 = off[t.e] + j * kNT;
        t.n = c - j * kNT < kNT ? c - j * kNT : kNT;
        t.o = run * a.pairs * kRows;
        const int64_t left = (a.Mo - t.o + kRows - 1) / kRows;
        t.np = left < a.pairs ? static_cast<int>(left) : a.pairs;
    };

    struct Buf { uint32_t w[kRows][8]; uint32_t d[kRows]; };
    Buf bufA[kU], bufB[kU];

    Unit iu;
    iu.ui = 0;
    locate(0, iu);
    int iq = 0, ist = 0;
    auto issue = [&](Buf(&buf)[kU]) {
#pragma unroll
        for (int k = 0; k < kU; ++k) {
            if (iq < nq) {
                const int64_t blk = static_cast<int64_t>(ist) * 32 + lane;
                const int64_t row = static_cast<int64_t>(iu.e) * a.Mo + iu.o;
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    buf[k].d[r] = 0u;
                    if (blk < nblk && iu.o + r < a.Mo) {
                        load32<LB>(a.Wq + (row + r) * a.K + 32 * blk, buf[k].w[r], pol);
                        StreamLoad<2>::run(a.Wd + (row + r) * nblk + blk, &buf[k].d[r], pol);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) buf[k].w[r][i] = 0u;
                    }
                }
                if (++ist == nsteps) {
                    ist = 0;
                    if (--iu.np > 0) iu.o += kRows;
                    else if (++iq < nq) locate(iq, iu);
                }
            }
        }
    };

    Unit cu = {0, 0, 0, 0, 0, 0};
    locate(0, cu);
    int cq = 0, cst = 0, cseg = 0;
    float acc[kRows][kNT], tot[kRows][kNT];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < kNT; ++t) acc[r][t] = tot[r][t] = 0.0f;
    int mrow[kNT];
#pragma unroll
    for (int t = 0; t < kNT; ++t) mrow[t] = t < cu.n ? list[cu.tok0 + t] : 0;

    auto compute = [&](const Buf(&buf)[kU]) {
#pragma unroll
        for (int k = 0; k < kU; ++k) {
            if (cq < nq) {
                const int64_t blk = static_cast<int64_t>(cst) * 32 + lane;
                const bool in = blk < nblk;
                float wdf[kRows];
#pragma unroll
                for (int r = 0; r < kRows; ++r) wdf[r] = q8d::half_bits(buf[k].d[r]);
#pragma unroll
                for (int t = 0; t < kNT; ++t) {
                    if (t < cu.n) {  // warp-uniform
                        uint32_t x[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                        uint32_t xdb = 0u;
                        if (in) {
                            load32_l1<LB>(a.xq + static_cast<int64_t>(mrow[t]) * a.K + 32 * blk, x);
                            xdb = __ldg(a.xd + static_cast<int64_t>(mrow[t]) * nblk + blk);
                        }
                        const uint4 x0 = make_uint4(x[0], x[1], x[2], x[3]);
                        const uint4 x1 = make_uint4(x[4], x[5], x[6], x[7]);
                        const float xdf = q8d::half_bits(xdb);
                        // fp32(Wd) * fp32(xd) is exact, so converting once per step is the
                        // same arithmetic as q8d::accumulate
#pragma unroll
                        for (int r = 0; r < kRows; ++r)
                            acc[r][t] = fmaf(wdf[r] * xdf, static_cast<float>(q8d::dot32(buf[k].w[r], x0, x1)), acc[r][t]);
                    }
                }
                const bool seg_end =
                    SPLIT ? cst + 1 == sg::seg_begin(cseg + 1, nsteps, a.log2_seg) : cst + 1 == nsteps;
                if (seg_end) {
#pragma unroll
                    for (int r = 0; r < kRows; ++r)
#pragma unroll
                        for (int t = 0; t < kNT; ++t) {
                            if (t < cu.n && cu.o + r < a.Mo) {
                                const float p = q8d::warp_sum(acc[r][t]);
                                tot[r][t] = (!SPLIT || cseg == 0) ? p : tot[r][t] + p;
                            }
                            acc[r][t] = 0.0f;
                        }
                    ++cseg;
                }
                if (++cst == nsteps) {
#pragma unroll
                    for (int r = 0; r < kRows; ++r)
#pragma unroll
                        for (int t = 0; t < kNT; ++t)
                            if (t < cu.n && cu.o + r < a.Mo && lane == r * kNT + t)
                                a.y[static_cast<int64_t>(mrow[t]) * a.Mo + cu.o + r] = tot[r][t];
                    cst = 0;
                    cseg = 0;
                    if (--cu.np > 0) {
                        cu.o += kRows;
                    } else if (++cq < nq) {
                        locate(cq, cu);
#pragma unroll
                        for (int t = 0; t < kNT; ++t) mrow[t] = t < cu.n ? list[cu.tok0 + t] : 0;
                    }
                }
            }
        }
    };

    issue(bufA);
    issue(bufB);
    while (cq < nq) {
        compute(bufA);
        if (cq >= nq) break;
        issue(bufA);
        compute(bufB);
        if (cq >= nq) break;
        issue(bufB);
    }
}

template <int LB>
cudaError_t launch_cc(bool split, const MoeArgs &a, unsigned ctas, size_t smem, cudaStream_t s, bool pdl) {
    auto k = split ? moe_cc_kernel<LB, true> : moe_cc_kernel<LB, false>;
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k), static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch(k, dim3(ctas), dim3(kT), smem, s, pdl, a);
}

}  // namespace
}  // namespace wsw

extern "C" size_t wsw_moe_workspace_bytes(int64_t E, int64_t K, int64_t R) {
    if (R <= wsw::kTcMinRows) return 0;
    return wsw::moe_q8_tc_workspace_bytes(E, K, R);
}

extern "C" int wsw_moe_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K,
                                 const int8_t *xq, const uint16_t *xd, const int32_t *ids, int64_t R,
                                 float *y, int32_t *err_flag, void *ws, size_t ws_bytes, void *stream,
                                 const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (E < 0 || Mo < 0 || K < 0 || R < 0 || K % 32 != 0) return WSW_ERR_INVALID_ARG;
    if (E > kMaxE || R > kMaxR) return WSW_ERR_UNSUPPORTED;
    if (R == 0 || Mo == 0) return WSW_OK;
    if (!ids || !y || E == 0) return WSW_ERR_INVALID_ARG;
    if (K == 0) return WSW_ERR_INVALID_ARG;
    if (!Wq || !Wd || !xq || !xd) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Wd) & 1) || (reinterpret_cast<uintptr_t>(xd) & 1) ||
        (reinterpret_cast<uintptr_t>(y) & 3) || (reinterpret_cast<uintptr_t>(ids) & 3) ||
        (reinterpret_cast<uintptr_t>(err_flag) & 3))
        return WSW_ERR_MISALIGNED;
    if (K > (int64_t(1) << 24) || Mo > (int64_t(1) << 24)) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (moe_q8_gather_takes(R)) {
        const int gs = moe_q8_gather_launch(Wq, Wd, E, Mo, K, xq, xd, ids, R, y, err_flag, o, di, s);
        if (gs != WSW_ERR_UNSUPPORTED) return gs;
    }
    if (R > kTcMinRows) {
        MoeTcArgs t;
        t.Wq = Wq; t.Wd = Wd; t.E = E; t.Mo = Mo; t.K = K; t.xq = xq; t.xd = xd; t.ids = ids; t.R = R;
        t.y = y; t.err = err_flag; t.ws = ws; t.ws_bytes = ws_bytes;
        if (moe_q8_tc_supported(t)) return moe_q8_tc_launch(t, di.sm_count, s, o.pdl);
    }
    MoeArgs a;
    a.Wq = Wq; a.Wd = Wd; a.E = E; a.Mo = Mo; a.K = K; a.xq = xq; a.xd = xd; a.ids = ids; a.R = R;
    a.y = y; a.err = err_flag;
    a.nsteps = static_cast<int>((K + 1023) / 1024);
    a.log2_seg = sg::choose_log2_seg(Mo, a.nsteps, di.sm_count, 8);  // the dense q8_0 model
    const int cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : 2;
    const unsigned ctas = static_cast<unsigned>(di.sm_count * cps);
    // Row pairs per unit: as many as keep about eight units per warp for the experts the
    // routed rows can use at most (runs amortise the unit's set-up over more weights).
    {
        const int64_t experts = R < E ? R : E;
        const int64_t pairs_total = experts * ((Mo + 1) / 2);
        const int64_t want = 8 * static_cast<int64_t>(ctas) * kW;
        int p = 1;
        while (p < 8 && pairs_total / (2 * p) >= want) p *= 2;
        a.pairs = p;
    }
    // ids[R], cnt, off, used, wbase[kW][E], list[R] (ints), then ubase[E + 1] (int64)
    const size_t ints = static_cast<size_t>(2 * R + (3 + kW) * E + 1) & ~static_cast<size_t>(1);
    const size_t smem = ints * 4 + static_cast<size_t>(E + 1) * 8;
    if (smem > static_cast<size_t>(di.max_smem_optin)) return WSW_ERR_UNSUPPORTED;
    // weight rows (K bytes) and activation rows (K bytes) share the load width
    int lb = load_width(Wq, K, o.load_bytes);
    const int lbx = load_width(xq, K, o.load_bytes);
    if (lbx < lb) lb = lbx;
    const bool split = a.log2_seg > 0;
    cudaError_t e;
    switch (lb) {
        case 32: e = launch_cc<32>(split, a, ctas, smem, s, o.pdl); break;
        case 16: e = launch_cc<16>(split, a, ctas, smem, s, o.pdl); break;
        case 8: e = launch_cc<8>(split, a, ctas, smem, s, o.pdl); break;
        case 4: e = launch_cc<4>(split, a, ctas, smem, s, o.pdl); break;
        default: e = launch_cc<2>(split, a, ctas, smem, s, o.pdl); break;
    }
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
