// stream_gemv.cuh -- the weight-streaming mat-vec skeleton shared by the bf16 and
// q8_0 decode GEMVs.
//
// Work decomposition (one wave, persistent, grid-stride):
//  * Rows form G = ceil(M / R) groups of R rows (R = rows per warp).  Every row is cut
//    into S = 2^ls K-segments; segment k covers warp steps [k*n/S, (k+1)*n/S) of the
//    row's n steps (a step is 32 lanes x 32 bytes = 1 KB of one row).  A unit is one
//    (group, segment) pair; units are numbered group-major, u = g*S + k.
//  * A CTA has NW warps (the format's choice: 8 or 16, i.e. two or one CTAs per SM).
//    Units form blocks of B = max(NW, S) consecutive units, i.e. whole groups.  CTA c
//    takes blocks c, c + C, c + 2C, ... (C CTAs), so at any moment the grid works on a
//    contiguous window of the matrix.  Inside a block the NW warps take one unit each
//    per NW positions; with split rows the position rotates from block to block so
//    that every warp sees segments of every length.
//  * A warp keeps two register batches of weight loads in flight (U = 4/R steps each,
//    both issued before the dependency wait, followed by an L2 prefetch of the next
//    kPrefetchSteps steps) and walks its units step by step; at the end of a unit it
//    reduces the lanes with a xor-butterfly.  Without splitting
//    (S = 1, the SPLIT = false kernel) the row sum is stored at once; split rows write
//    unit sums to shared memory and, after a barrier, one thread per row adds them in
//    segment order.
//
// The arithmetic of a row is fixed by M, K and the SM count (they fix S): lane l
// accumulates block 32*s + l of each step s of a segment in order, the butterfly fixes
// the lane order, and the segments are added first to last.  Rows per warp, load
// width, ctas_per_sm and PDL change which warp computes what and how bytes arrive,
// never a result bit.
//
// Format policy F provides Args (with a Common c), Buf, Acc, XVal, the warps per CTA,
// and load / row_ptr / row_bytes / prefetch_x / stage_x / load_x / accumulate /
// lane_total / store.  load_x also receives the first row of the group (a format whose
// activation differs by row picks it from there).  kWaitFirst: the weight addresses
// depend on data written by earlier kernels, so the dependency wait and the format's
// stage_route (which stages that data) come before the first weight load, and stage_x
// follows it.  A format whose Args has a NextLink `nx` also requests
// into L2, once its warps are done, what the next mat-vec of a chain reads first.
// A step is 1 KB of a row in both formats.
#pragma once

#include <type_traits>
#include <utility>

#include "common.cuh"

namespace wsw {
namespace sg {

constexpr int kWarps = 8;            // warps per CTA of the grouped (MoE) kernel
constexpr int kThreads = kWarps * 32;
constexpr int kMaxPartials = 4096;   // unit sums held in shared memory per batch
constexpr int kMaxLog2Seg = 6;       // at most 64 K-segments per row
constexpr int kPrefetchSteps = 1;    // steps prefetched into L2 before the dependency wait
constexpr int kStepBytes = 1024;

constexpr int log2_warps(int nw) { return nw == 16 ? 4 : 3; }

struct Common {
    int64_t M;        // rows
    int64_t groups;   // G = ceil(M / R)
    int64_t nblocks;  // ceil(G * S / B)
    int nsteps;       // warp steps per row
    int log2_seg;     // S = 2^log2_seg K-segments per row
    int log2_block;   // B = 2^log2_block units per block (B = max(8, S))
    int batch_blocks; // blocks of a CTA whose unit sums fit in shared memory at once
};

// First step of K-segment k of an n-step row cut into 2^ls segments.
__host__ __device__ __forceinline__ int seg_begin(int k, int n, int ls) {
    return static_cast<int>((static_cast<int64_t>(k) * n) >> ls);
}

// The next mat-vec of a chain, as far as its first loads go.
struct NextLink {
    const char *W;      // its weights; NULL: no next link, or nothing to prefetch
    int64_t pitch;      // row stride in bytes
    int64_t row_bytes;  // bytes of a row that are read
    Common c;           // its decomposition
    int ctas;           // its grid
    int R;              // its rows per warp
    int steps;          // steps of each warp's first unit to request
};

template <class F, class = void>
struct HasNextLink : std::false_type {};
template <class F>
struct HasNextLink<F, std::void_t<decltype(std::declval<typename F::Args>().nx)>> : std::true_type {};

// L2 prefetch of the next link's first loads ("cuda: prefetch the next PTQ1_0 mat-vec's
// weights into L2 from the last CTAs", Overview: CTAs that are done with the current
// mat-vec request the next one's weights while the rest drain).  The next launch's CTA
// n starts with block n, whose unit for warp w is (n << lb) + w; that warp first loads
// the first steps of the unit's rows.  Warp w of this launch's CTA c requests the first
// nx.steps steps of warp w's first unit for the next CTAs c, c + C, ... (both launches
// have NW warps per CTA).  Off unless the chain asks for it: on GB300 the chain ran
// slower with it, PDL's pre-wait loads already covering the transition.
template <int NW>
__device__ __forceinline__ void prefetch_next_link(const NextLink &nx, int wid, int lane) {
    if (nx.W == nullptr || nx.steps <= 0) return;
    constexpr int kLines = kStepBytes / 128;
    const int ls = nx.c.log2_seg, lb = nx.c.log2_block;
    for (int64_t n = blockIdx.x; n < nx.ctas; n += gridDim.x) {
        const int64_t u = (n << lb) + wid;
        const int64_t g = u >> ls;
        if (g >= nx.c.groups) continue;
        const int k = static_cast<int>(u & ((1 << ls) - 1));
        const int st = seg_begin(k, nx.c.nsteps, ls);
        const int se = seg_begin(k + 1, nx.c.nsteps, ls);
        const int ns = nx.steps < se - st ? nx.steps : se - st;
        for (int i = lane; i < nx.R * ns * kLines; i += 32) {
            const int line = i % kLines, rs = i / kLines;
            const int64_t row = g * nx.R + rs % nx.R;
            const int64_t off = static_cast<int64_t>(st + rs / nx.R) * kStepBytes + line * 128;
            if (row < nx.c.M && off < nx.row_bytes) prefetch_l2(nx.W + row * nx.pitch + off);
        }
    }
}

// The dependency protocol of one mat-vec launch: wait for the previous kernel in the
// stream (programmatic dependent launch), then let the next one be scheduled.
struct PdlWait {
    __device__ __forceinline__ void before() const { pdl_wait(); }
    __device__ __forceinline__ void after() const { pdl_launch_dependents(); }
};

// One mat-vec by one CTA, the body of stream_gemv_kernel.  `wait.before()` is where the
// CTA waits for the data an earlier kernel (or link) writes; every thread of the CTA
// calls it exactly once, after its first weight loads are in flight (before them for
// kWaitFirst formats).  `wait.after()` follows the staging of x.
template <class F, int R, int LB, bool XS, bool SPLIT, class Wait>
__device__ __forceinline__ void matvec_body(const typename F::Args &a, unsigned char *smem, const Wait &wait) {
    constexpr int U = 4 / R;  // steps per register batch
    constexpr int NW = F::kWarps;
    constexpr int LW = log2_warps(NW);
    static_assert(NW == 8 || NW == 16, "8 or 16 warps per CTA");
    float *part = reinterpret_cast<float *>(smem);
    unsigned char *xsm = smem + (SPLIT ? kMaxPartials * sizeof(float) : 0);

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int nsteps = a.c.nsteps;
    const int ls = SPLIT ? a.c.log2_seg : 0;
    const int lb = SPLIT ? a.c.log2_block : LW;
    const int wpb = 1 << (lb - LW);  // units of a warp per block
    const int64_t G = a.c.groups;
    const int64_t C = gridDim.x;
    const int64_t nbk = a.c.nblocks;
    const int64_t my_blocks = blockIdx.x < nbk ? (nbk - 1 - blockIdx.x) / C + 1 : 0;
    const int64_t bpb = SPLIT ? a.c.batch_blocks : (my_blocks > 0 ? my_blocks : 1);
    const uint64_t pol = policy_evict_first();
    bool started = false;

    typename F::Buf bufA[U][R], bufB[U][R];

    for (int64_t jb = 0; jb < my_blocks; jb += bpb) {
        const int64_t je = jb + bpb < my_blocks ? jb + bpb : my_blocks;

        // Unit q of this warp in this batch: its group, first and end step, and (split)
        // its slot among the batch's unit sums.  False when it lies past the last row.
        auto locate = [&](int q, int64_t &g, int &st, int &se, int &slot) -> bool {
            const int j = q >> (lb - LW);
            const int t = q & (wpb - 1);
            const int64_t blk = jb + j;
            const int pos = (SPLIT ? ((wid + static_cast<int>(blk)) & (NW - 1)) : wid) + (t << LW);
            const int64_t u = ((static_cast<int64_t>(blockIdx.x) + blk * C) << lb) + pos;
            g = u >> ls;
            const int k = static_cast<int>(u & ((1 << ls) - 1));
            st = SPLIT ? seg_begin(k, nsteps, ls) : 0;
            se = SPLIT ? seg_begin(k + 1, nsteps, ls) : nsteps;
            slot = (j << lb) + pos;
            return g < G;
        };

        // Only the grid's last block can hold units past the last row, and each warp has
        // at most one unit there (with more than one unit per block every unit is a
        // whole group's segment): it is the warp's last unit.
        int nq = static_cast<int>(je - jb) * wpb;
        {
            int64_t g;
            int st, se, slot;
            if (nq > 0 && !locate(nq - 1, g, st, se, slot)) --nq;
        }

        // Next unit of a cursor: without splitting the warp's groups are W = NW C apart
        // (one batch holds all of them), with splitting the unit is located afresh.
        const int64_t W = C * NW;
        auto next = [&](int q, int64_t &g, int &st, int &se, int &slot) {
            if constexpr (SPLIT) {
                locate(q, g, st, se, slot);
            } else {
                g += W;
                st = 0;
            }
        };

        int iq = 0, ist = 0, ise = 0, islot = 0;
        int64_t ig = 0;
        if (nq > 0) locate(0, ig, ist, ise, islot);

        auto issue = [&](typename F::Buf(&buf)[U][R]) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (iq < nq) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int64_t row = ig * R + r;
                        if (row < a.c.M) F::template load<LB>(a, row, ist, lane, buf[u][r], pol);
                        else F::zero(buf[u][r]);
                    }
                    if (++ist == ise && ++iq < nq) next(iq, ig, ist, ise, islot);
                }
            }
        };

        // The activation's lines are requested into L2 first (L2 is the point of
        // coherence, so this is safe while the previous kernel may still write them);
        // both register batches are then in flight before the dependency wait, i.e.
        // while the previous kernel in the stream drains, and the steps after them are
        // on their way into L2.
        // A kWaitFirst format waits first and stages what its weight addresses depend on
        // (stage_route); its weight loads are then in flight while it stages x.
        if (!started) {
            if constexpr (F::kWaitFirst) {
                wait.before();
                F::stage_route(a);
                __syncthreads();
            } else {
                F::prefetch_x(a);
            }
        }
        issue(bufA);
        issue(bufB);
        if (!started) {
            int q = iq, st = ist, se = ise, slot = islot;
            int64_t g = ig;
            const int64_t rb = F::row_bytes(a);
            for (int k = 0; k < kPrefetchSteps && q < nq; ++k) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int64_t row = g * R + r;
                    const int64_t off = static_cast<int64_t>(st) * kStepBytes + lane * 128;
                    if (lane < kStepBytes / 128 && row < a.c.M && off < rb) prefetch_l2(F::row_ptr(a, row) + off);
                }
                if (++st == se && ++q < nq) next(q, g, st, se, slot);
            }
        }
        if (!started) {
            if constexpr (!F::kWaitFirst) wait.before();
            F::template stage_x<XS>(a, xsm, nsteps);
            __syncthreads();
            wait.after();
            started = true;
        }

        typename F::Acc acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) F::clear(acc[r]);
        int cq = 0, cst = 0, cse = 0, cslot = 0;
        int64_t cg = 0;
        if (nq > 0) locate(0, cg, cst, cse, cslot);

        auto compute = [&](const typename F::Buf(&buf)[U][R]) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (cq < nq) {
                    const typename F::XVal xv = F::template load_x<XS>(a, xsm, cst, lane, nsteps, cg * R);
#pragma unroll
                    for (int r = 0; r < R; ++r) F::accumulate(acc[r], buf[u][r], xv);
                    if (++cst == cse) {
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            float s = F::lane_total(acc[r]);
#pragma unroll
                            for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(WSW_FULL_MASK, s, off);
                            if constexpr (SPLIT) {
                                if (lane == r) part[cslot * R + r] = s;
                            } else {
                                const int64_t row = cg * R + r;
                                if (lane == r && row < a.c.M) F::store(a, row, s);
                            }
                            F::clear(acc[r]);
                        }
                        if (++cq < nq) next(cq, cg, cst, cse, cslot);
                    }
                }
            }
        };

        while (cq < nq) {
            compute(bufA);
            if (cq >= nq) break;
            issue(bufA);
            compute(bufB);
            if (cq >= nq) break;
            issue(bufB);
        }
        if constexpr (SPLIT) {
            // Row sums of the batch's groups: segments added first to last.
            __syncthreads();
            const int S = 1 << ls;
            const int gpb = (1 << lb) >> ls;  // groups per block
            const int64_t nrows = (je - jb) * gpb * R;
            for (int64_t e = threadIdx.x; e < nrows; e += NW * 32) {
                const int64_t j = e / (static_cast<int64_t>(gpb) * R);
                const int rem = static_cast<int>(e - j * gpb * R);
                const int gl = rem / R, r = rem - gl * R;
                const int64_t blk = static_cast<int64_t>(blockIdx.x) + (jb + j) * C;
                const int64_t g = ((blk << lb) >> ls) + gl;
                const int64_t row = g * R + r;
                if (g < G && row < a.c.M) {
                    const float *p = part + ((j << lb) + static_cast<int64_t>(gl) * S) * R + r;
                    float s = p[0];
                    for (int k = 1; k < S; ++k) s += p[k * R];
                    F::store(a, row, s);
                }
            }
            __syncthreads();
        }
    }
    if (!started) {
        // A CTA without rows takes part in the dependency protocol all the same.
        wait.before();
        wait.after();
    }
    if constexpr (HasNextLink<F>::value) prefetch_next_link<NW>(a.nx, wid, lane);
}

template <class F, int R, int LB, bool XS, bool SPLIT>
__global__ void __launch_bounds__(F::kWarps * 32, 16 / F::kWarps) stream_gemv_kernel(const typename F::Args a) {
    extern __shared__ __align__(16) unsigned char smem[];
    matvec_body<F, R, LB, XS, SPLIT>(a, smem, PdlWait{});
}

// K-segments per row (log2) for an M x (nsteps warp steps) matrix on `sm_count` SMs and
// CTAs of nw warps.  The model: at the default launch (two rows per warp, 16 warps per
// SM) the kernel takes as long as its busiest warp, which streams
// ceil(blocks / CTAs) * B / nw units of
// n / S steps each, plus a fixed cost per unit for its butterfly; splitting must win
// by more than the cost of combining the sums, and matrices whose unsplit warps stream
// at most four steps (launch-bound) are not split.  Independent of every launch option,
// so the per-row arithmetic is too.
inline int choose_log2_seg(int64_t M, int nsteps, int sm_count, int nw) {
    constexpr double kUnitCost = 0.25;   // steps
    constexpr double kSplitCost = 1.05;  // split rows: shared-memory sums and a barrier
    constexpr double kMinSplit = 4.5;    // warps of at most four steps: launch-bound, not split
    const int64_t C = (16 / nw) * static_cast<int64_t>(sm_count > 0 ? sm_count : 1);
    const int64_t G = (M + 1) / 2;
    int best = 0;
    double best_cost = 0.0;
    for (int l = 0; l <= kMaxLog2Seg && (1 << l) <= nsteps; ++l) {
        const int64_t S = int64_t(1) << l, B = S > nw ? S : nw;
        const int64_t nblocks = (G * S + B - 1) / B;
        const int64_t per_cta = (nblocks + C - 1) / C;
        const double cost = static_cast<double>(per_cta) * static_cast<double>(B / nw) *
                            (static_cast<double>(nsteps) / static_cast<double>(S) + kUnitCost);
        if (l == 0 || cost * kSplitCost < best_cost) {
            best = l;
            best_cost = cost;
        }
        if (l == 0 && cost <= kMinSplit) break;
    }
    return best;
}

// Host side: fill Common for M rows of `nsteps` steps, R rows per warp group and CTAs
// of nw warps; the K-segments follow the model for CTAs of seg_nw warps (the format's
// own width, so that a variant with other CTAs computes the same bits).
inline Common make_common_seg(int64_t M, int nsteps, int R, int nw, int log2_seg) {
    Common c;
    c.M = M;
    c.groups = (M + R - 1) / R;
    c.nsteps = nsteps;
    c.log2_seg = log2_seg;
    const int lw = log2_warps(nw);
    c.log2_block = c.log2_seg > lw ? c.log2_seg : lw;
    const int64_t S = int64_t(1) << c.log2_seg, B = int64_t(1) << c.log2_block;
    c.nblocks = (c.groups * S + B - 1) / B;
    c.batch_blocks = static_cast<int>(kMaxPartials / (B * R));
    return c;
}

inline Common make_common(int64_t M, int nsteps, int R, int sm_count, int nw, int seg_nw) {
    return make_common_seg(M, nsteps, R, nw, choose_log2_seg(M, nsteps, sm_count, seg_nw));
}

// CTAs of a launch: at most max_ctas, and no more than needed for every CTA to take
// the same number of blocks as the busiest one.
inline unsigned grid_ctas(const Common &c, int64_t max_ctas) {
    if (c.nblocks <= 0) return 1;
    const int64_t per = (c.nblocks + max_ctas - 1) / max_ctas;
    return static_cast<unsigned>((c.nblocks + per - 1) / per);
}

// Host dispatch over the kernel's template parameters.  smem = shared bytes of the
// launch (unit sums when split, then the staged x).
template <class F, int R, int LB, bool XS, bool SPLIT>
cudaError_t launch_sg(const typename F::Args &a, unsigned ctas, size_t smem, cudaStream_t s, bool pdl) {
    auto k = stream_gemv_kernel<F, R, LB, XS, SPLIT>;
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k), static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch(k, dim3(ctas), dim3(F::kWarps * 32), smem, s, pdl, a);
}

template <class F, int R, int LB>
cudaError_t launch_sg_xs(bool xs, bool split, const typename F::Args &a, unsigned ctas, size_t smem,
                         cudaStream_t s, bool pdl) {
    if constexpr (F::kGlobalX) {
        if (!xs)
            return split ? launch_sg<F, R, LB, false, true>(a, ctas, smem, s, pdl)
                         : launch_sg<F, R, LB, false, false>(a, ctas, smem, s, pdl);
    }
    return split ? launch_sg<F, R, LB, true, true>(a, ctas, smem, s, pdl)
                 : launch_sg<F, R, LB, true, false>(a, ctas, smem, s, pdl);
}

template <class F, int R>
cudaError_t launch_sg_lb(int lb, bool xs, bool split, const typename F::Args &a, unsigned ctas, size_t smem,
                         cudaStream_t s, bool pdl) {
    switch (lb) {
        case 32: return launch_sg_xs<F, R, 32>(xs, split, a, ctas, smem, s, pdl);
        case 16: return launch_sg_xs<F, R, 16>(xs, split, a, ctas, smem, s, pdl);
        case 8: return launch_sg_xs<F, R, 8>(xs, split, a, ctas, smem, s, pdl);
        case 4: return launch_sg_xs<F, R, 4>(xs, split, a, ctas, smem, s, pdl);
        default: return launch_sg_xs<F, R, 2>(xs, split, a, ctas, smem, s, pdl);
    }
}

template <class F>
cudaError_t launch_stream_gemv(int R, int lb, bool xs, const typename F::Args &a, unsigned ctas, size_t x_smem,
                               cudaStream_t s, bool pdl) {
    const bool split = a.c.log2_seg > 0;
    const size_t smem = (split ? kMaxPartials * sizeof(float) : 0) + x_smem;
    switch (R) {
        case 1: return launch_sg_lb<F, 1>(lb, xs, split, a, ctas, smem, s, pdl);
        case 2: return launch_sg_lb<F, 2>(lb, xs, split, a, ctas, smem, s, pdl);
        default: return launch_sg_lb<F, 4>(lb, xs, split, a, ctas, smem, s, pdl);
    }
}

}  // namespace sg
}  // namespace wsw
