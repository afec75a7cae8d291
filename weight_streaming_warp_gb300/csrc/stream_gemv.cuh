// stream_gemv.cuh -- the weight-streaming mat-vec skeleton shared by the bf16 and
// q8_0 decode GEMVs.
//
// Work decomposition (one wave, persistent):
//  * The grid has exactly ctas_per_sm x SMs CTAs of 8 warps.  CTA c owns the row
//    groups [c*G/C, (c+1)*G/C) (G = ceil(M / R) groups of R rows), so CTAs differ by
//    at most one row group.
//  * Inside a CTA every row is cut into nseg K-segments of seg_steps warp steps (a step
//    is 32 lanes x 32 bytes = 1 KB of one row).  nseg depends only on M, K and the SM
//    count: rows are split only when a CTA would hold too few of them to give each of
//    its 8 warps several units (choose_seg_steps).  The CTA's (row group, segment)
//    units are split into 8 contiguous, equal runs, one per warp, so all warps of a CTA
//    stream the same number of bytes and each warp's run is one sequential stream.
//  * A warp keeps two register batches of weight loads in flight (U steps each, both
//    issued before the dependency wait) and walks its run step by step; at the end of
//    a segment it reduces the lanes with a xor-butterfly.  An unsplit row (one
//    segment, the SPLIT = false kernel) is stored at once; split rows write partial
//    sums to shared memory and, after a barrier, one thread per row adds them in
//    segment order.
//
// The arithmetic of a row is therefore fixed by M, K and the SM count: lane l
// accumulates chunk
// 32*s + l of steps s of a segment in order, the butterfly fixes the lane order, and
// the segments are added first to last.  Rows per warp, load width, ctas_per_sm and
// PDL change which warp computes what and how bytes arrive, never a result bit.
//
// Format policy F provides Args (with a Common c), Buf, Acc, XVal, the step size in
// elements, and load / stage_x / load_x / accumulate / lane_total / store.
#pragma once

#include "common.cuh"

namespace wsw {
namespace sg {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxPartials = 4096;   // partial sums held in shared memory per batch
constexpr int kUnitsPerCta = 40;     // target (row, segment) units per CTA

struct Common {
    int64_t M;             // rows
    int64_t groups;        // ceil(M / R)
    int64_t batch_groups;  // row groups per batch (partials fit in shared memory)
    int nsteps;            // warp steps per row
    int seg_steps;         // warp steps per K-segment
    int nseg;              // K-segments per row = ceil(nsteps / seg_steps)
};

template <class F, int R, int LB, bool XS, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2) stream_gemv_kernel(const typename F::Args a) {
    constexpr int U = 4 / R;  // steps per register batch
    extern __shared__ __align__(16) unsigned char smem[];
    float *part = reinterpret_cast<float *>(smem);
    unsigned char *xsm = smem + (SPLIT ? kMaxPartials * sizeof(float) : 0);

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int nsteps = a.c.nsteps;
    const int S = SPLIT ? a.c.nseg : 1;
    const int SS = SPLIT ? a.c.seg_steps : nsteps;
    const int64_t G = a.c.groups;
    const int64_t cg0 = static_cast<int64_t>(blockIdx.x) * G / gridDim.x;
    const int64_t cg1 = static_cast<int64_t>(blockIdx.x + 1) * G / gridDim.x;
    const uint64_t pol = policy_evict_first();
    bool started = false;

    typename F::Buf bufA[U][R], bufB[U][R];

    for (int64_t gb = cg0; gb < cg1; gb += a.c.batch_groups) {
        const int64_t ge = gb + a.c.batch_groups < cg1 ? gb + a.c.batch_groups : cg1;
        const int64_t nunits = (ge - gb) * S;
        const int64_t u0 = static_cast<int64_t>(wid) * nunits / kWarps;
        const int64_t u1 = static_cast<int64_t>(wid + 1) * nunits / kWarps;
        // Without splitting a unit is a row group and the cursor is (group, step);
        // with splitting it is (group, segment, step).
        const int nu = static_cast<int>(u1 - u0);  // units of this warp in this batch

        // issue cursor
        int iu = 0, iseg = SPLIT ? static_cast<int>(u0 % S) : 0;
        int64_t ig = gb + (SPLIT ? u0 / S : u0);
        int ist = iseg * SS;
        int iend = SPLIT ? (ist + SS < nsteps ? ist + SS : nsteps) : nsteps;

        auto issue = [&](typename F::Buf(&buf)[U][R]) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (iu < nu) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int64_t row = ig * R + r;
                        if (row < a.c.M) F::template load<LB>(a, row, ist, lane, buf[u][r], pol);
                        else F::zero(buf[u][r]);
                    }
                    if (++ist == iend) {
                        ++iu;
                        if constexpr (SPLIT) {
                            if (++iseg == S) { iseg = 0; ++ig; }
                            ist = iseg * SS;
                            iend = ist + SS < nsteps ? ist + SS : nsteps;
                        } else {
                            ist = 0;
                            ++ig;
                        }
                    }
                }
            }
        };

        // Both register batches are in flight before the dependency wait, i.e.
        // while the previous kernel in the stream drains.
        issue(bufA);
        issue(bufB);
        if (!started) {
            pdl_wait();
            F::template stage_x<XS>(a, xsm, nsteps);
            __syncthreads();
            pdl_launch_dependents();
            started = true;
        }

        typename F::Acc acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) F::clear(acc[r]);
        int cu = 0, cseg = iseg;
        cseg = SPLIT ? static_cast<int>(u0 % S) : 0;
        int64_t cgp = gb + (SPLIT ? u0 / S : u0);
        int cst = cseg * SS;
        int cend = SPLIT ? (cst + SS < nsteps ? cst + SS : nsteps) : nsteps;

        auto compute = [&](const typename F::Buf(&buf)[U][R]) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (cu < nu) {
                    const typename F::XVal xv = F::template load_x<XS>(a, xsm, cst, lane, nsteps);
#pragma unroll
                    for (int r = 0; r < R; ++r) F::accumulate(acc[r], buf[u][r], xv);
                    if (++cst == cend) {
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            float s = F::lane_total(acc[r]);
#pragma unroll
                            for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(WSW_FULL_MASK, s, off);
                            if constexpr (SPLIT) {
                                if (lane == r) part[((cgp - gb) * R + r) * S + cseg] = s;
                            } else {
                                const int64_t row = cgp * R + r;
                                if (lane == r && row < a.c.M) F::store(a, row, s);
                            }
                            F::clear(acc[r]);
                        }
                        ++cu;
                        if constexpr (SPLIT) {
                            if (++cseg == S) { cseg = 0; ++cgp; }
                            cst = cseg * SS;
                            cend = cst + SS < nsteps ? cst + SS : nsteps;
                        } else {
                            cst = 0;
                            ++cgp;
                        }
                    }
                }
            }
        };

        while (cu < nu) {
            compute(bufA);
            if (cu >= nu) break;
            issue(bufA);
            compute(bufB);
            if (cu >= nu) break;
            issue(bufB);
        }
        if constexpr (SPLIT) {
            __syncthreads();
            const int64_t nrows = (ge - gb) * R;
            for (int64_t lr = threadIdx.x; lr < nrows; lr += kThreads) {
                const int64_t row = gb * R + lr;
                if (row < a.c.M) {
                    float s = part[lr * S];
                    for (int g = 1; g < S; ++g) s += part[lr * S + g];
                    F::store(a, row, s);
                }
            }
            __syncthreads();
        }
    }
    if (!started) {
        // A CTA without rows takes part in the dependency protocol all the same.
        pdl_wait();
        pdl_launch_dependents();
    }
}

// K-segments per row for an M x (nsteps warp steps) matrix on `sm_count` SMs: enough
// that a CTA (at the default two per SM) holds about kUnitsPerCta units, segments of
// at least two steps, one segment when rows are plentiful.  Independent of every
// launch option, so the per-row arithmetic is too.
inline int choose_seg_steps(int64_t M, int nsteps, int sm_count) {
    const int64_t ctas = 2 * static_cast<int64_t>(sm_count);
    int64_t want = (kUnitsPerCta * ctas + M - 1) / (M > 0 ? M : 1);  // segments per row
    const int64_t max_seg = nsteps / 2 > 1 ? nsteps / 2 : 1;
    if (want > max_seg) want = max_seg;
    if (want < 1) want = 1;
    return static_cast<int>((nsteps + want - 1) / want);
}

// Host side: fill Common for M rows of `nsteps` steps and R rows per warp group.
inline Common make_common(int64_t M, int nsteps, int R, int sm_count) {
    Common c;
    c.M = M;
    c.groups = (M + R - 1) / R;
    c.nsteps = nsteps;
    c.seg_steps = choose_seg_steps(M, nsteps, sm_count);
    c.nseg = (nsteps + c.seg_steps - 1) / c.seg_steps;
    int64_t bg = kMaxPartials / (static_cast<int64_t>(c.nseg) * R);
    c.batch_groups = bg > 0 ? bg : 1;
    return c;
}

// Host dispatch over the kernel's template parameters.  smem = shared bytes of the
// launch (partial sums when split, then the staged x).
template <class F, int R, int LB, bool XS, bool SPLIT>
cudaError_t launch_sg(const typename F::Args &a, unsigned ctas, size_t smem, cudaStream_t s, bool pdl) {
    auto k = stream_gemv_kernel<F, R, LB, XS, SPLIT>;
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k), static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch(k, dim3(ctas), dim3(kThreads), smem, s, pdl, a);
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
    const bool split = a.c.nseg > 1;
    const size_t smem = (split ? kMaxPartials * sizeof(float) : 0) + x_smem;
    switch (R) {
        case 1: return launch_sg_lb<F, 1>(lb, xs, split, a, ctas, smem, s, pdl);
        case 2: return launch_sg_lb<F, 2>(lb, xs, split, a, ctas, smem, s, pdl);
        default: return launch_sg_lb<F, 4>(lb, xs, split, a, ctas, smem, s, pdl);
    }
}

}  // namespace sg
}  // namespace wsw
