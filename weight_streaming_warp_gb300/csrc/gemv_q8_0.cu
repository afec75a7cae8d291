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
// agree bit for bit): a lane owns whole blocks, block 32*s + lane in step s of a row
// (one 256-bit load of 32 int8 values); the exact block sum comes from eight dp4a; the
// lane multiplies the exact fp32 product Wd*xd by it and accumulates with an fp32 FMA,
// its blocks in increasing order; at the end of each K-segment a xor-butterfly reduces
// the lanes, and the segment sums are added first to last (the segments and the work
// decomposition are in stream_gemv.cuh).
#include <cuda_fp16.h>

#include "moe_tc.cuh"
#include "q8_math.cuh"
#include "stream_gemv.cuh"

namespace wsw {
namespace {

constexpr int kWarps = sg::kWarps;
constexpr int kThreads = sg::kThreads;

__device__ __forceinline__ int dot32(const uint32_t (&w)[8], const uint4 &x0, const uint4 &x1) {
    int s0 = 0, s1 = 0;
    s0 = __dp4a(static_cast<int>(w[0]), static_cast<int>(x0.x), s0);
    s1 = __dp4a(static_cast<int>(w[4]), static_cast<int>(x1.x), s1);
    s0 = __dp4a(static_cast<int>(w[1]), static_cast<int>(x0.y), s0);
    s1 = __dp4a(static_cast<int>(w[5]), static_cast<int>(x1.y), s1);
    s0 = __dp4a(static_cast<int>(w[2]), static_cast<int>(x0.z), s0);
    s1 = __dp4a(static_cast<int>(w[6]), static_cast<int>(x1.z), s1);
    s0 = __dp4a(static_cast<int>(w[3]), static_cast<int>(x0.w), s0);
    s1 = __dp4a(static_cast<int>(w[7]), static_cast<int>(x1.w), s1);
    return s0 + s1;  // exact: |sum| <= 32 * 127 * 127
}

__device__ __forceinline__ float half_bits(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// One block's contribution: (Wd * xd) is exact in fp32 (11 x 11 significant bits),
// the block sum is exact in fp32 (< 2^24); one fused multiply-add.
__device__ __forceinline__ float q8_accumulate(float acc, int isum, uint32_t wd_bits, uint32_t xd_bits) {
    return fmaf(half_bits(wd_bits) * half_bits(xd_bits), static_cast<float>(isum), acc);
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(WSW_FULL_MASK, s, off);
    return s;
}

// ---------------------------------------------------------------- dense ----

struct Q8 {
    static constexpr int kWarps = 8;  // warps per CTA
    static constexpr int kStepElems = 1024;
    static constexpr bool kGlobalX = false;  // x is always staged in shared memory
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
    // Shared memory: xq as two planes of 16-byte halves [2][nsteps * 32], then xd.
    template <bool XS>
    __device__ __forceinline__ static void stage_x(const Args &a, unsigned char *xsm, int nsteps) {
        uint4 *xs = reinterpret_cast<uint4 *>(xsm);
        const int64_t nslots = static_cast<int64_t>(nsteps) * 32;
        uint16_t *xs_d = reinterpret_cast<uint16_t *>(xs + 2 * nslots);
        const int64_t nblk = a.K / 32;
        const bool xvec = (reinterpret_cast<uintptr_t>(a.xq) & 15) == 0;
        for (int64_t h = threadIdx.x; h < 2 * nslots; h += blockDim.x) {
            // half h = bytes 16h .. 16h+15 = plane (h & 1) of block h >> 1
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (16 * h < a.K) {
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
        for (int64_t b = threadIdx.x; b < nslots; b += blockDim.x) xs_d[b] = b < nblk ? a.xd[b] : 0;
    }
    template <bool XS>
    __device__ __forceinline__ static XVal load_x(const Args &, const unsigned char *xsm, int step, int lane,
                                                  int nsteps) {
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
    template <bool XS>
    __device__ __forceinline__ static void stage_x(const Args &a, unsigned char *xsm, int nsteps) {
        constexpr int kB = 2;  // passes whose x loads are in flight together
        const int64_t nslots = static_cast<int64_t>(nsteps) * 32;
        uint16_t *xs_d = reinterpret_cast<uint16_t *>(xsm + 32 * nslots);
        const bool xvec = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
        const bool out = blockIdx.x == 0 && a.xq_out != nullptr;
        const bool ovec = (reinterpret_cast<uintptr_t>(a.xq_out) & 7) == 0;
        const int64_t nt = 4 * nslots;  // a multiple of 128: whole warps iterate together
        // Thread t quantizes values 8t .. 8t+7, quarter (t & 3) of block t >> 2 (block
        // amax uses shuffles, so every lane of a warp runs every pass).  Blocks past K
        // are zero: d = +0 and q = 0, as the padding of Q8.
        for (int64_t t0 = threadIdx.x; t0 < nt; t0 += kB * static_cast<int64_t>(blockDim.x)) {
            float v[kB][8];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int64_t e0 = 8 * (t0 + u * static_cast<int64_t>(blockDim.x));
                if (e0 < a.K) {  // K % 32 == 0: a block is entirely inside or outside
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
                const int64_t t = t0 + u * static_cast<int64_t>(blockDim.x);
                const float amax = q8m::block_amax<32>(v[u]);
                if (t >= nt) continue;  // warp-uniform
                const float d = q8m::scale(amax);
                uint32_t p[2];
                q8m::codes(v[u], amax, d, p);
                const int64_t b = t >> 2;
                const int qt = static_cast<int>(t & 3);
                // bytes 8 qt .. 8 qt + 7 of block b: plane qt >> 1, offset 8 (qt & 1)
                *reinterpret_cast<uint2 *>(xsm + ((qt >> 1) * nslots + b) * 16 + 8 * (qt & 1)) = make_uint2(p[0], p[1]);
                const uint16_t dbits = __half_as_ushort(__float2half_rn(d));
                if (qt == 0) xs_d[b] = dbits;
                const int64_t e0 = 8 * t;
                if (out && e0 < a.K) {
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

// ---------------------------------------------------------------- grouped ---
//
// Every CTA buckets the rows by expert in shared memory (counts, exclusive scan,
// scatter; no global scratch).  An expert's rows are cut into token batches of up to
// kMoeNT rows; the work units are (used expert, output row o, token batch j), ordered
// expert by expert, then by o, then by j, so the batches of one weight row follow each
// other and re-read that row from L2.  Units are split evenly over all warps of the
// grid; each warp streams its units with two register batches of weight loads in
// flight, like the dense kernel, and for each token of a unit follows the dense
// kernel's arithmetic exactly (lane blocks, K-segments of the dense kernel on an
// Mo x K matrix, butterfly, segments added in order).

constexpr int kMoeNT = 4;         // rows of one expert per pass over a weight row
constexpr int kMoeU = 4;          // steps per register batch
constexpr int kMoeMaxE = 1024;
constexpr int kMoeMaxR = 16384;
constexpr int64_t kMoeTcMinRows = 256;  // more rows than this: tensor-core form

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
    int nsteps;     // ceil(K / 1024)
    int log2_seg;   // K-segments (log2) as the dense kernel on one expert's Mo x K matrix
    int xs_cap;     // activation rows that fit the shared-memory staging area
    int64_t xs_off; // byte offset of that area in dynamic shared memory
};

// Shared memory: cnt[E], off[E], cur[E], nbt[E] (token batches), ubase[E+1] (first
// unit of each used expert, int64), used[E], list[R].
template <int LB>
__global__ void __launch_bounds__(kThreads, 2) moe_gemv_q8_0_kernel(const MoeArgs a) {
    extern __shared__ int moe_smem[];
    int *cnt = moe_smem;
    int *off = cnt + a.E;
    int *cur = off + a.E;
    int *nbt = cur + a.E;
    int64_t *ubase = reinterpret_cast<int64_t *>(nbt + a.E);  // 16 E bytes in: 8-byte aligned
    int *used = reinterpret_cast<int *>(ubase + a.E + 1);
    int *list = used + a.E;
    __shared__ int s_nused;

    pdl_wait();  // ids and the activation come from earlier kernels
    pdl_launch_dependents();

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
        // Exclusive scans (rows, units) and the list of used experts, in expert order.
        int run = 0, urun = 0;
        int64_t unit_run = 0;
        for (int64_t base = 0; base < a.E; base += 32) {
            const int64_t e = base + threadIdx.x;
            const int c = e < a.E ? cnt[e] : 0;
            const int nb = (c + kMoeNT - 1) / kMoeNT;
            int incl = c, uincl = c > 0;
            int64_t units = static_cast<int64_t>(nb) * a.Mo, uninc = units;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(WSW_FULL_MASK, incl, o);
                const int ut = __shfl_up_sync(WSW_FULL_MASK, uincl, o);
                const int64_t nt = __shfl_up_sync(WSW_FULL_MASK, uninc, o);
                if (threadIdx.x >= o) { incl += t; uincl += ut; uninc += nt; }
            }
            if (e < a.E) {
                off[e] = run + incl - c;
                nbt[e] = nb;
                if (c > 0) {
                    used[urun + uincl - 1] = static_cast<int>(e);
                    ubase[urun + uincl - 1] = unit_run + uninc - units;
                }
            }
            run += __shfl_sync(WSW_FULL_MASK, incl, 31);
            urun += __shfl_sync(WSW_FULL_MASK, uincl, 31);
            unit_run += __shfl_sync(WSW_FULL_MASK, uninc, 31);
        }
        if (threadIdx.x == 0) {
            s_nused = urun;
            ubase[urun] = unit_run;
        }
    }
    __syncthreads();
    // Stable scatter by warp 0: rows enter their expert's list in row order, so every
    // CTA builds the same list and the token batches (expert, row, j) that different
    // CTAs take are the same sets of rows.
    if (threadIdx.x < 32) {
        const int lane0 = threadIdx.x;
        for (int64_t base = 0; base < a.R; base += 32) {
            const int64_t m = base + lane0;
            const int e = m < a.R ? a.ids[m] : -1;
            const bool valid = e >= 0 && e < a.E;
            const int key = valid ? e : static_cast<int>(a.E) + lane0;  // invalid rows never group
            const unsigned peers = __match_any_sync(WSW_FULL_MASK, key);
            const int rank = __popc(peers & ((1u << lane0) - 1u));
            if (valid) list[off[e] + cur[e] + rank] = static_cast<int>(m);
            __syncwarp();
            if (valid && lane0 == __ffs(peers) - 1) cur[e] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int nused = s_nused;
    const int64_t total = ubase[nused];
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int64_t w0 = warp * total / nwarps, w1 = (warp + 1) * total / nwarps;
    const int nsteps = a.nsteps;
    const int64_t nblk = a.K / 32;
    const uint64_t pol = policy_evict_first();

    // used-expert index of a unit (binary search over ubase)
    auto find_unit = [&](int64_t u) {
        int lo = 0, hi = nused - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ubase[mid] <= u) lo = mid; else hi = mid - 1;
        }
        return lo;
    };

    // Stage the activation rows of the experts this CTA's units cover (a contiguous
    // range of the row lists) in shared memory, when they fit: two planes of 16-byte
    // halves [2][ntok][nblk] and the scales [ntok][nblk].
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kWarps * total / nwarps;
    const int64_t c1 = static_cast<int64_t>(blockIdx.x + 1) * kWarps * total / nwarps;
    int tl0 = 0, ntok = 0;
    if (c0 < c1) {
        const int ea = used[find_unit(c0)], eb = used[find_unit(c1 - 1)];
        tl0 = off[ea];
        ntok = off[eb] + cnt[eb] - tl0;
    }
    const bool staged = ntok > 0 && ntok <= a.xs_cap && (reinterpret_cast<uintptr_t>(a.xq) & 15) == 0;
    uint4 *xs = reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(moe_smem) + a.xs_off);
    uint16_t *xsd = reinterpret_cast<uint16_t *>(xs + 2 * static_cast<int64_t>(ntok) * nblk);
    if (staged) {
        for (int64_t h = threadIdx.x; h < 2 * ntok * nblk; h += kThreads) {
            const int64_t slot = h / (2 * nblk), rem = h - slot * 2 * nblk;  // rem = 2 * block + half
            const int64_t m = list[tl0 + slot];
            xs[((rem & 1) * ntok + slot) * nblk + (rem >> 1)] =
                __ldg(reinterpret_cast<const uint4 *>(a.xq + m * a.K) + rem);
        }
        for (int64_t h = threadIdx.x; h < ntok * nblk; h += kThreads) {
            const int64_t slot = h / nblk, b = h - slot * nblk;
            xsd[h] = a.xd[static_cast<int64_t>(list[tl0 + slot]) * nblk + b];
        }
    }
    __syncthreads();
    if (w0 >= w1) return;

    const int lo = find_unit(w0);
    struct Cursor {
        int ui;      // used-expert index
        int e, nb;   // expert, its token batches
        int64_t o;   // output row
        int j;       // token batch
        int st;      // step
    };
    Cursor ic;
    {
        const int64_t r = w0 - ubase[lo];
        ic.ui = lo; ic.e = used[lo]; ic.nb = nbt[ic.e];
        ic.o = r / ic.nb; ic.j = static_cast<int>(r - ic.o * ic.nb); ic.st = 0;
    }
    Cursor cc = ic;
    int64_t iu = w0, cu = w0;
    auto advance = [&](Cursor &c) {
        if (++c.st == nsteps) {
            c.st = 0;
            if (++c.j == c.nb) {
                c.j = 0;
                if (++c.o == a.Mo) {
                    c.o = 0;
                    if (++c.ui < nused) { c.e = used[c.ui]; c.nb = nbt[c.e]; }
                }
            }
            return true;
        }
        return false;
    };

    uint32_t wA[kMoeU][8], wB[kMoeU][8], dA[kMoeU], dB[kMoeU];
    auto issue = [&](uint32_t(&w)[kMoeU][8], uint32_t(&d)[kMoeU]) {
#pragma unroll
        for (int u = 0; u < kMoeU; ++u) {
            if (iu < w1) {
                const int64_t b = static_cast<int64_t>(ic.st) * 32 + lane;
                const int64_t row = static_cast<int64_t>(ic.e) * a.Mo + ic.o;
                d[u] = 0u;
                if (b < nblk) {
                    load32<LB>(a.Wq + row * a.K + 32 * b, w[u], pol);
                    StreamLoad<2>::run(a.Wd + row * nblk + b, &d[u], pol);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[u][i] = 0u;
                }
                if (advance(ic)) ++iu;
            }
        }
    };

    int m[kMoeNT];
    int cseg = 0;   // K-segment of the compute cursor's step
    int slot0 = 0;  // staging slot of the unit's first row (rows of a batch are consecutive)
    float acc[kMoeNT], tot[kMoeNT];
    auto load_tokens = [&]() {
        const int base = off[cc.e] + cc.j * kMoeNT;
        const int left = cnt[cc.e] - cc.j * kMoeNT;
        slot0 = base - tl0;
#pragma unroll
        for (int t = 0; t < kMoeNT; ++t) {
            m[t] = t < left ? list[base + t] : -1;
            acc[t] = 0.0f;
            tot[t] = 0.0f;
        }
    };
    load_tokens();
    auto compute = [&](const uint32_t(&w)[kMoeU][8], const uint32_t(&d)[kMoeU]) {
#pragma unroll
        for (int u = 0; u < kMoeU; ++u) {
            if (cu < w1) {
                const int s = cc.st;
                const int64_t b = static_cast<int64_t>(s) * 32 + lane;
                const bool valid = b < nblk;
                if (s == 0) cseg = 0;
                const bool seg_end = s + 1 == sg::seg_begin(cseg + 1, nsteps, a.log2_seg);
                const int seg = cseg;
                if (seg_end) ++cseg;
#pragma unroll
                for (int t = 0; t < kMoeNT; ++t) {
                    if (m[t] < 0) continue;  // warp-uniform
                    uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
                    uint32_t xdb = 0u;
                    if (valid && staged) {
                        const int64_t sl = slot0 + t;
                        x0 = xs[sl * nblk + b];
                        x1 = xs[(ntok + sl) * nblk + b];
                        xdb = xsd[sl * nblk + b];
                    } else if (valid) {
                        const int8_t *xr = a.xq + static_cast<int64_t>(m[t]) * a.K + 32 * b;
                        if ((reinterpret_cast<uintptr_t>(xr) & 15) == 0) {
                            x0 = __ldg(reinterpret_cast<const uint4 *>(xr));
                            x1 = __ldg(reinterpret_cast<const uint4 *>(xr) + 1);
                        } else {
                            uint32_t tt[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                            for (int i = 0; i < 32; ++i)
                                tt[i >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(xr[i])) << (8 * (i & 3));
                            x0 = make_uint4(tt[0], tt[1], tt[2], tt[3]);
                            x1 = make_uint4(tt[4], tt[5], tt[6], tt[7]);
                        }
                        xdb = __ldg(a.xd + static_cast<int64_t>(m[t]) * nblk + b);
                    }
                    acc[t] = q8_accumulate(acc[t], dot32(w[u], x0, x1), d[u], xdb);
                    if (seg_end) {
                        const float p = warp_sum(acc[t]);
                        tot[t] = seg == 0 ? p : tot[t] + p;
                        acc[t] = 0.0f;
                    }
                }
                if (s + 1 == nsteps) {
#pragma unroll
                    for (int t = 0; t < kMoeNT; ++t)
                        if (m[t] >= 0 && lane == t) a.y[static_cast<int64_t>(m[t]) * a.Mo + cc.o] = tot[t];
                }
                if (advance(cc)) {
                    ++cu;
                    if (cu < w1) load_tokens();
                }
            }
        }
    };

    issue(wA, dA);
    issue(wB, dB);
    while (cu < w1) {
        compute(wA, dA);
        if (cu >= w1) break;
        issue(wA, dA);
        compute(wB, dB);
        if (cu >= w1) break;
        issue(wB, dB);
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
    if (R > kMoeTcMinRows && moe_q8_tc_supported(E, Mo, K, R, Wq, Wd, xq, xd)) {
        MoeTcArgs t;
        t.Wq = Wq; t.Wd = Wd; t.E = E; t.Mo = Mo; t.K = K; t.xq = xq; t.xd = xd; t.ids = ids; t.R = R;
        t.y = y; t.err = err_flag;
        return moe_q8_tc_launch(t, s, o.pdl);
    }
    MoeArgs a;
    a.Wq = Wq; a.Wd = Wd; a.E = E; a.Mo = Mo; a.K = K; a.xq = xq; a.xd = xd; a.ids = ids; a.R = R;
    a.y = y; a.err = err_flag;
    a.nsteps = static_cast<int>((K + Q8::kStepElems - 1) / Q8::kStepElems);
    a.log2_seg = sg::choose_log2_seg(Mo, a.nsteps, di.sm_count, Q8::kWarps);
    // cnt, off, cur, nbt, ubase[E+1] (int64), used, list, then the activation staging area
    const size_t base_smem = (static_cast<size_t>(4 * E) * sizeof(int) + static_cast<size_t>(E + 1) * 8 +
                              static_cast<size_t>(E + R) * sizeof(int) + 15) & ~static_cast<size_t>(15);
    const size_t per_row = static_cast<size_t>(K) + static_cast<size_t>(K / 32) * 2;  // int8 + scales
    const size_t x_budget = 64 * 1024;
    a.xs_cap = static_cast<int>(x_budget / per_row);
    a.xs_off = static_cast<int64_t>(base_smem);
    const size_t smem = base_smem + static_cast<size_t>(a.xs_cap) * per_row;
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
        case 32: e = run(moe_gemv_q8_0_kernel<32>); break;
        case 16: e = run(moe_gemv_q8_0_kernel<16>); break;
        case 8: e = run(moe_gemv_q8_0_kernel<8>); break;
        case 4: e = run(moe_gemv_q8_0_kernel<4>); break;
        default: e = run(moe_gemv_q8_0_kernel<2>); break;
    }
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
