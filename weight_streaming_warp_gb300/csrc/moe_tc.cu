// moe_tc.cu -- grouped q8_0 MoE mat-vec on the tensor cores, for many rows per expert.
//
// Source: "QuantizeQ8KK is thread-per-superblock: 95.5us/call ..." (vllm.cpp issue),
// sections Cause and Scope: the MoE path quantizes m = T x top_k rows and runs a grouped
// GEMM over the experts.  With hundreds of rows the grouped product is a real dense
// contraction (about 60 integer operations per weight byte at T = 512), so it runs on
// tcgen05 instead of dp4a.
//
// Exactness.  q8_0 values are integers in [-127, 127], exact in fp16; a 32-value block
// product sum is at most 32 * 127^2 < 2^24, exact in the fp32 accumulator.  So one
// tcgen05.mma (kind::f16, K = 32 as two K = 16 steps) per block yields the exact integer
// block sums of a 128-row x (up to) 64-token tile.  The epilogue scales each block sum by
// fp32(Wd) * fp32(xd) (an exact product) and accumulates in fp32:
//   y[m][o] = sum_b (Wd[o][b] * xd[m][b]) * isum_b(o, m).
//
// Two launches.
//  * moe_q8_prep_kernel buckets the routing ids by expert (stable lists, each expert's
//    run padded to a multiple of 4 positions so that every later TMA coordinate stays
//    16-byte aligned) and writes into the caller's workspace, in that sorted order, the
//    activations as exact fp16 (Xh [Rp][K]) and their scales as fp32, block-major
//    (Xs [K/32][Rp]).  Each activation is converted once, not once per weight tile.
//  * moe_q8_tc_kernel, persistent (one CTA per SM), walks the work items i = blockIdx,
//    blockIdx + gridDim, ...; an item is (expert e, 128 output rows, up to 64 of e's
//    routed rows), ordered by expert, then row tile, then token tile, so the grid streams
//    one contiguous window of the expert weights.  A stage is 128 K-values (four blocks).
//    Warp roles (16 warps):
//      warp 0      TMA: raw int8 weight tiles (128 rows x 128 bytes, 128-byte swizzle)
//                  into a ring of kRaw stages
//      warp 1      tensor memory owner; one thread issues the MMAs: A from tensor memory,
//                  B from shared memory, D into a ring of kDPairs slots of two 64-column
//                  blocks.  Each barrier operation costs this thread about as much as an
//                  MMA, so it waits twice and commits three times per stage (8 MMAs)
//      warps 2-5   A converters: thread = weight row (its tensor-memory lane); reads its
//                  row's 128 bytes from the swizzled tile (conflict-free), converts int8
//                  -> fp16 and writes the 64 packed columns with tcgen05.st; they signal a
//                  stage only once its B tile has landed too
//      warp 6      TMA: the fp16 activation tile of each stage (64 sorted rows x 128
//                  values, two 128-byte-swizzled atoms) into a ring of kBS slots, and
//                  each item's scale tile
//      warp 7      cp.async of each item's 128 Wd rows (padded rows in shared memory)
//      warps 8-15  epilogue: two groups of four warps (one per lane quarter); tcgen05.ld
//                  of a block, scale and accumulate; with at most 32 routed rows group h
//                  takes the blocks of parity h and hands its sums to group 0 through
//                  shared memory, with more it takes every block for columns 32 h ..
//                  32 h + 31
//  * Every mbarrier wait gives up after about a second (tc_util.cuh).  A warp whose wait
//    ran out stops its role, the epilogue writes NaN into the rows of the CTA's
//    remaining items, and the kernel sets bit 1 (value 2) of the caller's error flag.
//    Bad expert ids set bit 0.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_tc.cuh"
#include "tc_util.cuh"

namespace wsw {
namespace {

using namespace tc;

constexpr int kRows = 128;      // output rows per item (MMA M)
constexpr int kNT = 64;         // routed rows per item (MMA N <= 64)
constexpr int kStageK = 128;    // K-values per stage (four blocks)
constexpr int kRaw = 4;         // raw weight stages (16 KB each)
constexpr int kAB = 2;          // A slots (tensor memory)
constexpr int kBS = 3;          // B slots (shared memory): the activation tile of a stage
constexpr int kDPairs = 3;      // accumulator slots of two blocks (64 columns each)
constexpr int kDStageBars = 3;  // accumulator-full barriers, one per stage (a ring)
constexpr int kMaxBlocks = 64;  // K <= 2048
constexpr int kMaxRows = 4096;  // routed rows
constexpr int kMaxE = 512;
constexpr int kMaxSorted = kMaxRows + 3 * kMaxE;  // sorted positions with per-expert padding
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kBucketWarps = 8;
constexpr int kPrepThreads = 512;

constexpr int kRawBytes = kRows * kStageK;       // 16 KB
constexpr int kBAtom = kNT * 128;                // one 64-value K-major atom of B: 8 KB
constexpr int kBBytes = 2 * kBAtom;              // 16 KB
constexpr int kScalePitch = 144;                 // bytes per staged Wd row (<= 64 binary16 + pad)
constexpr uint32_t kACol = 0;                    // A slots: columns 0 .. 127
constexpr uint32_t kDCol = 64 * kAB;             // D slots: columns 128 .. 511 (128 per pair)
constexpr uint32_t kTmemCols = 512;

// Workspace layout (byte offsets, each section 256-aligned).
struct WsLayout {
    int64_t Rp;         // sorted positions (a multiple of 4)
    size_t hdr;         // int: nitems, then cnt[E], off[E], ibase[E + 1]
    size_t list;        // int16 [Rp]: routed row at each sorted position, -1 for padding
    size_t xh;          // fp16 [Rp][K]
    size_t xs;          // fp32 [K/32][Rp]
    size_t bytes;
};

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(int64_t E, int64_t K, int64_t R) {
    WsLayout L;
    const int64_t pad = 3 * (E < R ? E : R);
    L.Rp = (R + pad + 3) & ~int64_t(3);
    L.hdr = 0;
    L.list = align256(static_cast<size_t>(1 + 3 * E + 1) * 4);
    L.xh = align256(L.list + static_cast<size_t>(L.Rp) * 2);
    L.xs = align256(L.xh + static_cast<size_t>(L.Rp) * K * 2);
    L.bytes = align256(L.xs + static_cast<size_t>(K / 32) * L.Rp * 4);
    return L;
}

struct Smem {
    unsigned char raw[kRaw][kRawBytes];        // 1024-aligned (first member)
    unsigned char bt[kBS][kBBytes];            // 1024-aligned
    unsigned char wd[2][kRows * kScalePitch];  // per item (double-buffered): Wd rows, padded
    float xs[2][kMaxBlocks][kNT];              // per item: xd as fp32, [block][token]
    float comb[32][kRows];                     // group 1 -> group 0 partial sums (<= 32 rows)
    int16_t list[kMaxSorted];
    int cnt[kMaxE];
    int off[kMaxE];
    int ibase[kMaxE + 1];
    uint64_t raw_full[kRaw], raw_empty[kRaw];
    uint64_t a_full[kAB], a_empty[kAB], b_full[kBS], b_empty[kBS];
    uint64_t d_full[kDStageBars], d_empty[kDPairs];
    uint64_t s_full[2], s_empty[2];
    uint32_t tmem_slot;
    int nitems;
    int timed_out;  // an epilogue wait ran out (a wait that runs out anywhere stops the
                    // data reaching the epilogue, so the epilogue's waits run out too)
};

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Two fp32 lanes in one 64-bit register, for the packed fp32 instructions of sm_100+
// (each lane rounds exactly as the scalar instruction does).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
// acc += (w * x) * d, lane by lane, with the product rounded before the fma
__device__ __forceinline__ void f2_scale_fma(uint64_t &acc, uint64_t w, uint64_t x, uint64_t d) {
    uint64_t s;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(w), "l"(x));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(s), "l"(d));
}

// 16 int8 values -> 16 fp16 values (exact), as 8 packed half2 words.  A byte q with its
// sign bit flipped is u = q + 128; the binary16 pattern 0x6400 | u is 1024 + u, and
// subtracting 1152 (0x6480) leaves q exactly.  Two byte permutes and two half2
// subtractions per four values.
__device__ __forceinline__ void i8x16_to_h(const uint4 &v, uint32_t *o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t u = w[i] ^ 0x80808080u;
        const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);  // u0, 0x64, u1, 0x64
        const uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);  // u2, 0x64, u3, 0x64
        const __half2 a = __hsub2(*reinterpret_cast<const __half2 *>(&lo), bias);
        const __half2 b = __hsub2(*reinterpret_cast<const __half2 *>(&hi), bias);
        o[2 * i] = *reinterpret_cast<const uint32_t *>(&a);
        o[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&b);
    }
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
        "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// D = A (tensor memory) x B (shared memory descriptor), kind::f16.
__device__ __forceinline__ void mma_ts(uint32_t dtmem, uint32_t atmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(dtmem),
        "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One work item of this CTA.
struct Item {
    int e;     // expert
    int m0;    // first output row
    int tok0;  // first sorted position of its routed rows
    int n;     // routed rows (1 .. kNT)
};

__device__ __forceinline__ void decode_item(const Smem &S, int i, int &ecur, Item &it) {
    while (S.ibase[ecur + 1] <= i) ++ecur;
    const int c = S.cnt[ecur];
    const int ntt = (c + kNT - 1) / kNT;
    const int local = i - S.ibase[ecur];
    const int mt = local / ntt, tt = local - mt * ntt;
    it.e = ecur;
    it.m0 = mt * kRows;
    it.tok0 = S.off[ecur] + tt * kNT;
    it.n = c - tt * kNT < kNT ? c - tt * kNT : kNT;
}

// ------------------------------------------------------------------- prepass --
// Every CTA buckets the ids (the same stable lists everywhere), CTA 0 writes the header
// and the sorted-position list, and every CTA converts its share of the routed rows.
// Dynamic shared memory: ids[R], wcnt[kBucketWarps][E], cnt[E], off[E], pos[R] (ints).
__global__ void __launch_bounds__(kPrepThreads, 1) moe_q8_prep_kernel(const MoeTcArgs a, const WsLayout L) {
    extern __shared__ int prep_smem[];
    const int E = static_cast<int>(a.E);
    const int R = static_cast<int>(a.R);
    const int nb = static_cast<int>(a.K / 32);
    const int m_tiles = static_cast<int>((a.Mo + kRows - 1) / kRows);
    int *ids_s = prep_smem;
    int *wcnt = ids_s + R;
    int *cnt = wcnt + kBucketWarps * E;
    int *off = cnt + E;
    int *pos = off + E;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned char *ws = static_cast<unsigned char *>(a.ws);
    int *hdr = reinterpret_cast<int *>(ws + L.hdr);
    int16_t *list = reinterpret_cast<int16_t *>(ws + L.list);
    __half *xh = reinterpret_cast<__half *>(ws + L.xh);
    float *xs = reinterpret_cast<float *>(ws + L.xs);

    pdl_wait();  // ids and activations come from earlier kernels
    pdl_launch_dependents();
    {
        bool bad = false;
        const bool vec = (reinterpret_cast<uintptr_t>(a.ids) & 15) == 0;
        const int nv = vec ? R / 4 : 0;  // ids read as int4 pieces, the rest one by one
        for (int q = threadIdx.x; q < nv; q += kPrepThreads) {
            const int4 v = __ldg(reinterpret_cast<const int4 *>(a.ids) + q);
            const int t[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool ok = t[i] >= 0 && t[i] < E;
                ids_s[4 * q + i] = ok ? t[i] : -1;
                bad |= !ok;
            }
        }
        for (int m = 4 * nv + threadIdx.x; m < R; m += kPrepThreads) {
            const int id = a.ids[m];
            const bool ok = id >= 0 && id < E;
            ids_s[m] = ok ? id : -1;
            bad |= !ok;
        }
        if (bad && blockIdx.x == 0 && a.err) atomicOr(a.err, 1);
        for (int i = threadIdx.x; i < kBucketWarps * E; i += kPrepThreads) wcnt[i] = 0;
    }
    // This CTA's share of the routed rows: the first kPre (row, 16-value chunk) pieces of
    // each thread and its scale pieces are requested now, so that their latency hides
    // behind the bucketing (whether a row is used is known only afterwards).
    const int m0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * R / gridDim.x);
    const int m1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * R / gridDim.x);
    // 32-bit piece indices: R <= kMaxRows and K / 16 <= 2 * kMaxBlocks
    const uint32_t chunks = static_cast<uint32_t>(a.K / 16);
    const uint32_t spr = static_cast<uint32_t>(nb / 8);  // scale pieces per row (8 binary16 a piece)
    const uint32_t work = static_cast<uint32_t>(m1 - m0) * chunks;
    const uint32_t swork = static_cast<uint32_t>(m1 - m0) * spr;
    constexpr int kPre = 8;
    uint4 pre[kPre], spre;
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
        const uint32_t w = threadIdx.x + static_cast<uint32_t>(u) * kPrepThreads;
        if (w < work) {
            const uint32_t r = w / chunks;
            pre[u] = __ldg(reinterpret_cast<const uint4 *>(a.xq + static_cast<int64_t>(m0 + r) * a.K) + (w - r * chunks));
        }
    }
    if (threadIdx.x < swork) {
        const uint32_t r = threadIdx.x / spr;
        spre = __ldg(reinterpret_cast<const uint4 *>(a.xd + static_cast<int64_t>(m0 + r) * nb) + (threadIdx.x - r * spr));
    }
    __syncthreads();
    const int r0 = warp < kBucketWarps ? static_cast<int>(static_cast<int64_t>(warp) * R / kBucketWarps) : 0;
    const int r1 = warp < kBucketWarps ? static_cast<int>(static_cast<int64_t>(warp + 1) * R / kBucketWarps) : 0;
    // per-warp counts of each expert (shared-memory atomics: a count does not depend on
    // the order; __match_any_sync costs a pass per distinct expert of the 32 ids)
    for (int base = r0; base < r1; base += 32) {
        const int m = base + lane;
        const int e = m < r1 ? ids_s[m] : -1;
        if (e >= 0) atomicAdd(&wcnt[warp * E + e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kPrepThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kBucketWarps; ++w) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
        cnt[e] = run;
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scans over the experts: padded offsets and item bases
        int run = 0, irun = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = e < E ? cnt[e] : 0;
            const int span = (c + 3) & ~3;
            const int items = m_tiles * ((c + kNT - 1) / kNT);
            int incl = span, iincl = items;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(WSW_FULL_MASK, incl, o);
                const int it = __shfl_up_sync(WSW_FULL_MASK, iincl, o);
                if (lane >= o) { incl += t; iincl += it; }
            }
            if (e < E) {
                off[e] = run + incl - span;
                if (blockIdx.x == 0) {
                    hdr[1 + e] = c;
                    hdr[1 + E + e] = run + incl - span;
                    hdr[1 + 2 * E + e] = irun + iincl - items;
                }
            }
            run += __shfl_sync(WSW_FULL_MASK, incl, 31);
            irun += __shfl_sync(WSW_FULL_MASK, iincl, 31);
        }
        if (blockIdx.x == 0 && lane == 0) {
            hdr[0] = irun;
            hdr[1 + 3 * E] = irun;
        }
    }
    __syncthreads();
    // stable positions: row m goes after the earlier rows of its expert in earlier warps
    // (the warp base), in earlier chunks of this warp (the running count) and at lower
    // lanes of its chunk (counted over the 32 lanes by shuffles)
    for (int base = r0; base < r1; base += 32) {
        const int m = base + lane;
        const int e = m < r1 ? ids_s[m] : -1;
        int below = 0;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            const int ej = __shfl_sync(WSW_FULL_MASK, e, j);
            below += (j < lane) & (ej == e);
        }
        const int run = e >= 0 ? wcnt[warp * E + e] : 0;
        __syncwarp();
        if (e >= 0) {
            pos[m] = off[e] + run + below;
            atomicAdd(&wcnt[warp * E + e], 1);
        }
        __syncwarp();
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int m = threadIdx.x; m < R; m += kPrepThreads)
            if (ids_s[m] >= 0) list[pos[m]] = static_cast<int16_t>(m);
        for (int e = threadIdx.x; e < E; e += kPrepThreads)
            for (int p = off[e] + cnt[e]; p < off[e] + ((cnt[e] + 3) & ~3); ++p) list[p] = -1;
    }
    // convert the preloaded pieces to fp16 at their sorted rows, then any remaining ones
    // (four loads in flight a pass)
    auto put = [&](uint32_t w, const uint4 &v) {
        const uint32_t r = w / chunks;
        const int m = m0 + static_cast<int>(r);
        if (ids_s[m] < 0) return;
        uint32_t h[8];
        i8x16_to_h(v, h);
        uint4 *dst = reinterpret_cast<uint4 *>(xh + static_cast<int64_t>(pos[m]) * a.K + 16 * (w - r * chunks));
        dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
        dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    };
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
        const uint32_t w = threadIdx.x + static_cast<uint32_t>(u) * kPrepThreads;
        if (w < work) put(w, pre[u]);
    }
    for (uint32_t w0 = threadIdx.x + static_cast<uint32_t>(kPre) * kPrepThreads; w0 < work; w0 += 4 * kPrepThreads) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t w = w0 + u * kPrepThreads;
            if (w < work) {
                const uint32_t r = w / chunks;
                v[u] = __ldg(reinterpret_cast<const uint4 *>(a.xq + static_cast<int64_t>(m0 + r) * a.K) + (w - r * chunks));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t w = w0 + u * kPrepThreads;
            if (w < work) put(w, v[u]);
        }
    }
    // scales: 8 per piece, fp32 at [block][sorted row]
    auto put_scales = [&](uint32_t w, const uint4 &v) {
        const uint32_t r = w / spr;
        const int m = m0 + static_cast<int>(r);
        if (ids_s[m] < 0) return;
        const int b0 = 8 * static_cast<int>(w - r * spr);
        const __half *hv = reinterpret_cast<const __half *>(&v);
#pragma unroll
        for (int i = 0; i < 8; ++i) xs[static_cast<int64_t>(b0 + i) * L.Rp + pos[m]] = __half2float(hv[i]);
    };
    if (threadIdx.x < swork) put_scales(threadIdx.x, spre);
    for (uint32_t w = threadIdx.x + kPrepThreads; w < swork; w += kPrepThreads) {
        const uint32_t r = w / spr;
        put_scales(w, __ldg(reinterpret_cast<const uint4 *>(a.xd + static_cast<int64_t>(m0 + r) * nb) + (w - r * spr)));
    }
}

// ---------------------------------------------------------------- main kernel --
__global__ void __launch_bounds__(kThreads, 1)
    moe_q8_tc_kernel(const __grid_constant__ CUtensorMap tmWq, const __grid_constant__ CUtensorMap tmXh,
                     const __grid_constant__ CUtensorMap tmXs, const MoeTcArgs a, const WsLayout L) {
    extern __shared__ unsigned char smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = static_cast<int>(a.E);
    const int nb = static_cast<int>(a.K / 32);       // blocks per row
    const int kst = static_cast<int>(a.K / kStageK); // stages per item
    const uint32_t xs_bytes = static_cast<uint32_t>(nb) * kNT * 4;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRaw; ++i) { mbar_init(&S.raw_full[i], 1); mbar_init(&S.raw_empty[i], 128); }
        for (int i = 0; i < kAB; ++i) { mbar_init(&S.a_full[i], 128); mbar_init(&S.a_empty[i], 1); }
        for (int i = 0; i < kBS; ++i) { mbar_init(&S.b_full[i], 1); mbar_init(&S.b_empty[i], 1); }
        for (int i = 0; i < kDStageBars; ++i) mbar_init(&S.d_full[i], 1);
        for (int i = 0; i < kDPairs; ++i) mbar_init(&S.d_empty[i], 8);
        // s_full: the 32 Wd-copy lanes plus the scale tile's transaction bytes
        for (int i = 0; i < 2; ++i) { mbar_init(&S.s_full[i], 33); mbar_init(&S.s_empty[i], 256); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();  // the workspace comes from the prepass
    const unsigned char *ws = static_cast<const unsigned char *>(a.ws);
    const int *hdr = reinterpret_cast<const int *>(ws + L.hdr);
    const int16_t *glist = reinterpret_cast<const int16_t *>(ws + L.list);
    for (int e = threadIdx.x; e < E; e += kThreads) {
        S.cnt[e] = hdr[1 + e];
        S.off[e] = hdr[1 + E + e];
        S.ibase[e] = hdr[1 + 2 * E + e];
    }
    // the list in 16-byte pieces (the workspace section is padded to 256 bytes)
    for (int64_t q = threadIdx.x; q < (L.Rp + 7) / 8; q += kThreads)
        reinterpret_cast<uint4 *>(S.list)[q] = __ldg(reinterpret_cast<const uint4 *>(glist) + q);
    if (threadIdx.x == 0) {
        S.ibase[E] = hdr[1 + 3 * E];
        S.nitems = hdr[0];
        S.timed_out = 0;
    }
    __syncthreads();
    pdl_launch_dependents();
    const int NI = S.nitems;
    const int C = static_cast<int>(gridDim.x);
    if (static_cast<int>(blockIdx.x) >= NI) return;  // no items: no tensor memory was taken
    const int my_items = (NI - 1 - static_cast<int>(blockIdx.x)) / C + 1;

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&S.tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_slot;
    bool ok = true;
    int ecur = 0;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA: weights
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmWq)) : "memory");
            uint64_t pol_first, pol_last;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_first));
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_last));
            for (int k = 0; k < my_items && ok; ++k) {
                Item it;
                decode_item(S, static_cast<int>(blockIdx.x) + k * C, ecur, it);
                // the tile is read again by the expert's next token tile unless this is its last
                const bool last_tt = it.tok0 + it.n >= S.off[it.e] + S.cnt[it.e];
                const uint64_t pol = last_tt ? pol_first : pol_last;
                const int y = static_cast<int>(it.e * a.Mo + it.m0);
                for (int s = 0; s < kst; ++s) {
                    const int g = k * kst + s, r = g % kRaw;
                    if (!mbar_wait(&S.raw_empty[r], ((g / kRaw) & 1u) ^ 1u)) { ok = false; break; }
                    mbar_expect_tx(&S.raw_full[r], kRawBytes);
                    tma_load_2d(S.raw[r], &tmWq, s * kStageK, y, &S.raw_full[r], pol);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // This thread's loop is the kernel's issue bottleneck, so every ring position
            // advances by counting (no division or modulo per stage) and the B descriptors
            // are a base plus the slot's offset.  Stage g (counted across items) uses A slot
            // g % kAB, B slot g % kBS, accumulator pairs 2g and 2g + 1 (mod kDPairs) and
            // barrier g % kDStageBars; the pair counter p1 = (2g + 1) mod 2 kDPairs gives
            // both the pair and its phase.
            static_assert(kAB == 2 && kDPairs == 3, "ring sizes");
            const uint64_t bd0 = sw128_desc(saddr(S.bt[0]));
            constexpr uint32_t kBSlot16 = kBBytes >> 4, kBAtom16 = kBAtom >> 4;
            int v = 0, u = 0, dsb = 0, p1 = 1;
            uint32_t pa = 0;  // A-slot phase
            for (int k = 0; k < my_items && ok; ++k) {
                Item it;
                decode_item(S, static_cast<int>(blockIdx.x) + k * C, ecur, it);
                const uint32_t idesc = instr_desc(kRows, (it.n + 15) & ~15, false);
                for (int s = 0; s < kst; ++s) {
                    // A full also means this stage's B tile has landed (the A converters
                    // wait for it), and the epilogue frees accumulator pairs in order, so
                    // one wait each covers the stage
                    const int pair1 = p1 < kDPairs ? p1 : p1 - kDPairs;  // pair 2g + 1
                    const uint32_t ph1 = p1 < kDPairs ? 0u : 1u;        // its round's parity
                    const int pair0 = pair1 == 0 ? kDPairs - 1 : pair1 - 1;
                    if (!mbar_wait(&S.a_full[v], pa) || !mbar_wait(&S.d_empty[pair1], ph1 ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = bd0 + static_cast<uint32_t>(u) * kBSlot16;
                    const uint32_t at0 = tmem + kACol + static_cast<uint32_t>(64 * v);
                    const uint32_t d0 = tmem + kDCol + static_cast<uint32_t>(128 * pair0);
                    const uint32_t d1 = tmem + kDCol + static_cast<uint32_t>(128 * pair1);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {  // block j of the stage: pair 2 g + j / 2, slot half j % 2
                        const uint32_t d = (j < 2 ? d0 : d1) + static_cast<uint32_t>(64 * (j & 1));
                        // atom j / 2 of the B tile, bytes 64 (j % 2) + {0, 32} of its rows
                        const uint64_t b0 = bd + static_cast<uint64_t>((j >> 1) * kBAtom16 + (j & 1) * 4);
                        mma_ts(d, at0 + 16 * j, b0, idesc, 0u);
                        mma_ts(d, at0 + 16 * j + 8, b0 + 2, idesc, 1u);
                    }
                    mma_commit(&S.d_full[dsb]);
                    mma_commit(&S.a_empty[v]);
                    mma_commit(&S.b_empty[u]);
                    v ^= 1;
                    if (v == 0) pa ^= 1u;
                    if (++u == kBS) u = 0;
                    if (++dsb == kDStageBars) dsb = 0;
                    p1 += 2;
                    if (p1 >= 2 * kDPairs) p1 -= 2 * kDPairs;
                }
            }
        }
        __syncwarp();
    } else if (warp <= 5) {
        // ---------------------------------------------------------- A converters
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16) + kACol;
        for (int k = 0; k < my_items && ok; ++k) {
            for (int s = 0; s < kst; ++s) {
                const int g = k * kst + s, r = g % kRaw, v = g % kAB;
                if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.raw_full[r], (g / kRaw) & 1u))) { ok = false; break; }
                uint4 raw[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) raw[c] = *reinterpret_cast<const uint4 *>(S.raw[r] + sw_off(row, c));
                if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.a_empty[v], ((g / kAB) & 1u) ^ 1u))) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t w[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) i8x16_to_h(raw[4 * h + c], &w[8 * c]);
                    tmem_st32(lane_addr + static_cast<uint32_t>(64 * v + 32 * h), w);
                }
                // The raw slot goes back to the TMA (async proxy) only after its values have
                // been consumed, with a proxy fence between the reads and the refill.
                fence_async_shared();
                mbar_arrive(&S.raw_empty[r]);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.b_full[g % kBS], (g / kBS) & 1u))) { ok = false; break; }
                mbar_arrive(&S.a_full[v]);
            }
        }
    } else if (warp == 6) {
        // ---------------------------------------------------------- TMA: activations
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmXh)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmXs)) : "memory");
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
            for (int k = 0; k < my_items && ok; ++k) {
                Item it;
                decode_item(S, static_cast<int>(blockIdx.x) + k * C, ecur, it);
                const int sb = k & 1;
                // the item's activation scales: fp32 [block][64 sorted rows] (x = tok0, a
                // multiple of 4, so the copy starts on a 16-byte boundary)
                if (!mbar_wait(&S.s_empty[sb], ((k >> 1) & 1u) ^ 1u)) { ok = false; break; }
                mbar_expect_tx(&S.s_full[sb], xs_bytes);
                tma_load_2d(&S.xs[sb][0][0], &tmXs, it.tok0, 0, &S.s_full[sb], pol);
                for (int s = 0; s < kst; ++s) {
                    const int g = k * kst + s, u = g % kBS;
                    if (!mbar_wait(&S.b_empty[u], ((g / kBS) & 1u) ^ 1u)) { ok = false; break; }
                    mbar_expect_tx(&S.b_full[u], kBBytes);
                    tma_load_2d(S.bt[u], &tmXh, s * kStageK, it.tok0, &S.b_full[u], pol);
                    tma_load_2d(S.bt[u] + kBAtom, &tmXh, s * kStageK + 64, it.tok0, &S.b_full[u], pol);
                }
            }
        }
        __syncwarp();
    } else if (warp == 7) {
        // ---------------------------------------------------------- Wd rows of each item
        const int pieces = nb / 8;  // 16-byte pieces of a scale row
        for (int k = 0; k < my_items && ok; ++k) {
            Item it;
            decode_item(S, static_cast<int>(blockIdx.x) + k * C, ecur, it);
            const int sb = k & 1;
            if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.s_empty[sb], ((k >> 1) & 1u) ^ 1u))) { ok = false; break; }
#pragma unroll 1
            for (int rr = 0; rr < 4; ++rr) {
                const int r = lane + 32 * rr;
                const int64_t o = it.m0 + r;
                const bool valid = o < a.Mo;
                const uint16_t *src = a.Wd + (it.e * a.Mo + (valid ? o : 0)) * nb;
                const uint32_t dst = saddr(S.wd[sb] + r * kScalePitch);
                for (int p = 0; p < pieces; ++p)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + 16 * p), "l"(src + 8 * p),
                                 "r"(valid ? 16u : 0u)
                                 : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            mbar_arrive(&S.s_full[sb]);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const int grp = (warp - 8) >> 2;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16) + kDCol;
        for (int k = 0; k < my_items; ++k) {
            Item it;
            decode_item(S, static_cast<int>(blockIdx.x) + k * C, ecur, it);
            const int sb = k & 1;
            const bool split_cols = it.n > 32;
            const int c0 = split_cols ? 32 * grp : 0;  // first accumulator column of this thread
            if (ok && !__all_sync(WSW_FULL_MASK, mbar_wait(&S.s_full[sb], (k >> 1) & 1u))) ok = false;
            uint64_t acc2[16];  // accumulators of columns c0 + 2 i, c0 + 2 i + 1
#pragma unroll
            for (int i = 0; i < 16; ++i) acc2[i] = 0ull;
            // acc += fl(Wd * xd) * isum per column: the scalar arithmetic, two columns an instruction
            auto scale_add = [&](int b, const uint32_t(&dv)[32]) {
                const float wd = __half2float(reinterpret_cast<const __half *>(S.wd[sb] + row * kScalePitch)[b]);
                const uint64_t ww = f2_pack(wd, wd);
                const float4 *xs4 = reinterpret_cast<const float4 *>(&S.xs[sb][b][c0]);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 xs = xs4[j4];
                    f2_scale_fma(acc2[2 * j4], ww, f2_pack(xs.x, xs.y),
                                 f2_pack(__uint_as_float(dv[4 * j4]), __uint_as_float(dv[4 * j4 + 1])));
                    f2_scale_fma(acc2[2 * j4 + 1], ww, f2_pack(xs.z, xs.w),
                                 f2_pack(__uint_as_float(dv[4 * j4 + 2]), __uint_as_float(dv[4 * j4 + 3])));
                }
            };
            // pair gp = 2 g + pp holds blocks 4 s + 2 pp and 4 s + 2 pp + 1 of stage s
            for (int s = 0; s < kst && ok; ++s) {
                const int g = k * kst + s;
                if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.d_full[g % kDStageBars], (g / kDStageBars) & 1u))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int pp = 0; pp < 2; ++pp) {
                    const int gp = 2 * g + pp, p = gp % kDPairs;
                    const uint32_t pa = lane_addr + static_cast<uint32_t>(128 * p);
                    uint32_t dv[32];
                    if (!split_cols) {
                        tmem_ld32(pa + static_cast<uint32_t>(64 * grp), dv);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&S.d_empty[p]);
                        scale_add(4 * s + 2 * pp + grp, dv);
                    } else {
                        tmem_ld32(pa + static_cast<uint32_t>(c0), dv);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                        scale_add(4 * s + 2 * pp, dv);
                        tmem_ld32(pa + static_cast<uint32_t>(64 + c0), dv);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&S.d_empty[p]);
                        scale_add(4 * s + 2 * pp + 1, dv);
                    }
                }
            }
            mbar_arrive(&S.s_empty[sb]);
            float acc[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) f2_unpack(acc2[i], acc[2 * i], acc[2 * i + 1]);
            const int64_t o = it.m0 + row;
            const float nan = __int_as_float(0x7fc00000);
            if (split_cols) {
                if (o < a.Mo) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < it.n)
                            a.y[static_cast<int64_t>(S.list[it.tok0 + c0 + j]) * a.Mo + o] = ok ? acc[j] : nan;
                }
            } else {
                // group 1 hands its sums to group 0
                if (grp == 1) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) S.comb[j][row] = ok ? acc[j] : nan;
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
                if (grp == 0 && o < a.Mo) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < it.n)
                            a.y[static_cast<int64_t>(S.list[it.tok0 + j]) * a.Mo + o] =
                                ok ? acc[j] + S.comb[j][row] : nan;
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
            }
        }
        if (!ok) S.timed_out = 1;  // the rows of the remaining items hold NaN
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && S.timed_out && a.err) atomicOr(a.err, 2);  // tell the host
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_moe() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_map_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base, uint64_t inner, uint64_t outer,
                 uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    auto fn = encode_fn_moe();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Sizes the tensor-core form takes: whole 128-value stages and 16-byte pieces of a scale
// row (K % 256), at most kMaxBlocks blocks; routed rows, experts and sorted positions
// that fit shared memory.
static bool tc_shape_ok(int64_t E, int64_t K, int64_t R) {
    return E > 0 && K > 0 && R > 0 && K % 256 == 0 && K / 32 <= kMaxBlocks && R <= kMaxRows && E <= kMaxE;
}

size_t moe_q8_tc_workspace_bytes(int64_t E, int64_t K, int64_t R) {
    return tc_shape_ok(E, K, R) ? ws_layout(E, K, R).bytes : 0;
}

// Whether the tensor-core path takes this problem (the caller falls back otherwise).
bool moe_q8_tc_supported(const MoeTcArgs &a) {
    // the sizes above, and a workspace of the layout's size, 256-byte aligned
    if (!tc_shape_ok(a.E, a.K, a.R) || a.E * a.Mo > 0x7fffffffLL) return false;
    if (((reinterpret_cast<uintptr_t>(a.Wq) | reinterpret_cast<uintptr_t>(a.Wd) | reinterpret_cast<uintptr_t>(a.xq) |
          reinterpret_cast<uintptr_t>(a.xd)) & 15) != 0)
        return false;
    return a.ws != nullptr && (reinterpret_cast<uintptr_t>(a.ws) & 255) == 0 &&
           a.ws_bytes >= ws_layout(a.E, a.K, a.R).bytes;
}

int moe_q8_tc_launch(const MoeTcArgs &a, int sm_count, cudaStream_t s, bool pdl) {
    const WsLayout L = ws_layout(a.E, a.K, a.R);
    unsigned char *ws = static_cast<unsigned char *>(a.ws);
    CUtensorMap mW, mXh, mXs;
    if (!make_map_2d(&mW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wq, a.K, a.E * a.Mo, a.K, kStageK, kRows,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&mXh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ws + L.xh, a.K, L.Rp, a.K * 2, 64, kNT,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&mXs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ws + L.xs, L.Rp, a.K / 32, L.Rp * 4, kNT,
                     static_cast<uint32_t>(a.K / 32), CU_TENSOR_MAP_SWIZZLE_NONE))
        return WSW_ERR_CUDA;
    // the prepass: one CTA per SM (at most one per routed row)
    const size_t prep_smem = static_cast<size_t>(2 * a.R + (kBucketWarps + 2) * a.E) * 4;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(moe_q8_prep_kernel), static_cast<int>(prep_smem));
    if (e != cudaSuccess) return WSW_ERR_CUDA;
    const unsigned prep_ctas = static_cast<unsigned>(a.R < sm_count ? a.R : sm_count);
    e = launch(moe_q8_prep_kernel, dim3(prep_ctas), dim3(kPrepThreads), prep_smem, s, pdl, a, L);
    if (e != cudaSuccess) return WSW_ERR_CUDA;
    // the product, programmatically dependent on the prepass
    const size_t smem = sizeof(Smem) + 1024;
    e = ensure_smem(reinterpret_cast<const void *>(moe_q8_tc_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return WSW_ERR_CUDA;
    e = launch(moe_q8_tc_kernel, dim3(static_cast<unsigned>(sm_count)), dim3(kThreads), smem, s, true, mW, mXh, mXs,
               a, L);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}

}  // namespace wsw
