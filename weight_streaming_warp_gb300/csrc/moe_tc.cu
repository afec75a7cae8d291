// moe_tc.cu -- grouped q8_0 MoE mat-vec on the tensor cores, for many rows per expert.
//
// Source: "QuantizeQ8KK is thread-per-superblock: 95.5us/call ..." (vllm.cpp issue),
// sections Cause and Scope: the MoE path quantizes m = T x top_k rows and runs a grouped
// GEMM over the experts.  With hundreds of rows the grouped product is a real dense
// contraction (about 60 integer operations per weight byte at T = 512), so it runs on
// tcgen05 instead of dp4a.
//
// Exactness.  q8_0 values are integers in [-127, 127], exact in fp16.  The weights enter
// the MMA as they are; an activation byte q enters biased, as the binary16 value 1152 + q
// (its bit pattern is 0x6400 | (q ^ 0x80), two byte permutes per four values).  Each
// block sum over 32 products is then I + 1152 * S with S the block's weight sum, at most
// 32 * 127 * 1279 < 2^23 in magnitude, so every partial sum is an integer exact in the
// fp32 accumulator.  One B row holds the constant 1152, so the MMA also yields the
// correction 1152 * S in its own column.  One tcgen05.mma (kind::f16, K = 32 as two K = 16
// steps) per block gives these exact sums for 128 weight rows x up to 62 routed rows; the
// epilogue subtracts the correction, scales by fp32(Wd) * fp32(xd) and accumulates in fp32:
//   y[m][o] = sum_b Wd[o][b] * xd[m][b] * isum_b(o, m).
//
// Persistent: one CTA per SM.  Every CTA buckets the routing ids by expert in shared
// memory (the same stable lists in every CTA), then walks the work items i = blockIdx,
// blockIdx + gridDim, ...; an item is (expert e, 128 output rows, up to 62 of e's routed
// rows), items ordered by expert, then row tile, then token tile, so the grid streams
// one contiguous window of the expert weights and the token tiles of one weight tile run
// side by side (the second read of the tile comes from L2).  A stage is 128 K-values
// (four blocks).  Warp roles (16 warps):
//   warp 0       TMA: raw int8 weight tiles (128 rows x 128 bytes, 128-byte swizzle) into
//                a ring of kRaw stages
//   warp 1       tensor memory owner; one thread issues the MMAs: A from tensor memory,
//                B from shared memory, D into a ring of kDPairs slots of two 64-column
//                blocks, and commits once per pair
//   warps 2-5    A converters: thread = weight row (its tensor-memory lane); reads its
//                row's 128 bytes from the swizzled tile (conflict-free), converts int8 ->
//                fp16 and writes the 64 packed columns with tcgen05.st
//   warps 6-7    B converters: thread = B row (a routed row, or a constant row); its
//                activation values by cp.async (one stage ahead), int8 -> biased fp16
//                into 128-byte-swizzled K-major B tiles;
//                halfway through an item they start the cp.async of the next item's
//                scale rows (Wd rows as they are, padded; xd rows), and at its first stage
//                turn the xd rows into fp32 [block][token]
//   warps 8-15   epilogue: two groups of four warps (one per lane quarter); tcgen05.ld of
//                a block, scale and accumulate; with at most 31 routed rows group h takes
//                the blocks of parity h (columns 0-31) and hands its sums to group 0
//                through shared memory, with more it takes every block for columns
//                32 h .. 32 h + 31.  Columns 0-30 and 32-62 are routed rows, columns 31
//                and 63 the corrections.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_tc.cuh"
#include "tc_util.cuh"

namespace wsw {
namespace {

using namespace tc;

constexpr int kRows = 128;      // output rows per item (MMA M)
constexpr int kCols = 64;       // B rows = accumulator columns of a block (MMA N <= 64)
constexpr int kNT = 62;         // routed rows per item: columns 0-30 and 32-62
constexpr int kHalf = 31;       // routed rows per 32-column half (column 31 / 63: correction)
constexpr int kStageK = 128;    // K-values per stage (four blocks)
constexpr int kRaw = 4;         // raw weight stages (16 KB each)
constexpr int kAB = 2;          // A (tensor memory) and B (shared memory) slots
constexpr int kDPairs = 3;      // accumulator slots of two blocks (64 columns each)
constexpr int kXAhead = 2;      // activation cp.async ring (stages)
constexpr int kMaxBlocks = 64;  // K <= 2048
constexpr int kMaxList = 4096;  // routed rows kept in shared memory
constexpr int kMaxE = 512;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kBucketWarps = 8;

constexpr int kRawBytes = kRows * kStageK;       // 16 KB
constexpr int kBAtom = kCols * 128;              // one 64-value K-major atom of B: 8 KB
constexpr int kBBytes = 2 * kBAtom;              // 16 KB
constexpr int kXRawBytes = kCols * kStageK;      // 8 KB
constexpr int kScalePitch = 144;                 // bytes per staged scale row (<= 64 binary16 + pad)
constexpr uint32_t kACol = 0;                    // A slots: columns 0 .. 127
constexpr uint32_t kDCol = 64 * kAB;             // D slots: columns 128 .. 511 (128 per pair)
constexpr uint32_t kTmemCols = 512;

struct Smem {
    unsigned char raw[kRaw][kRawBytes];     // 1024-aligned (first member); bucketing scratch first
    unsigned char bt[kAB][kBBytes];         // 1024-aligned
    unsigned char xraw[kXAhead][kXRawBytes];  // row t: 16-byte chunk j at (j ^ (t & 7))
    unsigned char wd[2][kRows * kScalePitch];  // per item (double-buffered): Wd rows, padded
    unsigned char xdr[kCols * kScalePitch];   // the next item's xd rows, padded
    float xs[2][kMaxBlocks][kCols];           // per item: xd as fp32, [block][column]
    float comb[32][kRows];                    // group 1 -> group 0 partial sums (<= 32 rows)
    uint16_t list[kMaxList];
    int cnt[kMaxE];
    int off[kMaxE];
    int ibase[kMaxE + 1];
    uint64_t raw_full[kRaw], raw_empty[kRaw];
    uint64_t a_full[kAB], b_full[kAB], ab_empty[kAB];
    uint64_t d_full[kDPairs], d_empty[kDPairs];
    uint64_t s_full[2], s_empty[2];
    uint32_t tmem_slot;
    int nitems;
};

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
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
    int tok0;  // first routed row in the expert-ordered list
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

// accumulator column of routed row t of an item, and back (-1: a correction column)
__device__ __forceinline__ int col_of(int t) { return t < kHalf ? t : t + 1; }
__device__ __forceinline__ int tok_of(int col) { return (col & 31) == kHalf ? -1 : (col < 32 ? col : col - 1); }
// MMA N of an item with n routed rows: one half (and its correction) or both
__device__ __forceinline__ int cols_of(int n) { return n <= kHalf ? 32 : 64; }

// 16 int8 values -> 16 biased binary16 values 1152 + q (exact), as 8 packed half2 words
__device__ __forceinline__ void i8x16_to_h_biased(const uint4 &v, uint32_t *o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t u = w[i] ^ 0x80808080u;
        o[2 * i] = __byte_perm(u, 0x64646464u, 0x4140);      // 1024 + u0, 1024 + u1
        o[2 * i + 1] = __byte_perm(u, 0x64646464u, 0x4342);  // 1024 + u2, 1024 + u3
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    moe_q8_tc_kernel(const __grid_constant__ CUtensorMap tmWq, const MoeTcArgs a) {
    extern __shared__ unsigned char smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = static_cast<int>(a.E);
    const int R = static_cast<int>(a.R);
    const int nb = static_cast<int>(a.K / 32);       // blocks per row
    const int kst = static_cast<int>(a.K / kStageK); // stages per item
    const int m_tiles = static_cast<int>((a.Mo + kRows - 1) / kRows);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRaw; ++i) { mbar_init(&S.raw_full[i], 1); mbar_init(&S.raw_empty[i], 128); }
        for (int i = 0; i < kAB; ++i) {
            mbar_init(&S.a_full[i], 128); mbar_init(&S.b_full[i], 64); mbar_init(&S.ab_empty[i], 1);
        }
        for (int i = 0; i < kDPairs; ++i) { mbar_init(&S.d_full[i], 1); mbar_init(&S.d_empty[i], 8); }
        for (int i = 0; i < 2; ++i) { mbar_init(&S.s_full[i], 64); mbar_init(&S.s_empty[i], 256); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }

    pdl_wait();  // ids and activations come from earlier kernels

    // ------------------------------------------------------------ bucketing
    // Stable per-expert lists of the routed rows (every CTA builds the same ones).
    int *ids_s = reinterpret_cast<int *>(&S.raw[0][0]);
    int *wcnt = ids_s + R;  // [kBucketWarps][E]
    {
        bool bad = false;
        for (int m = threadIdx.x; m < R; m += kThreads) {
            const int id = a.ids[m];
            const bool ok = id >= 0 && id < E;
            ids_s[m] = ok ? id : -1;
            bad |= !ok;
        }
        if (bad && blockIdx.x == 0 && a.err) atomicOr(a.err, 1);
        for (int i = threadIdx.x; i < kBucketWarps * E; i += kThreads) wcnt[i] = 0;
    }
    __syncthreads();
    const int r0 = warp < kBucketWarps ? static_cast<int>(static_cast<int64_t>(warp) * R / kBucketWarps) : 0;
    const int r1 = warp < kBucketWarps ? static_cast<int>(static_cast<int64_t>(warp + 1) * R / kBucketWarps) : 0;
    for (int base = r0; base < r1; base += 32) {
        const int m = base + lane;
        const int e = m < r1 ? ids_s[m] : -1;
        const unsigned peers = __match_any_sync(WSW_FULL_MASK, e >= 0 ? e : E + lane);
        if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kBucketWarps; ++w) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
        S.cnt[e] = run;
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scans over the experts: list offsets and item bases
        int run = 0, irun = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = e < E ? S.cnt[e] : 0;
            const int items = m_tiles * ((c + kNT - 1) / kNT);
            int incl = c, iincl = items;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(WSW_FULL_MASK, incl, o);
                const int it = __shfl_up_sync(WSW_FULL_MASK, iincl, o);
                if (lane >= o) { incl += t; iincl += it; }
            }
            if (e < E) {
                S.off[e] = run + incl - c;
                S.ibase[e] = irun + iincl - items;
            }
            run += __shfl_sync(WSW_FULL_MASK, incl, 31);
            irun += __shfl_sync(WSW_FULL_MASK, iincl, 31);
        }
        if (lane == 0) {
            S.ibase[E] = irun;
            S.nitems = irun;
        }
    }
    __syncthreads();
    for (int base = r0; base < r1; base += 32) {
        const int m = base + lane;
        const int e = m < r1 ? ids_s[m] : -1;
        const unsigned peers = __match_any_sync(WSW_FULL_MASK, e >= 0 ? e : E + lane);
        if (e >= 0) S.list[S.off[e] + wcnt[warp * E + e] + __popc(peers & ((1u << lane) - 1u))] = static_cast<uint16_t>(m);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();  // the raw ring is free again
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
        // ---------------------------------------------------------- TMA producer
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
            for (int k = 0; k < my_items && ok; ++k) {
                Item it;
                decode_item(S, static_cast<int>(blockIdx.x) + k * C, ecur, it);
                const uint32_t idesc = instr_desc(kRows, cols_of(it.n), false);
                for (int s = 0; s < kst && ok; ++s) {
                    const int g = k * kst + s, v = g % kAB;
                    const uint32_t ph = (g / kAB) & 1u;
                    if (!mbar_wait(&S.a_full[v], ph) || !mbar_wait(&S.b_full[v], ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = sw128_desc(saddr(S.bt[v]));
                    for (int pp = 0; pp < 2; ++pp) {
                        const int gp = 2 * g + pp, p = gp % kDPairs;
                        if (!mbar_wait(&S.d_empty[p], ((gp / kDPairs) & 1u) ^ 1u)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int j = 2 * pp + jj;  // block of the stage
                            const uint32_t d = tmem + kDCol + static_cast<uint32_t>(128 * p + 64 * jj);
                            const uint32_t at = tmem + kACol + static_cast<uint32_t>(64 * v + 16 * j);
                            // block j: atom j / 2 of the B tile, bytes 64 (j % 2) + {0, 32} of its rows
                            const uint64_t b0 = bd + static_cast<uint64_t>((j >> 1) * (kBAtom >> 4) + (j & 1) * 4);
                            mma_ts(d, at, b0, idesc, 0u);
                            mma_ts(d, at + 8, b0 + 2, idesc, 1u);
                        }
                        mma_commit(&S.d_full[p]);
                    }
                    mma_commit(&S.ab_empty[v]);
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
                if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.ab_empty[v], ((g / kAB) & 1u) ^ 1u))) { ok = false; break; }
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
                mbar_arrive(&S.a_full[v]);
            }
        }
    } else if (warp <= 7) {
        // ---------------------------------------------------------- B converters
        const int tt = threadIdx.x - 6 * 32;  // 0..63: B row = accumulator column
        const int tk = tok_of(tt);            // routed row of the item in this column, or -1
        // The correction rows (constant 1152) are written once into both B slots.
        if (tk < 0) {
            const uint32_t c1152 = 0x64806480u;
#pragma unroll
            for (int v = 0; v < kAB; ++v)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<uint4 *>(S.bt[v] + h * kBAtom + sw_off(tt, i)) =
                            make_uint4(c1152, c1152, c1152, c1152);
            fence_async_shared();
        }
        const int total = my_items * kst;
        const int pieces = nb / 8;            // 16-byte pieces of a scale row
        int kc = -1;  // item whose token row `xrow` describes
        Item cit;
        int ec2 = 0, ec3 = 0;
        const int8_t *xrow = nullptr;
        bool xzero = false;  // row inside the MMA's N but past the routed rows: zeros
        // the 128 activation values of token tt for global stage i -> xraw[i % kXAhead]
        auto copy_x = [&](int i) {
            if (i < total) {
                const int k = i / kst, s = i - k * kst;
                if (k != kc) {
                    decode_item(S, static_cast<int>(blockIdx.x) + k * C, ec2, cit);
                    kc = k;
                    xrow = tk >= 0 && tk < cit.n ? a.xq + static_cast<int64_t>(S.list[cit.tok0 + tk]) * a.K : nullptr;
                    xzero = tk >= cit.n && tt < cols_of(cit.n);
                }
                if (xrow || xzero) {
                    const int8_t *src = xrow ? xrow + s * kStageK : a.xq;
                    const uint32_t n = xrow ? 16u : 0u;
                    const uint32_t dst = saddr(S.xraw[i % kXAhead] + tt * kStageK);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + ((j ^ (tt & 7)) << 4)),
                                     "l"(src + 16 * j), "r"(n)
                                     : "memory");
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        // the scale rows of item kk (128 Wd rows into wd[kk % 2], this thread's xd row into
        // xdr) join the cp.async group committed next; buffer kk % 2 must be released by
        // the epilogue of item kk - 2 first
        auto copy_scales = [&](int kk) -> bool {
            if (kk >= my_items) return true;
            Item si;
            decode_item(S, static_cast<int>(blockIdx.x) + kk * C, ec3, si);
            if (!mbar_wait(&S.s_empty[kk & 1], ((kk >> 1) & 1u) ^ 1u)) return false;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = tt + 64 * rr;
                const int64_t o = si.m0 + r;
                const bool valid = o < a.Mo;
                const uint16_t *src = a.Wd + (si.e * a.Mo + (valid ? o : 0)) * nb;
                const uint32_t dst = saddr(S.wd[kk & 1] + r * kScalePitch);
                for (int p = 0; p < pieces; ++p)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + 16 * p), "l"(src + 8 * p),
                                 "r"(valid ? 16u : 0u)
                                 : "memory");
            }
            const bool valid = tk >= 0 && tk < si.n;
            const uint16_t *src = a.xd + static_cast<int64_t>(valid ? S.list[si.tok0 + tk] : 0) * nb;
            const uint32_t dst = saddr(S.xdr + tt * kScalePitch);
            for (int p = 0; p < pieces; ++p)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + 16 * p), "l"(src + 8 * p),
                             "r"(valid ? 16u : 0u)
                             : "memory");
            return true;
        };
        if (!copy_scales(0)) ok = false;
        for (int i = 0; i < kXAhead - 1; ++i) copy_x(i);
        for (int k = 0; k < my_items && ok; ++k) {
            Item it;
            decode_item(S, static_cast<int>(blockIdx.x) + k * C, ecur, it);
            const int N = cols_of(it.n);
            for (int s = 0; s < kst; ++s) {
                const int g = k * kst + s, v = g % kAB;
                if (s == kst / 2 && !copy_scales(k + 1)) { ok = false; break; }
                copy_x(g + kXAhead - 1);
                asm volatile("cp.async.wait_group %0;" ::"n"(kXAhead - 1) : "memory");
                if (s == 0) {
                    // this item's scale rows have landed: xd -> fp32 [block][token]
                    const unsigned char *xr = S.xdr + tt * kScalePitch;
                    for (int p = 0; p < pieces; ++p) {
                        const uint4 v4 = *reinterpret_cast<const uint4 *>(xr + 16 * p);
                        const __half *h = reinterpret_cast<const __half *>(&v4);
#pragma unroll
                        for (int i = 0; i < 8; ++i) S.xs[k & 1][8 * p + i][tt] = __half2float(h[i]);
                    }
                    mbar_arrive(&S.s_full[k & 1]);
                }
                const unsigned char *xr = S.xraw[g % kXAhead] + tt * kStageK;
                if (!mbar_wait(&S.ab_empty[v], ((g / kAB) & 1u) ^ 1u)) { ok = false; break; }
                if (tt < N && tk >= 0) {
                    // values 64 h .. 64 h + 63 of the stage = atom h of the B tile
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t w[32];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            i8x16_to_h_biased(*reinterpret_cast<const uint4 *>(xr + (((4 * h + j) ^ (tt & 7)) << 4)), &w[8 * j]);
                        unsigned char *B = S.bt[v] + h * kBAtom;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            *reinterpret_cast<uint4 *>(B + sw_off(tt, i)) =
                                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                    fence_async_shared();
                }
                mbar_arrive(&S.b_full[v]);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // ---------------------------------------------------------- epilogue
        // Two groups of four warps (one per lane quarter).  Items with at most 32 routed
        // rows: group h takes the blocks of parity h (32 columns each) and group 1 hands
        // its sums to group 0; items with more: group h takes every block, columns
        // 32 h .. 32 h + 31.
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const int grp = (warp - 8) >> 2;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16) + kDCol;
        for (int k = 0; k < my_items; ++k) {
            Item it;
            decode_item(S, static_cast<int>(blockIdx.x) + k * C, ecur, it);
            const int sb = k & 1;
            const bool split_cols = it.n > kHalf;
            const int c0 = split_cols ? 32 * grp : 0;  // first accumulator column of this thread
            if (ok && !__all_sync(WSW_FULL_MASK, mbar_wait(&S.s_full[sb], (k >> 1) & 1u))) ok = false;
            float acc[kHalf];
#pragma unroll
            for (int j = 0; j < kHalf; ++j) acc[j] = 0.0f;
            // block b's 32 columns c0 .. c0 + 31: routed rows, then the correction 1152 * S
            auto scale_add = [&](int b, const uint32_t(&dv)[32]) {
                const float wd = __half2float(reinterpret_cast<const __half *>(S.wd[sb] + row * kScalePitch)[b]);
                const float wdc = wd * __uint_as_float(dv[kHalf]);
                const float4 *xs4 = reinterpret_cast<const float4 *>(&S.xs[sb][b][c0]);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 xs = xs4[j4];
                    const float x[4] = {xs.x, xs.y, xs.z, xs.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int j = 4 * j4 + i;
                        if (j < kHalf)  // Wd * isum = Wd * (D - 1152 S), one rounding
                            acc[j] = fmaf(x[i], fmaf(__uint_as_float(dv[j]), wd, -wdc), acc[j]);
                    }
                }
            };
            // pair gp = 2 g + pp holds blocks 4 s + 2 pp and 4 s + 2 pp + 1 of stage s
            for (int s = 0; s < kst && ok; ++s) {
                for (int pp = 0; pp < 2 && ok; ++pp) {
                    const int gp = 2 * (k * kst + s) + pp, p = gp % kDPairs;
                    if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.d_full[p], (gp / kDPairs) & 1u))) { ok = false; break; }
                    tc_fence_after();
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
            const int64_t o = it.m0 + row;
            const float nan = __int_as_float(0x7fc00000);
            if (split_cols) {
                const int t0 = grp * kHalf;  // routed rows of columns c0 .. c0 + 30
                if (o < a.Mo) {
#pragma unroll
                    for (int j = 0; j < kHalf; ++j)
                        if (t0 + j < it.n)
                            a.y[static_cast<int64_t>(S.list[it.tok0 + t0 + j]) * a.Mo + o] = ok ? acc[j] : nan;
                }
            } else {
                // group 1 hands its sums to group 0
                if (grp == 1) {
#pragma unroll
                    for (int j = 0; j < kHalf; ++j) S.comb[j][row] = ok ? acc[j] : nan;
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
                if (grp == 0 && o < a.Mo) {
#pragma unroll
                    for (int j = 0; j < kHalf; ++j)
                        if (j < it.n)
                            a.y[static_cast<int64_t>(S.list[it.tok0 + j]) * a.Mo + o] =
                                ok ? acc[j] + S.comb[j][row] : nan;
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
            }
        }
    }
    tc_fence_before();
    __syncthreads();
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

}  // namespace

// Whether the tensor-core path takes this problem (the caller falls back otherwise).
bool moe_q8_tc_supported(int64_t E, int64_t Mo, int64_t K, int64_t R, const void *Wq, const void *Wd,
                         const void *xq, const void *xd) {
    // K: whole 128-value stages and 16-byte pieces of a scale row (K % 256), at most
    // kMaxBlocks blocks; the routing ids and per-warp counts fit the raw ring during
    // bucketing; the lists fit shared memory.
    return K % 256 == 0 && K / 32 <= kMaxBlocks && R <= kMaxList && E <= kMaxE &&
           (R + kBucketWarps * E) * 4 <= kRaw * kRawBytes && E * Mo <= 0x7fffffffLL &&
           ((reinterpret_cast<uintptr_t>(Wq) | reinterpret_cast<uintptr_t>(Wd) | reinterpret_cast<uintptr_t>(xq) |
             reinterpret_cast<uintptr_t>(xd)) & 15) == 0;
}

int moe_q8_tc_launch(const MoeTcArgs &a, int sm_count, cudaStream_t s, bool pdl) {
    auto fn = encode_fn_moe();
    if (!fn) return WSW_ERR_CUDA;
    CUtensorMap map;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.E * a.Mo)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K)};
    cuuint32_t box[2] = {kStageK, kRows};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(a.Wq), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return WSW_ERR_CUDA;
    const size_t smem = sizeof(Smem) + 1024;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(moe_q8_tc_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return WSW_ERR_CUDA;
    e = launch(moe_q8_tc_kernel, dim3(static_cast<unsigned>(sm_count)), dim3(kThreads), smem, s, pdl, map, a);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}

}  // namespace wsw
