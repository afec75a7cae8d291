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
// tcgen05.mma (kind::f16, fp16 inputs, K = 32 as two K = 16 steps) per block yields the
// exact integer block sums for a 128-row x NT-token tile.  The epilogue scales each
// block sum by fp32(Wd) * fp32(xd) (exact) and accumulates in fp32, blocks in order:
//   y[m][o] = sum_b (Wd[o][b] * xd[m][b]) * isum_b(o, m).
//
// One CTA per (expert, 128 output rows); the expert's rows are found by a stable scan of
// the routing ids and processed in token tiles of up to 64.  Pipeline (14 warps):
//   warp 0      TMA: raw int8 weight tiles (128 rows x 64 bytes) into a ring of 10 stages
//   warps 1-4   convert int8 -> fp16 into 128-byte-swizzled K-major A tiles, gather the
//               tile's activation rows (prefetched one stage ahead) into B tiles
//   warp 5      tensor memory; one thread issues the MMAs into a ring of 8 tensor-memory
//               slots (one 32-value block each) and commits
//   warps 6-13  epilogue, two warpgroups, each owning 32 token columns: tcgen05.ld of the
//               next block is in flight while the current one is scaled and accumulated;
//               a slot is released as soon as its values are in registers
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_tc.cuh"
#include "tc_util.cuh"

namespace wsw {
namespace {

using namespace tc;

constexpr int kRows = 128;     // output rows per CTA (MMA M)
constexpr int kNTMax = 64;     // tokens per tile (MMA N <= 64)
constexpr int kRaw = 10;       // raw weight stages (8 KB each)
constexpr int kCvt = 3;        // converted stages (A 16 KB + B 8 KB)
constexpr int kSlots = 8;      // tensor-memory slots (64 columns each): all 512 columns
constexpr int kThreadsM = 448;
constexpr int kMaxBlocks = 64;   // K <= 2048
constexpr int kMaxList = 4096;   // rows of one expert kept in shared memory

constexpr int kXAhead = 4;     // activation stages copied ahead (cp.async ring)
constexpr int kRawBytes = kRows * 64;
constexpr int kABytes = kRows * 128;
constexpr int kBBytes = kNTMax * 128;

struct Smem {
    unsigned char cvtA[kCvt][kABytes];   // 1024-aligned (first member)
    unsigned char cvtB[kCvt][kBBytes];
    unsigned char raw[kRaw][kRawBytes];
    unsigned char xraw[kXAhead][kNTMax * 64];  // int8 activation rows of a stage
    __half wscale[kRows][kMaxBlocks];
    float xscale[kMaxBlocks][kNTMax];  // transposed: one block's token scales are contiguous
    int list[kMaxList];
    uint64_t raw_full[kRaw], raw_empty[kRaw];
    uint64_t cvt_full[kCvt], cvt_empty[kCvt];
    uint64_t slot_full[kSlots], slot_empty[kSlots];
    uint32_t tmem_slot;
    int count;
};

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// 16 int8 values -> 16 fp16 values (exact), as 8 packed half2 words.  A byte q with its
// sign bit flipped is u = q + 128; the binary16 pattern 0x6400 | u is 1024 + u, and
// subtracting 1152 (0x6480) leaves q exactly.  Two byte permutes and two half2
// subtractions per four values.
__device__ __forceinline__ void i8x16_to_h(const uint4 &v, uint32_t (&o)[8]) {
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

__global__ void __launch_bounds__(kThreadsM, 1)
    moe_q8_tc_kernel(const __grid_constant__ CUtensorMap tmWq, const MoeTcArgs a, int m_tiles) {
    extern __shared__ unsigned char smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t e = blockIdx.x / m_tiles;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x % m_tiles) * kRows;
    const int nb = static_cast<int>(a.K / 32);  // 32-value blocks per row
    const int kst = nb / 2 + (nb & 1);          // 64-value stages per token tile

    pdl_wait();  // ids and activations come from earlier kernels
    if (blockIdx.x == 0 && a.err) {
        for (int64_t m = threadIdx.x; m < a.R; m += kThreadsM) {
            const int id = a.ids[m];
            if (id < 0 || id >= a.E) atomicOr(a.err, 1);
        }
    }
    // Routing ids into shared memory (coalesced, all threads; the converted-tile ring
    // is free until the main loop), then a stable list of this expert's rows.
    int *ids_s = reinterpret_cast<int *>(S.cvtA[0]);  // room for kCvt * kABytes / 4 ids
    if ((reinterpret_cast<uintptr_t>(a.ids) & 15) == 0) {
        const int64_t n4 = a.R / 4;
        for (int64_t i = threadIdx.x; i < n4; i += kThreadsM)
            reinterpret_cast<int4 *>(ids_s)[i] = __ldg(reinterpret_cast<const int4 *>(a.ids) + i);
        for (int64_t m = 4 * n4 + threadIdx.x; m < a.R; m += kThreadsM) ids_s[m] = a.ids[m];
    } else {
        for (int64_t m = threadIdx.x; m < a.R; m += kThreadsM) ids_s[m] = a.ids[m];
    }
    __syncthreads();
    if (warp == 0) {
        int n = 0;
        for (int64_t base = 0; base < a.R; base += 32) {
            const int64_t m = base + lane;
            const bool hit = m < a.R && ids_s[m] == static_cast<int>(e);
            const unsigned bal = __ballot_sync(WSW_FULL_MASK, hit);
            if (hit) {
                const int pos = n + __popc(bal & ((1u << lane) - 1u));
                if (pos < kMaxList) S.list[pos] = static_cast<int>(m);
            }
            n += __popc(bal);
        }
        if (lane == 0) S.count = n < kMaxList ? n : kMaxList;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRaw; ++i) { mbar_init(&S.raw_full[i], 1); mbar_init(&S.raw_empty[i], 128); }
        for (int i = 0; i < kCvt; ++i) { mbar_init(&S.cvt_full[i], 128); mbar_init(&S.cvt_empty[i], 1); }
        for (int i = 0; i < kSlots; ++i) { mbar_init(&S.slot_full[i], 1); mbar_init(&S.slot_empty[i], 256); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int n_e = S.count;
    pdl_launch_dependents();
    if (n_e == 0) return;  // expert unused: no tensor memory was taken

    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&S.tmem_slot)),
                     "r"(kSlots * kNTMax)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_slot;
    const int tiles = (n_e + kNTMax - 1) / kNTMax;
    const int total = tiles * kst;  // stages over all token tiles
    bool ok = true;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmWq)) : "memory");
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
            for (int i = 0; i < total && ok; ++i) {
                const int r = i % kRaw;
                if (!mbar_wait(&S.raw_empty[r], ((i / kRaw) & 1u) ^ 1u)) { ok = false; break; }
                mbar_expect_tx(&S.raw_full[r], kRawBytes);
                tma_load_2d(S.raw[r], &tmWq, (i % kst) * 64, static_cast<int>(e * a.Mo + m0), &S.raw_full[r], pol);
            }
        }
        __syncwarp();
    } else if (warp >= 1 && warp <= 4) {
        // ---------------------------------------------------------- converters
        const int c = threadIdx.x - 32;  // 0..127
        const int ch = c & 3;            // 16-byte chunk of a 64-byte raw row
        const int tt = c >> 1, hf = c & 1;  // B: token row, half of the 64 values
        // activation rows of stage i -> xraw[i % kXAhead], 32 bytes per thread, copied
        // kXAhead - 1 stages ahead; rows past the expert's count are zero-filled
        auto copy_x = [&](int i) {
            if (i < total) {
                const int tile = i / kst, ks = i % kst;
                const int t = tile * kNTMax + tt;
                const bool valid = t < n_e;
                const int8_t *src = valid ? a.xq + static_cast<int64_t>(S.list[t]) * a.K + ks * 64 + hf * 32 : a.xq;
                const uint32_t dst = saddr(S.xraw[i % kXAhead] + tt * 64 + hf * 32);
                const uint32_t n = valid ? 16u : 0u;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + 16), "l"(src + 16), "r"(n)
                             : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        for (int i = 0; i < kXAhead - 1; ++i) copy_x(i);
        for (int i = 0; i < total && ok; ++i) {
            const int r = i % kRaw, v = i % kCvt;
            copy_x(i + kXAhead - 1);
            if (!mbar_wait(&S.raw_full[r], (i / kRaw) & 1u)) { ok = false; break; }
            if (!mbar_wait(&S.cvt_empty[v], ((i / kCvt) & 1u) ^ 1u)) { ok = false; break; }
            unsigned char *A = S.cvtA[v];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int row = (c >> 2) + 32 * j;
                const uint4 raw = *reinterpret_cast<const uint4 *>(S.raw[r] + row * 64 + ch * 16);
                uint32_t h[8];
                i8x16_to_h(raw, h);
                *reinterpret_cast<uint4 *>(A + sw_off(row, 2 * ch)) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(A + sw_off(row, 2 * ch + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
            }
            mbar_arrive(&S.raw_empty[r]);
            // this stage's activation copy has landed (kXAhead - 1 newer groups may pend)
            asm volatile("cp.async.wait_group %0;" ::"n"(kXAhead - 1) : "memory");
            const uint4 x0 = *reinterpret_cast<const uint4 *>(S.xraw[i % kXAhead] + tt * 64 + hf * 32);
            const uint4 x1 = *reinterpret_cast<const uint4 *>(S.xraw[i % kXAhead] + tt * 64 + hf * 32 + 16);
            unsigned char *B = S.cvtB[v];
            uint32_t h0[8], h1[8];
            i8x16_to_h(x0, h0);
            i8x16_to_h(x1, h1);
            *reinterpret_cast<uint4 *>(B + sw_off(tt, 4 * hf)) = make_uint4(h0[0], h0[1], h0[2], h0[3]);
            *reinterpret_cast<uint4 *>(B + sw_off(tt, 4 * hf + 1)) = make_uint4(h0[4], h0[5], h0[6], h0[7]);
            *reinterpret_cast<uint4 *>(B + sw_off(tt, 4 * hf + 2)) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
            *reinterpret_cast<uint4 *>(B + sw_off(tt, 4 * hf + 3)) = make_uint4(h1[4], h1[5], h1[6], h1[7]);
            fence_async_shared();
            mbar_arrive(&S.cvt_full[v]);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == 5) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int g = 0;  // block counter over all tiles
            for (int i = 0; i < total && ok; ++i) {
                const int v = i % kCvt;
                const int tile = i / kst, ks = i % kst;
                const int nt_tok = n_e - tile * kNTMax < kNTMax ? n_e - tile * kNTMax : kNTMax;
                const int NT = (nt_tok + 15) & ~15;
                const uint32_t idesc = instr_desc(kRows, NT, false);
                if (!mbar_wait(&S.cvt_full[v], (i / kCvt) & 1u)) { ok = false; break; }
                tc_fence_after();
                const uint64_t dA = sw128_desc(saddr(S.cvtA[v]));
                const uint64_t dB = sw128_desc(saddr(S.cvtB[v]));
                const int nblk_here = (2 * ks + 1 < nb) ? 2 : 1;
                for (int j = 0; j < nblk_here; ++j, ++g) {
                    const int q = g % kSlots;
                    if (!mbar_wait(&S.slot_empty[q], ((g / kSlots) & 1u) ^ 1u)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d = tmem + static_cast<uint32_t>(q * kNTMax);
                    mma_bf16(d, dA + 4 * j, dB + 4 * j, idesc, 0u);          // values 32j .. 32j+15
                    mma_bf16(d, dA + 4 * j + 2, dB + 4 * j + 2, idesc, 1u);  // values 32j+16 .. 32j+31
                    mma_commit(&S.slot_full[q]);
                }
                mma_commit(&S.cvt_empty[v]);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const int wg = (warp - 6) >> 2;  // token columns 32*wg .. 32*wg+31
        const int64_t o = m0 + row;
        const int et = threadIdx.x - 192;  // 0..255 among the epilogue threads
        // this CTA's weight scales: each row's nb values are 2*nb contiguous bytes;
        // warpgroup wg loads 16-byte pieces wg, wg+2, ... (all issued before use)
        if (o < a.Mo) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.Wd + (e * a.Mo + o) * nb);
            uint4 v[kMaxBlocks / 16];
#pragma unroll
            for (int j = 0; j < kMaxBlocks / 16; ++j)
                if (8 * (2 * j + wg) < nb) v[j] = __ldg(src + 2 * j + wg);
#pragma unroll
            for (int j = 0; j < kMaxBlocks / 16; ++j)
                if (8 * (2 * j + wg) < nb) *reinterpret_cast<uint4 *>(&S.wscale[row][8 * (2 * j + wg)]) = v[j];
        }
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16) + static_cast<uint32_t>(32 * wg);
        int g = 0;
        for (int tile = 0; tile < tiles; ++tile) {
            const int nt_tok = n_e - tile * kNTMax < kNTMax ? n_e - tile * kNTMax : kNTMax;
            const bool mine = 32 * wg < nt_tok;  // this warpgroup has token columns in the tile
            // the tile's activation scales, fp32, transposed (named barrier 1: 256 threads)
            asm volatile("bar.sync 1, 256;" ::: "memory");
            {
                // token t's nb scales are 2*nb contiguous bytes: 16-byte pieces, two per thread
                constexpr int kPieces = kNTMax * kMaxBlocks / 8;  // 512 >= kNTMax * nb / 8
                uint4 v[kPieces / 256];
                int tk[kPieces / 256], pc[kPieces / 256];
#pragma unroll
                for (int j = 0; j < kPieces / 256; ++j) {
                    const int idx = et + 256 * j;
                    tk[j] = idx / (nb / 8);
                    pc[j] = idx % (nb / 8);
                    v[j] = make_uint4(0u, 0u, 0u, 0u);
                    if (tk[j] < nt_tok)
                        v[j] = __ldg(reinterpret_cast<const uint4 *>(
                                         a.xd + static_cast<int64_t>(S.list[tile * kNTMax + tk[j]]) * nb) + pc[j]);
                }
#pragma unroll
                for (int j = 0; j < kPieces / 256; ++j) {
                    if (tk[j] < kNTMax) {
                        const __half *h = reinterpret_cast<const __half *>(&v[j]);
#pragma unroll
                        for (int i = 0; i < 8; ++i) S.xscale[8 * pc[j] + i][tk[j]] = __half2float(h[i]);
                    }
                }
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            float acc[32];
#pragma unroll
            for (int t = 0; t < 32; ++t) acc[t] = 0.0f;
            float va[32], vb[32];
            // block b of this tile lives in slot (g + b) % kSlots
            auto fetch = [&](int b, float(&v)[32]) -> bool {
                const int gg = g + b, q = gg % kSlots;
                if (!ok || !mbar_wait(&S.slot_full[q], (gg / kSlots) & 1u)) { ok = false; return false; }
                tc_fence_after();
                if (mine) {
                    uint32_t r[32];
                    asm volatile(
                        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
                          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
                          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                        : "r"(lane_base + static_cast<uint32_t>(q * kNTMax)));
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                }
                return true;
            };
            auto release = [&](int b) {
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                tc_fence_before();
                mbar_arrive(&S.slot_empty[(g + b) % kSlots]);
            };
            auto scale_add = [&](int b, const float(&v)[32]) {
                if (!mine) return;
                const float wd = __half2float(S.wscale[row][b]);
                const float4 *xs4 = reinterpret_cast<const float4 *>(&S.xscale[b][32 * wg]);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 xs = xs4[j4];
                    acc[4 * j4 + 0] = fmaf(wd * xs.x, v[4 * j4 + 0], acc[4 * j4 + 0]);
                    acc[4 * j4 + 1] = fmaf(wd * xs.y, v[4 * j4 + 1], acc[4 * j4 + 1]);
                    acc[4 * j4 + 2] = fmaf(wd * xs.z, v[4 * j4 + 2], acc[4 * j4 + 2]);
                    acc[4 * j4 + 3] = fmaf(wd * xs.w, v[4 * j4 + 3], acc[4 * j4 + 3]);
                }
            };
            bool have = fetch(0, va);
            if (have) release(0);
            for (int b = 0; b < nb; b += 2) {
                // va holds block b; vb receives block b+1 while b is scaled
                const bool hb = (b + 1 < nb) && fetch(b + 1, vb);
                if (have) scale_add(b, va);
                if (hb) release(b + 1);
                const bool ha = (b + 2 < nb) && fetch(b + 2, va);
                if (hb) scale_add(b + 1, vb);
                if (ha) release(b + 2);
                have = ha;
            }
            g += nb;
            if (o < a.Mo && mine) {
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int tt = 32 * wg + t;
                    if (tt < nt_tok)
                        a.y[static_cast<int64_t>(S.list[tile * kNTMax + tt]) * a.Mo + o] =
                            ok ? acc[t] : __int_as_float(0x7fc00000);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kSlots * kNTMax)
                     : "memory");
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
    // K: whole 64-value stages, at most kMaxBlocks blocks; the scale rows (2 * K/32
    // bytes) split into 16-byte pieces; the routing ids fit the staging area.
    return K % 256 == 0 && K / 32 <= kMaxBlocks && R <= kMaxList && R * 4 <= kCvt * kABytes &&
           E * Mo <= 0x7fffffffLL &&
           ((reinterpret_cast<uintptr_t>(Wq) | reinterpret_cast<uintptr_t>(Wd) | reinterpret_cast<uintptr_t>(xq) |
             reinterpret_cast<uintptr_t>(xd)) & 15) == 0;
}

int moe_q8_tc_launch(const MoeTcArgs &a, cudaStream_t s, bool pdl) {
    auto fn = encode_fn_moe();
    if (!fn) return WSW_ERR_CUDA;
    CUtensorMap map;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.E * a.Mo)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K)};
    cuuint32_t box[2] = {64, kRows};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(a.Wq), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return WSW_ERR_CUDA;
    const int m_tiles = static_cast<int>((a.Mo + kRows - 1) / kRows);
    const size_t smem = sizeof(Smem) + 1024;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(moe_q8_tc_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return WSW_ERR_CUDA;
    e = launch(moe_q8_tc_kernel, dim3(static_cast<unsigned>(a.E * m_tiles)), dim3(kThreadsM), smem, s, pdl, map, a,
               m_tiles);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}

}  // namespace wsw
