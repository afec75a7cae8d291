// attn_prefill.cu -- causal prefill attention over a binary16 KV cache on the
// fifth-generation tensor cores: the pass that consumes the dequantized scratch.
//
// Source: "vulkan : dequant q8_0 KV once in coopmat1" (llama.cpp pull request),
// Overview (the flash-attention pass of prompt processing, pp512 at depth 32768 and
// 65536, reads the binary16 K and V) and the stride discussion (the cache keeps one
// head's rows head_dim * n_head_kv elements apart, the scratch back to back; both are
// read here through a 3-D tensor map with the caller's strides).
//
//   query i (0 <= i < nq) of query head (h, g) sits at position depth - nq + i and
//   attends to positions 0 .. depth - nq + i:
//     s_p = scale * q . K(h, p),  out = sum_p exp(s_p - m) V(h, p) / sum_p exp(s_p - m)
//
// Design (GB300, one CTA per (KV head, query head, tile of 128 queries)):
//  * warp 0       TMA: the query tile once (128 x 128 binary16, two 128-byte-swizzled
//                 boxes of 64 dims), then K tiles of 128 positions into a ring of kKS
//                 stages.
//  * warp 10      TMA: V tiles of 128 positions into a ring of kVS stages.  K and V have
//                 producers of their own, so that neither ring waits behind the other:
//                 a tile takes about 1.5 us to land, and K is needed a softmax earlier
//                 than V.
//  * warp 1       owns tensor memory (512 columns: O [0, 128), two score buffers S of
//                 128 columns, two P buffers of 64 columns) and one thread issues the
//                 MMAs: S_j = Q K_j^T (A = Q, B = K, both K-major in shared memory) and
//                 O += P_j V_j (A = P from tensor memory, binary16 pairs per column;
//                 B = V in its natural [position][dim] layout, an MN-major operand).
//                 S_{j+1} is issued before P_j is waited for, so the tensor core works
//                 on the next scores while the softmax runs.
//  * warps 2-9    softmax: a query row per thread (its tensor-memory lane) and one half
//                 of each tile's 128 positions per warp; the two warps of a lane quarter
//                 combine their tile maxima through shared memory.  Per tile: read the
//                 64 scores, mask the positions past the row's causal limit (only in the
//                 last tiles of a query tile), take the tile maximum in the log2 domain,
//                 write P = 2^(s scale log2(e) - m) as binary16 into tensor memory and
//                 add P to the row sum l (packed fp32x2 arithmetic).  The maximum m in
//                 use is raised (and O, l rescaled by 2^(m_old - m_new)) only when a
//                 tile's maximum exceeds it by more than 8; otherwise the stale maximum
//                 stays, P <= 2^8, and the final O / l is the same softmax.  At the end:
//                 O / l to fp32.
//  * Precision: Q, K, V and P are binary16 in the products, scores, O and l accumulate
//    in fp32 (l from the unrounded P).  P's rounding to binary16 (relative 2^-11) bounds
//    the error of an output element by about 2^-11 * sum_p w_p |V_p| / sum_p w_p.
//  * Every mbarrier wait is bounded (about a second); a role whose wait ran out stops,
//    the rows of the tile are written as NaN, the producer waits (bounded) for its
//    copies in flight, and tensor memory is still released.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_util.cuh"

namespace wsw {
namespace {

using namespace tc;

constexpr int kHD = 128;        // head_dim
constexpr int kBQ = 128;        // queries per tile (MMA M)
constexpr int kBP = 128;        // positions per KV tile (MMA N of S, K of P V)
constexpr int kKS = 3;          // K stages (a K tile is needed one softmax before its V tile)
constexpr int kVS = 2;          // V stages
constexpr int kSoftWarps = 8;   // two per tensor-memory lane quarter, one per half of a tile
constexpr int kVWarp = 2 + kSoftWarps;  // the V producer
// warp 0: Q and K TMA, warp 1: MMA, warps 2-9: softmax, warp 10: V TMA
constexpr int kThreadsA = 32 * (kVWarp + 1);
constexpr int kTile = kBP * kHD * 2;  // 32 KB: one K or V tile (two boxes of 64 dims)
constexpr int kBox = kTile / 2;       // 16 KB: 128 rows x 128 bytes
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 128, kColP = 384;
constexpr float kLazy = 8.0f;   // log2-domain headroom before the running maximum is raised

struct Smem {
    unsigned char q[kTile];
    unsigned char k[kKS][kTile];
    unsigned char v[kVS][kTile];
    uint64_t q_full;
    uint64_t k_full[kKS], k_empty[kKS];
    uint64_t v_full[kVS], v_empty[kVS];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full[2], pv_done[2];
    uint64_t o_final;
    uint64_t pair_max[2][4];  // the two warps of a lane quarter exchange tile maxima
    uint64_t pair_sum[4];     // ... and their halves of the row sums
    float red[2][2][kBQ];     // [tile parity][half][row]: partial tile maxima
    float lsum[2][kBQ];       // [half][row]: partial row sums
    uint32_t tmem_slot;
};

// One launch attends over the cache positions [pos0, pos0 + npos) of a cache of `depth`
// positions; K and V hold just those rows (a window of the cache, or all of it).  Between
// the windows of one batch the online-softmax state of every query row travels through
// `state`: fp32 [heads * group * nq][kStateStride] = (m, l, -, -, O[128]), O unnormalized
// and m the log2-domain maximum that P and O are relative to.
constexpr int kStateStride = 132;

struct AttnArgs {
    int64_t depth, nq;
    int64_t pos0, npos;  // the window of this launch
    int heads, group, qtiles;
    int first, last;     // first window (no incoming state), last window (write out)
    float scale_log2;    // scale * log2(e)
    float *out;
    float *state;        // NULL when first && last
};

// MN-major operand (V as B of P V): 128-byte swizzle, 64-element atoms along N
// `lbo` bytes apart, groups of 8 K-rows 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t addr, uint32_t lbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(saddr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(saddr(bar)), "l"(policy)
        : "memory");
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
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x (MUFU); results below 2^-126 flush to zero, which no probability here needs
// (the largest probability of a row is at least 2^-8).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}

__global__ void __launch_bounds__(kThreadsA, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
    extern __shared__ unsigned char smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // work item: (KV head h, query head g of its group, query tile t)
    const int t = static_cast<int>(blockIdx.x % a.qtiles);
    const int hg = static_cast<int>(blockIdx.x / a.qtiles);
    const int h = hg / a.group;
    const int64_t q0 = static_cast<int64_t>(t) * kBQ;
    const int64_t rows = a.nq - q0 < kBQ ? a.nq - q0 : kBQ;
    const int64_t base = a.depth - a.nq;           // position of query 0
    const int64_t lim0 = base + q0;                 // last position row 0 sees
    const int64_t lim_last = base + q0 + rows - 1;  // last position any row sees
    // KV tiles of this window that some row sees, and the first one that row 0 may not
    // see whole (past its causal limit, or past the window's last row)
    const int64_t wtiles = (a.npos + kBP - 1) / kBP;
    int64_t nkv64 = lim_last < a.pos0 ? 0 : (lim_last - a.pos0) / kBP + 1;
    if (nkv64 > wtiles) nkv64 = wtiles;
    const int nkv = static_cast<int>(nkv64);
    int64_t fm = lim0 + 1 - a.pos0 < 0 ? 0 : (lim0 + 1 - a.pos0) / kBP;
    if (fm > a.npos / kBP) fm = a.npos / kBP;
    const int first_masked = static_cast<int>(fm);

    if (threadIdx.x == 0) {
        mbar_init(&S.q_full, 1);
        for (int i = 0; i < kKS; ++i) { mbar_init(&S.k_full[i], 1); mbar_init(&S.k_empty[i], 1); }
        for (int i = 0; i < kVS; ++i) { mbar_init(&S.v_full[i], 1); mbar_init(&S.v_empty[i], 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&S.s_full[i], 1);
            mbar_init(&S.s_free[i], kSoftWarps);
            mbar_init(&S.p_full[i], kSoftWarps);
            mbar_init(&S.pv_done[i], 1);
            for (int qd = 0; qd < 4; ++qd) mbar_init(&S.pair_max[i][qd], 2);
        }
        for (int qd = 0; qd < 4; ++qd) mbar_init(&S.pair_sum[qd], 2);
        mbar_init(&S.o_final, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
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

    if (nkv == 0) {
        // no position of this window is visible to the tile: only the last window has
        // work, the output from the incoming state
        if (warp >= 2 && warp < kVWarp && a.last) {
            pdl_wait();  // the state is written by the window before, maybe still running
            const int qd = warp & 3, hf = (warp - 2) >> 2;
            const int r = 32 * qd + lane;
            if (r < rows) {
                const int64_t row = static_cast<int64_t>(hg) * a.nq + q0 + r;
                const float *st = a.state + row * kStateStride;
                const float inv = 1.0f / st[1];
                float *dst = a.out + row * kHD + 64 * hf;
#pragma unroll
                for (int i = 0; i < 64; i += 4) {
                    const float4 o = *reinterpret_cast<const float4 *>(st + 4 + 64 * hf + i);
                    *reinterpret_cast<float4 *>(dst + i) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
                }
            }
        }
    } else if (warp == 0) {
        if (lane == 0) {
            uint64_t pol_q, pol_kv;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_q));
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_kv));
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
            pdl_wait();  // Q and K may be written by earlier kernels in the stream
            mbar_expect_tx(&S.q_full, kTile);
            for (int b = 0; b < 2; ++b)
                tma_load_3d(S.q + b * kBox, &tmQ, 64 * b, static_cast<int>(q0), hg, &S.q_full, pol_q);
            int issued = 0;
            for (int j = 0; j < nkv && ok; ++j) {
                const int ks = j % kKS;
                if (j >= kKS && !mbar_wait(&S.k_empty[ks], ((j / kKS) - 1) & 1u)) { ok = false; break; }
                mbar_expect_tx(&S.k_full[ks], kTile);
                for (int b = 0; b < 2; ++b)
                    tma_load_3d(S.k[ks] + b * kBox, &tmK, 64 * b, j * kBP, h, &S.k_full[ks], pol_kv);
                issued = j + 1;
            }
            if (!ok) {
                // the copies still in flight land before the CTA may exit (bounded waits)
                for (int j = issued - kKS; j < issued; ++j)
                    if (j >= 0) mbar_wait(&S.k_full[j % kKS], (j / kKS) & 1u);
                mbar_wait(&S.q_full, 0);
            }
        }
        __syncwarp();
    } else if (warp == kVWarp) {
        if (lane == 0) {
            uint64_t pol_kv;
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_kv));
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
            pdl_wait();  // V may be written by earlier kernels in the stream
            int issued = 0;
            for (int j = 0; j < nkv && ok; ++j) {
                const int vs = j % kVS;
                if (j >= kVS && !mbar_wait(&S.v_empty[vs], ((j / kVS) - 1) & 1u)) { ok = false; break; }
                mbar_expect_tx(&S.v_full[vs], kTile);
                for (int b = 0; b < 2; ++b)
                    tma_load_3d(S.v[vs] + b * kBox, &tmV, 64 * b, j * kBP, h, &S.v_full[vs], pol_kv);
                issued = j + 1;
            }
            if (!ok) {
                for (int j = issued - kVS; j < issued; ++j)
                    if (j >= 0) mbar_wait(&S.v_full[j % kVS], (j / kVS) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id_s = instr_desc(kBQ, kBP, false);
            const uint32_t id_pv = instr_desc(kBQ, kHD, false) | (1u << 16);  // B (V) MN-major
            auto issue_s = [&](int j) -> bool {
                const int ks = j % kKS, sb = j & 1;
                if (!mbar_wait(&S.k_full[ks], (j / kKS) & 1u)) return false;
                if (j >= 2 && !mbar_wait(&S.s_free[sb], ((j >> 1) - 1) & 1u)) return false;
                tc_fence_after();
                for (int b = 0; b < 2; ++b) {
                    const uint64_t dq = sw128_desc(saddr(S.q + b * kBox));
                    const uint64_t dk = sw128_desc(saddr(S.k[ks] + b * kBox));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + kColS + 128 * sb, dq + 2 * kk, dk + 2 * kk, id_s, (b | kk) != 0);
                }
                mma_commit(&S.k_empty[ks]);
                mma_commit(&S.s_full[sb]);
                return true;
            };
            ok = mbar_wait(&S.q_full, 0);
            if (ok) ok = issue_s(0);
            for (int j = 0; j < nkv && ok; ++j) {
                if (j + 1 < nkv && !issue_s(j + 1)) { ok = false; break; }
                const int vs = j % kVS, pb = j & 1;
                if (!mbar_wait(&S.p_full[pb], (j >> 1) & 1u)) { ok = false; break; }
                if (!mbar_wait(&S.v_full[vs], (j / kVS) & 1u)) { ok = false; break; }
                tc_fence_after();
                const uint64_t dv = sw128_mn_desc(saddr(S.v[vs]), kBox);
#pragma unroll
                for (int kk = 0; kk < kBP / 16; ++kk)  // 16 positions per MMA: 8 P columns, 2 KB of V
                    mma_ts(tmem + kColO, tmem + kColP + 64 * pb + 8 * kk, dv + 128 * kk, id_pv,
                           (j | kk) != 0 || !a.first);
                mma_commit(&S.v_empty[vs]);
                mma_commit(&S.pv_done[pb]);
            }
            if (ok) mma_commit(&S.o_final);  // completes once every MMA issued above has
        }
        __syncwarp();
    } else {
        // softmax: thread = query row r (its tensor-memory lane) and half hf of each tile
        // (positions 64 hf .. 64 hf + 63); the two warps of a lane quarter combine their
        // tile maxima through shared memory, so both use the same maximum for the row
        const int qd = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int r = 32 * qd + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        const int64_t lim = base + q0 + (r < rows ? r : rows - 1);  // last visible position
        // last visible row of the window for this thread's row
        const int64_t lim_w = (lim - a.pos0 < a.npos - 1 ? lim - a.pos0 : a.npos - 1);
        const int64_t srow = static_cast<int64_t>(hg) * a.nq + q0 + (r < rows ? r : rows - 1);
        const float cs = a.scale_log2;
        const uint64_t cs2 = f2_pack(cs, cs);
        float m = -INFINITY;
        // four partial sums of the row's probabilities (two fp32 pairs, so that the
        // additions of a tile form two independent chains)
        uint64_t l2 = 0ull, l2b = 0ull;
        if (!a.first) {  // the state of the earlier windows: m, and l in half 0's sum
            pdl_wait();  // written by the window before, maybe still running
            m = a.state[srow * kStateStride];
            if (hf == 0) l2 = f2_pack(a.state[srow * kStateStride + 1], 0.0f);
        }
        for (int j = 0; j < nkv; ++j) {
            const int sb = j & 1;
            if (!__all_sync(WSW_FULL_MASK, ok && mbar_wait(&S.s_full[sb], (j >> 1) & 1u))) { ok = false; break; }
            tc_fence_after();
            uint32_t sv[2][32];
            tmem_ld32(lane_base + kColS + 128 * sb + 64 * hf, sv[0]);
            tmem_ld32(lane_base + kColS + 128 * sb + 64 * hf + 32, sv[1]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.s_free[sb]);
            if (j >= first_masked) {
                // positions past the row's causal limit or the window's end read as -inf
                const int64_t lc = lim_w - (static_cast<int64_t>(j) * kBP + 64 * hf);
                const int last = lc < 0 ? -1 : (lc > 63 ? 63 : static_cast<int>(lc));
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c > last) sv[c >> 5][c & 31] = 0xff800000u;
            }
            // tile maximum as four independent chains of 16
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 64; ++c) mq[c & 3] = fmaxf(mq[c & 3], __uint_as_float(sv[c >> 5][c & 31]));
            const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            S.red[sb][hf][r] = mx;
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.pair_max[sb][qd]);
            if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.pair_max[sb][qd], (j >> 1) & 1u))) { ok = false; break; }
            // scale > 0, so the maximum of the scaled scores is the scaled maximum
            const float mt = fmaxf(S.red[sb][0][r], S.red[sb][1][r]) * cs;
            // raise the maximum in use only when this tile exceeds it by more than kLazy
            // (both warps of the quarter decide alike: same inputs)
            const bool raise = mt > m + kLazy;
            if (j == 0 && !a.first) {
                // O of the earlier windows into tensor memory, rescaled to the maximum in use
                const float alpha = raise ? ex2(m - mt) : 1.0f;
                const float *so = a.state + srow * kStateStride + 4 + 64 * hf;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(so[32 * c + i] * alpha);
                    tmem_st32(lane_base + kColO + 64 * hf + 32 * c, o);
                }
                const uint64_t al2 = f2_pack(alpha, alpha);
                asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(l2) : "l"(al2));
                asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(l2b) : "l"(al2));
            } else if (j > 0 && __any_sync(WSW_FULL_MASK, raise)) {
                // O must hold P_{j-1} V_{j-1} before it is rescaled
                if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1u))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float alpha = raise ? ex2(m - mt) : 1.0f;
                const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kColO + 64 * hf + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        uint64_t v = f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1]));
                        asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(v) : "l"(al2));
                        float x0, x1;
                        f2_unpack(v, x0, x1);
                        o[i] = __float_as_uint(x0);
                        o[i + 1] = __float_as_uint(x1);
                    }
                    tmem_st32(lane_base + kColO + 64 * hf + 32 * c, o);
                }
                asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(l2) : "l"(al2));
                asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(l2b) : "l"(al2));
            }
            if (raise) m = mt;
            // P_j into its tensor-memory slot, free once P_{j-2} V_{j-2} has completed
            if (j >= 2 && !__all_sync(WSW_FULL_MASK, mbar_wait(&S.pv_done[sb], ((j >> 1) - 1) & 1u))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t nm2 = f2_pack(-m, -m);
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int e = 2 * i;
                uint64_t t = f2_pack(__uint_as_float(sv[e >> 5][e & 31]), __uint_as_float(sv[(e + 1) >> 5][(e + 1) & 31]));
                asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(t) : "l"(cs2), "l"(nm2));  // s log2(e) scale - m
                float t0, t1;
                f2_unpack(t, t0, t1);
                const float p0 = ex2(t0), p1 = ex2(t1);
                const __half2 hp = __floats2half2_rn(p0, p1);
                pk[i] = *reinterpret_cast<const uint32_t *>(&hp);
                if (i & 1) asm("add.rn.f32x2 %0, %0, %1;" : "+l"(l2b) : "l"(f2_pack(p0, p1)));
                else asm("add.rn.f32x2 %0, %0, %1;" : "+l"(l2) : "l"(f2_pack(p0, p1)));
            }
            tmem_st32(lane_base + kColP + 64 * sb + 32 * hf, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.p_full[sb]);
        }
        // epilogue: the row sum from both halves, then this half of O / l
        float l0, l1, l2f, l3;
        f2_unpack(l2, l0, l1);
        f2_unpack(l2b, l2f, l3);
        S.lsum[hf][r] = (l0 + l1) + (l2f + l3);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.pair_sum[qd]);
        const bool have = __all_sync(WSW_FULL_MASK, ok && mbar_wait(&S.pair_sum[qd], 0) && mbar_wait(&S.o_final, 0));
        tc_fence_after();
        const float lrow = S.lsum[0][r] + S.lsum[1][r];
        if (!a.last) {
            // hand the state on: m, l and this half of the unnormalized O
            float *st = a.state + srow * kStateStride;
            if (r < rows && hf == 0) {
                st[0] = have ? m : __int_as_float(0x7fc00000);
                st[1] = have ? lrow : __int_as_float(0x7fc00000);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t o[32];
                if (have) {
                    tmem_ld32(lane_base + kColO + 64 * hf + 32 * c, o);
                    tmem_wait_ld();
                }
                if (r < rows) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        float4 w;
                        w.x = have ? __uint_as_float(o[i]) : __int_as_float(0x7fc00000);
                        w.y = have ? __uint_as_float(o[i + 1]) : __int_as_float(0x7fc00000);
                        w.z = have ? __uint_as_float(o[i + 2]) : __int_as_float(0x7fc00000);
                        w.w = have ? __uint_as_float(o[i + 3]) : __int_as_float(0x7fc00000);
                        *reinterpret_cast<float4 *>(st + 4 + 64 * hf + 32 * c + i) = w;
                    }
                }
            }
        }
        const float inv = 1.0f / lrow;
        float *dst = a.out + ((static_cast<int64_t>(hg) * a.nq) + q0 + r) * kHD + 64 * hf;
#pragma unroll
        for (int c = 0; c < 2 && a.last; ++c) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(lane_base + kColO + 64 * hf + 32 * c, o);
                tmem_wait_ld();
            }
            if (r < rows) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    float4 w;
                    w.x = have ? __uint_as_float(o[i]) * inv : __int_as_float(0x7fc00000);
                    w.y = have ? __uint_as_float(o[i + 1]) * inv : __int_as_float(0x7fc00000);
                    w.z = have ? __uint_as_float(o[i + 2]) * inv : __int_as_float(0x7fc00000);
                    w.w = have ? __uint_as_float(o[i + 3]) * inv : __int_as_float(0x7fc00000);
                    *reinterpret_cast<float4 *>(dst + 32 * c + i) = w;
                }
            }
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// --------------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_attn() {
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

// 3-D binary16 map over rows of 128 values: dims (128, d1, d2) with byte strides
// (s1, s2); box (64, 128, 1) with 128-byte swizzle; out-of-range rows read as zero.
bool make_map3(CUtensorMap *map, const void *base, int64_t d1, int64_t d2, int64_t s1_bytes, int64_t s2_bytes) {
    auto fn = encode_fn_attn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(d1), static_cast<cuuint64_t>(d2)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(s1_bytes), static_cast<cuuint64_t>(s2_bytes)};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBP), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One launch over the window [pos0, pos0 + npos) of the cache (K and V hold its rows);
// arguments already validated.
int attn_launch(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t depth, int64_t heads,
                int64_t group, int64_t nq, int64_t kps, int64_t khs, int64_t vps, int64_t vhs, int64_t pos0,
                int64_t npos, bool first, bool last, float *state, float scale, float *out, cudaStream_t s,
                bool pdl, const DeviceInfo &di) {
    const size_t smem = sizeof(Smem) + 1024;
    if (smem > static_cast<size_t>(di.max_smem_optin)) return WSW_ERR_UNSUPPORTED;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(attn_prefill_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return WSW_ERR_CUDA;
    CUtensorMap tmQ, tmK, tmV;
    const int64_t hs_k = heads > 1 ? khs : kps * npos;
    const int64_t hs_v = heads > 1 ? vhs : vps * npos;
    if (!make_map3(&tmQ, q, nq, heads * group, kHD * 2, nq * kHD * 2) ||
        !make_map3(&tmK, k, npos, heads, kps * 2, hs_k * 2) || !make_map3(&tmV, v, npos, heads, vps * 2, hs_v * 2))
        return WSW_ERR_CUDA;
    AttnArgs a;
    a.depth = depth;
    a.nq = nq;
    a.pos0 = pos0;
    a.npos = npos;
    a.heads = static_cast<int>(heads);
    a.group = static_cast<int>(group);
    a.qtiles = static_cast<int>((nq + kBQ - 1) / kBQ);
    a.first = first ? 1 : 0;
    a.last = last ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.out = out;
    a.state = state;
    const unsigned grid = static_cast<unsigned>(a.qtiles * heads * group);
    e = launch(attn_prefill_kernel, dim3(grid), dim3(kThreadsA), smem, s, pdl, tmQ, tmK, tmV, a);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}

// Checks shared by the two entry points (q, out, the shape and the scale).
int check_common(const uint16_t *q, float *out, int64_t depth, int64_t heads, int64_t group, int64_t nq,
                 int64_t head_dim, float scale) {
    if (heads < 0 || group < 1 || nq < 1 || depth < nq || head_dim < 1) return WSW_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !(scale < 3.0e38f)) return WSW_ERR_INVALID_ARG;  // finite and positive
    if (heads == 0) return WSW_OK;
    if (!q || !out) return WSW_ERR_INVALID_ARG;
    if (head_dim != kHD) return WSW_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return WSW_ERR_MISALIGNED;
    if (depth >= (int64_t(1) << 31) || heads * group > 65535 || (nq + kBQ - 1) / kBQ * heads * group > 0x7fffffffLL)
        return WSW_ERR_UNSUPPORTED;
    return WSW_OK;
}

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// Workspace of the windowed q8_0 pass: binary16 scratch for one window of K and of V,
// then (with more than one window) the carried state.
size_t q8_ws_bytes(int64_t depth, int64_t heads, int64_t group, int64_t nq, int64_t window, int64_t *nwin) {
    const int64_t w = window < depth ? window : depth;
    *nwin = (depth + window - 1) / window;
    size_t n = 2 * align256(static_cast<size_t>(heads) * w * kHD * 2);
    if (*nwin > 1) n += align256(static_cast<size_t>(heads) * group * nq * kStateStride * 4);
    return n;
}

}  // namespace
}  // namespace wsw

extern "C" int wsw_attn_prefill_f16(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t depth,
                                    int64_t heads, int64_t group, int64_t nq, int64_t head_dim,
                                    int64_t k_pos_stride, int64_t k_head_stride, int64_t v_pos_stride,
                                    int64_t v_head_stride, float scale, float *out, void *stream,
                                    const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    st = check_common(q, out, depth, heads, group, nq, head_dim, scale);
    if (st != WSW_OK || heads == 0) return st;
    if (!k || !v) return WSW_ERR_INVALID_ARG;
    if (k_pos_stride < 1 || k_head_stride < 0 || v_pos_stride < 1 || v_head_stride < 0) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k) & 15) || (reinterpret_cast<uintptr_t>(v) & 15) || (k_pos_stride % 8) ||
        (k_head_stride % 8) || (v_pos_stride % 8) || (v_head_stride % 8))
        return WSW_ERR_MISALIGNED;
    if ((k_head_stride == 0 || v_head_stride == 0) && heads > 1) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    return attn_launch(q, k, v, depth, heads, group, nq, k_pos_stride, k_head_stride, v_pos_stride, v_head_stride, 0,
                       depth, true, true, nullptr, scale, out, static_cast<cudaStream_t>(stream), o.pdl, di);
}

extern "C" size_t wsw_attn_prefill_q8_0_workspace_bytes(int64_t depth, int64_t heads, int64_t group, int64_t nq,
                                                        int64_t window) {
    using namespace wsw;
    if (depth < 1 || heads < 1 || group < 1 || nq < 1 || window < kBP || window % kBP != 0) return 0;
    int64_t nwin;
    return q8_ws_bytes(depth, heads, group, nq, window, &nwin);
}

extern "C" int wsw_attn_prefill_q8_0(const uint16_t *q, const int8_t *kq, const uint16_t *kd, const int8_t *vq,
                                     const uint16_t *vd, int64_t depth, int64_t heads, int64_t group, int64_t nq,
                                     int64_t head_dim, float scale, int64_t window, void *ws, size_t ws_bytes,
                                     float *out, void *stream, const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    st = check_common(q, out, depth, heads, group, nq, head_dim, scale);
    if (st != WSW_OK || heads == 0) return st;
    if (!kq || !kd || !vq || !vd) return WSW_ERR_INVALID_ARG;
    if (window < kBP || window % kBP != 0) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kd) & 1) || (reinterpret_cast<uintptr_t>(vd) & 1)) return WSW_ERR_MISALIGNED;
    int64_t nwin;
    const size_t need = q8_ws_bytes(depth, heads, group, nq, window, &nwin);
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)) return WSW_ERR_WORKSPACE;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t w = window < depth ? window : depth;
    uint16_t *sk = static_cast<uint16_t *>(ws);
    uint16_t *sv = reinterpret_cast<uint16_t *>(static_cast<char *>(ws) + align256(static_cast<size_t>(heads) * w * kHD * 2));
    float *state = nwin > 1 ? reinterpret_cast<float *>(static_cast<char *>(ws) +
                                                        2 * align256(static_cast<size_t>(heads) * w * kHD * 2))
                            : nullptr;
    wsw_launch_opts dq = {0, 0, o.pdl ? 1 : 0, 0, 0};
    for (int64_t i = 0; i < nwin; ++i) {
        const int64_t pos0 = i * window;
        const int64_t npos = depth - pos0 < window ? depth - pos0 : window;
        // this window of K and V, dequantized into the per-head scratch [heads][npos][128]
        st = wsw_dequant_q8_0_kv(kq + pos0 * heads * kHD, kd + pos0 * heads * (kHD / 32), npos, heads, kHD, sk, stream,
                                 &dq);
        if (st != WSW_OK) return st;
        st = wsw_dequant_q8_0_kv(vq + pos0 * heads * kHD, vd + pos0 * heads * (kHD / 32), npos, heads, kHD, sv, stream,
                                 &dq);
        if (st != WSW_OK) return st;
        st = attn_launch(q, sk, sv, depth, heads, group, nq, kHD, npos * kHD, kHD, npos * kHD, pos0, npos, i == 0,
                         i == nwin - 1, state, scale, out, s, o.pdl, di);
        if (st != WSW_OK) return st;
    }
    return WSW_OK;
}
