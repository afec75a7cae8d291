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
//                 boxes of 64 dims), then K and V tiles of 128 positions into rings of
//                 kKS and kVS stages.
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
constexpr int kKS = 2;          // K stages
constexpr int kVS = 3;          // V stages (a V tile is used one softmax later than its K tile)
constexpr int kSoftWarps = 8;   // two per tensor-memory lane quarter, one per half of a tile
constexpr int kThreadsA = 64 + 32 * kSoftWarps;  // warp 0: TMA, warp 1: MMA, warps 2-9: softmax
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

struct AttnArgs {
    int64_t depth, nq;
    int heads, group, qtiles;
    float scale_log2;  // scale * log2(e)
    float *out;
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
    const int64_t base = a.depth - a.nq;                  // position of query 0
    const int64_t lim_last = base + q0 + rows - 1;         // last position any row sees
    const int nkv = static_cast<int>(lim_last / kBP) + 1;  // KV tiles of this CTA
    const int first_masked = static_cast<int>((base + q0) / kBP);  // first tile row 0 may not fully see

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

    if (warp == 0) {
        if (lane == 0) {
            uint64_t pol_q, pol_kv;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_q));
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_kv));
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
            pdl_wait();  // Q, K and V may be written by earlier kernels in the stream
            mbar_expect_tx(&S.q_full, kTile);
            for (int b = 0; b < 2; ++b)
                tma_load_3d(S.q + b * kBox, &tmQ, 64 * b, static_cast<int>(q0), hg, &S.q_full, pol_q);
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < nkv && ok; ++j) {
                const int ks = j % kKS, vs = j % kVS;
                if (j >= kKS && !mbar_wait(&S.k_empty[ks], ((j / kKS) - 1) & 1u)) { ok = false; break; }
                mbar_expect_tx(&S.k_full[ks], kTile);
                for (int b = 0; b < 2; ++b)
                    tma_load_3d(S.k[ks] + b * kBox, &tmK, 64 * b, j * kBP, h, &S.k_full[ks], pol_kv);
                issued_k = j + 1;
                if (j >= kVS && !mbar_wait(&S.v_empty[vs], ((j / kVS) - 1) & 1u)) { ok = false; break; }
                mbar_expect_tx(&S.v_full[vs], kTile);
                for (int b = 0; b < 2; ++b)
                    tma_load_3d(S.v[vs] + b * kBox, &tmV, 64 * b, j * kBP, h, &S.v_full[vs], pol_kv);
                issued_v = j + 1;
            }
            if (!ok) {
                // the copies still in flight land before the CTA may exit (bounded waits)
                for (int j = issued_k - kKS; j < issued_k; ++j)
                    if (j >= 0) mbar_wait(&S.k_full[j % kKS], (j / kKS) & 1u);
                for (int j = issued_v - kVS; j < issued_v; ++j)
                    if (j >= 0) mbar_wait(&S.v_full[j % kVS], (j / kVS) & 1u);
                mbar_wait(&S.q_full, 0);
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
                    mma_ts(tmem + kColO, tmem + kColP + 64 * pb + 8 * kk, dv + 128 * kk, id_pv, (j | kk) != 0);
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
        const float cs = a.scale_log2;
        const uint64_t cs2 = f2_pack(cs, cs);
        float m = -INFINITY;
        uint64_t l2 = 0ull;  // two partial sums of the row's probabilities (fp32 pair)
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
                // positions past the row's causal limit read as -inf
                const int64_t lc = lim - (static_cast<int64_t>(j) * kBP + 64 * hf);
                const int last = lc < 0 ? -1 : (lc > 63 ? 63 : static_cast<int>(lc));
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c > last) sv[c >> 5][c & 31] = 0xff800000u;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) mx = fmaxf(mx, __uint_as_float(sv[c >> 5][c & 31]));
            S.red[sb][hf][r] = mx;
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.pair_max[sb][qd]);
            if (!__all_sync(WSW_FULL_MASK, mbar_wait(&S.pair_max[sb][qd], (j >> 1) & 1u))) { ok = false; break; }
            // scale > 0, so the maximum of the scaled scores is the scaled maximum
            const float mt = fmaxf(S.red[sb][0][r], S.red[sb][1][r]) * cs;
            // raise the maximum in use only when this tile exceeds it by more than kLazy
            // (both warps of the quarter decide alike: same inputs)
            const bool raise = mt > m + kLazy;
            if (j > 0 && __any_sync(WSW_FULL_MASK, raise)) {
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
                asm("add.rn.f32x2 %0, %0, %1;" : "+l"(l2) : "l"(f2_pack(p0, p1)));
            }
            tmem_st32(lane_base + kColP + 64 * sb + 32 * hf, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.p_full[sb]);
        }
        // epilogue: the row sum from both halves, then this half of O / l
        float l0, l1;
        f2_unpack(l2, l0, l1);
        S.lsum[hf][r] = l0 + l1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.pair_sum[qd]);
        const bool have = __all_sync(WSW_FULL_MASK, ok && mbar_wait(&S.pair_sum[qd], 0) && mbar_wait(&S.o_final, 0));
        tc_fence_after();
        const float inv = 1.0f / (S.lsum[0][r] + S.lsum[1][r]);
        float *dst = a.out + ((static_cast<int64_t>(hg) * a.nq) + q0 + r) * kHD + 64 * hf;
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
    if (heads < 0 || group < 1 || nq < 1 || depth < nq || head_dim < 1) return WSW_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !(scale < 3.0e38f)) return WSW_ERR_INVALID_ARG;  // finite and positive
    if (heads == 0) return WSW_OK;
    if (!q || !k || !v || !out) return WSW_ERR_INVALID_ARG;
    if (head_dim != kHD) return WSW_ERR_UNSUPPORTED;
    if (k_pos_stride < 1 || k_head_stride < 0 || v_pos_stride < 1 || v_head_stride < 0) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(k) & 15) ||
        (reinterpret_cast<uintptr_t>(v) & 15) || (reinterpret_cast<uintptr_t>(out) & 15) || (k_pos_stride % 8) ||
        (k_head_stride % 8) || (v_pos_stride % 8) || (v_head_stride % 8))
        return WSW_ERR_MISALIGNED;
    if (depth >= (int64_t(1) << 31) || heads * group > 65535 || (nq + kBQ - 1) / kBQ * heads * group > 0x7fffffffLL)
        return WSW_ERR_UNSUPPORTED;
    if (k_head_stride == 0 && heads > 1) return WSW_ERR_INVALID_ARG;
    if (v_head_stride == 0 && heads > 1) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;

    const size_t smem = sizeof(Smem) + 1024;
    if (smem > static_cast<size_t>(di.max_smem_optin)) return WSW_ERR_UNSUPPORTED;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(attn_prefill_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return WSW_ERR_CUDA;

    CUtensorMap tmQ, tmK, tmV;
    const int64_t hs_k = heads > 1 ? k_head_stride : k_pos_stride * depth;
    const int64_t hs_v = heads > 1 ? v_head_stride : v_pos_stride * depth;
    if (!make_map3(&tmQ, q, nq, heads * group, kHD * 2, nq * kHD * 2) ||
        !make_map3(&tmK, k, depth, heads, k_pos_stride * 2, hs_k * 2) ||
        !make_map3(&tmV, v, depth, heads, v_pos_stride * 2, hs_v * 2))
        return WSW_ERR_CUDA;

    AttnArgs a;
    a.depth = depth;
    a.nq = nq;
    a.heads = static_cast<int>(heads);
    a.group = static_cast<int>(group);
    a.qtiles = static_cast<int>((nq + kBQ - 1) / kBQ);
    a.scale_log2 = scale * 1.4426950408889634f;
    a.out = out;
    const unsigned grid = static_cast<unsigned>(a.qtiles * heads * group);
    e = launch(attn_prefill_kernel, dim3(grid), dim3(kThreadsA), smem, static_cast<cudaStream_t>(stream), o.pdl,
               tmQ, tmK, tmV, a);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
