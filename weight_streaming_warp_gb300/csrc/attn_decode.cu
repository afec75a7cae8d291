// attn_decode.cu -- one decoding step of attention over a binary16 KV cache: the
// consumer of the dequantized KV scratch.
//
// Source: "vulkan : dequant q8_0 KV once in coopmat1" (llama.cpp PR).  Overview: the
// flash-attention pass reads the f16 K and V of every cached position; the stride
// discussion: in the cache one head's rows are head_dim * n_head_kv elements apart (a
// 256-on / 768-off walk for 4 heads of 128), in the scratch they are back to back.  The
// call takes both layouts through its (position, head) strides.
//
//   s_p          = scale * q[h][g] . K(h, p)
//   out[h][g][i] = sum_p exp(s_p - m) V(h, p)[i] / sum_p exp(s_p - m),  m = max_p s_p
//
// Design (GB300), flash decoding in one launch:
//  * attn_decode_warp_kernel: grid (splits, heads) of about one CTA per SM, 256 threads.
//    A CTA takes a chunk of positions of one KV head for all G query heads of its group,
//    so every K and V byte is read once per step.  Each of its eight warps walks its own
//    run of 16-position steps through a private three-stage cp.async ring and keeps its
//    own online softmax, so the loop has no block barrier; the warps' partials are
//    merged once at the end, and the CTA writes (m, l = sum of weights, acc[128]) of each
//    query to the workspace.  Scores are kept in the log2 domain (scale * log2 e folded
//    into q), so the weights are exp2f(s - m).
//  * The last CTA of a head to finish (an arrival counter per head in the workspace)
//    rescales every chunk's record to the common maximum, adds them in a fixed order and
//    divides, so the result does not depend on the launch; it then sets the counter back
//    to zero.  A second launch for this merge measured 4-5 us slower per call: its
//    dependency hop sat on the critical path.
//  * Groups of one and two query heads run on the CUDA cores: the dot products and the
//    value sums use packed fp32x2 FMAs (even and odd dimensions in the two lanes), and
//    the loop is bound by memory.  Groups of four and eight run the two products of a
//    step on the tensor cores (m16n8k16, fp32 accumulation): on the CUDA cores their
//    loop was bound by instruction issue, 1.7x slower.  The fp32 queries and weights
//    enter as a binary16 high part plus a binary16 residual, in the two halves of the
//    16-row operand, so their products keep about 22 bits.
// The split count is a function of (depth, heads) alone, never of the device or the
// launch options.
#include <cuda_fp16.h>

#include <cmath>

#include "common.cuh"

namespace wsw {
namespace {

constexpr int kDh = 128;                // head_dim
constexpr int kThreads = 256;           // 8 warps
constexpr int kRowBytes = kDh * 2;      // one K or V row in shared memory
constexpr int kPart = kDh + 4;          // floats per (chunk, head, query): m, l, 2 pad, acc
constexpr float kLog2e = 1.4426950408889634f;

struct AttnArgs {
    const float *q;
    const __half *k, *v;
    int64_t depth, kps, khs, vps, vhs;  // strides in elements
    float qscale;                       // scale * log2(e)
    int chunk;                          // positions per CTA (whole 16-position steps)
    int splits;
    int heads;
    unsigned *cnt;                      // [heads] arrival counters (zero between calls)
    float *part;                        // [heads][splits][G][kPart] partial records
    float *out;
};

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Two fp32 lanes in one 64-bit register, for the packed fp32 FMA of sm_100 and newer.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float f2_sum(uint64_t r) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
    return lo + hi;
}
__device__ __forceinline__ void f2_split(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ void fma2(uint64_t &acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t h2_to_f2(uint32_t h) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    return f2(f.x, f.y);
}

// Warp-streaming form: each of the eight warps walks its own run of whole 16-position
// steps of the CTA's chunk through a private three-stage cp.async ring (8 KB a stage:
// 16 K rows, then 16 V rows), and keeps its own running maximum, weight sum and value
// sums; the loop has no block barrier.  Lane (hf = lane / 16, c = lane % 16) copies
// piece c (dimensions 8 c .. 8 c + 7) of rows hf, hf + 2, ...; a row's 16-byte pieces
// sit XOR-swizzled (piece c of row r in slot c ^ (r mod 8)), so that eight rows' equal
// pieces fall in distinct banks.  The CUDA-core form below reads only the lane's own
// pieces, so no lane waits on another's copies; the tensor-core form reads the stage
// by ldmatrix after a warp barrier.
// CUDA-core form:
//   scores:  the lane's partial dots with its eight rows, summed over the half-warp by a
//            butterfly that halves the values in flight at each of its four shuffles
//            (8 shuffles for 8 rows); lanes 2 i and 2 i + 1 of half hf end with the
//            score of row 2 i + hf
//   softmax: the step's maximum over the warp, then each lane's weight exp2(s - m)
//   values:  each row's weight is shuffled from the lane that holds it
// At the end the warps' partials are merged once in shared memory (one barrier) and the
// CTA writes its (m, l, acc) record; the last CTA of the head merges the records.
constexpr int kWBatch = 16;                                // positions per warp step
constexpr int kWStages = 3;
constexpr int kWWarps = kThreads / 32;
constexpr int kWStageBytes = 2 * kWBatch * kRowBytes;       // K and V rows of one step
constexpr int kWSmem = kWWarps * kWStages * kWStageBytes;   // 192 KB: one CTA per SM
constexpr int kWTargetCtas = 152;                          // one CTA per SM of a 152-SM part
constexpr int kRed = kDh + 4;  // floats per warp partial in the merge: m, l, 2 pad, acc (16-byte aligned)

__device__ __forceinline__ uint32_t h2_bits(__half2 x) { return *reinterpret_cast<uint32_t *>(&x); }
// D += A B for one m16n8k16 tile: binary16 operands, fp32 accumulation
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p)))
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p)))
                 : "memory");
}

// 16-byte copy that writes zeros and reads nothing when !valid (src must still be mapped)
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

// The merge of one head's chunks, by the last CTA to finish.  Thread (slice, query,
// 16-byte column) takes the chunks s = slice, slice + 8 / G, ... in order, loading each
// chunk's maximum, weight sum and four values in one round and keeping a running
// maximum (what it has added so far is rescaled when the maximum grows); the 8 / G
// slices are then merged in a fixed order.  The result depends on neither the CTA that
// merges nor the launch.  sm: 1040 floats of shared memory (kSl G = 8).
template <int G>
__device__ __forceinline__ void merge_chunks(const AttnArgs &a, int h, float *sm) {
    constexpr int kSl = kWWarps / G;  // slices of the chunk list
    const int tid = threadIdx.x;
    const int S = a.splits;
    float *sums = sm;                          // [kSl][G][kDh]
    float *msl = sums + kSl * G * kDh;         // [kSl][G]
    float *lsl = msl + kSl * G;                // [kSl][G]
    const float *part = a.part + static_cast<int64_t>(h) * S * G * kPart;  // [S][G][kPart]
    const int sl = tid / (G * 32), gq = tid - sl * (G * 32);
    const int g = gq >> 5, c4 = gq & 31;  // query, 16-byte column (dimensions 4 c4 .. 4 c4 + 3)
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // deeper for the large groups, whose threads walk 8 / kSl times more records (the
    // small groups measured slower with it: their main loop is larger)
    constexpr int kUnroll = G >= 4 ? 16 : 8;
#pragma unroll kUnroll
    for (int sidx = sl; sidx < S; sidx += kSl) {
        const float *r = part + (static_cast<int64_t>(sidx) * G + g) * kPart;
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(r));
        const float4 x = __ldcg(reinterpret_cast<const float4 *>(r + 4) + c4);
        const float mn = fmaxf(m, ml.x);
        const float fo = m == -INFINITY ? 0.f : exp2f(m - mn);     // rescales what was added
        const float fn = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mn);
        m = mn;
        l = l * fo + ml.y * fn;
        acc.x = acc.x * fo + x.x * fn;
        acc.y = acc.y * fo + x.y * fn;
        acc.z = acc.z * fo + x.z * fn;
        acc.w = acc.w * fo + x.w * fn;
    }
    reinterpret_cast<float4 *>(sums + (sl * G + g) * kDh)[c4] = acc;
    if (c4 == 0) {
        msl[sl * G + g] = m;
        lsl[sl * G + g] = l;
    }
    __syncthreads();
    for (int i = tid; i < G * kDh; i += kThreads) {
        const int gg = i / kDh;
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < kSl; ++k) mx = fmaxf(mx, msl[k * G + gg]);
        float n = 0.f, dn = 0.f;
#pragma unroll
        for (int k = 0; k < kSl; ++k) {
            const float ms = msl[k * G + gg];
            const float f = ms == -INFINITY ? 0.f : exp2f(ms - mx);
            n = fmaf(sums[k * G * kDh + i], f, n);
            dn = fmaf(lsl[k * G + gg], f, dn);
        }
        a.out[static_cast<int64_t>(h) * G * kDh + i] = n / dn;
    }
}

template <int G, bool TC>
__global__ void __launch_bounds__(kThreads, 1) attn_decode_warp_kernel(const AttnArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hf = lane >> 4, c = lane & 15;
    const int h = blockIdx.y;
    const int64_t p0 = static_cast<int64_t>(blockIdx.x) * a.chunk;
    const int64_t pend = p0 + a.chunk < a.depth ? p0 + a.chunk : a.depth;
    const int nb = a.chunk / kWBatch;  // steps in a chunk; warp w takes [w nb / 8, (w + 1) nb / 8)
    const int64_t w0 = p0 + static_cast<int64_t>(warp * nb / kWWarps) * kWBatch;
    const int64_t wl = p0 + static_cast<int64_t>((warp + 1) * nb / kWWarps) * kWBatch;
    const int64_t w1 = wl < pend ? wl : pend;
    const int nsteps = w1 > w0 ? static_cast<int>((w1 - w0 + kWBatch - 1) / kWBatch) : 0;
    const __half *kh = a.k + h * a.khs, *vh = a.v + h * a.vhs;
    unsigned char *ring = smem + warp * (kWStages * kWStageBytes);

    // the first two steps' lines into L2 before the dependency wait (L2 is the point of
    // coherence, so this is safe while an earlier kernel may still write them)
    for (int j = lane; j < 2 * 4 * kWBatch; j += 32) {
        const int64_t p = w0 + (j >> 2);
        if (p < w1) prefetch_l2(((j & 2) ? vh + p * a.vps : kh + p * a.kps) + 64 * (j & 1));
    }
    pdl_wait();

    int ist = 0;  // ring stage of the next step to copy
    auto issue = [&](int t) {
        if (t < nsteps) {
            unsigned char *stg = ring + ist * kWStageBytes;
            const int64_t pb = w0 + static_cast<int64_t>(t) * kWBatch;
#pragma unroll
            for (int i = 0; i < kWBatch / 2; ++i) {
                const int r = 2 * i + hf;
                const bool ok = pb + r < w1;
                const int64_t p = ok ? pb + r : w0;
                const int sw = (c ^ (r & 7)) * 16;  // piece c of row r, XOR-swizzled
                cp_async16_zfill(stg + r * kRowBytes + sw, kh + p * a.kps + c * 8, ok);
                cp_async16_zfill(stg + (kWBatch + r) * kRowBytes + sw, vh + p * a.vps + c * 8, ok);
            }
            if (++ist == kWStages) ist = 0;
        }
        cp_async_commit();  // one group per step, empty past the end
    };
    issue(0);
    issue(1);

    float *red = reinterpret_cast<float *>(smem);  // the warps' partials [8][G][kRed], after the loop
    if constexpr (!TC) {
        // this lane's eight dimensions of every query, in the log2 domain
        uint64_t qv[G][4];
    #pragma unroll
        for (int g = 0; g < G; ++g) {
            const float *qp = a.q + (static_cast<int64_t>(h) * G + g) * kDh + c * 8;  // 4-byte aligned
    #pragma unroll
            for (int k = 0; k < 4; ++k) qv[g][k] = f2(qp[2 * k] * a.qscale, qp[2 * k + 1] * a.qscale);
        }
        pdl_launch_dependents();

        float m[G], l[G];
        uint64_t acc[G][4];
    #pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
            acc[g][0] = acc[g][1] = acc[g][2] = acc[g][3] = 0ull;
        }
        const bool b3 = c & 8, b2 = c & 4, b1 = c & 2;
        const int row = 2 * (c >> 1) + hf;  // the row whose score this lane ends with

        int rst = 0;  // ring stage of the step being used
        for (int t = 0; t < nsteps; ++t) {
            issue(t + 2);
            cp_async_wait<2>();
            const unsigned char *stg = ring + rst * kWStageBytes;
            if (++rst == kWStages) rst = 0;
            const bool valid = w0 + static_cast<int64_t>(t) * kWBatch + row < w1;

            uint64_t kf[kWBatch / 2][4];
    #pragma unroll
            for (int i = 0; i < kWBatch / 2; ++i) {
                const int r = 2 * i + hf;
                const uint4 kv = *reinterpret_cast<const uint4 *>(stg + r * kRowBytes + ((c ^ (r & 7)) << 4));
                kf[i][0] = h2_to_f2(kv.x);
                kf[i][1] = h2_to_f2(kv.y);
                kf[i][2] = h2_to_f2(kv.z);
                kf[i][3] = h2_to_f2(kv.w);
            }
            float w[G];
    #pragma unroll
            for (int g = 0; g < G; ++g) {
                float d[kWBatch / 2];
    #pragma unroll
                for (int i = 0; i < kWBatch / 2; ++i) {
                    uint64_t x = 0ull;
                    fma2(x, qv[g][0], kf[i][0]);
                    fma2(x, qv[g][1], kf[i][1]);
                    fma2(x, qv[g][2], kf[i][2]);
                    fma2(x, qv[g][3], kf[i][3]);
                    d[i] = f2_sum(x);
                }
                // butterfly over the half-warp: after the shuffle at distance 8 a lane keeps
                // rows 0..3 or 4..7 (by bit 3 of c), at 4 two of those, at 2 one, and the
                // shuffle at 1 completes the sum
                float e4[4], e2[2];
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float send = b3 ? d[k] : d[k + 4], keep = b3 ? d[k + 4] : d[k];
                    e4[k] = keep + __shfl_xor_sync(WSW_FULL_MASK, send, 8);
                }
    #pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float send = b2 ? e4[k] : e4[k + 2], keep = b2 ? e4[k + 2] : e4[k];
                    e2[k] = keep + __shfl_xor_sync(WSW_FULL_MASK, send, 4);
                }
                const float send = b1 ? e2[0] : e2[1], keep = b1 ? e2[1] : e2[0];
                const float e1 = keep + __shfl_xor_sync(WSW_FULL_MASK, send, 2);
                float s = e1 + __shfl_xor_sync(WSW_FULL_MASK, e1, 1);
                if (!valid) s = -INFINITY;
                // online softmax: the step's maximum over the warp (lane pairs hold equal scores)
                float mt = s;
    #pragma unroll
                for (int off = 2; off <= 16; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(WSW_FULL_MASK, mt, off));
                const float mn = fmaxf(m[g], mt);
                const bool none = mn == -INFINITY;
                const float al = none ? 1.f : exp2f(m[g] - mn);
                w[g] = none ? 0.f : exp2f(s - mn);
                m[g] = mn;
                l[g] = l[g] * al + w[g];
                const uint64_t al2 = f2(al, al);
    #pragma unroll
                for (int k = 0; k < 4; ++k) asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(acc[g][k]) : "l"(al2));
            }
            // values: row 2 i + hf, piece c; its weight sits in lane 16 hf + 2 i
    #pragma unroll
            for (int i = 0; i < kWBatch / 2; ++i) {
                const int r = 2 * i + hf;
                const uint4 vv = *reinterpret_cast<const uint4 *>(stg + (kWBatch + r) * kRowBytes + ((c ^ (r & 7)) << 4));
                const uint64_t v01 = h2_to_f2(vv.x), v23 = h2_to_f2(vv.y), v45 = h2_to_f2(vv.z), v67 = h2_to_f2(vv.w);
    #pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float wi = __shfl_sync(WSW_FULL_MASK, w[g], (lane & 16) | (2 * i));
                    const uint64_t w2 = f2(wi, wi);
                    fma2(acc[g][0], w2, v01);
                    fma2(acc[g][1], w2, v23);
                    fma2(acc[g][2], w2, v45);
                    fma2(acc[g][3], w2, v67);
                }
            }
        }
        cp_async_wait<0>();

        // the warp's partial: the two half-warps' value sums added, the weight sum over the
        // lanes of one parity of each pair (pairs hold equal weights)
        __syncthreads();  // every warp is past its ring: it becomes the merge area
    #pragma unroll
        for (int g = 0; g < G; ++g) {
            float lv = l[g];
    #pragma unroll
            for (int off = 2; off <= 16; off <<= 1) lv += __shfl_xor_sync(WSW_FULL_MASK, lv, off);
            float v8[8];
    #pragma unroll
            for (int k = 0; k < 4; ++k) {
                f2_split(acc[g][k], v8[2 * k], v8[2 * k + 1]);
                v8[2 * k] += __shfl_xor_sync(WSW_FULL_MASK, v8[2 * k], 16);
                v8[2 * k + 1] += __shfl_xor_sync(WSW_FULL_MASK, v8[2 * k + 1], 16);
            }
            float *r = red + (warp * G + g) * kRed;
            if (hf == 0) {
                reinterpret_cast<float4 *>(r + 4 + 8 * c)[0] = make_float4(v8[0], v8[1], v8[2], v8[3]);
                reinterpret_cast<float4 *>(r + 4 + 8 * c)[1] = make_float4(v8[4], v8[5], v8[6], v8[7]);
            }
            if (lane == 0) {
                r[0] = m[g];
                r[1] = lv;
            }
        }
    } else {
        // Tensor-core form (m16n8k16, fp32 accumulation).  A holds 16 rows: the binary16
        // high parts of the G queries in rows 0..7 and their residuals q - hi in rows
        // 8..15 (rows past G are zero), so row g plus row g + 8 of a product is the fp32
        // query's product to about 2^-22.  Scores: S = [q_hi; q_lo] K^T over 8 k-steps of
        // 16 dimensions, two 8-position column blocks; the weights P take the same
        // high / residual split as the A operand of O += [P_hi; P_lo] V.  K and V come
        // from the swizzled ring by ldmatrix (V transposed).  Thread (group gq = lane / 4,
        // tq = lane % 4) owns query gq and positions 8 n + 2 tq + {0, 1} of each block.
        const int gq = lane >> 2, tq = lane & 3;
        uint32_t qa[kDh / 16][4];
#pragma unroll
        for (int kt = 0; kt < kDh / 16; ++kt) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float x0 = 0.f, x1 = 0.f;
                if (gq < G) {
                    const float *qp = a.q + (static_cast<int64_t>(h) * G + gq) * kDh + 16 * kt + 8 * half + 2 * tq;
                    x0 = qp[0] * a.qscale;
                    x1 = qp[1] * a.qscale;
                }
                const __half2 hi = __floats2half2_rn(x0, x1);
                const __half2 lo = __floats2half2_rn(x0 - __low2float(hi), x1 - __high2float(hi));
                qa[kt][2 * half] = h2_bits(hi);
                qa[kt][2 * half + 1] = h2_bits(lo);
            }
        }
        pdl_launch_dependents();

        float m = -INFINITY, l = 0.f;
        float o[kDh / 8][4];
#pragma unroll
        for (int n = 0; n < kDh / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        // ldmatrix row addresses: lane L points at row L % 8 of matrix L / 8
        const int mi = lane >> 3, mr = lane & 7;
        const int kpos = 8 * (mi >> 1) + mr, kchunk = mi & 1;  // K: (block, k-half) per matrix
        const int vpos = 8 * (mi & 1) + mr, vnt = mi >> 1;     // V: (position half, dims) per matrix

        int rst = 0;
        for (int t = 0; t < nsteps; ++t) {
            __syncwarp();  // every lane is done reading the stage that step t + 2 reuses
            issue(t + 2);
            cp_async_wait<2>();
            __syncwarp();  // the step's pieces copied by every lane are visible
            const unsigned char *stg = ring + rst * kWStageBytes;
            if (++rst == kWStages) rst = 0;
            const int64_t pb = w0 + static_cast<int64_t>(t) * kWBatch;

            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kt = 0; kt < kDh / 16; ++kt) {
                uint32_t b[4];
                const int ch = 2 * kt + kchunk;
                ldsm_x4(b, stg + kpos * kRowBytes + ((ch ^ (kpos & 7)) << 4));
                mma16816(sc[0], qa[kt], b[0], b[1]);
                mma16816(sc[1], qa[kt], b[2], b[3]);
            }
            float sv[4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const bool ok = pb + 8 * n + 2 * tq + j < w1;
                    sv[2 * n + j] = ok ? sc[n][j] + sc[n][2 + j] : -INFINITY;
                }
            float mt = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
            mt = fmaxf(mt, __shfl_xor_sync(WSW_FULL_MASK, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(WSW_FULL_MASK, mt, 2));
            const float mn = fmaxf(m, mt);
            const bool none = mn == -INFINITY;
            const float al = none ? 1.f : exp2f(m - mn);
            float p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = none ? 0.f : exp2f(sv[i] - mn);
            m = mn;
            l = l * al + ((p[0] + p[1]) + (p[2] + p[3]));
            if (__any_sync(WSW_FULL_MASK, al != 1.f)) {
#pragma unroll
                for (int n = 0; n < kDh / 8; ++n) {
                    o[n][0] *= al;
                    o[n][1] *= al;
                    o[n][2] *= al;
                    o[n][3] *= al;
                }
            }
            uint32_t pa[4];
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const __half2 hi = __floats2half2_rn(p[2 * n], p[2 * n + 1]);
                const __half2 lo = __floats2half2_rn(p[2 * n] - __low2float(hi), p[2 * n + 1] - __high2float(hi));
                pa[2 * n] = h2_bits(hi);
                pa[2 * n + 1] = h2_bits(lo);
            }
#pragma unroll
            for (int j = 0; j < kDh / 16; ++j) {
                uint32_t b[4];
                const int ch = 2 * j + vnt;
                ldsm_x4_trans(b, stg + (kWBatch + vpos) * kRowBytes + ((ch ^ (vpos & 7)) << 4));
                mma16816(o[2 * j], pa, b[0], b[1]);
                mma16816(o[2 * j + 1], pa, b[2], b[3]);
            }
        }
        cp_async_wait<0>();
        __syncthreads();  // every warp is past its ring: it becomes the merge area
        l += __shfl_xor_sync(WSW_FULL_MASK, l, 1);
        l += __shfl_xor_sync(WSW_FULL_MASK, l, 2);
        if (gq < G) {
            float *r = red + (warp * G + gq) * kRed;
#pragma unroll
            for (int n = 0; n < kDh / 8; ++n)
                *reinterpret_cast<float2 *>(r + 4 + 8 * n + 2 * tq) = make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
            if (tq == 0) {
                r[0] = m;
                r[1] = l;
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < G * (kDh + 1); i += kThreads) {
        const int g = i / (kDh + 1), e = i - g * (kDh + 1);
        float mx = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < kWWarps; ++ww) mx = fmaxf(mx, red[(ww * G + g) * kRed]);
        float sum = 0.f;
#pragma unroll
        for (int ww = 0; ww < kWWarps; ++ww) {
            const float *r = red + (ww * G + g) * kRed;
            const float f = r[0] == -INFINITY ? 0.f : exp2f(r[0] - mx);
            sum = fmaf(e < kDh ? r[4 + e] : r[1], f, sum);
        }
        float *dst = a.part + ((static_cast<int64_t>(h) * a.splits + blockIdx.x) * G + g) * kPart;
        if (e < kDh) dst[4 + e] = sum;
        else {
            dst[0] = mx;
            dst[1] = sum;
        }
    }

    // The last CTA of the head to arrive merges every chunk's record.  The block barrier
    // orders the CTA's record writes before thread 0's arrival, whose release (cumulative)
    // publishes them at GPU scope; its acquire, and the barrier after it, order the
    // merge's reads after every other CTA's arrival.
    __shared__ int last;
    __syncthreads();
    if (tid == 0) {
        unsigned old;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.cnt + h) : "memory");
        last = old == static_cast<unsigned>(a.splits - 1);
    }
    __syncthreads();
    if (!last) return;
    merge_chunks<G>(a, h, reinterpret_cast<float *>(smem));
    if (tid == 0) a.cnt[h] = 0u;  // ready for the next call
}

// The workspace: one arrival counter per head (padded to 16 bytes), then the records.
size_t counter_bytes(int64_t heads) { return static_cast<size_t>((heads * 4 + 15) / 16 * 16); }

// Positions per CTA and CTAs per head: about kWTargetCtas CTAs over all heads, chunks a
// whole number of 16-position steps.
void attn_split(int64_t depth, int64_t heads, int *chunk, int *splits) {
    const int64_t want = kWTargetCtas / heads > 1 ? kWTargetCtas / heads : 1;
    int64_t c = (depth + want - 1) / want;
    c = (c + kWBatch - 1) / kWBatch * kWBatch;
    *chunk = static_cast<int>(c);
    *splits = static_cast<int>((depth + c - 1) / c);
}

// groups of four and eight query heads take the tensor-core form, smaller ones the
// CUDA-core form (there the loop is bound by memory, not by issue)
template <int G>
cudaError_t launch_warp(const AttnArgs &a, cudaStream_t s, bool pdl) {
    constexpr bool tc = G >= 4;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(attn_decode_warp_kernel<G, tc>), kWSmem);
    if (e != cudaSuccess) return e;
    return launch(attn_decode_warp_kernel<G, tc>, dim3(a.splits, a.heads), dim3(kThreads), kWSmem, s, pdl, a);
}

}  // namespace
}  // namespace wsw

extern "C" size_t wsw_attn_decode_workspace_bytes(int64_t depth, int64_t heads, int64_t group) {
    using namespace wsw;
    if (depth <= 0 || heads <= 0 || heads > 65535 || group <= 0 || group > 8 || depth > (int64_t(1) << 31))
        return 0;
    int chunk, splits;
    attn_split(depth, heads, &chunk, &splits);
    return counter_bytes(heads) + static_cast<size_t>(splits) * heads * group * kPart * sizeof(float);
}

extern "C" int wsw_attn_decode_f16(const float *q, const uint16_t *k, const uint16_t *v, int64_t depth,
                                   int64_t heads, int64_t group, int64_t head_dim, int64_t k_pos_stride,
                                   int64_t k_head_stride, int64_t v_pos_stride, int64_t v_head_stride,
                                   float scale, float *out, void *ws, size_t ws_bytes, void *stream,
                                   const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (!q || !k || !v || !out || !ws || depth <= 0 || heads <= 0 || head_dim <= 0) return WSW_ERR_INVALID_ARG;
    if (group != 1 && group != 2 && group != 4 && group != 8) return WSW_ERR_UNSUPPORTED;
    if (head_dim != kDh || heads > 65535 || depth > (int64_t(1) << 31) || heads * group > (int64_t(1) << 31))
        return WSW_ERR_UNSUPPORTED;
    if (k_pos_stride < 0 || k_head_stride < 0 || v_pos_stride < 0 || v_head_stride < 0 || !std::isfinite(scale))
        return WSW_ERR_INVALID_ARG;
    const uintptr_t al = reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
                         static_cast<uintptr_t>(k_pos_stride * 2) | static_cast<uintptr_t>(k_head_stride * 2) |
                         static_cast<uintptr_t>(v_pos_stride * 2) | static_cast<uintptr_t>(v_head_stride * 2) |
                         reinterpret_cast<uintptr_t>(ws);
    if ((al & 15) || (reinterpret_cast<uintptr_t>(q) & 3) || (reinterpret_cast<uintptr_t>(out) & 3))
        return WSW_ERR_MISALIGNED;
    if (ws_bytes < wsw_attn_decode_workspace_bytes(depth, heads, group)) return WSW_ERR_WORKSPACE;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    AttnArgs a;
    a.q = q;
    a.k = reinterpret_cast<const __half *>(k);
    a.v = reinterpret_cast<const __half *>(v);
    a.depth = depth;
    a.kps = k_pos_stride; a.khs = k_head_stride; a.vps = v_pos_stride; a.vhs = v_head_stride;
    a.qscale = scale * kLog2e;
    attn_split(depth, heads, &a.chunk, &a.splits);
    a.heads = static_cast<int>(heads);
    a.cnt = static_cast<unsigned *>(ws);
    a.part = reinterpret_cast<float *>(static_cast<unsigned char *>(ws) + counter_bytes(heads));
    a.out = out;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (group) {
        case 1: e = launch_warp<1>(a, s, o.pdl); break;
        case 2: e = launch_warp<2>(a, s, o.pdl); break;
        case 4: e = launch_warp<4>(a, s, o.pdl); break;
        default: e = launch_warp<8>(a, s, o.pdl); break;
    }
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
