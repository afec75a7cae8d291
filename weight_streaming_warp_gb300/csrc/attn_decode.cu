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
// Design (GB300), flash decoding in two launches:
//  * attn_decode_split_kernel: grid (splits, heads), 256 threads, two CTAs per SM.  A
//    CTA takes a chunk of positions of one KV head for all G query heads of its group,
//    so every K and V byte is read once per step.  Tiles of 64 positions of K and V
//    (2 x 16 KB) are copied with 16-byte cp.async into a three-stage ring (two tiles in
//    flight while one is used); the 16-byte chunks of odd rows are XOR-swizzled so that
//    the reads below hit distinct banks.
//      scores:  four lanes per position, each a quarter of the 128 dimensions, for all
//               G queries at once (each K value is read from shared memory once),
//               reduced with two xor shuffles; scores are kept in the log2 domain
//               (scale * log2 e folded into q), so the weights are exp2f(s - m)
//      softmax: warp g takes query g's 64 scores, the running maximum and the factor
//               exp2f(m_old - m_new) that rescales what was accumulated so far
//      values:  warp w takes every eighth position (w, w + 8, ...) for all G queries;
//               a lane owns four dimensions, so a warp reads whole 256-byte V rows
//    At the end of its chunk the CTA adds its warps' partial sums and writes
//    (m, l = sum of weights, acc[128]) of each query to the workspace.
//  * attn_decode_combine_kernel (PDL-linked): one CTA per (head, query); rescales every
//    chunk's partials to the global maximum, adds them in a fixed order and divides, so
//    the result does not depend on the launch.
//  * The dot products and the value sums use packed fp32x2 FMAs (even and odd
//    dimensions in the two lanes), which halves their instruction count.
// The split count is a function of (depth, heads) alone, never of the device or the
// launch options.
#include <cuda_fp16.h>

#include <cmath>

#include "common.cuh"

namespace wsw {
namespace {

constexpr int kDh = 128;                // head_dim
constexpr int kTile = 64;               // positions per tile
constexpr int kThreads = 256;           // 8 warps
constexpr int kRowBytes = kDh * 2;      // one K or V row in shared memory
constexpr int kTileBytes = kTile * kRowBytes;
constexpr int kStages = 3;              // tiles in the ring: two in flight while one is used
constexpr int kTargetCtas = 320;        // about two CTAs per SM on a 152-SM part
constexpr int kPart = kDh + 2;          // floats per (chunk, head, query): m, l, acc
constexpr float kLog2e = 1.4426950408889634f;

struct AttnArgs {
    const float *q;
    const __half *k, *v;
    int64_t depth, kps, khs, vps, vhs;  // strides in elements
    float qscale;                       // scale * log2(e)
    int chunk;                          // positions per CTA (multiple of kTile)
    int splits;
    int heads;
    float *ws;
    float *out;
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
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

// Byte offset of 16-byte chunk c (0..15) of row r in a tile: bit 2 of the chunk index
// flips on odd rows.  The score pass reads 16-byte chunks, a quarter-warp at a time: two
// rows, four chunks each, which land on eight distinct chunk positions of 128 bytes,
// i.e. distinct banks.  The value pass reads 8 bytes a lane, a half-warp at a time: one
// row's 128 bytes, whose chunks the swizzle only permutes.
__device__ __forceinline__ int chunk_off(int r, int c) { return r * kRowBytes + ((c ^ ((r & 1) << 2)) << 4); }

template <int G>
__global__ void __launch_bounds__(kThreads, 2) attn_decode_split_kernel(const AttnArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *kt = smem;                            // [kStages][kTile][kRowBytes]
    unsigned char *vt = smem + kStages * kTileBytes;     // [kStages][kTile][kRowBytes]
    float *qs = reinterpret_cast<float *>(smem + 2 * kStages * kTileBytes);  // [G][kDh], log2 domain
    float *sw = qs + G * kDh;                  // [G][kTile] scores; weights then [kTile][G]
    float *wt = sw + G * kTile;                // [kTile][G] weights
    float *mrun = wt + G * kTile;              // [G] running maximum
    float *alpha = mrun + G;                   // [G] rescale factor of the current tile

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.y;
    const int64_t p0 = static_cast<int64_t>(blockIdx.x) * a.chunk;
    const int64_t p1 = p0 + a.chunk < a.depth ? p0 + a.chunk : a.depth;
    const int ntiles = static_cast<int>((p1 - p0 + kTile - 1) / kTile);
    const __half *kh = a.k + h * a.khs, *vh = a.v + h * a.vhs;

    // the first tile's lines into L2 before the dependency wait (L2 is the point of
    // coherence, so this is safe while an earlier kernel may still write them)
    {
        const int r = tid >> 2, part = tid & 3;  // 64 rows x (2 lines of K, 2 of V)
        if (p0 + r < p1) {
            const __half *base = part < 2 ? kh + (p0 + r) * a.kps : vh + (p0 + r) * a.vps;
            prefetch_l2(base + 64 * (part & 1));
        }
    }
    pdl_wait();

    auto load_tile = [&](int t) {
        if (t < ntiles) {
            const int st = t % kStages;
            const int64_t pb = p0 + static_cast<int64_t>(t) * kTile;
            for (int i = tid; i < kTile * 16; i += kThreads) {
                const int r = i >> 4, c = i & 15;
                if (pb + r < p1) {
                    cp_async16(kt + st * kTileBytes + chunk_off(r, c), kh + (pb + r) * a.kps + c * 8);
                    cp_async16(vt + st * kTileBytes + chunk_off(r, c), vh + (pb + r) * a.vps + c * 8);
                }
            }
        }
        cp_async_commit();  // one group per tile, empty past the end
    };
    load_tile(0);
    load_tile(1);
    // q after the first tiles' copies are on their way (its load would hold them up)
    for (int i = tid; i < G * kDh; i += kThreads) qs[i] = a.q[static_cast<int64_t>(h) * G * kDh + i] * a.qscale;
    if (tid < G) mrun[tid] = -INFINITY;
    pdl_launch_dependents();

    // value pass: this thread's dimensions 4 lane .. 4 lane + 3 for every query, over the
    // positions warp, warp + 8, ... of each tile
    uint64_t acc[G][2];
    float l[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        acc[g][0] = acc[g][1] = 0ull;
        l[g] = 0.f;
    }

    for (int t = 0; t < ntiles; ++t) {
        const int st = t % kStages;
        load_tile(t + 2);  // into the stage that tile t - 1 used
        const int64_t left = p1 - (p0 + static_cast<int64_t>(t) * kTile);
        const int nv = left < kTile ? static_cast<int>(left) : kTile;
        cp_async_wait<2>();
        __syncthreads();
        // scores: position p = tid / 4, chunks 4 j + sub (dimensions 8 c .. 8 c + 7),
        // j = 0..3; even and odd dimensions in the two lanes of a packed accumulator
        {
            const int p = tid >> 2, sub = tid & 3;
            uint64_t d[G];
#pragma unroll
            for (int g = 0; g < G; ++g) d[g] = 0ull;
            const unsigned char *ktile = kt + st * kTileBytes;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 4 * j + sub;
                const uint4 kv = *reinterpret_cast<const uint4 *>(ktile + chunk_off(p, c));
                const uint64_t k01 = h2_to_f2(kv.x), k23 = h2_to_f2(kv.y), k45 = h2_to_f2(kv.z), k67 = h2_to_f2(kv.w);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const ulonglong2 qa = *reinterpret_cast<const ulonglong2 *>(qs + g * kDh + c * 8);
                    const ulonglong2 qb = *reinterpret_cast<const ulonglong2 *>(qs + g * kDh + c * 8 + 4);
                    fma2(d[g], qa.x, k01);
                    fma2(d[g], qa.y, k23);
                    fma2(d[g], qb.x, k45);
                    fma2(d[g], qb.y, k67);
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float e = f2_sum(d[g]);
                e += __shfl_xor_sync(WSW_FULL_MASK, e, 1);
                e += __shfl_xor_sync(WSW_FULL_MASK, e, 2);
                if (sub == 0) sw[g * kTile + p] = p < nv ? e : -INFINITY;
            }
        }
        __syncthreads();
        // softmax of the tile: warp g handles query g; weights go out position-major
        if (warp < G) {
            const float *s = sw + warp * kTile;
            const float s0 = s[lane], s1 = s[lane + 32];
            float mt = fmaxf(s0, s1);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(WSW_FULL_MASK, mt, off));
            const float mo = mrun[warp];
            const float mn = fmaxf(mo, mt);
            const bool none = mn == -INFINITY;  // nothing seen yet: no weight, nothing to rescale
            wt[lane * G + warp] = none ? 0.f : exp2f(s0 - mn);
            wt[(lane + 32) * G + warp] = none ? 0.f : exp2f(s1 - mn);
            if (lane == 0) {
                alpha[warp] = none ? 1.f : exp2f(mo - mn);
                mrun[warp] = mn;
            }
        }
        __syncthreads();
        // values: positions warp, warp + 8, ... of the tile, every query
        {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float al = alpha[g];
                const uint64_t al2 = f2(al, al);
                l[g] *= al;
                asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(acc[g][0]) : "l"(al2));
                asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(acc[g][1]) : "l"(al2));
            }
            const unsigned char *vtile = vt + st * kTileBytes;
            for (int p = warp; p < nv; p += 8) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(vtile + chunk_off(p, lane >> 1) + (lane & 1) * 8);
                const uint64_t v01 = h2_to_f2(raw.x), v23 = h2_to_f2(raw.y);
                float w[G];
#pragma unroll
                for (int g4 = 0; g4 < (G + 3) / 4; ++g4) {
                    if constexpr (G >= 4) {
                        const float4 w4 = *reinterpret_cast<const float4 *>(wt + p * G + 4 * g4);
                        w[4 * g4] = w4.x;
                        w[4 * g4 + 1] = w4.y;
                        w[4 * g4 + 2] = w4.z;
                        w[4 * g4 + 3] = w4.w;
                    } else {
#pragma unroll
                        for (int g = 0; g < G; ++g) w[g] = wt[p * G + g];
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const uint64_t w2 = f2(w[g], w[g]);
                    l[g] += w[g];
                    fma2(acc[g][0], w2, v01);
                    fma2(acc[g][1], w2, v23);
                }
            }
        }
        __syncthreads();  // stage st is free for tile t + 3
    }
    cp_async_wait<0>();

    // add the eight warps' partials (in warp order) into the workspace
    float *red = reinterpret_cast<float *>(smem);  // [8 warps][G][kDh + 1]; the tiles are done
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float *r = red + (warp * G + g) * (kDh + 1);
        f2_split(acc[g][0], r[4 * lane], r[4 * lane + 1]);
        f2_split(acc[g][1], r[4 * lane + 2], r[4 * lane + 3]);
        if (lane == 0) r[kDh] = l[g];
    }
    __syncthreads();
    for (int i = tid; i < G * (kDh + 1); i += kThreads) {
        const int g = i / (kDh + 1), e = i - g * (kDh + 1);
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sum += red[(w * G + g) * (kDh + 1) + e];
        float *dst = a.ws + ((static_cast<int64_t>(h) * a.splits + blockIdx.x) * G + g) * kPart;
        if (e < kDh) dst[2 + e] = sum;
        else {
            dst[0] = mrun[g];
            dst[1] = sum;
        }
    }
}

// One CTA per (head, query) of 512 threads: the global maximum and the factor
// exp2(m_s - m) of every chunk first, then four slices of 128 threads (one per
// dimension) add the chunks s = slice, slice + 4, ... in order, and the slices are added
// in a fixed order.  Many chunks' loads are in flight at once.
constexpr int kCombThreads = 4 * kDh;

__global__ void __launch_bounds__(kCombThreads) attn_decode_combine_kernel(const AttnArgs a, int G) {
    __shared__ float fac[kTargetCtas];  // splits <= kTargetCtas
    __shared__ float wmax[kCombThreads / 32];
    __shared__ float num_s[4][kDh], den_s[4];
    const int hg = blockIdx.x;  // h * G + g
    const int h = hg / G, g = hg - h * G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    const float *part = a.ws + (static_cast<int64_t>(h) * a.splits * G + g) * kPart;
    const int64_t step = static_cast<int64_t>(G) * kPart;  // from one chunk to the next
    float m = -INFINITY;
    for (int s = tid; s < a.splits; s += kCombThreads) m = fmaxf(m, part[s * step]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(WSW_FULL_MASK, m, off));
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    m = wmax[0];
#pragma unroll
    for (int w = 1; w < kCombThreads / 32; ++w) m = fmaxf(m, wmax[w]);
    for (int s = tid; s < a.splits; s += kCombThreads) fac[s] = exp2f(part[s * step] - m);
    __syncthreads();
    const int sl = tid / kDh, d = tid % kDh;
    float num = 0.f, den = 0.f;
#pragma unroll 8
    for (int s = sl; s < a.splits; s += 4) {
        const float *ps = part + s * step;
        num = fmaf(ps[2 + d], fac[s], num);
        den = fmaf(ps[1], fac[s], den);
    }
    num_s[sl][d] = num;
    if (d == 0) den_s[sl] = den;
    __syncthreads();
    pdl_launch_dependents();
    if (sl == 0) {
        const float n = (num_s[0][d] + num_s[1][d]) + (num_s[2][d] + num_s[3][d]);
        const float dn = (den_s[0] + den_s[1]) + (den_s[2] + den_s[3]);
        a.out[static_cast<int64_t>(hg) * kDh + d] = n / dn;
    }
}

// Positions per CTA and CTAs per head: about kTargetCtas CTAs over all heads, chunks a
// whole number of tiles.
void attn_split(int64_t depth, int64_t heads, int *chunk, int *splits) {
    const int64_t want = kTargetCtas / heads > 1 ? kTargetCtas / heads : 1;
    int64_t c = (depth + want - 1) / want;
    c = (c + kTile - 1) / kTile * kTile;
    *chunk = static_cast<int>(c);
    *splits = static_cast<int>((depth + c - 1) / c);
}

template <int G>
cudaError_t launch_split(const AttnArgs &a, cudaStream_t s, bool pdl) {
    const int smem = 2 * kStages * kTileBytes + (G * kDh + 2 * G * kTile + 2 * G) * 4;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(attn_decode_split_kernel<G>), smem);
    if (e != cudaSuccess) return e;
    return launch(attn_decode_split_kernel<G>, dim3(a.splits, a.heads), dim3(kThreads), smem, s, pdl, a);
}

}  // namespace
}  // namespace wsw

extern "C" size_t wsw_attn_decode_workspace_bytes(int64_t depth, int64_t heads, int64_t group) {
    using namespace wsw;
    if (depth <= 0 || heads <= 0 || heads > 65535 || group <= 0 || group > 8 || depth > (int64_t(1) << 31))
        return 0;
    int chunk, splits;
    attn_split(depth, heads, &chunk, &splits);
    return static_cast<size_t>(splits) * heads * group * kPart * sizeof(float);
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
    a.ws = static_cast<float *>(ws);
    a.out = out;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (group) {
        case 1: e = launch_split<1>(a, s, o.pdl); break;
        case 2: e = launch_split<2>(a, s, o.pdl); break;
        case 4: e = launch_split<4>(a, s, o.pdl); break;
        default: e = launch_split<8>(a, s, o.pdl); break;
    }
    if (e != cudaSuccess) return WSW_ERR_CUDA;
    e = launch(attn_decode_combine_kernel, dim3(static_cast<unsigned>(heads * group)), dim3(kCombThreads), 0, s,
               true, a, static_cast<int>(group));
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
