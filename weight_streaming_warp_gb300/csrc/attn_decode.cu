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
//    (2 x 16 KB) are copied with 16-byte cp.async into a two-stage ring, rows padded to
//    320 bytes so that the per-position reads below hit distinct banks.
//      scores:  four lanes per position, each a quarter of the 128 dimensions, for all
//               G queries at once (each K value is read from shared memory once),
//               reduced with two xor shuffles; scores are kept in the log2 domain
//               (scale * log2 e folded into q), so the weights are exp2f(s - m)
//      softmax: warp g takes query g's 64 scores, the running maximum and the factor
//               exp2f(m_old - m_new) that rescales what was accumulated so far
//      values:  warp w takes query w / (8 / G) and every (8 / G)-th position; a lane
//               owns four dimensions, so a warp reads whole 256-byte V rows
//    At the end of its chunk the CTA adds its warps' partial sums and writes
//    (m, l = sum of weights, acc[128]) of each query to the workspace.
//  * attn_decode_combine_kernel (PDL-linked): one CTA per (head, query), one thread per
//    dimension; rescales every chunk's partials to the global maximum and divides, in
//    chunk order, so the result does not depend on the launch.
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
constexpr int kPitch = 320;             // bytes per row in shared memory (256 + 64)
constexpr int kTileBytes = kTile * kPitch;
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

template <int G>
__global__ void __launch_bounds__(kThreads, 2) attn_decode_split_kernel(const AttnArgs a) {
    constexpr int WQ = 8 / G;  // warps per query in the value pass
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *kt = smem;                  // [2][kTile][kPitch]
    unsigned char *vt = smem + 2 * kTileBytes;  // [2][kTile][kPitch]
    float *qs = reinterpret_cast<float *>(smem + 4 * kTileBytes);  // [G][kDh], log2 domain
    float *sw = qs + G * kDh;                  // [G][kTile]: scores, then weights
    float *mrun = sw + G * kTile;              // [G] running maximum
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
    for (int i = tid; i < G * kDh; i += kThreads) qs[i] = a.q[static_cast<int64_t>(h) * G * kDh + i] * a.qscale;
    if (tid < G) mrun[tid] = -INFINITY;

    auto load_tile = [&](int t) {
        if (t < ntiles) {
            const int st = t & 1;
            const int64_t pb = p0 + static_cast<int64_t>(t) * kTile;
            for (int i = tid; i < kTile * 16; i += kThreads) {
                const int r = i >> 4, c = i & 15;
                if (pb + r < p1) {
                    cp_async16(kt + st * kTileBytes + r * kPitch + c * 16, kh + (pb + r) * a.kps + c * 8);
                    cp_async16(vt + st * kTileBytes + r * kPitch + c * 16, vh + (pb + r) * a.vps + c * 8);
                }
            }
        }
        cp_async_commit();  // one group per tile, empty past the end
    };
    load_tile(0);
    load_tile(1);
    pdl_launch_dependents();

    const int qg = warp / WQ, qsub = warp % WQ;  // value pass: query and position phase
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, l = 0.f;

    for (int t = 0; t < ntiles; ++t) {
        const int st = t & 1;
        const int64_t left = p1 - (p0 + static_cast<int64_t>(t) * kTile);
        const int nv = left < kTile ? static_cast<int>(left) : kTile;
        cp_async_wait<1>();
        __syncthreads();
        // scores: position p = tid / 4, dimensions (4 j + sub) * 8 .. + 7, j = 0..3
        {
            const int p = tid >> 2, sub = tid & 3;
            float d[G];
#pragma unroll
            for (int g = 0; g < G; ++g) d[g] = 0.f;
            const unsigned char *krow = kt + st * kTileBytes + p * kPitch;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 4 * j + sub;
                const uint4 kv = *reinterpret_cast<const uint4 *>(krow + c * 16);
                const __half2 *k2 = reinterpret_cast<const __half2 *>(&kv);
                float kf[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(k2[e]);
                    kf[2 * e] = f.x;
                    kf[2 * e + 1] = f.y;
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float4 qa = *reinterpret_cast<const float4 *>(qs + g * kDh + c * 8);
                    const float4 qb = *reinterpret_cast<const float4 *>(qs + g * kDh + c * 8 + 4);
                    d[g] = fmaf(qa.x, kf[0], d[g]);
                    d[g] = fmaf(qa.y, kf[1], d[g]);
                    d[g] = fmaf(qa.z, kf[2], d[g]);
                    d[g] = fmaf(qa.w, kf[3], d[g]);
                    d[g] = fmaf(qb.x, kf[4], d[g]);
                    d[g] = fmaf(qb.y, kf[5], d[g]);
                    d[g] = fmaf(qb.z, kf[6], d[g]);
                    d[g] = fmaf(qb.w, kf[7], d[g]);
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                d[g] += __shfl_xor_sync(WSW_FULL_MASK, d[g], 1);
                d[g] += __shfl_xor_sync(WSW_FULL_MASK, d[g], 2);
                if (sub == 0) sw[g * kTile + p] = p < nv ? d[g] : -INFINITY;
            }
        }
        __syncthreads();
        // softmax of the tile: warp g handles query g
        if (warp < G) {
            float *s = sw + warp * kTile;
            const float s0 = s[lane], s1 = s[lane + 32];
            float mt = fmaxf(s0, s1);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(WSW_FULL_MASK, mt, off));
            const float mo = mrun[warp];
            const float mn = fmaxf(mo, mt);
            const bool none = mn == -INFINITY;  // nothing seen yet: no weight, nothing to rescale
            s[lane] = none ? 0.f : exp2f(s0 - mn);
            s[lane + 32] = none ? 0.f : exp2f(s1 - mn);
            __syncwarp();
            if (lane == 0) {
                alpha[warp] = none ? 1.f : exp2f(mo - mn);
                mrun[warp] = mn;
            }
        }
        __syncthreads();
        // values: warp (qg, qsub) adds positions qsub, qsub + WQ, ... for query qg
        {
            const float al = alpha[qg];
            l *= al;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] *= al;
            const float *w = sw + qg * kTile;
            const unsigned char *vb = vt + st * kTileBytes + lane * 8;
            for (int p = qsub; p < nv; p += WQ) {
                const float wv = w[p];
                const uint2 raw = *reinterpret_cast<const uint2 *>(vb + p * kPitch);
                const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
                const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
                l += wv;
                acc[0] = fmaf(wv, v01.x, acc[0]);
                acc[1] = fmaf(wv, v01.y, acc[1]);
                acc[2] = fmaf(wv, v23.x, acc[2]);
                acc[3] = fmaf(wv, v23.y, acc[3]);
            }
        }
        __syncthreads();  // stage st is free again
        load_tile(t + 2);
    }
    cp_async_wait<0>();

    // add the partials of the WQ warps of each query (in warp order) into the workspace
    float *red = reinterpret_cast<float *>(smem);  // [8 warps][kDh + 1]; the tiles are done
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 4; ++e) red[warp * (kDh + 1) + 4 * lane + e] = acc[e];
    if (lane == 0) red[warp * (kDh + 1) + kDh] = l;
    __syncthreads();
    for (int i = tid; i < G * (kDh + 1); i += kThreads) {
        const int g = i / (kDh + 1), e = i - g * (kDh + 1);
        float s = 0.f;
        for (int w = 0; w < WQ; ++w) s += red[(g * WQ + w) * (kDh + 1) + e];
        float *dst = a.ws + ((static_cast<int64_t>(h) * a.splits + blockIdx.x) * G + g) * kPart;
        if (e < kDh) dst[2 + e] = s;
        else {
            dst[0] = mrun[g];
            dst[1] = s;
        }
    }
}

__global__ void __launch_bounds__(kDh) attn_decode_combine_kernel(const AttnArgs a, int G) {
    const int hg = blockIdx.x;  // h * G + g
    const int h = hg / G, g = hg - h * G, d = threadIdx.x;
    pdl_wait();
    const float *part = a.ws + (static_cast<int64_t>(h) * a.splits * G + g) * kPart;
    const int64_t step = static_cast<int64_t>(G) * kPart;  // from one chunk to the next
    float m = -INFINITY;
    for (int s = 0; s < a.splits; ++s) m = fmaxf(m, part[s * step]);
    float den = 0.f, num = 0.f;
    for (int s = 0; s < a.splits; ++s) {
        const float *ps = part + s * step;
        const float f = exp2f(ps[0] - m);
        den = fmaf(ps[1], f, den);
        num = fmaf(ps[2 + d], f, num);
    }
    pdl_launch_dependents();
    a.out[static_cast<int64_t>(hg) * kDh + d] = num / den;
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
    const int smem = 4 * kTileBytes + (G * kDh + G * kTile + 2 * G) * 4;
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
    e = launch(attn_decode_combine_kernel, dim3(static_cast<unsigned>(heads * group)), dim3(kDh), 0, s, true, a,
               static_cast<int>(group));
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
