// gemm_bf16.cu -- small-batch prefill product Y[n][r] = sum_k W[r][k] * X[n][k] on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Source: "ggml-cuda: pad matmul weight rows to avoid cache-set aliasing" (AMD-Ecosystem
// llama.cpp PR), Overview and Results: in small-batch prefill a short run of output
// rows streams the whole weight matrix; the weight's row stride may carry one extra
// 128-byte line and the matmul takes its leading dimension from the row stride.
//
// Design (GB300):
//  * A CTA owns a tile of 128 weight rows x NT batch rows (NT a multiple of 16, at most
//    256; fewer batch rows are zero-filled by the tensor-memory-access engine).  K is
//    walked in stages of one or two 64-element boxes (128 bytes of bf16 = one 128-byte
//    swizzle row per box); the memory-bound small-NT tiles take two, so that 256
//    consecutive bytes of each weight row are requested together.
//  * Warp 0 streams W boxes and warp 2 X boxes with cp.async.bulk.tensor (TMA) into a
//    ring of shared-memory stages guarded by mbarriers.  Two issuing threads, because on
//    GB300 a thread that issues a TMA tile load is held for about 550 cycles whatever the
//    box size: one thread issuing both boxes of a stage took twice as long per stage as
//    the MMAs of a 128 x 256 tile.  Warp 1 allocates tensor memory and one of its threads
//    issues tcgen05.mma (M = 128, N = NT, K = 16, bf16 in, fp32 accumulate) and
//    tcgen05.commit to release stages; warps 2-5 are the epilogue, reading the
//    accumulator with tcgen05.ld (each warp owns its 32 tensor-memory lanes).
//  * Tiles are few (20 for a 2560-row weight at NT <= 256), so K is split over a
//    thread-block cluster of S CTAs (S chosen on the host from the cluster occupancy):
//    each CTA accumulates its share of K, writes the partial tile to its own shared
//    memory, and after a cluster barrier every rank adds a slice of the tile from all S
//    ranks through distributed shared memory, ranks first to last.  The reduction order
//    is fixed, so results are deterministic and do not depend on the row stride.
//  * Every mbarrier wait is bounded; a wait that runs out marks the tile with NaN and
//    the CTA still reaches its tensor-memory release.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <utility>

#include "tc_util.cuh"

namespace wsw {
namespace {

using namespace tc;

constexpr int kBM = 128;            // weight rows per tile (MMA M)
constexpr int kAtom = 64;           // K elements per 128-byte swizzle atom (one TMA box)
constexpr int kThreadsG = 192;      // warp 0: TMA, warp 1: TMEM + MMA, warps 2-5: epilogue
constexpr int kSmemBudget = 200 * 1024;
constexpr int kAtomA = kBM * kAtom * 2;  // 16 KB: one weight box
constexpr int kMaxSplit = 8;            // cluster size limit (portable)

struct GemmArgs {
    int64_t M, N, K;
    float *Y;
    int nt;       // batch rows per tile
    int n_tiles;  // ceil(N / nt)
    int atoms;    // 64-element boxes per stage (1 or 2)
    int kblocks;  // ceil(K / (64 * atoms))
    int stages;
};

__global__ void __launch_bounds__(kThreadsG, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        const GemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stages = a.stages;
    const int nt = a.nt;
    const int atoms = a.atoms;
    const uint32_t a_bytes = static_cast<uint32_t>(atoms) * kAtomA;
    const uint32_t b_bytes = static_cast<uint32_t>(atoms) * nt * kAtom * 2;
    unsigned char *sA = smem;
    unsigned char *sB = smem + static_cast<size_t>(stages) * a_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + static_cast<size_t>(stages) * b_bytes);
    uint64_t *empty = full + stages;
    uint64_t *accum = empty + stages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
    float *part = reinterpret_cast<float *>(smem);  // reuses the stages after the main loop

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t S = cluster_size();
    const uint32_t rank = cluster_rank();
    const int64_t tile = blockIdx.x / S;
    const int64_t m_tile = tile / a.n_tiles;
    const int n_tile = static_cast<int>(tile % a.n_tiles);
    const int64_t m0 = m_tile * kBM;
    const int n0 = n_tile * nt;
    const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * a.kblocks / S);
    const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * a.kblocks / S);
    const int nk = kb1 - kb0;
    const uint32_t tcols = nt <= 32 ? 32 : (nt <= 64 ? 64 : (nt <= 128 ? 128 : 256));

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                     "r"(tcols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // W: stage i's boxes (consecutive 128-byte pieces of each weight row, requested
            // back to back); this thread also arms full[i % stages] with the bytes of W and
            // X.  The weights do not come from earlier kernels, so the first ring of W
            // stages is in flight before anything waits for the previous kernel.
            uint64_t pol_w;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
            uint32_t s = 0, phase = 0;
            for (int i = 0; i < nk; ++i) {
                if (i >= stages && !mbar_wait(&empty[s], phase ^ 1u)) break;
                mbar_expect_tx(&full[s], a_bytes + b_bytes);
                const int k = (kb0 + i) * kAtom * atoms;
                for (int j = 0; j < atoms; ++j)
                    tma_load_2d(sA + s * a_bytes + j * kAtomA, &tmW, k + j * kAtom, static_cast<int>(m0), &full[s],
                                pol_w);
                if (++s == static_cast<uint32_t>(stages)) {
                    s = 0;
                    phase ^= 1u;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // One thread keeps the tensor core fed, so its loop is kept short: the stage
            // and its phase advance by counting, and the descriptors of stage s are the
            // stage-0 descriptors plus s stage sizes (start addresses are in 16-byte units
            // and stay inside the 14-bit field: shared memory is below 256 KB).
            const uint32_t idesc = instr_desc(kBM, nt);
            const uint64_t da0 = sw128_desc(saddr(sA)), db0 = sw128_desc(saddr(sB));
            const uint32_t a_stage = a_bytes >> 4, b_stage = b_bytes >> 4;
            const uint32_t a_box = kAtomA >> 4, b_box = (static_cast<uint32_t>(nt) * kAtom * 2) >> 4;
            uint32_t s = 0, phase = 0;
            for (int i = 0; i < nk; ++i) {
                if (!mbar_wait(&full[s], phase)) break;
                tc_fence_after();
                const uint64_t da = da0 + s * a_stage, db = db0 + s * b_stage;
                if (atoms == 1) {
#pragma unroll
                    for (int kk = 0; kk < kAtom / 16; ++kk)  // K = 16 per MMA: +32 bytes within the atom
                        mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, (i | kk) != 0);
                } else {
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int kk = 0; kk < kAtom / 16; ++kk)
                            mma_bf16(tmem, da + j * a_box + 2 * kk, db + j * b_box + 2 * kk, idesc, (i | j | kk) != 0);
                }
                mma_commit(&empty[s]);
                if (++s == static_cast<uint32_t>(stages)) {
                    s = 0;
                    phase ^= 1u;
                }
            }
            mma_commit(accum);
        }
        __syncwarp();
    } else {
        if (warp == 2 && lane == 0) {
            // X: written by earlier kernels, so after the dependency wait
            uint64_t pol_x;
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
            pdl_wait();
            uint32_t s = 0, phase = 0;
            for (int i = 0; i < nk; ++i) {
                if (i >= stages && !mbar_wait(&empty[s], phase ^ 1u)) break;
                const int k = (kb0 + i) * kAtom * atoms;
                for (int j = 0; j < atoms; ++j)
                    tma_load_2d(sB + s * b_bytes + j * (nt * kAtom * 2), &tmX, k + j * kAtom, n0, &full[s], pol_x);
                if (++s == static_cast<uint32_t>(stages)) {
                    s = 0;
                    phase ^= 1u;
                }
            }
        }
        __syncwarp();
        // epilogue: warp w owns tensor-memory lanes 32*(w % 4) .. +31 = tile rows
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const int64_t m = m0 + row;
        const bool have = mbar_wait(accum, 0);
        tc_fence_after();
        for (int c = 0; c < nt; c += 16) {
            float v[16];
            if (have) {
                tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(c), v);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = __int_as_float(0x7fc00000);
            }
            if (S == 1) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int64_t n = n0 + c + j;
                    if (n < a.N && m < a.M) a.Y[n * a.M + m] = v[j];
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) part[(c + j) * kBM + row] = v[j];
            }
        }
    }

    pdl_launch_dependents();
    if (S > 1) {
        // Split-K: every rank adds a slice of the tile from all ranks, in rank order.
        cluster_sync();
        const int quads = nt * kBM / 4;  // 4 consecutive tile rows of one batch row
        const int q0 = static_cast<int>(static_cast<int64_t>(rank) * quads / S);
        const int q1 = static_cast<int>(static_cast<int64_t>(rank + 1) * quads / S);
        const bool vec_store = (a.M % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.Y) & 15) == 0);
        for (int qd = q0 + threadIdx.x; qd < q1; qd += kThreadsG) {
            float4 v[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < static_cast<int>(S)) v[r] = ld_dsmem4(part + 4 * qd, static_cast<uint32_t>(r));
            float4 sum = v[0];
#pragma unroll
            for (int r = 1; r < 8; ++r) {
                if (r < static_cast<int>(S)) {
                    sum.x += v[r].x;
                    sum.y += v[r].y;
                    sum.z += v[r].z;
                    sum.w += v[r].w;
                }
            }
            const int64_t n = n0 + (4 * qd) / kBM;
            const int64_t m = m0 + (4 * qd) % kBM;
            if (n < a.N) {
                float *dst = a.Y + n * a.M + m;
                if (vec_store && m + 3 < a.M) {
                    *reinterpret_cast<float4 *>(dst) = sum;
                } else {
                    const float t[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (m + i < a.M) dst[i] = t[i];
                }
            }
        }
        cluster_sync();  // peers keep their shared memory until every rank has read it
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols) : "memory");
    }
}

// --------------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2-D bf16 tensor map: `rows` rows of `cols` elements, row pitch `ld` elements, box
// of 64 x box_rows with 128-byte swizzle; out-of-range elements read as zero.
bool make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kAtom), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t smem_bytes(int stages, int nt, int atoms) {
    return 1024 + static_cast<size_t>(stages) * atoms * (kAtomA + static_cast<size_t>(nt) * kAtom * 2) +
           static_cast<size_t>(2 * stages + 1) * 8 + 16;
}

// Clusters of `s` CTAs that fit on the device at once (cached per size and smem).
int max_clusters(int s, size_t smem) {
    static std::map<std::pair<int, size_t>, int> cache;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(s * 64 + dev, smem);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s) * 32);
    cfg.blockDim = dim3(kThreadsG);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(s);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(gemm_bf16_tc_kernel), &cfg) != cudaSuccess)
        n = 0;
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = n;
    return n;
}

}  // namespace
}  // namespace wsw

extern "C" int wsw_gemm_bf16(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const uint16_t *X,
                             int64_t N, int64_t ldx, float *Y, void *stream, const wsw_launch_opts *opts) {
    using namespace wsw;
    Opts o;
    int st = resolve_opts(opts, &o);
    if (st != WSW_OK) return st;
    if (M < 0 || N < 0 || K < 0 || ld < K || ldx < K) return WSW_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return WSW_OK;
    if (!W || !X || !Y) return WSW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15) || (reinterpret_cast<uintptr_t>(X) & 15) ||
        (reinterpret_cast<uintptr_t>(Y) & 3) || (K % 8) || (ld % 8) || (ldx % 8))
        return WSW_ERR_MISALIGNED;
    if (M > (int64_t(1) << 31) || N > (int64_t(1) << 31) || K > (int64_t(1) << 31)) return WSW_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di, &st)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return cudaMemsetAsync(Y, 0, static_cast<size_t>(M) * N * 4, s) == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;

    GemmArgs a;
    a.M = M; a.N = N; a.K = K; a.Y = Y;
    a.n_tiles = static_cast<int>((N + 255) / 256);
    a.nt = static_cast<int>(((N + a.n_tiles - 1) / a.n_tiles + 15) / 16 * 16);
    // Memory-bound tiles (few batch rows) read 256 bytes of each weight row per stage;
    // compute-bound ones keep 128-byte stages and more of them.
    a.atoms = a.nt <= 128 ? 2 : 1;
    a.kblocks = static_cast<int>((K + kAtom * a.atoms - 1) / (kAtom * a.atoms));
    const int stage_bytes = a.atoms * (kAtomA + a.nt * kAtom * 2);
    a.stages = (kSmemBudget - 2048) / stage_bytes;
    if (a.stages > 8) a.stages = 8;
    if (a.stages < 2) return WSW_ERR_UNSUPPORTED;
    // the partial tile of a split must fit in the stage buffers
    if (static_cast<size_t>(a.nt) * kBM * 4 > static_cast<size_t>(a.stages) * stage_bytes) return WSW_ERR_UNSUPPORTED;
    const size_t smem = smem_bytes(a.stages, a.nt, a.atoms);
    const int64_t tiles = ((M + kBM - 1) / kBM) * a.n_tiles;
    if (tiles * 8 > 0x7fffffffLL) return WSW_ERR_UNSUPPORTED;

    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(gemm_bf16_tc_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return WSW_ERR_CUDA;

    // Split-K cluster size: the fewest waves x K-blocks per CTA (ties: smaller S).
    int best_s = 1;
    int64_t best_cost = -1;
    for (int sp = 1; sp <= kMaxSplit && sp <= a.kblocks; ++sp) {
        const int cap = max_clusters(sp, smem);
        if (cap <= 0) continue;
        const int64_t waves = (tiles + cap - 1) / cap;
        const int64_t cost = waves * ((a.kblocks + sp - 1) / sp) + (sp > 1 ? 2 : 0);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_s = sp; }
    }

    CUtensorMap tmW, tmX;
    if (!make_map(&tmW, W, M, K, ld, kBM) || !make_map(&tmX, X, N, K, ldx, a.nt)) return WSW_ERR_CUDA;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * best_s));
    cfg.blockDim = dim3(kThreadsG);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(best_s);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int nattr = 1;
    if (o.pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        nattr = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    e = cudaLaunchKernelEx(&cfg, gemm_bf16_tc_kernel, tmW, tmX, a);
    return e == cudaSuccess ? WSW_OK : WSW_ERR_CUDA;
}
