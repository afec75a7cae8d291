/*
 * wsw.h -- C ABI of libwsw.so, the decode-time weight-streaming hot path for one
 * NVIDIA GB300 (sm_103a).
 *
 * The calls cover the memory-bound mat-vec y = W.x that streams every weight byte
 * once per decoded token, the block quantizer that turns the activation into int8
 * blocks with absmax scales in front of the quantized mat-vec, the grouped MoE
 * form of that mat-vec, the one-pass q8_0 KV-cache dequantizer and the
 * small-batch prefill GEMM.  Each call is one or more hand-written CUDA kernels.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "vulkan : dequant q8_0 KV once in coopmat1" (llama.cpp pull request)
 *   [P2] "ggml-cuda: pad matmul weight rows to avoid cache-set aliasing"
 *   [P3] "QuantizeQ8KK is thread-per-superblock: 95.5us/call against llama.cpp's
 *        1.6us, and 41% of the ROCm decode gap"
 *   [P4] "perf(vulkan): decode GEMV reads four elements per load, and the row lever
 *        is dead"
 *   [P5] "cuda: prefetch the next PTQ1_0 mat-vec's weights into L2 from the last CTAs"
 *
 * Conventions shared by every call
 *   - Every pointer is a CUDA device pointer owned by the caller.  The library
 *     allocates nothing and keeps no state between calls apart from per-device
 *     kernel attributes set on first use.
 *   - bf16 and binary16 (fp16) data travel as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous and stream-ordered; none synchronizes the host.
 *   - Arguments are validated on the host before anything is launched.  A rejected
 *     call returns a nonzero wsw_status and launches nothing.  A launch failure
 *     returns WSW_ERR_CUDA (the CUDA error is not cleared; query it with
 *     cudaGetLastError).  No kernel traps, asserts or spins without a bound.
 *   - Row strides (ld, ldq, ldx) are in elements.  The elements between the row
 *     length and the stride are padding and are never read ([P2] Overview: the
 *     pad is zero-filled by the uploader, the kernels take the stride as given).
 *   - A pointer or stride that is not aligned for 32-byte loads does not fail:
 *     the weight load width degrades 32 -> 16 -> 8 -> 4 -> 2 bytes until aligned,
 *     and the result is bit-identical to the 32-byte path ([P4] "What shipped": the
 *     load width degrades one step at a time when an offset is misaligned).
 *     The exception is wsw_gemm_bf16, whose TMA tile loads need 16-byte
 *     alignment (WSW_ERR_MISALIGNED otherwise).
 *   - Results do not depend on wsw_launch_opts: any rows_per_warp, load_bytes,
 *     pdl or ctas_per_sm gives bit-identical output ([P4] "What did NOT work":
 *     rows-per-workgroup variants verified bit-identical by full-output hash).
 */
#ifndef WSW_H
#define WSW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WSW_ABI_VERSION 7

typedef enum wsw_status {
    WSW_OK = 0,
    WSW_ERR_INVALID_ARG = 1, /* null pointer, bad size, stride or block size */
    WSW_ERR_MISALIGNED = 2,  /* alignment that the call cannot degrade around */
    WSW_ERR_UNSUPPORTED = 3, /* device is not sm_103 / shape beyond a stated limit */
    WSW_ERR_WORKSPACE = 4,   /* a required caller workspace is absent or too small */
    WSW_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
    WSW_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up (read on the
                                device: wsw_bounded_wait_check, bit 1 of the MoE
                                error flag) */
} wsw_status;

/* Steps of the next link that a chain link prefetches into L2 by default: 0 = off.
 * Programmatic dependent launch already issues each link's first loads while the one
 * before drains; on GB300 the 257-link 27B-shaped chain ran 0.4% (2 steps) to 3.8%
 * (16 steps) slower with the prefetch on. */
#define WSW_CHAIN_L2_PREFETCH_STEPS 0

/* Launch knobs.  Pass NULL for the defaults.  0 in a field means "choose". */
typedef struct wsw_launch_opts {
    int32_t rows_per_warp; /* output rows one warp reduces together: 1, 2 or 4
                              (the pages' rows per workgroup, [P4] "What did NOT
                              work"); 0 = the library's choice (2; 4 for bf16
                              mat-vecs of at least 16384 rows) */
    int32_t load_bytes;    /* cap on the weight load width: 32, 16, 8, 4 or 2;
                              0 = 32 (one 256-bit load per lane) */
    int32_t pdl;           /* 1 = launch with programmatic dependent launch: the
                              kernel issues its first weight loads before waiting
                              for the previous kernel in the stream ([P5]
                              "Additional information": PDL on sm_90 and newer) */
    int32_t ctas_per_sm;   /* resident CTAs per SM for persistent grids; 0 = auto */
    int32_t l2_prefetch_steps; /* wsw_gemv_bf16_chain only: once done with a link,
                              its warps request into L2 the first this-many 1 KB steps
                              of every warp's first unit of the next link ([P5]
                              Overview); 1..64, -1 = off, 0 = the library's choice
                              (WSW_CHAIN_L2_PREFETCH_STEPS) */
} wsw_launch_opts;

/* Human-readable name of a wsw_status value (static storage, never NULL). */
const char *wsw_status_string(int status);

/* ABI version of the loaded library (WSW_ABI_VERSION it was built with). */
int wsw_abi_version(void);

/*
 * wsw_quantize_q8 -- block quantizer for the activation ([P3] Cause: the amax
 * scan over one superblock; [P3] Scope: quantize, then the quantized mat-vec).
 *
 * For each block of `block` consecutive values of a row:
 *   amax = max |x|;  d = amax / 127 (fp32 division);
 *   q = round_half_away_from_zero(x / d) (fp32 division by the fp32 d), in
 *   [-127, 127];  an all-zero block gives d = +0 and q = 0.
 * One thread per 8 elements and a warp-shuffle reduction of amax; each element is
 * loaded once (the page's second defect, a second load per element, is avoided).
 *
 *   x       fp32 [rows][ldx]; the first n values of each row are quantized.
 *   rows    >= 0;  n >= 0, a multiple of `block`;  ldx >= n.
 *   block   32 (q8_0) or 256 (superblock).
 *   q       int8 [rows][n], packed.
 *   scales  block 32: binary16 [rows][n/32]; block 256: fp32 [rows][n/256].
 * rows == 0 or n == 0 launches nothing and returns WSW_OK.
 */
int wsw_quantize_q8(const float *x, int64_t rows, int64_t n, int64_t ldx, int32_t block,
                    int8_t *q, void *scales, void *stream, const wsw_launch_opts *opts);

/*
 * wsw_gemv_bf16 -- decode mat-vec with bf16 weights ([P4] opening paragraph: the
 * decode GEMV streams ~52 GB of bf16 weights once per token and is bound by DRAM
 * bandwidth; [P2] Overview: the row stride may exceed the row).
 *
 *   y[r] = alpha * sum_{k<K} W[r*ld + k] * x[k],  r < M,
 * with bf16 x fp32 products accumulated in fp32.
 *
 *   W      bf16 [M][ld], row-major;  ld >= K.
 *   x      fp32 [K] (not rounded to bf16).
 *   y      fp32 [M]; must not overlap x.
 * M == 0 launches nothing; K == 0 writes y = 0.
 */
int wsw_gemv_bf16(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const float *x,
                  float alpha, float *y, void *stream, const wsw_launch_opts *opts);

/*
 * One link of a decode chain: y = alpha * W . x, as wsw_gemv_bf16.  x may point
 * into an earlier link's y ([P5] Overview: consecutive mat-vecs of the decode
 * graph, each paying a ramp-up and ramp-down in which DRAM idles).
 */
typedef struct wsw_gemv_link {
    const uint16_t *W;
    int64_t M, K, ld;
    const float *x;
    float alpha;
    float *y;
} wsw_gemv_link;

/*
 * wsw_gemv_bf16_chain -- launch n_links bf16 mat-vecs back to back on one stream,
 * each one programmatically dependent on the one before ([P5] "Additional
 * information": programmatic dependent launch is the sm_90+ tool for the idle
 * window between chained mat-vecs).  Every link is validated before the first
 * launch; the results equal n_links separate wsw_gemv_bf16 calls, bit for bit.
 * opts->pdl = 0 turns the dependency off (plain stream order).
 */
int wsw_gemv_bf16_chain(int64_t n_links, const wsw_gemv_link *links, void *stream,
                        const wsw_launch_opts *opts);

/* The launch that wsw_gemv_bf16 (or one link of wsw_gemv_bf16_chain) makes. */
typedef struct wsw_gemv_plan {
    int32_t load_bytes;    /* bytes per weight load of a lane: 32, 16, 8, 4 or 2 */
    int32_t rows_per_warp; /* 1, 2 or 4 */
    int32_t pdl;           /* 1 = programmatic dependent launch */
    int32_t ctas;          /* CTAs in the grid; 0 = no kernel (M == 0, or K == 0,
                              where y is zero-filled by a memset) */
    int32_t threads;       /* threads per CTA */
    int32_t log2_segments; /* each row's K is cut into 2^log2_segments segments
                              whose sums are combined in a fixed order */
    int32_t x_in_smem;     /* 1 = x is staged in shared memory, 0 = read via L1 */
    int32_t l2_prefetch_steps; /* chain links: steps of the next link's first units
                              requested into L2 (0 = none; the last link has no next) */
} wsw_gemv_plan;

/*
 * wsw_gemv_bf16_plan -- the launch choices of wsw_gemv_bf16 (chain == 0) or of a link
 * of wsw_gemv_bf16_chain (chain == 1) for these arguments, without launching anything
 * or calling CUDA ([P4] "What shipped": the load width follows the alignment of the
 * weight base and row pitch and degrades one step at a time; [P4] "Gates": a
 * variant-selection test pins what the launcher picks).  The launchers take their
 * choices from the same host function.
 *
 *   W          only its address is used (alignment); it is never dereferenced.
 *   M, K, ld   as wsw_gemv_bf16, validated the same way.
 *   sm_count   multiprocessors of the target device (> 0; 152 on GB300).
 *   chain      0 or 1.
 *   opts       as the call (NULL = defaults).
 *   out        host struct, written on WSW_OK.
 */
int wsw_gemv_bf16_plan(const uint16_t *W, int64_t M, int64_t K, int64_t ld, int32_t sm_count,
                       int32_t chain, const wsw_launch_opts *opts, wsw_gemv_plan *out);

/*
 * wsw_gemv_q8_0 -- decode mat-vec with q8_0 weights and a q8_0 activation ([P3]
 * Scope: the quantized mat-vec behind the quantizer).
 *
 *   y[r] = sum_b fp32(Wd[r][b]) * fp32(xd[b]) * (sum_{i<32} Wq[r*ldq + 32b+i] * xq[32b+i])
 * with the block sums in exact int32 and the rest in fp32.
 *
 *   Wq   int8 [M][ldq];  K % 32 == 0, ldq % 32 == 0 and ldq >= K (a quantized
 *        row stride must divide exactly into blocks, [P2] Overview).
 *   Wd   binary16 [M][K/32], packed.
 *   xq   int8 [K];  xd binary16 [K/32]  (as written by wsw_quantize_q8, block 32).
 *   y    fp32 [M].
 */
int wsw_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t M, int64_t K, int64_t ldq,
                  const int8_t *xq, const uint16_t *xd, float *y, void *stream,
                  const wsw_launch_opts *opts);

/*
 * wsw_quantize_gemv_q8_0 -- the batch-1 decode step of [P3] Scope (quantize the
 * activation to q8_0, then the quantized mat-vec) in one launch: every CTA quantizes
 * the fp32 x itself while its first weight loads are in flight, so no separate
 * quantizer kernel sits between two chained mat-vecs.
 *
 *   y = wsw_gemv_q8_0(Wq, Wd, M, K, ldq, q(x), d(x))  with (q(x), d(x)) =
 *       wsw_quantize_q8(x, 1, K, K, 32), bit for bit.
 *
 *   Wq, Wd, M, K, ldq, y   as wsw_gemv_q8_0.
 *   x        fp32 [K], 4-byte aligned.
 *   xq_out   int8 [K] and xd_out binary16 [K/32]: both NULL, or both set to receive
 *            the quantized activation (the bytes wsw_quantize_q8 writes).
 */
int wsw_quantize_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t M, int64_t K, int64_t ldq,
                           const float *x, int8_t *xq_out, uint16_t *xd_out, float *y, void *stream,
                           const wsw_launch_opts *opts);

/*
 * wsw_moe_workspace_bytes -- bytes of device workspace that wsw_moe_gemv_q8_0 can use
 * for E experts, row length K and R routed rows (0: that call needs none).  With the
 * workspace, calls with more than 256 routed rows run on the tensor cores; without it
 * they run on the CUDA cores.
 */
size_t wsw_moe_workspace_bytes(int64_t E, int64_t K, int64_t R);

/*
 * wsw_moe_gemv_q8_0 -- grouped MoE mat-vec over per-expert q8_0 weights ([P3]
 * Cause and Scope: the MoE path quantizes m = T x top_k rows, then runs a grouped
 * GEMM over the experts).
 *
 * For each row m < R with e = ids[m] in [0, E):
 *   y[m][o] = gemv_q8_0(W_e, x_m)[o],  o < Mo,
 * bit-identical to wsw_gemv_q8_0 on expert e's matrix and row m for R <= 256.
 * Each expert that some row uses is streamed from DRAM once per call; experts no row
 * uses are not read.  (For R <= 16 each routed row streams its own expert's rows; a
 * repeated expert's second pass is served by L2 while the routed experts' weights fit
 * in it, as they do for 16 rows of 128 x 1536 x 2048 experts.)  For R > 256 with a workspace, a prepass sorts
 * and converts the activations into the workspace and the rows of an expert are
 * multiplied on the tensor cores with exact integer block sums; results then agree
 * with the CUDA-core form within fp32 rounding, not bit for bit.
 *
 *   Wq   int8 [E][Mo][K];  Wd binary16 [E][Mo][K/32];  K % 32 == 0.
 *   xq   int8 [R][K];  xd binary16 [R][K/32].
 *   ids  int32 [R] (device).  A row whose id is outside [0, E) is skipped, its y
 *        row is left untouched, and bit 0 of *err_flag (if err_flag != NULL) is
 *        set.  Bit 1 is set if a bounded wait of the tensor-core form gave up (a
 *        WSW_ERR_TIMEOUT condition); the y rows that CTA had not finished are then
 *        NaN.  The library only ORs bits in; it never clears *err_flag.
 *   y    fp32 [R][Mo].
 *   ws   device workspace of ws_bytes >= wsw_moe_workspace_bytes(E, K, R) bytes,
 *        256-byte aligned, owned by the caller and overwritten by the call; NULL (or
 *        too small) keeps every row count on the CUDA cores.  Two calls in flight at
 *        once need two workspaces.
 *   R <= 16384 and E <= 1024, else WSW_ERR_UNSUPPORTED.
 */
int wsw_moe_gemv_q8_0(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K,
                      const int8_t *xq, const uint16_t *xd, const int32_t *ids, int64_t R,
                      float *y, int32_t *err_flag, void *ws, size_t ws_bytes, void *stream,
                      const wsw_launch_opts *opts);

/*
 * wsw_moe_gemv_q8_0_noalloc -- wsw_moe_gemv_q8_0 for callers that cannot allocate device
 * memory, such as a plugin or custom-operator interface that receives only its input
 * and output buffers, a runtime that reserves all device memory in its own pool at
 * start-up, or a path that cannot accept cudaMalloc's device synchronisation.  The pages
 * have no counterpart: this is a convenience of this library.
 *
 * Arguments, results and errors are those of wsw_moe_gemv_q8_0, except that there is
 * no ws / ws_bytes.  The workspace is a fixed 8 MiB scratch array inside the library,
 * which every GPU that loads the library holds until the process exits.  Sizes whose
 * wsw_moe_workspace_bytes(E, K, R) exceeds 8 MiB return WSW_ERR_UNSUPPORTED and launch
 * nothing (for example E = 128 takes R up to 1540 routed rows at K = 2048, and up to
 * 4096 at K = 768, the tensor-core limit).  The call
 * performs no cudaMalloc, cudaFree or other allocation.
 *
 *   - The first call on a device looks up the scratch array's device address on that
 *     device (it must be the current device).  Make that first call before any stream
 *     capture.
 *   - Every call on a device shares the one scratch array and leaves its contents
 *     behind.  Nothing in it needs to start at zero, because each call writes what it
 *     reads.  Calls whose executions overlap on the GPU (for example on two streams)
 *     race on the scratch; calls on one stream do not.
 */
int wsw_moe_gemv_q8_0_noalloc(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K,
                              const int8_t *xq, const uint16_t *xd, const int32_t *ids, int64_t R,
                              float *y, int32_t *err_flag, void *stream, const wsw_launch_opts *opts);

/*
 * wsw_dequant_q8_0_kv -- dequantize one layer's q8_0 K (or V) cache once into a
 * per-head-contiguous binary16 buffer ([P1] Overview and the stride discussion:
 * the cache walks [dim][position][head] with a position stride of
 * head_dim * heads elements; the scratch puts one head's positions back to back).
 *
 *   out[h][p][i] = f16_rn(fp32(d[p][h][i/32]) * q[p][h][i])
 *
 *   q     int8 [depth][heads][head_dim];  head_dim % 32 == 0.
 *   d     binary16 [depth][heads][head_dim/32].
 *   out   binary16 [heads][depth][head_dim]; must not overlap the inputs.
 * Returns WSW_ERR_INVALID_ARG for negative sizes, head_dim % 32 != 0, depth > 2^32,
 * heads or head_dim > 65536, or more than 2^45 values; WSW_ERR_MISALIGNED for an odd d
 * or out address.  Any size of zero is a no-op.
 */
int wsw_dequant_q8_0_kv(const int8_t *q, const uint16_t *d, int64_t depth, int64_t heads,
                        int64_t head_dim, uint16_t *out, void *stream,
                        const wsw_launch_opts *opts);

/*
 * wsw_attn_decode_f16 -- one decoding step of attention over a binary16 KV cache, the
 * consumer of the dequantized scratch ([P1] Overview: the flash-attention pass reads
 * the f16 K and V; the stride discussion: the cache keeps one head's rows
 * head_dim * n_head_kv elements apart, the scratch back to back).
 *
 *   s_p          = scale * sum_i q[h][g][i] * K(h, p)[i]
 *   out[h][g][i] = sum_p exp(s_p - m) * V(h, p)[i] / sum_p exp(s_p - m),  m = max_p s_p
 * over every position p < depth, for `heads` KV heads with `group` query heads each.
 * K(h, p) is the row of head_dim binary16 values at k + h * k_head_stride +
 * p * k_pos_stride (elements); V likewise.  The per-head-contiguous scratch that
 * wsw_dequant_q8_0_kv writes has (pos, head) strides (head_dim, depth * head_dim), the
 * position-major cache (heads * head_dim, head_dim).  Groups of 1 and 2 compute in fp32;
 * groups of 4 and 8 on the tensor cores, with q and the softmax weights entering as a
 * binary16 high part plus a binary16 residual (about 22 bits) and fp32 accumulation.
 * Either way results agree with fp64 within 1e-4 (normwise per output row) and do not
 * depend on the launch options.
 *
 *   q      fp32 [heads][group][head_dim].
 *   k, v   binary16; 16-byte aligned, strides multiples of 8 elements.
 *   out    fp32 [heads][group][head_dim]; must not overlap the inputs.
 *   ws     device workspace of ws_bytes >= wsw_attn_decode_workspace_bytes(depth,
 *          heads, group) bytes (WSW_ERR_WORKSPACE otherwise), 16-byte aligned.  It
 *          starts with one arrival counter per head, which must be zero before the
 *          first call; every call that completes leaves them zero, so a workspace is
 *          zero-filled once and then reused.  The rest is overwritten.  Two calls in
 *          flight at once need two workspaces.
 *   depth >= 1;  group in {1, 2, 4, 8};  head_dim == 128;  heads <= 65535
 *   (WSW_ERR_UNSUPPORTED otherwise).
 * One launch: chunks of positions in parallel; the last chunk of a head to finish
 * merges that head's chunks.
 */
size_t wsw_attn_decode_workspace_bytes(int64_t depth, int64_t heads, int64_t group);
int wsw_attn_decode_f16(const float *q, const uint16_t *k, const uint16_t *v, int64_t depth,
                        int64_t heads, int64_t group, int64_t head_dim, int64_t k_pos_stride,
                        int64_t k_head_stride, int64_t v_pos_stride, int64_t v_head_stride,
                        float scale, float *out, void *ws, size_t ws_bytes, void *stream,
                        const wsw_launch_opts *opts);

/*
 * wsw_attn_prefill_f16 -- causal prefill attention over a binary16 KV cache on the tensor
 * cores: the flash-attention pass of prompt processing that reads the dequantized
 * scratch ([P1] Overview: pp512 at depth 32768 and 65536 over the binary16 K and V; the
 * stride discussion: the cache keeps one head's rows head_dim * n_head_kv elements
 * apart, the scratch back to back).
 *
 * A batch of nq queries at the end of a cache of `depth` positions: query i of query
 * head (h, g) sits at position depth - nq + i and attends to positions
 * 0 .. depth - nq + i:
 *   s_p          = scale * sum_d q[h][g][i][d] * K(h, p)[d]
 *   out[h][g][i] = sum_p exp(s_p - m) V(h, p) / sum_p exp(s_p - m),  m = max_p s_p
 * K(h, p) is the row of head_dim binary16 values at k + h * k_head_stride +
 * p * k_pos_stride (elements); V likewise (the per-head scratch of
 * wsw_dequant_q8_0_kv: strides (head_dim, depth * head_dim); the position-major cache:
 * (heads * head_dim, head_dim)).  Products of binary16 values (q, K, V and the
 * probabilities P, rounded to binary16) accumulate in fp32; P's rounding bounds an
 * output element's error by about 2^-11 * sum_p w_p |V(h, p)| / sum_p w_p.
 *
 *   q      binary16 [heads][group][nq][head_dim], 16-byte aligned.
 *   k, v   binary16, 16-byte aligned; strides multiples of 8 elements.
 *   out    fp32 [heads][group][nq][head_dim], 16-byte aligned; must not overlap inputs.
 *   scale  finite and > 0.
 *   1 <= nq <= depth < 2^31;  head_dim == 128;  heads * group <= 65535
 *   (WSW_ERR_UNSUPPORTED / WSW_ERR_INVALID_ARG otherwise).  heads == 0 does nothing.
 * One launch; a bounded wait that gives up leaves NaN in the rows of its query tile.
 */
int wsw_attn_prefill_f16(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t depth,
                         int64_t heads, int64_t group, int64_t nq, int64_t head_dim, int64_t k_pos_stride,
                         int64_t k_head_stride, int64_t v_pos_stride, int64_t v_head_stride, float scale,
                         float *out, void *stream, const wsw_launch_opts *opts);

/*
 * wsw_attn_prefill_q8_0 -- the same causal prefill attention over a q8_0 KV cache, with a
 * scratch of bounded size: the cache is dequantized and attended one window of
 * positions at a time ([P1] author's reply, "A few directions ... as follow-ups":
 * bounding the scratch with a chunked / streamed scratch that caps the peak, instead of
 * one binary16 layer of K and V for the whole depth; the dequantization is [P1]'s
 * dequant-once pass, wsw_dequant_q8_0_kv, applied to each window).
 *
 * For each window of `window` positions (the last one may be shorter): dequantize the
 * window's K and V rows into the per-head binary16 scratch, then attend over them,
 * carrying every query row's online-softmax state (running maximum, sum and unnormalized
 * output) from window to window.  Three launches per window, PDL-linked with opts->pdl.
 * The result equals wsw_dequant_q8_0_kv of K and V followed by wsw_attn_prefill_f16
 * within that call's stated error bound (not bit for bit: the maximum the
 * probabilities are taken against can differ between the two).
 *
 *   q        binary16 [heads][group][nq][head_dim], 16-byte aligned.
 *   kq, vq   int8 [depth][heads][head_dim];  kd, vd binary16 [depth][heads][head_dim/32]
 *            (the cache layout wsw_dequant_q8_0_kv reads).
 *   window   positions per window: a multiple of 128, at least 128.
 *   ws       device workspace of ws_bytes >= wsw_attn_prefill_q8_0_workspace_bytes(...)
 *            bytes, 256-byte aligned, overwritten (WSW_ERR_WORKSPACE otherwise): the K and
 *            V scratch of one window (2 * heads * min(window, depth) * head_dim * 2 bytes)
 *            and, with more than one window, the state (heads * group * nq * 528 bytes).
 *            Two calls in flight at once need two workspaces.
 *   out      as wsw_attn_prefill_f16.
 * Other limits as wsw_attn_prefill_f16.
 */
size_t wsw_attn_prefill_q8_0_workspace_bytes(int64_t depth, int64_t heads, int64_t group, int64_t nq,
                                             int64_t window);
int wsw_attn_prefill_q8_0(const uint16_t *q, const int8_t *kq, const uint16_t *kd, const int8_t *vq,
                          const uint16_t *vd, int64_t depth, int64_t heads, int64_t group, int64_t nq,
                          int64_t head_dim, float scale, int64_t window, void *ws, size_t ws_bytes, float *out,
                          void *stream, const wsw_launch_opts *opts);

/*
 * wsw_gemm_bf16 -- small-batch prefill product on the tensor cores ([P2] Results:
 * small-batch prefill streams the whole weight matrix for a short run of output
 * rows; the weight's row stride may carry one extra 128-byte line).
 *
 *   Y[n][r] = sum_{k<K} W[r*ld + k] * X[n*ldx + k],  r < M, n < N,
 * bf16 products accumulated in fp32.  Y row stride = M.
 *
 *   W   bf16 [M][ld];  X bf16 [N][ldx];  Y fp32 [N][M].
 *   W and X 16-byte aligned; K, ld and ldx multiples of 8 (WSW_ERR_MISALIGNED
 *   otherwise).
 */
int wsw_gemm_bf16(const uint16_t *W, int64_t M, int64_t K, int64_t ld, const uint16_t *X,
                  int64_t N, int64_t ldx, float *Y, void *stream, const wsw_launch_opts *opts);

/*
 * wsw_bounded_wait_check -- run the bounded mbarrier wait of the tensor-core kernels
 * on its own, one thread of one CTA.  The library has no device-side fault injection:
 * this call is how the give-up path of a wait is exercised on a GPU.
 *
 *   arrive = 1   the barrier's phase completes before the wait: *status = WSW_OK.
 *   arrive = 0   nothing completes the phase: the wait gives up after about one
 *                second and *status = WSW_ERR_TIMEOUT.  The kernel then returns
 *                normally and the context stays usable.
 *   status       int32 on the device, written by the kernel.
 */
int wsw_bounded_wait_check(int32_t arrive, int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* WSW_H */
