/*
 * fp8g.h -- C ABI of the GB300 (sm_103a) FP8 GEMM library.
 *
 * Compute entry points:
 *
 *   fp8_gemm_nt              D[M,N] = A[M,K] . B[N,K]^T
 *   fp8_gemm_grouped_masked  D[g,m,n] = A[g,m,:] . B[g,n,:]  for m < masked_m[g]
 *   ..._scaled               the same times per-tensor / per-channel scales
 *   ..._blockscaled          UE8M0 scales per row per 32/128-element K group
 *   ..._ex                   any of those plus a fused epilogue (alpha, beta*C,
 *                            bias, ReLU, rounding mode)
 *   fp8_gemm_grouped_contiguous  groups' token rows concatenated along M
 *   fp8_gemm_nt_noalloc      dense small-token form that allocates nothing
 *
 * A and B hold FP8 codes (E4M3 or E5M2, chosen per operand), products are
 * accumulated in FP32 by the tensor cores, and D is BF16 (round to nearest
 * even).  Sources:
 *   "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
 *     (sheratonhq.com/news/187119) -- §1.3 (FP8 inputs, E4M3/E5M2
 *     selectable, FP32 accumulator), §3.1 (the two formats), §6.2-6.4
 *     (K tails and edge shapes must be handled exactly).
 *   "一次“转置”，半张算力：DeepSeek SwapAB 漂流史" (hwcomputing.csdn.net)
 *     -- §3.1 (m_grouped_fp8_gemm_nt_masked: masked grouped FP8 GEMM for
 *     MoE decode, ENABLE_SWAPAB switch), §3.2 (SwapAB: weights on the
 *     instruction's M side, tokens on N), §3.3 (runtime N in the
 *     instruction descriptor shrinks the tail to the valid tokens), §3.5
 *     (swap pays for small token counts only; selection is per shape).
 *   "MLS 三个访存 Bug 深度剖析" (chatdocs.ruinique.com) -- Bug 1 (64-bit
 *     address arithmetic), Bug 2 (a fully masked tail issues no load),
 *     Bug 3 (invalid padding must not reach valid outputs).
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library keeps no reference once the enqueued work has completed.
 *  - Calls enqueue work on `stream` and return without synchronising.
 *  - The return value is an fp8g_status code.  Invalid arguments are
 *    rejected before anything is enqueued.  Errors found on the device
 *    (a bounded wait that ran out, masked_m out of range) are recorded in a
 *    per-device status word read by fp8g_get_device_status().
 *  - Offsets are computed in 64 bits throughout.
 *  - Calls on different streams may run at the same time on the GPU.  The
 *    scratch memory a launch needs beyond its operands (the stream-K
 *    partial tiles and arrival counters of the SwapAB kernel and of split
 *    SM-pair tiles; "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
 *    §6.4 on accumulation across CTAs) is kept per (device, stream), so
 *    launches on unordered streams never share it; launches on one stream
 *    are ordered by the stream.  A CUDA graph captured from a stream uses
 *    that stream's scratch: replay it ordered with the stream's other
 *    library work (on that stream, or after an event on it).  The
 *    per-thread default stream counts as one stream per host thread.
 *    Before destroying a stream whose library work may still be running,
 *    call fp8g_release_stream() on it (or synchronise it): the runtime may
 *    hand the same handle to a new stream.
 *  - fp8_gemm_nt_noalloc is the exception: all of its calls on a device
 *    share one fixed array (see there).
 *  - Host cost: the TMA tensor maps of a call are cached by (base address,
 *    extents, box), so repeated calls on the same buffers encode none; the
 *    masked_m / group_offsets pointer of the grouped calls is checked to be
 *    device memory once per address.  A buffer freed and reallocated at the
 *    same address with the same extents gets the same, still correct map.
 *  - Not thread-safe for concurrent calls from several host threads on the
 *    same device while fp8g_set_wait_timeout_ns() is being changed.
 */
#ifndef FP8G_H
#define FP8G_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (same declaration as driver_types.h). */
struct CUstream_st;
typedef struct CUstream_st *cudaStream_t;

/* FP8 element formats of A and B. */
typedef enum {
    FP8G_E4M3 = 0, /* 1 sign, 4 exponent (bias 7), 3 mantissa; max 448     */
    FP8G_E5M2 = 1  /* 1 sign, 5 exponent (bias 15), 2 mantissa; max 57344  */
} fp8g_dtype;

/* Status codes. */
typedef enum {
    FP8G_OK = 0,
    FP8G_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad dtype, ...  */
    FP8G_ERR_MISALIGNED = 2,    /* a pointer is not 16-byte aligned                  */
    FP8G_ERR_UNSUPPORTED = 3,   /* shape outside the supported range, not sm_103     */
    FP8G_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed              */
    FP8G_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out; kernel returned   */
    FP8G_ERR_NO_DEVICE = 6,     /* no CUDA device is visible                         */
    FP8G_ERR_MASKED_M_RANGE = 7 /* device: a masked_m entry was outside [0, M_max]
                                   and was clamped                                   */
} fp8g_status;

/* `flags` bits 0-1: operand placement (the pages' ENABLE_SWAPAB switch). */
#define FP8G_SWAP_AUTO 0u  /* library picks by token count (the default)          */
#define FP8G_SWAP_ON 1u    /* weights (B) on the MMA M side, tokens (A) on N       */
#define FP8G_SWAP_OFF 2u   /* tokens (A) on the MMA M side, weights (B) on N       */
#define FP8G_SWAP_MASK 3u
/* Tuning overrides (0 = the library's choice).  Results stay correct for
 * every value; only speed (and the last bits of rounding) change.
 *   FP8G_WHOLE_TILES  SwapAB kernel: each CTA takes whole output tiles in
 *                     turn instead of an equal stream-K range of K blocks;
 *                     SM-pair kernel: never split the last wave's tiles
 *   FP8G_STREAM_K     SM-pair dense kernel: split the tiles of the last,
 *                     partial wave stream-K over all pairs (default: whole
 *                     tiles round-robin)
 *   FP8G_TILE_N(n)    non-swapped kernel: N tile of n (32..256, multiple of 32) */
#define FP8G_WHOLE_TILES 0x100u
#define FP8G_STREAM_K 0x800u
/*   FP8G_SPLIT_TAIL   SM-pair dense kernel: split each tile of the last partial
 *                     wave 2 to 4 ways along K whenever that is possible (by
 *                     default the split competes with whole tiles in a cost
 *                     model and needs a whole wave to overlap its sums).
 *                     FP8G_WHOLE_TILES also turns the default split off.    */
#define FP8G_SPLIT_TAIL 0x80u
/*   FP8G_SINGLE_SM_TILES  non-swapped dense kernel: 128-row tiles on one SM
 *                     each instead of 256-row tiles on a pair of SMs         */
#define FP8G_SINGLE_SM_TILES 0x200u
/*   FP8G_NO_PDL       launch without programmatic dependent launch (by
 *                     default a launch may begin its set-up while the
 *                     previous launch in the stream finishes; it waits for
 *                     that launch before any load or store of its operands.
 *                     A dense launch may issue L2 prefetches of its first B
 *                     tiles before that wait -- of all of them from the CTAs
 *                     that start on SMs the launch leaves idle, when the
 *                     weights fit in half of L2: L2 is coherent, so the loads
 *                     after the wait still see what the previous launch
 *                     wrote)                                                */
#define FP8G_NO_PDL 0x400u
/*   FP8G_PAIR_TILES   dense problems with more than 128 token rows: always use
 *                     SM-pair tiles (the automatic choice skips them for
 *                     block-scaled problems, where single-SM tiles measured
 *                     faster). */
#define FP8G_PAIR_TILES 0x4000u
/*   FP8G_ONE_MMA_ISSUER  block-scaled SwapAB, single-SM and SM-pair kernels: one
 *                     thread issues every MMA (default: two threads alternate
 *                     K blocks, each into its own accumulator, when each has
 *                     two accumulator buffers in TMEM -- token chunks or
 *                     tiles up to 112 wide -- and, single-SM tiles with
 *                     32-element groups, also with one buffer each) */
#define FP8G_ONE_MMA_ISSUER 0x8000u
/*   FP8G_TWO_MMA_ISSUERS  block-scaled single-SM and SM-pair tiles: two
 *                     issuers even when each has only one accumulator buffer */
#define FP8G_TWO_MMA_ISSUERS 0x2000u
/*   FP8G_STAGES(n)    at most n shared-memory pipeline stages (1..15)       */
#define FP8G_STAGES(n) ((((uint32_t)(n)) & 15u) << 20)
/*   FP8G_SHARE_SM     SwapAB kernel with <= 128 tokens per chunk: half the
 *                     shared memory and TMEM per CTA, so the next launch's
 *                     CTAs can become resident while this one drains (the
 *                     default for dense problems of up to 16 tokens)
 *   FP8G_NO_SHARE_SM  never share an SM that way                            */
#define FP8G_SHARE_SM 0x1000u
#define FP8G_NO_SHARE_SM 0x40u
#define FP8G_TILE_N(n) (((((uint32_t)(n)) / 32u) & 15u) << 16)
/*   FP8G_TOKEN_BOX(n) SwapAB kernel: n token rows per TMA copy of a chunk (a
 *                     multiple of 16 up to 240 that divides the chunk; other
 *                     values are ignored)                                   */
#define FP8G_TOKEN_BOX(n) (((((uint32_t)(n)) / 16u) & 15u) << 24)
/* Debug bits (bench and tests only; never needed for correct results). */
#define FP8G_DEBUG_ONE_STAGE 0x10u       /* one shared-memory stage: load,
                                            compute, load ... (isolates races
                                            from address bugs)                  */
#define FP8G_DEBUG_DROP_FIRST_LOAD 0x20u /* block 0's producer skips its first
                                            load, so its consumer's bounded wait
                                            runs out: exercises the timeout
                                            path; the call's output is invalid  */

/*
 * fp8_gemm_nt -- dense D = A . B^T.
 *   A  [M, K] FP8 codes, row-major, K contiguous (row stride K bytes).
 *   B  [N, K] FP8 codes, row-major, K contiguous (row stride K bytes).
 *   D  [M, N] BF16, row-major (row stride 2N bytes); every element written.
 *   M, N, K  >= 1;  K % 16 == 0 (16-byte row stride for the tensor copy
 *            engine);  N % 8 == 0 (16-byte rows of D);  each < 2^31.
 *   a_dtype, b_dtype  fp8g_dtype of A and B (mixed pairs allowed).
 *   flags  FP8G_SWAP_* (plus debug bits).
 *   stream  CUDA stream to enqueue on (0 = legacy default stream).  A
 *           SwapAB or split-tile launch uses this stream's own stream-K
 *           scratch (allocated on the stream's first such call, or by
 *           fp8g_init), so calls on other streams may overlap with it.
 * Returns FP8G_OK or an error code; on error nothing is enqueued.
 */
int fp8_gemm_nt(const void *A, const void *B, void *D, int64_t M, int64_t N,
                int64_t K, int a_dtype, int b_dtype, uint32_t flags,
                cudaStream_t stream);

/*
 * fp8_gemm_grouped_masked -- MoE-decode masked grouped GEMM.
 *   A         [G, M_max, K] FP8 token rows; only rows m < masked_m[g] of
 *             group g are valid (padding rows may hold any bytes, NaN codes
 *             included, and never affect valid outputs).
 *   B         [G, N, K] FP8 expert weights, K contiguous.
 *   D         [G, M_max, N] BF16.  Rows m < masked_m[g] are written; rows
 *             m >= masked_m[g] are NOT touched.
 *   masked_m  DEVICE pointer to G int32 valid-row counts, read on the device
 *             (no host synchronisation).  Entries outside [0, M_max] are
 *             clamped and flagged FP8G_ERR_MASKED_M_RANGE in the device status.
 *   G         1 .. 1024 groups.  M_max >= 1.
 *   max_m_hint  host-side upper bound the caller expects for masked_m (0 =
 *             unknown, taken as M_max).  It only sizes the token tile; groups
 *             above it are still computed correctly.
 *   N % 8 == 0, K % 16 == 0, sizes < 2^31, dtypes and flags as above.
 *   stream    as fp8_gemm_nt: the SwapAB kernel's stream-K scratch belongs
 *             to this stream, so grouped calls and dense calls on other
 *             streams may run at the same time.
 * Returns FP8G_OK or an error code; on error nothing is enqueued.
 */
int fp8_gemm_grouped_masked(const void *A, const void *B, void *D,
                            const int32_t *masked_m, int64_t G, int64_t M_max,
                            int64_t N, int64_t K, int64_t max_m_hint,
                            int a_dtype, int b_dtype, uint32_t flags,
                            cudaStream_t stream);

/*
 * fp8_gemm_nt_scaled / fp8_gemm_grouped_masked_scaled -- the same products
 * multiplied back by FP32 scales before the BF16 rounding:
 *   D[m,n]   = bf16( sa(m) * sb(n) * sum_k A[m,k] B[n,k] )            (dense)
 *   D[g,m,n] = bf16( sa(g,m) * sb(g,n) * sum_k A[g,m,k] B[g,n,k] )    (grouped)
 * Source: "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
 * §3.1 (the scale is computed beforehand and multiplied back at the
 * output) and §5.2 (per-tensor or per-channel scales).
 *   scale_a  DEVICE float array: scale_a_len == G (one per tensor / group)
 *            or G*rows (rows = M dense, M_max grouped: one per token row).
 *   scale_b  DEVICE float array: scale_b_len == G or G*N (one per output
 *            channel).  Dense problems have G = 1.
 *   Both 16-byte aligned.  Computed in FP32 as (acc * sa) * sb, or with the
 *   per-tensor factor folded first.  Other arguments, layouts and errors as
 *   the unscaled calls.
 */
int fp8_gemm_nt_scaled(const void *A, const void *B, void *D, int64_t M, int64_t N,
                       int64_t K, int a_dtype, int b_dtype, const float *scale_a,
                       int64_t scale_a_len, const float *scale_b, int64_t scale_b_len,
                       uint32_t flags, cudaStream_t stream);
int fp8_gemm_grouped_masked_scaled(const void *A, const void *B, void *D,
                                   const int32_t *masked_m, int64_t G, int64_t M_max,
                                   int64_t N, int64_t K, int64_t max_m_hint, int a_dtype,
                                   int b_dtype, const float *scale_a, int64_t scale_a_len,
                                   const float *scale_b, int64_t scale_b_len,
                                   uint32_t flags, cudaStream_t stream);

/*
 * fp8_gemm_nt_blockscaled / fp8_gemm_grouped_masked_blockscaled -- block-
 * scaled products: every K group of `sf_group_k` (32 or 128) elements of
 * each row of A and of B carries its own UE8M0 scale (2^(e-127); e = 255 is
 * NaN), applied to the products before they are summed:
 *   D[g,m,n] = bf16( sum_k A[g,m,k] B[g,n,k]
 *                    * 2^(sf_a[g][k/gs][m] - 127) * 2^(sf_b[g][k/gs][n] - 127) )
 * Source: "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
 * §5.2 (scales per group of 128 elements); "一次“转置”，半张算力：DeepSeek
 * SwapAB 漂流史" §5 (UE8M0 scales on SM100) and §3.4 (the Blackwell MMA
 * takes A- and B-side scale factors).  The tensor core applies
 * the scales (tcgen05.mma kind::mxf8f6f4.block_scale).
 *   sf_a   DEVICE bytes [G][ceil(K/gs)][sf_a_ld]: the scale of row m of A
 *          (token row) for K group j at sf_a[(g*ks + j)*sf_a_ld + m];
 *          sf_a_ld >= M (dense) or M_max (grouped), a multiple of 16.
 *   sf_b   DEVICE bytes [G][ceil(K/gs)][sf_b_ld], row n of B likewise;
 *          sf_b_ld >= N, a multiple of 16.  128x128 weight blocks are
 *          expressed by repeating a block's scale over its 128 rows.
 *   Both 16-byte aligned; padding bytes past M / N are never read.
 * Dense problems run on SM-pair tiles (128-element groups, K > 4096, or with
 * FP8G_PAIR_TILES) or single-SM tiles, N tile <= 224, or SwapAB with token
 * chunks <= 224.  Other arguments, layouts and errors as the unscaled calls.
 */
int fp8_gemm_nt_blockscaled(const void *A, const void *B, void *D, int64_t M, int64_t N,
                            int64_t K, int a_dtype, int b_dtype, const uint8_t *sf_a,
                            int64_t sf_a_ld, const uint8_t *sf_b, int64_t sf_b_ld,
                            int sf_group_k, uint32_t flags, cudaStream_t stream);
int fp8_gemm_grouped_masked_blockscaled(const void *A, const void *B, void *D,
                                        const int32_t *masked_m, int64_t G, int64_t M_max,
                                        int64_t N, int64_t K, int64_t max_m_hint, int a_dtype,
                                        int b_dtype, const uint8_t *sf_a, int64_t sf_a_ld,
                                        const uint8_t *sf_b, int64_t sf_b_ld, int sf_group_k,
                                        uint32_t flags, cudaStream_t stream);

/*
 * fp8_gemm_nt_ex / fp8_gemm_grouped_masked_ex -- the general forms: any
 * combination of output scales, block scales and a fused epilogue.
 *
 *   value  = sum_k A B (* block scales)  * sa * sb  (output scales)
 *   D      = round( act( alpha * value + beta * C + bias[g][n] ) )
 *
 * The fused epilogue follows "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法
 * 内核优化实践" §3.3: alpha * AB + beta * C + per-channel bias and ReLU inside
 * the GEMM (no extra pass over HBM), with a choice of rounding for the final
 * conversion (nearest even, toward zero, toward +inf; toward -inf added for
 * symmetry).  Evaluated in FP32 as fma(alpha, value, fma(beta, C, bias)).
 *
 * `scales` (NULL: none) -- out_a/out_b as in the ..._scaled calls (both or
 * neither), block_a/block_b as in the ..._blockscaled calls (both or
 * neither, with block_k 32 or 128).
 * `epilogue` (NULL: D = round-to-nearest-even(value)) --
 *   alpha, beta  FP32 multipliers;
 *   c            DEVICE BF16 shaped like D (may be D itself), or NULL (no
 *                beta term);
 *   bias         DEVICE FP32 [G][N] (dense: [N]), or NULL;
 *   activation   FP8G_ACT_NONE or FP8G_ACT_RELU (negative results become
 *                +0, NaN stays NaN);
 *   round_mode   FP8G_ROUND_RN / _RZ / _RU / _RD.
 *   c and bias must be 16-byte aligned.  Masked-out rows of the grouped
 *   form are neither read from c nor written.
 */
typedef struct {
    const float *out_a;
    int64_t out_a_len;
    const float *out_b;
    int64_t out_b_len;
    const uint8_t *block_a;
    int64_t block_a_ld;
    const uint8_t *block_b;
    int64_t block_b_ld;
    int32_t block_k;
} fp8g_scales;

#define FP8G_ACT_NONE 0
#define FP8G_ACT_RELU 1
#define FP8G_ROUND_RN 0 /* to nearest, ties to even  */
#define FP8G_ROUND_RZ 1 /* toward zero               */
#define FP8G_ROUND_RU 2 /* toward +infinity          */
#define FP8G_ROUND_RD 3 /* toward -infinity          */

typedef struct {
    float alpha;
    float beta;
    const void *c;
    const float *bias;
    int32_t activation;
    int32_t round_mode;
} fp8g_epilogue;

int fp8_gemm_nt_ex(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                   int a_dtype, int b_dtype, const fp8g_scales *scales,
                   const fp8g_epilogue *epilogue, uint32_t flags, cudaStream_t stream);
int fp8_gemm_grouped_masked_ex(const void *A, const void *B, void *D, const int32_t *masked_m,
                               int64_t G, int64_t M_max, int64_t N, int64_t K,
                               int64_t max_m_hint, int a_dtype, int b_dtype,
                               const fp8g_scales *scales, const fp8g_epilogue *epilogue,
                               uint32_t flags, cudaStream_t stream);

/*
 * fp8_gemm_grouped_contiguous / _ex -- grouped GEMM with the groups' token
 * rows concatenated along M (the MoE prefill form, beside the masked decode
 * form; "一次“转置”，半张算力：DeepSeek SwapAB 漂流史" §5 counts four grouped
 * layouts on SM100 without describing them -- this is the plainest reading):
 *   D[r, n] = sum_k A[r, k] * B[g, n, k]   for group_offsets[g] <= r < group_offsets[g+1]
 *   A              [M_total, K] FP8 codes, row-major.
 *   B              [G, N, K] FP8 codes.
 *   D              [M_total, N] BF16; rows outside every group are not written.
 *   group_offsets  DEVICE int32 [G+1], nondecreasing, 0 <= offsets[0],
 *                  offsets[G] <= M_total; group boundaries need no alignment.
 *                  A group whose extent breaks this is skipped and reported as
 *                  FP8G_ERR_MASKED_M_RANGE by fp8g_get_device_status().
 *   max_m_hint     expected largest group (0: M_total); picks SwapAB under AUTO.
 * Output scales (out_a: G or M_total entries, out_b: G or G*N) and the fused
 * epilogue (bias [G][N], C shaped like D) as in the _ex calls; block scales
 * are not supported with this layout (FP8G_ERR_UNSUPPORTED).
 */
int fp8_gemm_grouped_contiguous(const void *A, const void *B, void *D,
                                const int32_t *group_offsets, int64_t G, int64_t M_total,
                                int64_t N, int64_t K, int64_t max_m_hint, int a_dtype,
                                int b_dtype, uint32_t flags, cudaStream_t stream);
int fp8_gemm_grouped_contiguous_ex(const void *A, const void *B, void *D,
                                   const int32_t *group_offsets, int64_t G, int64_t M_total,
                                   int64_t N, int64_t K, int64_t max_m_hint, int a_dtype,
                                   int b_dtype, const fp8g_scales *scales,
                                   const fp8g_epilogue *epilogue, uint32_t flags,
                                   cudaStream_t stream);

/*
 * fp8g_get_device_status -- synchronise `stream`, then read and clear the
 * status word of the current device.  info[0] = first fp8g_status recorded
 * on the device since the last read (FP8G_OK if none), info[1] = block
 * index, info[2] = role (0 loader, 1 MMA issuer, 2 epilogue, 3 scheduler),
 * info[3] = detail (pipeline stage or group).  `info` is host memory of 4
 * int32.  Returns FP8G_OK or FP8G_ERR_CUDA / FP8G_ERR_INVALID_ARG.
 */
int fp8g_get_device_status(int32_t *info, cudaStream_t stream);

/*
 * fp8g_init -- allocate, on the current device, the stream-K workspace of
 * `stream` at its largest size: partial tiles for every SM (2 x SMs x 128 x
 * 256 FP32, 39.8 MB on 152 SMs) and arrival counters for up to `max_tiles`
 * output tiles of one launch (0 = 65536; 64 bytes a tile).  A stream-K
 * launch is one with SwapAB (output tiles = groups x token chunks x
 * ceil(N / 128)) or split SM-pair tiles (ceil(M / 256) x ceil(N / tile)).
 * The calls allocate a stream's workspace themselves on its first need;
 * after fp8g_init, calls on that stream whose launches fit allocate
 * nothing, so they can be recorded into a CUDA graph captured from that
 * stream from the start.  Idempotent; never shrinks.
 * Returns FP8G_OK, FP8G_ERR_INVALID_ARG (max_tiles < 0 or > 2^31 - 1),
 * FP8G_ERR_NO_DEVICE, FP8G_ERR_UNSUPPORTED (not sm_103) or FP8G_ERR_CUDA
 * (allocation failed).
 *
 * fp8g_release_stream -- synchronise `stream` and free its stream-K
 * workspace on the current device (nothing to do if it has none).  Call it
 * before destroying a stream that ran library work.  Returns FP8G_OK or
 * FP8G_ERR_CUDA.
 *
 * fp8g_shutdown -- free the stream-K workspaces of every stream on every
 * device (cudaFree waits for the device's work).  Call it with no library
 * work being enqueued or captured on another thread; later calls allocate
 * again on first need.  The fixed array of fp8_gemm_nt_noalloc is not
 * affected.  Returns FP8G_OK or FP8G_ERR_CUDA.
 */
int fp8g_init(int64_t max_tiles, cudaStream_t stream);
int fp8g_release_stream(cudaStream_t stream);
int fp8g_shutdown(void);

/*
 * fp8g_set_wait_timeout_ns -- limit, in nanoseconds of device time, of every
 * barrier wait inside the kernels launched after this call (default 2e9).
 * A wait that runs out records FP8G_ERR_TIMEOUT, stops the block's pipeline,
 * drains its in-flight copies and tensor-core work, frees its tensor memory
 * and returns.  0 restores the default.  Returns the previous value.
 */
uint64_t fp8g_set_wait_timeout_ns(uint64_t ns);

/*
 * fp8_gemm_nt_noalloc -- dense D = A . B^T for small token counts that
 * allocates no device memory.  (Not from the pages: they have no
 * counterpart.)
 *
 * For callers that cannot have a library call cudaMalloc: a framework whose
 * caching allocator must own every device byte, or a serving loop that cannot
 * take cudaMalloc's device-wide synchronisation.  fp8_gemm_nt may
 * allocate its stream-K workspace on first use; this call instead keeps that
 * scratch in one fixed device array of FP8G_NOALLOC_SCRATCH_BYTES (32 MiB)
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  It runs the SwapAB stream-K kernel of fp8_gemm_nt's
 * small-token path, with one difference in configuration: it always gives
 * each CTA a whole SM (all of its shared memory, 512 TMEM columns), where
 * fp8_gemm_nt shares an SM between two launches for problems of up to 16
 * tokens (measured about 5 % slower than that shared-SM form there).
 *
 *   A [M, K], B [N, K], D [M, N] and the dtypes: as fp8_gemm_nt.
 *   M  1..256 tokens, else FP8G_ERR_UNSUPPORTED.
 *   Scratch a call needs: its arrival counters, 32 bytes per 128 rows of N
 *   (rounded up to 256 bytes), then its partial tiles, 2 x grid x 128 x
 *   round16(M) x 4 bytes, where grid = min(SMs, ceil(N/128) x ceil(K/128)).
 *   A problem that needs more than FP8G_NOALLOC_SCRATCH_BYTES returns
 *   FP8G_ERR_UNSUPPORTED before anything is enqueued.  On 152 SMs every
 *   problem of up to 208 tokens fits (for N up to 4.7 million rows); 209
 *   to 256 tokens (chunks of 224, 240, 256) fit only launches of fewer CTAs.
 *   No cudaMalloc, cudaFree or allocating library routine is called.  The
 *   first call on a device looks up the array's device address and the
 *   device limits (once per device, with that device current).  Each call
 *   clears the scratch's arrival counters with cudaMemsetAsync on `stream`
 *   before its launch.
 *   All calls on a device share the array: calls that overlap on the GPU
 *   (unordered streams) race on it and give wrong results.
 *   Bounded waits use the default 2 s limit.
 * Returns FP8G_OK or an error code.  On an argument or size error nothing
 * is enqueued; FP8G_ERR_CUDA from the launch itself can follow the
 * counters' clearing memset, which is then harmless.
 */
#define FP8G_NOALLOC_SCRATCH_BYTES (32u << 20)
int fp8_gemm_nt_noalloc(const void *A, const void *B, void *D, int64_t M, int64_t N,
                        int64_t K, int a_dtype, int b_dtype, cudaStream_t stream);

/*
 * fp8g_describe_plan -- the launch the library would make for a problem,
 * without touching memory or enqueueing anything (the kernel choice of
 * FP8G_SWAP_AUTO and of the tile planners, for inspection and tuning).
 *   layout      0: dense fp8_gemm_nt (G must be 1); 1: masked grouped
 *               (rows = M_max); 2: contiguous grouped (rows = M_total).
 *   G, rows, N, K, token_hint, flags: as the corresponding call takes them
 *               (token_hint: max_m_hint of the masked call, 0 = rows; the
 *               contiguous layout uses rows / G, the dense one rows).
 *   sf_group_k  0 (no block scales), 32 or 128: as the block-scaled calls.
 *   sms, smem_optin: the device to plan for (SM count, opt-in shared memory
 *               per block in bytes); both 0: the current device.
 *   out         caller-owned; filled on FP8G_OK.
 * Returns FP8G_OK, FP8G_ERR_INVALID_ARG (null out, sizes <= 0, bad layout,
 * flags or group size), FP8G_ERR_UNSUPPORTED, or a device-query error
 * when sms and smem_optin are 0.  Shape limits of the GEMM calls (K % 16,
 * N % 8) are checked as they are there.
 */
#define FP8G_KERNEL_TOKEN_TILES 0   /* 128-row token tiles on one SM each */
#define FP8G_KERNEL_SM_PAIRS 1      /* 256-row token tiles on an SM pair (cta_group::2) */
#define FP8G_KERNEL_SWAP_AB 2       /* weights on the MMA's M side, tokens on a runtime N */
typedef struct fp8g_plan {
    int32_t kernel;      /* FP8G_KERNEL_* */
    int32_t tile_n;      /* N tile (token tiles, SM pairs) or token chunk (SwapAB) */
    int32_t stages;      /* shared-memory pipeline stages */
    int32_t stream_k;    /* 1: some tiles' K blocks split over several CTAs (stream-K or a
                            split last wave); 0: whole tiles */
    int32_t mma_issuers; /* threads issuing MMAs per tile: 1 or 2 */
    int32_t shared_sm;   /* 1: half the shared memory, two CTAs may share an SM */
    int32_t token_box;   /* token rows per TMA copy (SwapAB; token tiles: A rows) */
    int32_t grid;        /* CTAs launched */
    int32_t k_split;     /* SM pairs: 1 whole tiles; s >= 2: each tile of the last partial wave
                            split s ways along K (run first, summed by its last contributor);
                            0: that wave stream-K over every pair.  Other kernels: 1, or 0 for
                            stream-K */
} fp8g_plan;
int fp8g_describe_plan(int layout, int64_t G, int64_t rows, int64_t N, int64_t K, int64_t token_hint,
                       int sf_group_k, uint32_t flags, int sms, int smem_optin, fp8g_plan *out);

/* Human-readable name of a status code (static string). */
const char *fp8g_status_string(int code);

/* Library ABI version: major*10000 + minor*100 + patch. */
int fp8g_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8G_H */
